/*
 * moe_debug.h -- entry points of the debug build of the library only
 * (libmoe_gb300_debug.so, compiled with MOE_DEBUG=1; the release library
 * does not export them).
 *
 * The debug build checks, in every expert kernel, the grouping the routing
 * kernels hand it before using it: the grouped-row offsets must start at 0,
 * never decrease and end at T*k (a kernel given anything else does no work),
 * and every token index a row gather or an output scatter reads must lie in
 * [0, T) (an index outside is not used).  Either failure is recorded in the
 * call's device status word, which moe_check (include/moe.h) reports as
 * MOE_ERR_DEVICE_CHECK.  The outputs of a call that failed a check are
 * undefined; calls that pass every check give bit for bit the release
 * build's results.
 */
#ifndef MOE_GB300_DEBUG_H
#define MOE_GB300_DEBUG_H

#include "moe.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Test hook: the next moe_forward-family call made after this one (any
 * thread) adds 1 to offsets[E] in its workspace between its grouping step and
 * its expert kernels -- a grouping that no longer accounts for T*k rows --
 * so that the expert kernels' offset checks fail (MOE_ERR_DEVICE_CHECK from
 * moe_check on that call's workspace).  The change is one store inside the
 * workspace; no kernel reads or writes out of bounds.  Returns MOE_OK.
 */
MOE_API moe_status moe_debug_corrupt_next_offsets(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_DEBUG_H */
