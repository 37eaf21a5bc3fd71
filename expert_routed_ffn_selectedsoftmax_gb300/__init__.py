"""GB300-native (sm_103a) mixture-of-experts FFN layer with SelectedSoftmax routing.

The layer (router projection, SelectedSoftmax top-k, token grouping, SwiGLU
expert GEMMs, weighted combine) runs in the hand-written CUDA kernels of
libmoe_gb300.so behind the C ABI of include/moe.h; `binding` marshals torch
tensors to it.  Importing this package loads no CUDA code.
"""
from .binding import (EXPORTS, MOE_BF16, MOE_F32, MOE_PATH_AUTO, MOE_PATH_DECODE,  # noqa: F401
                      MOE_PATH_PREFILL, MOE_PATH_DECODE_SIMT, MOE_Q4_A64, MOE_Q4_K, MOE_Q6_K, MOE_Q8_0, MOE_FP8,
                      MoeError, library_path, load_library, moe_pack_q4_a64, moe_q4_a64_packed_size,
                      moe_pack_q4_k, moe_q4_k_packed_size, moe_pack_q6_k, moe_q6_k_packed_size,
                      moe_pack_fp8, moe_fp8_packed_size,
                      MOE_SCORE_SELECTED_SOFTMAX, MOE_SCORE_SIGMOID, MOE_SCORE_SOFTMAX,
                      moe_check, moe_check_noalloc, moe_ffn_dense, moe_forward,
                      moe_forward_noalloc, moe_pack_q8_0, moe_permute, moe_q8_0_packed_size,
                      moe_route, moe_workspace_size, moe_workspace_views, read_routing,
                      VIEW_NAMES)
