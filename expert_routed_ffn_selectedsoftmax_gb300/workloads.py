"""Seeded synthetic inputs for the MoE FFN layer with SelectedSoftmax routing.

This module only draws random numbers and encodes them in the storage formats
the layer consumes (fp32, bf16 bit patterns, Q8_0 blocks).  It holds none of
the layer's arithmetic: no router projection, no top-k, no softmax, no expert
FFN.  Both the CUDA path and the CPU oracle read the bytes produced here.

Shapes follow the two backbones described on the source pages:
  * ZONOS2 ("zonos2.cpp internals", §Model architecture): n_embd 2048,
    16 experts, top-1.
  * ZONOS3-Mini ("New Community Model: ZONOS3-Mini (Zyphra) - #1271",
    §Summary): width 1024, top-2 of 64 experts on layers 1-10.
Expert ffn widths (512, 2816) are not printed on the pages; they are the
workload definitions of this library's benchmark suite.

Value recipe (all seeded with numpy.random.default_rng(seed)):
  x ~ N(0, 1); W_r, W_g, W_u ~ N(0, 1/d) (standard deviation 1/sqrt(fan_in));
  W_d ~ N(0, 1/F); selection bias ~ N(0, bias_sd), or, for the Zipf workload,
  b_e = ZIPF_ALPHA * log(p_rank(e)) with p_r proportional to r^-1.1 and ranks
  assigned to experts by a seeded permutation.  Draws are made in float32 and
  rounded to nearest-even bf16 where the workload is bf16.  Q8_0 blocks hold
  32 consecutive values along the contiguous (reduction) axis: an fp16 scale
  max|w|/127 followed by 32 int8 values round-half-away-from-zero(w/scale).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

F32, BF16, Q8_0, Q4_A64, Q4_K, Q6_K, FP8 = 0, 1, 2, 3, 4, 5, 6
DTYPE_NAMES = {F32: "f32", BF16: "bf16", Q8_0: "q8_0", Q4_A64: "q4_a64", Q4_K: "q4_k", Q6_K: "q6_k",
               FP8: "fp8_e4m3"}
FP8_MAX = 448.0          # largest finite E4M3 value
Q4_K_BLOCK = 256
Q4_K_BLOCK_BYTES = 144
Q6_K_BLOCK = 256
Q6_K_BLOCK_BYTES = 210
Q4_A64_GROUP = 64
Q4_A64_BLOCK_BYTES = 36
Q8_0_BLOCK = 32
Q8_0_BLOCK_BYTES = 34

# Scale on log(p_rank) for the Zipf-skewed workload's analytic bias (used
# where no fitted bias exists: other sizes and seeds).  With router logits
# close to N(0, 1), 0.65 puts ~25% of the top-2 assignments on the busiest
# expert, the head share of Zipf(s=1.1) over 64 ranks; the tail falls off
# faster than Zipf.  The benchmark's full-size Zipf layers instead use a bias
# fitted to their own inputs (zipf_host_inputs; fitted with the oracle's
# routing by tests/golden/fit_zipf_bias.py) so that the loads follow
# Zipf(s=1.1) over all ranks.
ZIPF_S = 1.1
ZIPF_ALPHA = 0.65
ZIPF_HOST_SEED = 7100   # host seed of layer i's x and W_r: ZIPF_HOST_SEED + i


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int
    d: int
    E: int
    k: int
    F: int
    act_dtype: int      # dtype of x and W_r (F32 or BF16)
    w_dtype: int        # dtype of expert weights (F32, BF16, Q8_0, Q4_A64)
    bias: str           # "normal" or "zipf"
    bias_sd: float
    layers: int         # layers run back to back in one benchmark step
    description: str


WORKLOADS = {
    "tiny_fp32": Workload(
        "tiny_fp32", T=8, d=64, E=8, k=2, F=128, act_dtype=F32, w_dtype=F32,
        bias="normal", bias_sd=0.1, layers=1,
        description="tiny fp32 MoE layer, T=8 d=64 E=8 top-2 F=128"),
    "zonos3_mini_decode": Workload(
        "zonos3_mini_decode", T=128, d=1024, E=64, k=2, F=512, act_dtype=BF16,
        w_dtype=BF16, bias="normal", bias_sd=0.5, layers=10,
        description="ZONOS3-Mini-shaped decode step: 128 rows (64 streams x "
                    "speaker-CFG pair), d=1024, E=64, top-2, F=512, bf16, "
                    "10 MoE layers back to back"),
    "zonos2_decode": Workload(
        "zonos2_decode", T=64, d=2048, E=16, k=1, F=2816, act_dtype=BF16,
        w_dtype=BF16, bias="normal", bias_sd=0.1, layers=28,
        description="ZONOS2-shaped decode step: d=2048, E=16, top-1, F=2816, "
                    "bf16, T in {1, 8, 64}, 28-layer weight rotation"),
    "zonos3_mini_prefill": Workload(
        "zonos3_mini_prefill", T=8192, d=1024, E=64, k=2, F=512, act_dtype=BF16,
        w_dtype=BF16, bias="zipf", bias_sd=0.0, layers=4,
        description="ZONOS3-Mini-shaped prefill: T=8192, d=1024, E=64, top-2, "
                    "F=512, bf16, Zipf(1.1)-skewed expert loads (4 independent "
                    "layers per benchmark step so weights come from HBM)"),
    "zonos2_prefill_q8": Workload(
        "zonos2_prefill_q8", T=4096, d=2048, E=16, k=1, F=2816, act_dtype=BF16,
        w_dtype=Q8_0, bias="normal", bias_sd=0.1, layers=4,
        description="ZONOS2-shaped prefill with Q8_0 experts: T=4096, d=2048, "
                    "E=16, top-1, F=2816, bf16 activations and router (4 "
                    "independent layers per benchmark step)"),
    "zonos2_decode_q4": Workload(
        "zonos2_decode_q4", T=8, d=2048, E=16, k=1, F=2816, act_dtype=BF16,
        w_dtype=Q4_A64, bias="normal", bias_sd=0.1, layers=28,
        description="ZONOS2-shaped decode step with affine 4-bit group-64 experts "
                    "(the format of the pages' MLX figures): d=2048, E=16, top-1, "
                    "F=2816, T in {1, 8, 64}, 28-layer weight rotation"),
    "zonos2_prefill_q4": Workload(
        "zonos2_prefill_q4", T=4096, d=2048, E=16, k=1, F=2816, act_dtype=BF16,
        w_dtype=Q4_A64, bias="normal", bias_sd=0.1, layers=4,
        description="ZONOS2-shaped prefill with affine 4-bit group-64 experts (the "
                    "MLX build's expert format): T=4096, d=2048, E=16, top-1, "
                    "F=2816, bf16 activations and router (4 independent layers "
                    "per benchmark step)"),
    "zonos2_decode_q4k": Workload(
        "zonos2_decode_q4k", T=8, d=2048, E=16, k=1, F=2816, act_dtype=BF16,
        w_dtype=Q4_K, bias="normal", bias_sd=0.1, layers=28,
        description="ZONOS2-shaped decode step with Q4_K experts (the K-quant the "
                    "pages recommend for the expert stacks): d=2048, E=16, top-1, "
                    "F=2816, T in {1, 8, 64}, 28-layer weight rotation"),
    "zonos2_decode_q8": Workload(
        "zonos2_decode_q8", T=8, d=2048, E=16, k=1, F=2816, act_dtype=BF16,
        w_dtype=Q8_0, bias="normal", bias_sd=0.1, layers=28,
        description="ZONOS2-shaped decode step with Q8_0 experts (the port's "
                    "effectively lossless default): d=2048, E=16, top-1, F=2816, "
                    "T in {1, 8, 64}, 28-layer weight rotation"),
    "zonos2_decode_q6k": Workload(
        "zonos2_decode_q6k", T=8, d=2048, E=16, k=1, F=2816, act_dtype=BF16,
        w_dtype=Q6_K, bias="normal", bias_sd=0.1, layers=28,
        description="ZONOS2-shaped decode step with Q6_K experts (the K-quant ladder's "
                    "sweet spot): d=2048, E=16, top-1, F=2816, T in {1, 8, 64}, "
                    "28-layer weight rotation"),
    "zonos2_decode_fp8": Workload(
        "zonos2_decode_fp8", T=8, d=2048, E=16, k=1, F=2816, act_dtype=BF16,
        w_dtype=FP8, bias="normal", bias_sd=0.1, layers=28,
        description="ZONOS2-shaped decode step with fp8 (E4M3, one scale per row) "
                    "experts (the serving configs' fp8): d=2048, E=16, top-1, "
                    "F=2816, T in {1, 8, 64}, 28-layer weight rotation"),
    "zonos2_prefill_fp8": Workload(
        "zonos2_prefill_fp8", T=4096, d=2048, E=16, k=1, F=2816, act_dtype=BF16,
        w_dtype=FP8, bias="normal", bias_sd=0.1, layers=4,
        description="ZONOS2-shaped prefill with fp8 (E4M3, one scale per row) "
                    "experts: T=4096, d=2048, E=16, top-1, F=2816, bf16 "
                    "activations and router (4 independent layers per benchmark step)"),
    "zonos2_prefill_q6k": Workload(
        "zonos2_prefill_q6k", T=4096, d=2048, E=16, k=1, F=2816, act_dtype=BF16,
        w_dtype=Q6_K, bias="normal", bias_sd=0.1, layers=4,
        description="ZONOS2-shaped prefill with Q6_K experts: T=4096, d=2048, E=16, "
                    "top-1, F=2816, bf16 activations and router (4 independent "
                    "layers per benchmark step)"),
    "zonos2_prefill_q4k": Workload(
        "zonos2_prefill_q4k", T=4096, d=2048, E=16, k=1, F=2816, act_dtype=BF16,
        w_dtype=Q4_K, bias="normal", bias_sd=0.1, layers=4,
        description="ZONOS2-shaped prefill with Q4_K experts: T=4096, d=2048, E=16, "
                    "top-1, F=2816, bf16 activations and router (4 independent "
                    "layers per benchmark step)"),
}


@dataclasses.dataclass
class Layer:
    """One MoE layer's inputs as raw storage arrays (host numpy)."""
    T: int
    d: int
    E: int
    k: int
    F: int
    act_dtype: int
    w_dtype: int
    x: np.ndarray        # [T, d] float32 or uint16 (bf16 bits)
    w_router: np.ndarray  # [E, d] same storage as x
    bias: np.ndarray     # [E] float32
    w_gate: np.ndarray   # [E, F, d] (Q8_0: uint8 [E, F, d/32, 34])
    w_up: np.ndarray     # [E, F, d]
    w_down: np.ndarray   # [E, d, F] (Q8_0: uint8 [E, d, F/32, 34])


def f32_to_bf16_bits(a) -> np.ndarray:
    """Round float32 values to the nearest bf16 (ties to even); return bits."""
    a32 = np.ascontiguousarray(a, dtype=np.float32)
    u = a32.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def bf16_bits_to_f32(b) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def q8_0_quantize(w) -> np.ndarray:
    """Encode w[..., K] (K % 32 == 0) as Q8_0 blocks: uint8 [..., K/32, 34].

    Block layout: bytes 0-1 the fp16 scale (little endian), bytes 2-33 the
    int8 values.  scale = max|w|/127 (float32, stored rounded to fp16);
    q = round-half-away-from-zero(w / scale) clamped to [-127, 127]; an
    all-zero block has scale 0 and q 0.
    """
    w = np.asarray(w, dtype=np.float32)
    K = w.shape[-1]
    if K % Q8_0_BLOCK:
        raise ValueError("Q8_0 needs the contiguous axis to be a multiple of 32")
    blocks = w.reshape(w.shape[:-1] + (K // Q8_0_BLOCK, Q8_0_BLOCK))
    amax = np.abs(blocks).max(axis=-1)
    scale = (amax / np.float32(127.0)).astype(np.float32)
    inv = np.zeros_like(scale)
    nz = scale > 0
    inv[nz] = np.float32(1.0) / scale[nz]
    v = blocks * inv[..., None]
    q = np.sign(v) * np.floor(np.abs(v) + np.float32(0.5))
    q = np.clip(q, -127, 127).astype(np.int8)
    out = np.empty(blocks.shape[:-1] + (Q8_0_BLOCK_BYTES,), dtype=np.uint8)
    out[..., 0:2] = scale.astype(np.float16).view(np.uint8).reshape(scale.shape + (2,))
    out[..., 2:] = q.view(np.uint8)
    return out


def q4_a64_quantize(w) -> np.ndarray:
    """Encode w[..., K] (K % 64 == 0) as affine 4-bit blocks: uint8 [..., K/64, 36].

    Block layout: bytes 0-1 the fp16 scale, bytes 2-3 the fp16 bias (little
    endian), bytes 4-35 the 64 codes, value 2j in the low nibble of byte 4+j and
    2j+1 in the high nibble; value = scale * q + bias.  Per group of 64:
    scale = (max - min) / 15, bias = min (both stored rounded to fp16);
    q = round-half-away-from-zero((w - bias) / scale) with the stored fp16
    scale and bias, clamped to [0, 15]; a constant group has scale 0, q 0.
    """
    w = np.asarray(w, dtype=np.float32)
    K = w.shape[-1]
    if K % Q4_A64_GROUP:
        raise ValueError("affine 4-bit needs the contiguous axis to be a multiple of 64")
    g = w.reshape(w.shape[:-1] + (K // Q4_A64_GROUP, Q4_A64_GROUP))
    mn, mx = g.min(axis=-1), g.max(axis=-1)
    scale16 = ((mx - mn) / np.float32(15.0)).astype(np.float16)
    bias16 = mn.astype(np.float16)
    sc, bi = scale16.astype(np.float32), bias16.astype(np.float32)
    inv = np.zeros_like(sc)
    nz = sc > 0
    inv[nz] = np.float32(1.0) / sc[nz]
    v = (g - bi[..., None]) * inv[..., None]
    q = np.clip(np.sign(v) * np.floor(np.abs(v) + np.float32(0.5)), 0, 15).astype(np.uint8)
    out = np.empty(g.shape[:-1] + (Q4_A64_BLOCK_BYTES,), dtype=np.uint8)
    out[..., 0:2] = scale16.view(np.uint8).reshape(scale16.shape + (2,))
    out[..., 2:4] = bias16.view(np.uint8).reshape(bias16.shape + (2,))
    out[..., 4:] = q[..., 0::2] | (q[..., 1::2] << 4)
    return out


def q4_k_pack_scales(sc, m) -> np.ndarray:
    """Six-bit sub-block scales sc[..., 8] and mins m[..., 8] -> the 12 bytes of
    a Q4_K super-block: bytes 0-3 hold sc[0..3] in their low 6 bits and the top
    2 bits of sc[4..7]; bytes 4-7 likewise m[0..3] and the top bits of m[4..7];
    bytes 8-11 hold the low nibbles of sc[4..7] (low) and m[4..7] (high)."""
    sc = np.asarray(sc, np.uint8)
    m = np.asarray(m, np.uint8)
    out = np.empty(sc.shape[:-1] + (12,), np.uint8)
    out[..., 0:4] = (sc[..., 0:4] & 63) | ((sc[..., 4:8] >> 4) << 6)
    out[..., 4:8] = (m[..., 0:4] & 63) | ((m[..., 4:8] >> 4) << 6)
    out[..., 8:12] = (sc[..., 4:8] & 15) | ((m[..., 4:8] & 15) << 4)
    return out


def q4_k_quantize(w) -> np.ndarray:
    """Encode w[..., K] (K % 256 == 0) as Q4_K super-blocks: uint8 [..., K/256, 144].

    Block: fp16 d, fp16 dmin, 12 bytes of six-bit sub-block scales and mins
    (q4_k_pack_scales), 128 bytes of codes (the 32-byte run c holds sub-block
    2c in its low nibbles and 2c+1 in its high nibbles); sub-block j (values
    32j .. 32j+31) decodes as d * sc[j] * q - dmin * m[j].  This encoder: per
    sub-block min' = max(0, -min w) and step s = (max w + min') / 15; d =
    max s / 63 and dmin = max min' / 63 rounded to fp16; sc = round(s / d),
    m = round(min' / dmin) clamped to [0, 63]; q = round-half-away((w + dmin
    m) / (d sc)) clamped to [0, 15] with the stored d and dmin (0 where d sc = 0).
    """
    w = np.asarray(w, dtype=np.float32)
    K = w.shape[-1]
    if K % Q4_K_BLOCK:
        raise ValueError("Q4_K needs the contiguous axis to be a multiple of 256")
    g = w.reshape(w.shape[:-1] + (K // Q4_K_BLOCK, 8, 32)).astype(np.float64)
    mn = np.maximum(0.0, -g.min(axis=-1))
    step = (g.max(axis=-1) + mn) / 15.0
    d16 = (step.max(axis=-1) / 63.0).astype(np.float16)
    dmin16 = (mn.max(axis=-1) / 63.0).astype(np.float16)
    d, dmin = d16.astype(np.float64), dmin16.astype(np.float64)
    safe = lambda a: np.where(a > 0, a, 1.0)
    sc = np.where(d[..., None] > 0, np.clip(np.floor(step / safe(d)[..., None] + 0.5), 0, 63), 0)
    m = np.where(dmin[..., None] > 0, np.clip(np.floor(mn / safe(dmin)[..., None] + 0.5), 0, 63), 0)
    a = d[..., None] * sc                    # effective step per sub-block
    b = dmin[..., None] * m                  # effective offset per sub-block
    v = (g + b[..., None]) / safe(a)[..., None]
    q = np.where(a[..., None] > 0, np.clip(np.sign(v) * np.floor(np.abs(v) + 0.5), 0, 15), 0)
    q = q.astype(np.uint8)
    out = np.empty(g.shape[:-2] + (Q4_K_BLOCK_BYTES,), dtype=np.uint8)
    out[..., 0:2] = d16.view(np.uint8).reshape(d16.shape + (2,))
    out[..., 2:4] = dmin16.view(np.uint8).reshape(dmin16.shape + (2,))
    out[..., 4:16] = q4_k_pack_scales(sc.astype(np.uint8), m.astype(np.uint8))
    runs = q.reshape(q.shape[:-2] + (4, 2, 32))       # [..., run c, sub-block 2c / 2c+1, value]
    out[..., 16:] = (runs[..., 0, :] | (runs[..., 1, :] << 4)).reshape(q.shape[:-2] + (128,))
    return out


def q6_k_pack(q, sc, d16) -> np.ndarray:
    """6-bit codes q[..., 256] (0..63), int8 scales sc[..., 16] and fp16 d[...]
    -> 210-byte Q6_K super-blocks [..., 210]: ql[128] (low 4 bits), qh[64] (top
    2 bits), int8 scales[16], fp16 d.  Value v = 128 h + 32 g + l: low bits in
    the low (g < 2) or high (g >= 2) nibble of ql[64 h + l + 32 (g % 2)], top
    bits in bits 2g, 2g+1 of qh[32 h + l]."""
    q = np.asarray(q, np.uint8).reshape(np.shape(q)[:-1] + (2, 4, 32))   # [..., h, g, l]
    lo, hi = q & 15, (q >> 4) & 3
    ql = np.concatenate([lo[..., 0, :] | (lo[..., 2, :] << 4), lo[..., 1, :] | (lo[..., 3, :] << 4)], axis=-1)
    qh = hi[..., 0, :] | (hi[..., 1, :] << 2) | (hi[..., 2, :] << 4) | (hi[..., 3, :] << 6)
    lead = q.shape[:-3]
    out = np.empty(lead + (Q6_K_BLOCK_BYTES,), np.uint8)
    out[..., 0:128] = ql.reshape(lead + (128,))
    out[..., 128:192] = qh.reshape(lead + (64,))
    out[..., 192:208] = np.asarray(sc, np.int8).view(np.uint8)
    d16 = np.ascontiguousarray(np.asarray(d16, np.float16))
    out[..., 208:210] = d16.reshape(d16.shape + (1,)).view(np.uint8)
    return out


def q6_k_quantize(w) -> np.ndarray:
    """Encode w[..., K] (K % 256 == 0) as Q6_K super-blocks: uint8 [..., K/256, 210]
    (q6_k_pack); value v decodes as d * scales[v / 16] * (q - 32).  This
    encoder: per 16-value group step s = max|w| / 31; d = max s / 127 rounded
    to fp16; scale = round(s / d) clamped to [0, 127]; q - 32 =
    round-half-away(w / (d scale)) clamped to [-32, 31] with the stored d (0
    where d scale = 0)."""
    w = np.asarray(w, dtype=np.float32)
    K = w.shape[-1]
    if K % Q6_K_BLOCK:
        raise ValueError("Q6_K needs the contiguous axis to be a multiple of 256")
    g = w.reshape(w.shape[:-1] + (K // Q6_K_BLOCK, 16, 16)).astype(np.float64)
    step = np.abs(g).max(axis=-1) / 31.0
    d16 = (step.max(axis=-1) / 127.0).astype(np.float16)
    d = d16.astype(np.float64)
    safe = lambda a: np.where(a > 0, a, 1.0)
    sc = np.where(d[..., None] > 0, np.clip(np.floor(step / safe(d)[..., None] + 0.5), 0, 127), 0)
    a = d[..., None] * sc
    v = g / safe(a)[..., None]
    q = np.where(a[..., None] > 0, np.clip(np.sign(v) * np.floor(np.abs(v) + 0.5), -32, 31), 0) + 32
    return q6_k_pack(q.reshape(q.shape[:-2] + (256,)).astype(np.uint8), sc.astype(np.int8), d16)


def fp8_quantize(w) -> np.ndarray:
    """Encode w[..., K] as fp8 rows: uint8 [..., 4 + K] = {fp32 scale (little
    endian), E4M3 codes[K]}; value = scale * E4M3(code).  This encoder: scale =
    max|w| / 448 of the row in fp32 (1 for an all-zero row), codes = w / scale
    (fp32, clamped to +-448) rounded to nearest-even E4M3 (torch's float8_e4m3fn
    cast)."""
    import torch
    w = np.ascontiguousarray(np.asarray(w, dtype=np.float32))
    t = torch.from_numpy(w)
    return fp8_quantize_torch(t).numpy()


def fp8_quantize_torch(w):
    """fp8 rows of a float32 tensor [..., K] (fp8_quantize), on w's device."""
    import torch
    w = w.float()
    K = w.shape[-1]
    s = w.abs().amax(-1, keepdim=True) / FP8_MAX
    s = torch.where(s > 0, s, torch.ones_like(s))
    q = torch.clamp(w / s, -FP8_MAX, FP8_MAX).to(torch.float8_e4m3fn).view(torch.uint8)
    out = torch.empty(*w.shape[:-1], 4 + K, dtype=torch.uint8, device=w.device)
    out[..., 0:4] = s.contiguous().view(torch.uint8).reshape(*w.shape[:-1], 4)
    out[..., 4:] = q
    return out


def _encode(a: np.ndarray, dtype: int) -> np.ndarray:
    if dtype == F32:
        return np.ascontiguousarray(a, dtype=np.float32)
    if dtype == BF16:
        return f32_to_bf16_bits(a)
    if dtype == Q8_0:
        return q8_0_quantize(a)
    if dtype == Q4_A64:
        return q4_a64_quantize(a)
    if dtype == Q4_K:
        return q4_k_quantize(a)
    if dtype == Q6_K:
        return q6_k_quantize(a)
    if dtype == FP8:
        return fp8_quantize(a)
    raise ValueError(dtype)


def zipf_bias(E: int, rng: np.random.Generator, s: float = ZIPF_S,
              alpha: float = ZIPF_ALPHA) -> np.ndarray:
    """Selection bias whose log-shares follow Zipf(s) over a seeded ranking."""
    ranks = np.arange(1, E + 1, dtype=np.float64)
    p = ranks ** (-s)
    p /= p.sum()
    order = rng.permutation(E)          # order[r] = expert holding rank r+1
    b = np.empty(E, dtype=np.float64)
    b[order] = alpha * np.log(p)
    return b.astype(np.float32)


def zipf_targets(E: int, T: int, k: int, s: float = ZIPF_S) -> np.ndarray:
    """Target assignments per rank: T*k * r^-s / sum_r r^-s, r = 1..E."""
    p = np.arange(1, E + 1, dtype=np.float64) ** (-s)
    return T * k * p / p.sum()


def zipf_host_inputs(w: Workload, layer: int):
    """Layer `layer` of a full-size Zipf workload, drawn on the host: x [T, d]
    and W_r [E, d] as float32 (same distributions as make_layer) and the
    seeded permutation order[r] = expert holding rank r + 1."""
    rng = np.random.default_rng(ZIPF_HOST_SEED + layer)
    f32 = np.float32
    x = rng.standard_normal((w.T, w.d), dtype=f32)
    wr = rng.standard_normal((w.E, w.d), dtype=f32) * f32(1.0 / math.sqrt(w.d))
    order = rng.permutation(w.E)
    return x, wr, order


def make_layer(w: Workload, seed: int, T: Optional[int] = None,
               d: Optional[int] = None, E: Optional[int] = None,
               k: Optional[int] = None, F: Optional[int] = None) -> Layer:
    """Draw one layer's inputs for workload ``w`` (sizes may be overridden)."""
    T = w.T if T is None else T
    d = w.d if d is None else d
    E = w.E if E is None else E
    k = w.k if k is None else k
    F = w.F if F is None else F
    rng = np.random.default_rng(seed)
    f32 = np.float32
    x = rng.standard_normal((T, d), dtype=f32)
    wr = rng.standard_normal((E, d), dtype=f32) * f32(1.0 / math.sqrt(d))
    if w.bias == "zipf":
        bias = zipf_bias(E, rng)
    else:
        bias = (rng.standard_normal(E, dtype=f32) * f32(w.bias_sd)).astype(f32)
    wg = rng.standard_normal((E, F, d), dtype=f32) * f32(1.0 / math.sqrt(d))
    wu = rng.standard_normal((E, F, d), dtype=f32) * f32(1.0 / math.sqrt(d))
    wd = rng.standard_normal((E, d, F), dtype=f32) * f32(1.0 / math.sqrt(F))
    return Layer(T=T, d=d, E=E, k=k, F=F, act_dtype=w.act_dtype,
                 w_dtype=w.w_dtype, x=_encode(x, w.act_dtype),
                 w_router=_encode(wr, w.act_dtype), bias=bias,
                 w_gate=_encode(wg, w.w_dtype), w_up=_encode(wu, w.w_dtype),
                 w_down=_encode(wd, w.w_dtype))


def make_custom_layer(seed: int, T: int, d: int, E: int, k: int, F: int,
                      act_dtype: int, w_dtype: int, bias_sd: float = 0.1,
                      bias: str = "normal") -> Layer:
    """A layer with arbitrary sizes (edge-case and ragged-size tests)."""
    w = Workload("custom", T, d, E, k, F, act_dtype, w_dtype, bias, bias_sd, 1, "")
    return make_layer(w, seed)


def weight_bytes_per_expert(d: int, F: int, w_dtype: int) -> int:
    """Storage bytes of one expert's W_g + W_u + W_d in ``w_dtype``."""
    n = 3 * d * F
    if w_dtype == F32:
        return 4 * n
    if w_dtype == BF16:
        return 2 * n
    if w_dtype == Q4_A64:
        return n // Q4_A64_GROUP * Q4_A64_BLOCK_BYTES
    if w_dtype == Q4_K:
        return n // Q4_K_BLOCK * Q4_K_BLOCK_BYTES
    if w_dtype == Q6_K:
        return n // Q6_K_BLOCK * Q6_K_BLOCK_BYTES
    if w_dtype == FP8:   # one byte per weight and an fp32 scale per row (2F + d rows)
        return n + 4 * (2 * F + d)
    return n // Q8_0_BLOCK * Q8_0_BLOCK_BYTES


def act_bytes(dtype: int) -> int:
    return 4 if dtype == F32 else 2


# ---------------------------------------------------------------- device draws
def q8_0_quantize_torch(w):
    """Device twin of q8_0_quantize for benchmark weights: float32 [..., K] ->
    uint8 blocks [..., K/32, 34] (same block layout and rounding rule)."""
    import torch
    K = w.shape[-1]
    b = w.reshape(*w.shape[:-1], K // Q8_0_BLOCK, Q8_0_BLOCK).float()
    amax = b.abs().amax(-1)
    scale = amax / 127.0
    inv = torch.where(scale > 0, 1.0 / torch.where(scale > 0, scale, torch.ones_like(scale)),
                      torch.zeros_like(scale))
    v = b * inv[..., None]
    q = (torch.sign(v) * torch.floor(v.abs() + 0.5)).clamp(-127, 127).to(torch.int8)
    out = torch.empty(*b.shape[:-1], Q8_0_BLOCK_BYTES, dtype=torch.uint8, device=w.device)
    out[..., 0:2] = scale.to(torch.float16).contiguous().view(torch.uint8).reshape(*scale.shape, 2)
    out[..., 2:] = q.view(torch.uint8)
    return out


def q4_a64_quantize_torch(w):
    """Device twin of q4_a64_quantize: float32 [..., K] -> uint8 blocks
    [..., K/64, 36] (same layout and rounding rule)."""
    import torch
    K = w.shape[-1]
    g = w.reshape(*w.shape[:-1], K // Q4_A64_GROUP, Q4_A64_GROUP).float()
    mn, mx = g.amin(-1), g.amax(-1)
    scale16 = ((mx - mn) / 15.0).to(torch.float16)
    bias16 = mn.to(torch.float16)
    sc, bi = scale16.float(), bias16.float()
    inv = torch.where(sc > 0, 1.0 / torch.where(sc > 0, sc, torch.ones_like(sc)), torch.zeros_like(sc))
    v = (g - bi[..., None]) * inv[..., None]
    q = (torch.sign(v) * torch.floor(v.abs() + 0.5)).clamp(0, 15).to(torch.uint8)
    out = torch.empty(*g.shape[:-1], Q4_A64_BLOCK_BYTES, dtype=torch.uint8, device=w.device)
    out[..., 0:2] = scale16.contiguous().view(torch.uint8).reshape(*scale16.shape, 2)
    out[..., 2:4] = bias16.contiguous().view(torch.uint8).reshape(*bias16.shape, 2)
    out[..., 4:] = q[..., 0::2] | (q[..., 1::2] << 4)
    return out


def q4_k_quantize_torch(w):
    """Device twin of q4_k_quantize: float32 [..., K] -> uint8 super-blocks
    [..., K/256, 144] (same layout and rounding rules)."""
    import torch
    K = w.shape[-1]
    g = w.reshape(*w.shape[:-1], K // Q4_K_BLOCK, 8, 32).double()
    mn = torch.clamp(-g.amin(-1), min=0.0)
    step = (g.amax(-1) + mn) / 15.0
    d16 = (step.amax(-1) / 63.0).to(torch.float16)
    dmin16 = (mn.amax(-1) / 63.0).to(torch.float16)
    d, dmin = d16.double(), dmin16.double()
    one = torch.ones_like(d)
    sd = torch.where(d > 0, d, one)[..., None]
    smin = torch.where(dmin > 0, dmin, one)[..., None]
    sc = torch.where(d[..., None] > 0, torch.clamp(torch.floor(step / sd + 0.5), 0, 63), torch.zeros_like(step))
    m = torch.where(dmin[..., None] > 0, torch.clamp(torch.floor(mn / smin + 0.5), 0, 63), torch.zeros_like(mn))
    a = d[..., None] * sc
    b = dmin[..., None] * m
    v = (g + b[..., None]) / torch.where(a > 0, a, torch.ones_like(a))[..., None]
    q = torch.where(a[..., None] > 0, torch.clamp(torch.sign(v) * torch.floor(v.abs() + 0.5), 0, 15),
                    torch.zeros_like(v)).to(torch.uint8)
    sc8, m8 = sc.to(torch.uint8), m.to(torch.uint8)
    out = torch.empty(*g.shape[:-2], Q4_K_BLOCK_BYTES, dtype=torch.uint8, device=w.device)
    out[..., 0:2] = d16.contiguous().view(torch.uint8).reshape(*d16.shape, 2)
    out[..., 2:4] = dmin16.contiguous().view(torch.uint8).reshape(*dmin16.shape, 2)
    out[..., 4:8] = (sc8[..., 0:4] & 63) | ((sc8[..., 4:8] >> 4) << 6)
    out[..., 8:12] = (m8[..., 0:4] & 63) | ((m8[..., 4:8] >> 4) << 6)
    out[..., 12:16] = (sc8[..., 4:8] & 15) | ((m8[..., 4:8] & 15) << 4)
    runs = q.reshape(*q.shape[:-2], 4, 2, 32)
    out[..., 16:] = (runs[..., 0, :] | (runs[..., 1, :] << 4)).reshape(*q.shape[:-2], 128)
    return out


def q6_k_quantize_torch(w):
    """Device twin of q6_k_quantize: float32 [..., K] -> uint8 super-blocks
    [..., K/256, 210] (same layout and rounding rules)."""
    import torch
    K = w.shape[-1]
    g = w.reshape(*w.shape[:-1], K // Q6_K_BLOCK, 16, 16).double()
    step = g.abs().amax(-1) / 31.0
    d16 = (step.amax(-1) / 127.0).to(torch.float16)
    d = d16.double()
    sd = torch.where(d > 0, d, torch.ones_like(d))[..., None]
    sc = torch.where(d[..., None] > 0, torch.clamp(torch.floor(step / sd + 0.5), 0, 127), torch.zeros_like(step))
    a = d[..., None] * sc
    v = g / torch.where(a > 0, a, torch.ones_like(a))[..., None]
    q = (torch.where(a[..., None] > 0, torch.clamp(torch.sign(v) * torch.floor(v.abs() + 0.5), -32, 31),
                     torch.zeros_like(v)) + 32).to(torch.uint8)
    q = q.reshape(*q.shape[:-2], 2, 4, 32)                 # [..., h, g, l]
    lo, hi = q & 15, (q >> 4) & 3
    ql = torch.cat([lo[..., 0, :] | (lo[..., 2, :] << 4), lo[..., 1, :] | (lo[..., 3, :] << 4)], dim=-1)
    qh = hi[..., 0, :] | (hi[..., 1, :] << 2) | (hi[..., 2, :] << 4) | (hi[..., 3, :] << 6)
    lead = q.shape[:-3]
    out = torch.empty(*lead, Q6_K_BLOCK_BYTES, dtype=torch.uint8, device=w.device)
    out[..., 0:128] = ql.reshape(*lead, 128)
    out[..., 128:192] = qh.reshape(*lead, 64)
    out[..., 192:208] = sc.to(torch.int8).view(torch.uint8)
    out[..., 208:210] = d16.contiguous().view(torch.uint8).reshape(*d16.shape, 2)
    return out


def make_device_stack(w: Workload, seed: int, layers: int, T: Optional[int] = None,
                      device="cuda", zipf_biases=None):
    """Draw ``layers`` independent layers directly in device memory.

    Used for benchmark stacks whose weights (GBs) are too large to draw on the
    host.  Same distributions as make_layer, drawn with torch's seeded device
    generator; returns a list of dicts of torch tensors: x / W_r as
    torch.bfloat16, expert weights as torch.bfloat16 or, for Q8_0 workloads,
    uint8 Q8_0 blocks [E, rows, cols/32, 34].  ``zipf_biases`` (a Zipf
    workload at its full size): per layer, a selection bias fitted to the
    layer's host-drawn x and W_r (zipf_host_inputs), which are used then.
    """
    import torch
    if (w.act_dtype, w.w_dtype) not in ((BF16, BF16), (BF16, Q8_0), (BF16, Q4_A64), (BF16, Q4_K),
                                        (BF16, Q6_K), (BF16, FP8), (F32, F32)):
        raise ValueError("device stacks: bf16/bf16, bf16 with Q8_0, Q4_A64, Q4_K, Q6_K or fp8 "
                         "experts, or fp32/fp32")
    act = torch.float32 if w.act_dtype == F32 else torch.bfloat16
    T = w.T if T is None else T
    g = torch.Generator(device=device)
    out = []
    for layer in range(layers):
        g.manual_seed(seed * 1000003 + layer)

        def rn(*shape, sd=1.0, q8=False):
            t = torch.randn(*shape, generator=g, device=device, dtype=torch.float32) * sd
            if q8:
                return {Q4_A64: q4_a64_quantize_torch, Q4_K: q4_k_quantize_torch,
                        Q6_K: q6_k_quantize_torch, Q8_0: q8_0_quantize_torch,
                        FP8: fp8_quantize_torch}[w.w_dtype](t)
            return t.to(act)
        d, E, F = w.d, w.E, w.F
        x = rn(T, d)
        wr = rn(E, d, sd=1.0 / math.sqrt(d))
        if zipf_biases is not None and w.bias == "zipf" and T == w.T:
            hx, hwr, _ = zipf_host_inputs(w, layer)
            x = torch.from_numpy(hx).to(device).to(act)
            wr = torch.from_numpy(hwr).to(device).to(act)
            b = torch.from_numpy(np.asarray(zipf_biases[layer], dtype=np.float32)).to(device)
        elif w.bias == "zipf":
            rng = np.random.default_rng(seed * 1000003 + layer)
            b = torch.from_numpy(zipf_bias(E, rng)).to(device)
        else:
            b = torch.randn(E, generator=g, device=device, dtype=torch.float32) * w.bias_sd
        q8 = w.w_dtype in (Q8_0, Q4_A64, Q4_K, Q6_K, FP8)   # quantised expert weights
        wg = rn(E, F, d, sd=1.0 / math.sqrt(d), q8=q8)
        wu = rn(E, F, d, sd=1.0 / math.sqrt(d), q8=q8)
        wd = rn(E, d, F, sd=1.0 / math.sqrt(F), q8=q8)
        out.append(dict(x=x, w_router=wr, bias=b, w_gate=wg, w_up=wu, w_down=wd))
    return out
