"""DeepSeek-style blockwise FP8 quantization oracle (1x128 and 128x128).

TEST INFRASTRUCTURE ONLY (see the package docstring).

Follows "Add ROCm Triton blockwise FP8 grouped GEMM" (ROCm TransformerEngine
PR #716): activations are quantized in 1x128 blocks along K, weights in
128x128 blocks, and the wgrad operand column-wise (1x128 along tokens) with
every expert's segment padded to a multiple of 128 rows.  Its review thread
"Clamp block amax to 1e-4" fixes the amax floor.  The pages keep fp32 scales
unless the power-of-two option is chosen.  The fp32 form, with arithmetic in
float32 exactly as the method states:

    a = max(amax, 1e-4f)          (fp32)
    s = a / 448                   (fp32, correctly rounded division)
    q = RNE_satfinite_E4M3(x / s) (x / s correctly rounded in fp32 first)

The power-of-two form (the `pow2` option of the pages' quantizers, TE's
`power_2_scale` default of its blockwise recipe): the same a, and s the
smallest power of two with 448 * s >= a, i.e. a / 448 rounded up to a power of
two, so that every |x / s| <= 448; x / s is then exact.

s is the dequantization scale: x ~= decode(q) * s.
"""

from __future__ import annotations

import numpy as np

from .mx import bf16_to_f64, round_to_grid, decode, padded_offsets

BW = 128
AMAX_FLOOR = np.float32(1e-4)
E4M3_MAX = np.float32(448.0)


def _bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    return bf16_to_f64(bits).astype(np.float32)   # exact


def pow2_scale(a32: np.ndarray) -> np.ndarray:
    """Smallest power of two s with 448 * s >= a, for fp32 a > 0 (exact:
    448 * 2^k and a are both exact in float64)."""
    a = np.asarray(a32, dtype=np.float64)
    k = np.ceil(np.log2(a / 448.0)).astype(np.int64)
    k = np.where(448.0 * np.ldexp(1.0, k) < a, k + 1, k)          # too small: go up
    k = np.where(448.0 * np.ldexp(1.0, k - 1) >= a, k - 1, k)     # not minimal: go down
    return np.ldexp(np.float32(1.0), k).astype(np.float32)


def _quantize_blocks(v32: np.ndarray, amax32: np.ndarray, bshape_axes, pow2: bool = False):
    """v32: float32 values; amax32: per-block amax broadcastable against v32
    after expanding ``bshape_axes``."""
    a = np.maximum(amax32, AMAX_FLOOR)
    s = pow2_scale(a) if pow2 else (a / E4M3_MAX).astype(np.float32)
    sb = np.expand_dims(s, bshape_axes)
    q32 = (v32 / sb).astype(np.float32)
    codes = round_to_grid(q32.astype(np.float64), "e4m3")
    return codes, s


def quantize_bw_1x128(x_bits: np.ndarray, pow2: bool = False):
    """BF16 [R, C] (C % 128 == 0) -> (E4M3 codes [R, C], fp32 scales [R, C/128])."""
    R, C = x_bits.shape
    if C % BW:
        raise ValueError("cols must be a multiple of 128")
    v = _bf16_to_f32(x_bits).reshape(R, C // BW, BW)
    amax = np.abs(v).max(axis=-1)
    codes, s = _quantize_blocks(v, amax, (-1,), pow2)
    return codes.reshape(R, C), s


def quantize_bw_128x128(w_bits: np.ndarray, pow2: bool = False):
    """BF16 weights [G, N, K] (N, K % 128 == 0) -> (E4M3 codes [G, N, K],
    fp32 scales [G, N/128, K/128]); one scale per 128x128 tile."""
    G, N, K = w_bits.shape
    if N % BW or K % BW:
        raise ValueError("N and K must be multiples of 128")
    v = _bf16_to_f32(w_bits).reshape(G, N // BW, BW, K // BW, BW)
    amax = np.abs(v).max(axis=(2, 4))
    codes, s = _quantize_blocks(v, amax, (2, 4), pow2)
    return codes.reshape(G, N, K), s


def transpose_bw_128x128(codes: np.ndarray, s: np.ndarray):
    """The dgrad copy of a 128x128-quantized weight: the same blocks with the
    same scales, transposed ([G, K, N] codes, [G, K/128, N/128] scales)."""
    return np.ascontiguousarray(np.swapaxes(codes, 1, 2)), np.ascontiguousarray(np.swapaxes(s, 1, 2))


def quantize_bw_colwise_padded(x_bits: np.ndarray, m_splits, pow2: bool = False):
    """Column-wise wgrad operand: BF16 [S, C] with experts' rows concatenated
    -> E4M3 codes [C, Spad], fp32 scales [C, Spad/128], poff [G+1]; expert g
    occupies columns [poff_g, poff_g + m_g) followed by zero padding up to the
    next multiple of 128, and blocks start at poff_g."""
    m = np.asarray(m_splits, dtype=np.int64)
    S, C = x_bits.shape
    if m.sum() != S or (m < 0).any():
        raise ValueError("invalid splits")
    off = np.concatenate([[0], np.cumsum(m)])
    poff = padded_offsets(m, BW)
    spad = int(poff[-1])
    codes = np.zeros((C, spad), dtype=np.uint8)
    scale = np.zeros((C, spad // BW), dtype=np.float32)
    for g in range(m.shape[0]):
        p_g = int(poff[g + 1] - poff[g])
        if p_g == 0:
            continue
        seg = np.zeros((C, p_g), dtype=np.uint16)
        seg[:, : m[g]] = x_bits[off[g]: off[g + 1]].T
        cg, sg = quantize_bw_1x128(seg, pow2)
        codes[:, poff[g]: poff[g + 1]] = cg
        scale[:, poff[g] // BW: poff[g + 1] // BW] = sg
    return codes, scale, poff


def dequantize_bw_1x128(codes: np.ndarray, s: np.ndarray) -> np.ndarray:
    v = decode(codes, "e4m3")
    R, C = v.shape
    return (v.reshape(R, C // BW, BW) * s.astype(np.float64)[..., None]).reshape(R, C)


def dequantize_bw_128x128(codes: np.ndarray, s: np.ndarray) -> np.ndarray:
    v = decode(codes, "e4m3")
    G, N, K = v.shape
    vb = v.reshape(G, N // BW, BW, K // BW, BW)
    return (vb * s.astype(np.float64)[:, :, None, :, None]).reshape(G, N, K)
