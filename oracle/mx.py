"""MX (OCP microscaling) quantization oracle: BF16 -> E2M1 / E4M3 + UE8M0.

TEST INFRASTRUCTURE ONLY (see the package docstring).

What is computed, per block of 32 consecutive elements along the quantization
axis (OCP MX v1.0, "shared scale" rule; the pages use it for MXFP4 weights and
activations in "Triton mxfp4 (and a8w4) grouped GEMM kernel", PR #723, and for
the MXFP8 E4M3 reference quantizer of PR #745):

1. amax = max |x_i| over the block (BF16 values, subnormals honoured).
2. e = floor(log2(amax)) - emax, emax = 2 for E2M1 (largest value 6 = 1.5*2^2)
   and 8 for E4M3 (largest value 448 = 1.75*2^8).  An all-zero block has no
   finite log2; the exponent then takes the floor of the allowed range.
3. e is clamped to [-127, 127].  The lower clamp is the rule stated in PR #745's
   review "Clamp tiny block scales to preserve nonzero values": a block whose
   amax is 2^-126 quantizes to the E4M3 element value 2 with exponent -127,
   rather than losing its values.  The scale byte is the UE8M0 encoding e+127.
4. Each element is divided by 2^e (exact in float64) and rounded to the nearest
   representable element value, ties to the even code, saturating at the
   largest finite magnitude (6 for E2M1, 448 for E4M3 "fn", whose code 0x7F is
   NaN and never produced).  The sign is kept, also for values that round to 0.
5. E2M1 codes are packed two per byte, element 2j in the low nibble.

Readings where the pages are silent (all written out in the design notes):
all-zero blocks get scale byte 0x00 and zero codes; negative values that round
to zero keep their sign bit; NaN/Inf inputs are outside the contract.

Selectable scale rule ``rule="round_up"``: the TransformerEngine recipe that the
same PR #745 review describes (the scale is amax / 448 taken to E8M0, i.e. a
power of two that never lets an element saturate, with the same -127 floor):
e is the smallest integer with maxval * 2^e >= amax (maxval 448 for E4M3, 6 for
E2M1), clamped to [-127, 127]; -127 for an all-zero block.  It differs from
the OCP rule only when amax's mantissa exceeds maxval's (1.75 / 1.5), where the
OCP rule saturates the largest elements and this one takes the next exponent.
"""

from __future__ import annotations

import numpy as np

E2M1_MAGNITUDES = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=np.float64)
BLOCK = 32
EMAX = {"e2m1": 2, "e4m3": 8}
MAXVAL = {"e2m1": 6.0, "e4m3": 448.0}
RULES = ("ocp", "round_up")
SIGN_SHIFT = {"e2m1": 3, "e4m3": 7}


def e4m3_magnitudes() -> np.ndarray:
    """Values of the non-negative finite E4M3 ("fn") codes 0x00..0x7E, indexed
    by code: 4 exponent bits (bias 7), 3 mantissa bits, subnormals m*2^-9."""
    vals = []
    for code in range(0x7F):
        E, m = code >> 3, code & 7
        if E == 0:
            vals.append(m * 2.0 ** -9)
        else:
            vals.append((1.0 + m / 8.0) * 2.0 ** (E - 7))
    return np.array(vals, dtype=np.float64)


_E4M3 = e4m3_magnitudes()


def _magnitudes(elem: str) -> np.ndarray:
    if elem == "e2m1":
        return E2M1_MAGNITUDES
    if elem == "e4m3":
        return _E4M3
    raise ValueError(elem)


def decode(codes: np.ndarray, elem: str) -> np.ndarray:
    """Element code -> float64 value (sign bit 3 for E2M1, bit 7 for E4M3)."""
    codes = np.asarray(codes).astype(np.int64)
    sh = SIGN_SHIFT[elem]
    mag = _magnitudes(elem)[codes & ((1 << sh) - 1)]
    return np.where((codes >> sh) & 1, -mag, mag)


def round_to_grid(v: np.ndarray, elem: str) -> np.ndarray:
    """Round float64 values to the nearest element code, ties to the even code,
    saturating at the largest finite magnitude; the sign bit follows the sign
    of v (so -0.0 and small negatives give the negative-zero code)."""
    v = np.asarray(v, dtype=np.float64)
    grid = _magnitudes(elem)                   # ascending; code == index
    n = grid.shape[0]
    mag = np.abs(v)
    hi = np.searchsorted(grid, mag, side="left")
    hi_c = np.minimum(hi, n - 1)
    lo_c = np.maximum(hi_c - 1, 0)
    d_lo = mag - grid[lo_c]
    d_hi = grid[hi_c] - mag
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi_c % 2 == 0))
    idx = np.where(pick_hi, hi_c, lo_c)
    idx = np.where(mag >= grid[-1], n - 1, idx)   # saturate
    idx = np.where(mag == 0.0, 0, idx)
    sign = np.signbit(v).astype(np.int64)
    return (idx | (sign << SIGN_SHIFT[elem])).astype(np.uint8)


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def shared_exponent(amax: np.ndarray, elem: str, rule: str = "ocp") -> np.ndarray:
    """OCP: floor(log2(amax)) - emax.  round_up: the smallest e with
    maxval * 2^e >= amax.  Both clamped to [-127, 127]; -127 for amax == 0."""
    if rule not in RULES:
        raise ValueError(rule)
    amax = np.asarray(amax, dtype=np.float64)
    _, ex = np.frexp(amax)                     # amax = f * 2^ex, f in [0.5, 1)
    e = (ex.astype(np.int64) - 1) - EMAX[elem]
    if rule == "round_up":
        # maxval * 2^(e - 1) < 2^floor(log2 amax) <= amax, so the smallest
        # exponent that covers amax is e or e + 1 (exact float64 comparison)
        e = np.where(np.ldexp(MAXVAL[elem], e) >= amax, e, e + 1)
    e = np.where(amax == 0.0, -127, e)
    return np.clip(e, -127, 127)


def quantize_mx(x_bits: np.ndarray, elem: str, rule: str = "ocp"):
    """Quantize BF16 bits along the last axis in blocks of 32 (scale rule
    ``rule``, see ``shared_exponent``).

    Returns (codes uint8 [..., C], scale bytes uint8 [..., C/32]).  Codes are
    one per element (unpacked); see ``pack_e2m1``."""
    x = bf16_to_f64(x_bits)
    C = x.shape[-1]
    if C % BLOCK:
        raise ValueError("quantization axis must be a multiple of 32")
    xb = x.reshape(x.shape[:-1] + (C // BLOCK, BLOCK))
    amax = np.abs(xb).max(axis=-1)
    e = shared_exponent(amax, elem, rule)
    y = np.ldexp(xb, -e[..., None])            # exact: power-of-two rescale
    codes = round_to_grid(y, elem).reshape(x.shape)
    return codes, (e + 127).astype(np.uint8)


def dequantize_mx(codes: np.ndarray, scale: np.ndarray, elem: str) -> np.ndarray:
    """codes [..., C] (unpacked) and scale bytes [..., C/32] -> float64."""
    v = decode(codes, elem)
    C = v.shape[-1]
    e = scale.astype(np.int64) - 127
    vb = v.reshape(v.shape[:-1] + (C // BLOCK, BLOCK))
    return np.ldexp(vb, e[..., None]).reshape(v.shape)


def pack_e2m1(codes: np.ndarray) -> np.ndarray:
    """[..., C] 4-bit codes -> [..., C/2] bytes, element 2j in the low nibble."""
    c = np.asarray(codes, dtype=np.uint8)
    return (c[..., 0::2] & 0xF) | ((c[..., 1::2] & 0xF) << 4)


def unpack_e2m1(packed: np.ndarray) -> np.ndarray:
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out


def quantize_mx_rowwise(x_bits: np.ndarray, elem: str, rule: str = "ocp"):
    """Row-wise operand of a K-major GEMM: BF16 [R, C] quantized along C.

    Returns (data, scale) in the plain interchange layout: data [R, C/2]
    packed E2M1 or [R, C] E4M3 bytes, scale [R, C/32] UE8M0 bytes.  This is the
    ``_row_operand`` bridge of PR #723 ((N, K/2) data, (N, K/32) scales)."""
    codes, scale = quantize_mx(x_bits, elem, rule)
    data = pack_e2m1(codes) if elem == "e2m1" else codes
    return data, scale


def padded_offsets(m_splits, pad: int) -> np.ndarray:
    """Exclusive prefix sum of ceil(m_g/pad)*pad, length G+1 (int64)."""
    m = np.asarray(m_splits, dtype=np.int64)
    p = ((m + pad - 1) // pad) * pad
    return np.concatenate([[0], np.cumsum(p)]).astype(np.int64)


def quantize_mx_colwise_segment_padded(x_bits: np.ndarray, m_splits, pad: int, elem: str,
                                       rule: str = "ocp"):
    """Columnwise, segment-padded operand of the variable-K wgrad (PR #723,
    ``_col_operand_grouped_padded``: (C, Mpad/2) data + scales).

    x is BF16 [S, C] with experts' rows concatenated in order.  Expert g's rows
    [off_g, off_g + m_g) are transposed to [C, m_g], zero-padded on the right to
    p_g = ceil(m_g/pad)*pad columns and quantized along that axis in blocks of
    32 that start at the expert's padded origin poff_g, so no block straddles
    two experts.  Returns (data [C, Spad(/2)], scale [C, Spad/32], poff[G+1])."""
    if pad <= 0 or pad % BLOCK:
        raise ValueError("pad must be a positive multiple of 32")
    m = np.asarray(m_splits, dtype=np.int64)
    S, C = x_bits.shape
    if m.sum() != S or (m < 0).any():
        raise ValueError("invalid splits")
    off = np.concatenate([[0], np.cumsum(m)])
    poff = padded_offsets(m, pad)
    spad = int(poff[-1])
    codes = np.zeros((C, spad), dtype=np.uint8)
    scale = np.zeros((C, spad // BLOCK), dtype=np.uint8)
    for g in range(m.shape[0]):
        p_g = int(poff[g + 1] - poff[g])
        if p_g == 0:
            continue
        seg = np.zeros((C, p_g), dtype=np.uint16)        # +0.0 padding
        seg[:, : m[g]] = x_bits[off[g]: off[g + 1]].T
        cg, sg = quantize_mx(seg, elem, rule)
        codes[:, poff[g]: poff[g + 1]] = cg
        scale[:, poff[g] // BLOCK: poff[g + 1] // BLOCK] = sg
    data = pack_e2m1(codes) if elem == "e2m1" else codes
    return data, scale, poff
