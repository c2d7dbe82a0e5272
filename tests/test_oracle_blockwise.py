"""Pins for the blockwise-FP8 quantization oracle (CPU only): closed-form
blocks, an exact-rational restatement of the fp32 arithmetic, tile
structure of the 128x128 weight scales, and segment isolation of the
column-wise operand."""

import os

import numpy as np

import oracle
from oracle import scalar
from oracle.blockwise import transpose_bw_128x128
import synth
from conftest import parse_value, read_records


def f32_bits(x):
    return int(np.array([x], dtype=np.float32).view(np.uint32)[0])


def test_golden_constant_blocks(golden_dir):
    recs = read_records(os.path.join(golden_dir, "blockwise_blocks.txt"))
    assert len(recs) == 3
    for name, val, s_hex, code_hex in recs:
        v = parse_value(val)
        x = synth.f32_to_bf16_bits(np.full((2, 256), v, dtype=np.float32))
        codes, s = oracle.quantize_bw_1x128(x)
        assert s.shape == (2, 2)
        assert all(f32_bits(t) == int(s_hex, 16) for t in s.ravel()), name
        assert (codes == int(code_hex, 16)).all(), name


def test_matches_exact_rational_formulation():
    rng = np.random.default_rng(21)
    x = synth.normal_bf16(rng, (6, 256), std=1.0, outlier_frac=0.02)
    v = synth.bf16_bits_to_f32(x)
    # a row of tiny values (below the 1e-4 floor) and a row with a zero block
    x[4] = synth.f32_to_bf16_bits(v[4] * np.float32(1e-7))
    x[5, :128] = 0
    codes, s = oracle.quantize_bw_1x128(x)
    for r in range(x.shape[0]):
        for b in range(2):
            blk = [int(t) for t in x[r, 128 * b: 128 * b + 128]]
            sf, cs = scalar.quantize_block_bw(blk)
            assert float(sf) == float(s[r, b])
            assert list(codes[r, 128 * b: 128 * b + 128]) == cs, (r, b)


def test_weight_tiles_and_transpose():
    rng = np.random.default_rng(22)
    w = synth.normal_bf16(rng, (2, 256, 384))
    codes, s = oracle.quantize_bw_128x128(w)
    assert s.shape == (2, 2, 3)
    # one tile checked against the exact-rational formulation
    tile = w[1, 128:256, 256:384]
    sf, cs = scalar.quantize_block_bw([int(t) for t in tile.ravel()])
    assert float(sf) == float(s[1, 1, 2])
    assert list(codes[1, 128:256, 256:384].ravel()) == cs
    # each tile's scale depends only on that tile's amax
    w2 = w.copy()
    w2[0, :128, :128] = synth.f32_to_bf16_bits(np.full((128, 128), 1000.0, dtype=np.float32))
    _, s2 = oracle.quantize_bw_128x128(w2)
    changed = s2 != s
    assert changed[0, 0, 0] and changed.sum() == 1
    ct, st = transpose_bw_128x128(codes, s)
    assert np.array_equal(ct[1], codes[1].T) and np.array_equal(st[1], s[1].T)
    deq = oracle.dequantize_bw_128x128(codes, s)
    assert np.allclose(deq, synth.bf16_bits_to_f32(w), rtol=2 ** -3, atol=float(s.max()) * 2 ** -9)


def test_colwise_padded_segments():
    splits = np.array([200, 0, 1, 128, 55], dtype=np.int32)
    consts = [2.0 ** 8, 1.0, -2.0 ** -9, 3.0, 2.0 ** 14]
    C = 128
    x = synth.f32_to_bf16_bits(np.concatenate(
        [np.full((m, C), c, dtype=np.float32) for m, c in zip(splits, consts)]))
    codes, s, poff = oracle.quantize_bw_colwise_padded(x, splits)
    assert s.shape == (C, int(poff[-1]) // 128)
    for g, (m, c) in enumerate(zip(splits, consts)):
        assert poff[g + 1] - poff[g] == -(-m // 128) * 128
        for b in range(int(poff[g]) // 128, int(poff[g + 1]) // 128):
            # a constant block's dequant scale is fl32(|c|/448)
            want = np.float32(np.float32(abs(c)) / np.float32(448.0))
            assert (s[:, b] == want).all(), (g, b)
        j0 = int(poff[g])
        seg = codes[:, j0: j0 + m]
        assert (seg == (0xFE if c < 0 else 0x7E)).all()
        assert (codes[:, j0 + m: int(poff[g + 1])] == 0).all()


# ---------------------------------------------------------------- power-of-two scales

def test_pow2_scale_hand_worked_values():
    """s = the smallest power of two with 448 * s >= max(amax, 1e-4), worked by hand:
    448 -> 1 (exact fit), 449 -> 2, 447.99 -> 1, 896 -> 2, 0.875 = 448 * 2^-9 -> 2^-9,
    3 -> 2^-7 (448/128 = 3.5 >= 3 > 1.75), 1e-4 (the floor) -> 2^-22 (448 * 2^-22 =
    1.07e-4 >= 1e-4 > 5.3e-5)."""
    a = np.array([448.0, 449.0, 447.99, 896.0, 0.875, 3.0, 1e-4], dtype=np.float32)
    want = [1.0, 2.0, 1.0, 2.0, 2.0 ** -9, 2.0 ** -7, 2.0 ** -22]
    assert oracle.pow2_scale(a).tolist() == want


def test_pow2_block_codes_hand_worked():
    """A 1x128 block with amax 3: s = 2^-7, so 3 -> 384 = 1.5 * 2^8 (E4M3 0x7C),
    -1 -> -128 = -2^7 (0xF0), 0.5 -> 64 = 2^6 (0x68), 0 -> 0x00."""
    row = np.zeros(128, dtype=np.float32)
    row[:4] = [3.0, -1.0, 0.5, 0.0]
    codes, s = oracle.quantize_bw_1x128(synth.f32_to_bf16_bits(row[None, :]), pow2=True)
    assert s.tolist() == [[2.0 ** -7]]
    assert codes[0, :4].tolist() == [0x7C, 0xF0, 0x68, 0x00]


def test_pow2_matches_exact_rational_formulation():
    rng = np.random.default_rng(23)
    x = synth.normal_bf16(rng, (6, 256), std=3.0, outlier_frac=0.02)
    v = synth.bf16_bits_to_f32(x)
    x[4] = synth.f32_to_bf16_bits(v[4] * np.float32(1e-7))   # below the floor
    x[5, :128] = 0                                           # zero block
    x[5, 128] = synth.f32_to_bf16_bits(np.array([448.0], dtype=np.float32))[0]  # exact fit
    codes, s = oracle.quantize_bw_1x128(x, pow2=True)
    for r in range(x.shape[0]):
        for b in range(2):
            blk = [int(t) for t in x[r, 128 * b: 128 * b + 128]]
            sf, cs = scalar.quantize_block_bw(blk, pow2=True)
            assert float(sf) == float(s[r, b]), (r, b)
            assert list(codes[r, 128 * b: 128 * b + 128]) == cs, (r, b)


def test_pow2_scale_brackets_the_fp32_scale():
    """The power-of-two scale is the fp32 scale a/448 rounded up to a power of
    two: s_fp32 <= s_pow2 < 2 s_fp32 (up to the rounding of s_fp32), blockwise."""
    rng = np.random.default_rng(24)
    w = synth.normal_bf16(rng, (3, 256, 384), std=5.0, outlier_frac=0.05)
    _, s32 = oracle.quantize_bw_128x128(w)
    _, s2 = oracle.quantize_bw_128x128(w, pow2=True)
    m, _ = np.frexp(s2.astype(np.float64))
    assert (m == 0.5).all()                                   # powers of two
    r = s2.astype(np.float64) / s32.astype(np.float64)
    assert (r >= 1.0 - 2.0 ** -23).all() and (r < 2.0).all()


def test_pow2_colwise_segments_match_rowwise_of_each_expert():
    rng = np.random.default_rng(25)
    splits = np.array([130, 0, 5, 256], dtype=np.int32)
    x = synth.normal_bf16(rng, (int(splits.sum()), 96), std=2.0, outlier_frac=0.02)
    codes, s, poff = oracle.quantize_bw_colwise_padded(x, splits, pow2=True)
    off = np.concatenate([[0], np.cumsum(splits)])
    for g in range(len(splits)):
        p_g = int(poff[g + 1] - poff[g])
        if p_g == 0:
            continue
        seg = np.zeros((96, p_g), dtype=np.uint16)
        seg[:, : splits[g]] = x[off[g]: off[g + 1]].T
        cg, sg = oracle.quantize_bw_1x128(seg, pow2=True)
        assert np.array_equal(codes[:, poff[g]: poff[g + 1]], cg)
        assert np.array_equal(s[:, poff[g] // 128: poff[g + 1] // 128], sg)


# --------------------------------------------------------------------------
# Dequantizer pins ("Add ROCm Triton blockwise FP8 grouped GEMM", PR #716:
# the value is the E4M3 code times the fp32 scale of its own 1x128 block, or of
# its own 128x128 tile).  The scale arrays have as many blocks on each axis so
# that a transposed or shifted broadcast still has the right shape and must be
# caught by value.  E4M3 codes used: 0x38 = 1.0, 0xB8 = -1.0, 0x7E = 448,
# 0x01 = 2^-9, 0x00 = 0.
# --------------------------------------------------------------------------
def _pin_dequant_1x128(fn):
    codes = np.full((3, 384), 0x38, dtype=np.uint8)
    codes[1, 130] = 0xB8
    codes[2, 300] = 0x7E
    codes[0, 5] = 0x01
    codes[2, 0] = 0x00
    # row r, block b: 2^(3r + b) -- nine distinct scales
    s = np.array([[1.0, 2.0, 4.0], [8.0, 16.0, 32.0], [64.0, 128.0, 256.0]], dtype=np.float32)
    d = fn(codes, s)
    assert d.shape == (3, 384)
    # hand-worked elements: (row, col) -> code value x its block's scale
    expect = {(0, 0): 1.0, (0, 127): 1.0, (0, 128): 2.0, (0, 200): 2.0, (0, 383): 4.0,
              (1, 0): 8.0, (1, 130): -16.0, (1, 256): 32.0,
              (2, 0): 0.0, (2, 1): 64.0, (2, 255): 128.0, (2, 300): 448.0 * 256.0,
              (0, 5): 2.0 ** -9}
    for (r, c), v in expect.items():
        assert d[r, c] == v, ((r, c), d[r, c], v)
    # every other element of a block equals that block's scale
    for r in range(3):
        for b in range(3):
            blk = d[r, 128 * b: 128 * b + 128]
            others = np.delete(blk, [i for i in range(128) if (r, 128 * b + i) in expect])
            assert (others == 2.0 ** (3 * r + b)).all(), (r, b)


def _pin_dequant_128x128(fn):
    G, N, K = 2, 384, 384
    codes = np.full((G, N, K), 0x38, dtype=np.uint8)
    codes[0, 10, 300] = 0xB8
    codes[1, 383, 0] = 0x7E
    # expert g, tile (i, j): 2^(3i + j + 16g) -- eighteen distinct scales
    s = np.array([[[2.0 ** (3 * i + j + 16 * g) for j in range(3)] for i in range(3)] for g in range(G)],
                 dtype=np.float32)
    d = fn(codes, s)
    assert d.shape == (G, N, K)
    expect = {(0, 0, 0): 1.0, (0, 10, 300): -4.0, (0, 300, 10): 64.0, (0, 200, 200): 16.0,
              (0, 127, 128): 2.0, (0, 128, 127): 8.0, (1, 0, 0): 65536.0,
              (1, 383, 0): 448.0 * 2.0 ** 22, (1, 383, 383): 2.0 ** 24}
    for idx, v in expect.items():
        assert d[idx] == v, (idx, d[idx], v)
    for g in range(G):
        for i in range(3):
            for j in range(3):
                t = d[g, 128 * i: 128 * i + 128, 128 * j: 128 * j + 128]
                n_special = sum(1 for (gg, n, k) in expect
                                if gg == g and n // 128 == i and k // 128 == j and expect[(gg, n, k)] != 2.0 ** (3 * i + j + 16 * g))
                assert (t == 2.0 ** (3 * i + j + 16 * g)).sum() == 128 * 128 - n_special, (g, i, j)


def test_dequantize_1x128_hand_worked():
    _pin_dequant_1x128(oracle.dequantize_bw_1x128)


def test_dequantize_128x128_hand_worked():
    _pin_dequant_128x128(oracle.dequantize_bw_128x128)


def test_dequantize_pins_catch_planted_axis_swaps():
    """The pins above are not vacuous: a dequantizer that broadcasts its
    scales along the wrong axis (transposed block grid, or tiles read
    [K/128, N/128]) fails them."""
    def swapped_1x128(codes, s):
        return oracle.dequantize_bw_1x128(codes, np.ascontiguousarray(s.T))

    def swapped_128x128(codes, s):
        return oracle.dequantize_bw_128x128(codes, np.ascontiguousarray(np.swapaxes(s, 1, 2)))

    def shifted_128x128(codes, s):   # expert axis misread
        return oracle.dequantize_bw_128x128(codes, np.ascontiguousarray(s[::-1]))

    for planted, pin in ((swapped_1x128, _pin_dequant_1x128), (swapped_128x128, _pin_dequant_128x128),
                         (shifted_128x128, _pin_dequant_128x128)):
        try:
            pin(planted)
        except AssertionError:
            continue
        raise AssertionError(f"pin did not catch {planted.__name__}")


def test_dequantize_inverts_exact_constant_tiles():
    """Tiles of constant 7 * 2^k quantize exactly (s = 2^k / 64 is exact in
    fp32, the code is 448 = 0x7E), so dequantization must give back every
    element exactly, tile by tile, for both schemes."""
    ks = np.array([[-3, 0, 5], [9, -7, 2], [11, 1, -12]])
    w = np.empty((1, 384, 384), dtype=np.float32)
    for i in range(3):
        for j in range(3):
            w[0, 128 * i: 128 * i + 128, 128 * j: 128 * j + 128] = 7.0 * 2.0 ** ks[i, j]
    w[0, 200:210, 130:140] *= -1.0
    bits = synth.f32_to_bf16_bits(w)
    codes, s = oracle.quantize_bw_128x128(bits)
    assert (codes[0] & 0x7F == 0x7E).all()
    assert np.array_equal(oracle.dequantize_bw_128x128(codes, s), w.astype(np.float64))
    rows = bits[0, :3]                     # 3 rows x 3 blocks of 1x128
    c1, s1 = oracle.quantize_bw_1x128(rows)
    assert np.array_equal(oracle.dequantize_bw_1x128(c1, s1), w[0, :3].astype(np.float64))
