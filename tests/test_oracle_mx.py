"""Pins for the MX quantization oracle (CPU only).

The oracle is checked against things other than itself: hand-worked blocks
(one of them the value printed in the PR #745 review), a second scalar
formulation (bit-field exponent, IEEE-style rounding on exact rationals), the
defining nearest-value property over all finite BF16 patterns, and algebraic
invariants (idempotence, sign symmetry, power-of-two covariance, segment
isolation)."""

import os

import numpy as np
import pytest

import oracle
from oracle import scalar
import synth
from conftest import parse_value, read_records


def bits_of(values):
    a = np.array(values, dtype=np.float32)
    b = synth.f32_to_bf16_bits(a)
    assert np.array_equal(synth.bf16_bits_to_f32(b), a), "golden value not exact in BF16"
    return b


def test_golden_blocks(golden_dir):
    recs = read_records(os.path.join(golden_dir, "mx_blocks.txt"))
    assert len(recs) >= 12
    for name, elem, scale_hex, data_hex, vals in recs:
        toks = vals.split()
        v = [parse_value(t) for t in toks] + [0.0] * (32 - len(toks))
        bits = bits_of(v)
        for i, t in enumerate(toks):
            if t == "-0":
                bits[i] = 0x8000
        data, scale = oracle.quantize_mx_rowwise(bits[None, :], elem)
        assert scale[0].tobytes().hex() == scale_hex, name
        assert data[0].tobytes().hex() == data_hex, name
        # the scalar formulation agrees
        sb, codes = scalar.quantize_block_mx([int(b) for b in bits], elem)
        assert sb == int(scale_hex, 16), name
        c = np.array(codes, dtype=np.uint8)
        packed = oracle.pack_e2m1(c) if elem == "e2m1" else c
        assert packed.tobytes().hex() == data_hex, name


def _finite_bf16():
    b = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    return b[((b >> 7) & 0xFF) != 0xFF]


@pytest.mark.parametrize("elem", ["e2m1", "e4m3"])
def test_single_value_blocks_match_scalar_formulation(elem):
    """Every finite BF16 value alone in a block: scale and code agree with the
    bit-field / exact-rational formulation."""
    b = _finite_bf16()
    blocks = np.zeros((b.shape[0], 32), dtype=np.uint16)
    blocks[:, 0] = b
    codes, scale = oracle.quantize_mx(blocks, elem)
    assert (codes[:, 1:] == 0).all()
    from fractions import Fraction
    for i in range(0, b.shape[0], 7):      # every 7th pattern: all binades, both signs
        bb = int(b[i])
        e = scalar.mx_scale_exponent([bb], elem)
        assert scale[i, 0] == e + 127, hex(bb)
        want = scalar.encode(scalar.bf16_value(bb) / Fraction(2) ** e, elem, bool(bb >> 15))
        assert codes[i, 0] == want, hex(bb)


@pytest.mark.parametrize("elem,anchor", [("e2m1", 6.0), ("e2m1", 2.0 ** -120),
                                         ("e2m1", 1.5 * 2.0 ** 100), ("e4m3", 448.0),
                                         ("e4m3", 2.0 ** -118), ("e4m3", 2.0 ** 90)])
def test_nearest_value_property_all_bf16(elem, anchor):
    """With the block's scale fixed by an anchor element, every BF16 value
    |b| <= anchor decodes to the nearest element value (ties: even code),
    saturating at the largest magnitude, sign kept."""
    b = _finite_bf16()
    vals = synth.bf16_bits_to_f32(b).astype(np.float64)
    b = b[np.abs(vals) <= anchor]
    vals = np.abs(synth.bf16_bits_to_f32(b).astype(np.float64))
    blocks = np.zeros((b.shape[0], 32), dtype=np.uint16)
    blocks[:, 0] = bits_of([anchor])[0]
    blocks[:, 1] = b
    codes, scale = oracle.quantize_mx(blocks, elem)
    e = int(scale[0, 0]) - 127
    assert (scale == scale[0, 0]).all()
    fl = int(np.floor(np.log2(anchor)))
    emax = 2 if elem == "e2m1" else 8
    assert e == max(-127, min(127, fl - emax))
    c = codes[:, 1].astype(np.int64)
    sb = 3 if elem == "e2m1" else 7
    assert np.array_equal((c >> sb) & 1, (b >> 15).astype(np.int64))
    grid = oracle.E2M1_MAGNITUDES if elem == "e2m1" else oracle.e4m3_magnitudes()
    got = grid[c & ((1 << sb) - 1)]
    y = np.ldexp(vals, -e)
    dist_all = np.abs(grid[None, :] - y[:, None])
    best = dist_all.min(axis=1)
    assert np.all(np.abs(got - y) == best), "not a nearest value"
    ties = (dist_all == best[:, None]).sum(axis=1) > 1
    assert np.all(((c & ((1 << sb) - 1))[ties] % 2) == 0), "tie not to even code"


def test_idempotence_and_symmetry():
    rng = np.random.default_rng(7)
    for elem in ("e2m1", "e4m3"):
        x = synth.normal_bf16(rng, (64, 256), std=3.0, outlier_frac=0.02)
        codes, scale = oracle.quantize_mx(x, elem)
        deq = oracle.dequantize_mx(codes, scale, elem)
        back = synth.f32_to_bf16_bits(deq.astype(np.float32))
        assert np.array_equal(synth.bf16_bits_to_f32(back).astype(np.float64), deq)
        c2, s2 = oracle.quantize_mx(back, elem)
        assert np.array_equal(s2, scale) and np.array_equal(c2, codes)
        # sign symmetry: negating flips every code's sign bit, scales unchanged
        cn, sn = oracle.quantize_mx(x ^ np.uint16(0x8000), elem)
        sb = np.uint8(0x8 if elem == "e2m1" else 0x80)
        assert np.array_equal(sn, scale) and np.array_equal(cn, codes ^ sb)


def test_power_of_two_covariance():
    rng = np.random.default_rng(8)
    x = synth.normal_bf16(rng, (32, 128))
    v = synth.bf16_bits_to_f32(x)
    for elem in ("e2m1", "e4m3"):
        c0, s0 = oracle.quantize_mx(x, elem)
        for j in (-20, -3, 5, 40):
            xs = synth.f32_to_bf16_bits(v * np.float32(2.0 ** j))
            c, s = oracle.quantize_mx(xs, elem)
            assert np.array_equal(c, c0)
            assert np.array_equal(s.astype(int), s0.astype(int) + j)


def test_pack_roundtrip():
    rng = np.random.default_rng(9)
    c = rng.integers(0, 16, size=(5, 64)).astype(np.uint8)
    p = oracle.pack_e2m1(c)
    assert p.shape == (5, 32)
    assert np.array_equal(p & 0xF, c[:, 0::2])
    assert np.array_equal(oracle.unpack_e2m1(p), c)


def test_colwise_segments_do_not_straddle():
    """Each expert holds one constant with a very different magnitude; with
    blocks starting at every expert's padded origin, dequantization returns
    each constant exactly and the padding is zero.  A block crossing an
    expert boundary would crush the smaller constant to zero."""
    splits = np.array([37, 0, 5, 64, 33], dtype=np.int32)
    consts = [2.0 ** 10, 1.0, 2.0 ** -12, 3.0, 2.0 ** 20]
    C = 64
    rows = []
    for m, c in zip(splits, consts):
        rows.append(np.full((m, C), c, dtype=np.float32))
    x = synth.f32_to_bf16_bits(np.concatenate(rows))
    for elem in ("e2m1", "e4m3"):
        for pad in (32, 64, 128):
            data, scale, poff = oracle.quantize_mx_colwise_segment_padded(x, splits, pad, elem)
            codes = oracle.unpack_e2m1(data) if elem == "e2m1" else data
            deq = oracle.dequantize_mx(codes, scale, elem)
            assert deq.shape == (C, int(poff[-1]))
            for g, (m, c) in enumerate(zip(splits, consts)):
                seg = deq[:, poff[g]: poff[g + 1]]
                assert seg.shape[1] == -(-m // pad) * pad
                assert (seg[:, :m] == c).all()
                assert (seg[:, m:] == 0).all()
            assert poff[-1] <= synth.padded_rows_capacity(int(splits.sum()), len(splits), pad)


def test_colwise_matches_scalar_per_column():
    rng = np.random.default_rng(11)
    splits = np.array([3, 40, 0, 29], dtype=np.int32)
    S, C = int(splits.sum()), 8
    x = synth.normal_bf16(rng, (S, C), std=2.0, outlier_frac=0.05)
    off = np.concatenate([[0], np.cumsum(splits)])
    for elem in ("e2m1", "e4m3"):
        data, scale, poff = oracle.quantize_mx_colwise_segment_padded(x, splits, 32, elem)
        codes = oracle.unpack_e2m1(data) if elem == "e2m1" else data
        for g in range(len(splits)):
            col_vals = x[off[g]: off[g + 1]]
            p = int(poff[g + 1] - poff[g])
            for c in range(C):
                seg = [int(v) for v in col_vals[:, c]] + [0] * (p - splits[g])
                for blk in range(p // 32):
                    sb, cs = scalar.quantize_block_mx(seg[32 * blk: 32 * blk + 32], elem)
                    j = int(poff[g]) + 32 * blk
                    assert scale[c, j // 32] == sb
                    assert list(codes[c, j: j + 32]) == cs


def test_colwise_pad_invariance():
    rng = np.random.default_rng(12)
    splits = np.array([70, 1, 0, 130, 31], dtype=np.int32)
    x = synth.normal_bf16(rng, (int(splits.sum()), 96))
    for elem in ("e2m1", "e4m3"):
        outs = []
        for pad in (32, 128):
            data, scale, poff = oracle.quantize_mx_colwise_segment_padded(x, splits, pad, elem)
            codes = oracle.unpack_e2m1(data) if elem == "e2m1" else data
            deq = oracle.dequantize_mx(codes, scale, elem)
            outs.append([deq[:, poff[g]: poff[g] + splits[g]] for g in range(len(splits))])
        for a, b in zip(*outs):
            assert np.array_equal(a, b)


def test_colwise_rejects_bad_splits():
    x = np.zeros((10, 32), dtype=np.uint16)
    with pytest.raises(ValueError):
        oracle.quantize_mx_colwise_segment_padded(x, [5, 4], 32, "e2m1")
    with pytest.raises(ValueError):
        oracle.quantize_mx_colwise_segment_padded(x, [12, -2], 32, "e2m1")
    with pytest.raises(ValueError):
        oracle.quantize_mx_colwise_segment_padded(x, [10], 48, "e2m1")


# ---------------------------------------------------------------- round-up scale rule

def test_golden_blocks_round_up(golden_dir):
    recs = read_records(os.path.join(golden_dir, "mx_roundup_blocks.txt"))
    assert len(recs) >= 8
    for name, elem, scale_hex, data_hex, vals in recs:
        toks = vals.split()
        v = [parse_value(t) for t in toks] + [0.0] * (32 - len(toks))
        bits = bits_of(v)
        data, scale = oracle.quantize_mx_rowwise(bits[None, :], elem, rule="round_up")
        assert scale[0].tobytes().hex() == scale_hex, name
        assert data[0].tobytes().hex() == data_hex, name
        sb, codes = scalar.quantize_block_mx([int(b) for b in bits], elem, rule="round_up")
        assert sb == int(scale_hex, 16), name


@pytest.mark.parametrize("elem", ["e2m1", "e4m3"])
def test_round_up_exponent_is_the_smallest_covering_power(elem):
    """Over every finite positive BF16 amax: maxval * 2^e >= amax, and 2^(e-1)
    would not cover it (unless e sits at the -127 floor)."""
    bits = np.arange(1, 0x7F80, dtype=np.uint16)
    amax = oracle.mx.bf16_to_f64(bits)
    e = oracle.shared_exponent(amax, elem, rule="round_up")
    mv = 6.0 if elem == "e2m1" else 448.0
    assert (np.ldexp(mv, e) >= amax).all()
    assert ((e == -127) | (np.ldexp(mv, e - 1) < amax)).all()
    # against the OCP exponent: equal, or one more exactly where OCP saturates the amax
    eo = oracle.shared_exponent(amax, elem)
    over = np.ldexp(mv, eo) < amax
    assert np.array_equal(e, np.clip(eo + over, -127, 127))


@pytest.mark.parametrize("elem", ["e2m1", "e4m3"])
def test_round_up_never_saturates_and_matches_scalar(elem):
    rng = np.random.default_rng(17)
    x = synth.normal_bf16(rng, (64, 32), std=3.0, outlier_frac=0.05)
    x[:4] = synth.f32_to_bf16_bits(np.float32(2.0) ** rng.integers(-140, 120, size=(4, 32)).astype(np.float32))
    codes, scale = oracle.quantize_mx(x, elem, rule="round_up")
    e = scale.astype(np.int64) - 127
    xs = oracle.mx.bf16_to_f64(x).reshape(64, 1, 32)
    mv = 6.0 if elem == "e2m1" else 448.0
    assert (np.abs(np.ldexp(xs, -e[..., None])) <= mv).all()
    for r in range(0, 64, 7):
        sb, cs = scalar.quantize_block_mx([int(b) for b in x[r]], elem, rule="round_up")
        assert sb == int(scale[r, 0]) and cs == [int(c) for c in codes[r]]


def test_round_up_colwise_matches_rowwise_of_the_transposed_segments():
    rng = np.random.default_rng(23)
    splits = [5, 0, 40, 33]
    x = synth.normal_bf16(rng, (sum(splits), 64), std=2.0, outlier_frac=0.05)
    d, s, poff = oracle.quantize_mx_colwise_segment_padded(x, splits, 32, "e4m3", rule="round_up")
    off = np.concatenate([[0], np.cumsum(splits)])
    for g, m in enumerate(splits):
        if m == 0:
            continue
        seg = np.zeros((64, int(poff[g + 1] - poff[g])), dtype=np.uint16)
        seg[:, :m] = x[off[g]: off[g + 1]].T
        dg, sg = oracle.quantize_mx_rowwise(seg, "e4m3", rule="round_up")
        assert np.array_equal(d[:, poff[g]: poff[g + 1]], dg)
        assert np.array_equal(s[:, poff[g] // 32: poff[g + 1] // 32], sg)
