"""GPU quantizers vs the oracle: bytes and scales must be bit-exact."""

import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu

from gpu_util import bf16_to_dev, i32_to_dev  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()


def _mxg():
    import fp8_bf16_mxfp4_gb300 as mxg
    return mxg


@pytest.mark.parametrize("elem", ["e2m1", "e4m3"])
@pytest.mark.parametrize("shape", [(1, 32), (7, 96), (257, 512), (1000, 4128), (3, 14336)])
def test_rowwise_random(elem, shape):
    rng = np.random.default_rng(shape[0] * 7 + shape[1])
    x = synth.normal_bf16(rng, shape, std=2.0, outlier_frac=0.02)
    op = _mxg().mx_quantize_rowwise(bf16_to_dev(x), elem)
    torch.cuda.synchronize()
    d, s = oracle.quantize_mx_rowwise(x, elem)
    assert np.array_equal(op.data.cpu().numpy(), d)
    assert np.array_equal(op.scale.cpu().numpy(), s)


@pytest.mark.parametrize("elem", ["e2m1", "e4m3"])
def test_rowwise_strided_input_and_outputs(elem):
    rng = np.random.default_rng(5)
    x = synth.normal_bf16(rng, (33, 512))
    xd = bf16_to_dev(x)
    big = torch.zeros((33, 640), dtype=torch.bfloat16, device=xd.device)
    big[:, :512] = xd
    mxg = _mxg()
    cb = 256 if elem == "e2m1" else 512
    q = torch.full((33, cb + 48), 0xAB, dtype=torch.uint8, device=xd.device)
    s = torch.full((33, 16 + 16), 0xCD, dtype=torch.uint8, device=xd.device)
    op = mxg.mx_quantize_rowwise(big[:, :512], elem, q=q[:, :cb], s=s[:, :16])
    torch.cuda.synchronize()
    d, sc = oracle.quantize_mx_rowwise(x, elem)
    assert np.array_equal(op.data.cpu().numpy(), d)
    assert np.array_equal(op.scale.cpu().numpy(), sc)
    assert (q[:, cb:] == 0xAB).all() and (s[:, 16:] == 0xCD).all()   # nothing outside


def _anchored_blocks(anchor_bits: int, rest: np.ndarray) -> np.ndarray:
    blocks = np.zeros((rest.shape[0], 32), dtype=np.uint16)
    blocks[:, 0] = anchor_bits
    blocks[:, 1] = rest
    blocks[:, 2] = rest ^ 0x8000        # its negation too
    return blocks


@pytest.mark.parametrize("elem", ["e2m1", "e4m3"])
def test_every_finite_bf16_value(elem):
    """All finite BF16 patterns, alone in a block and next to anchors that fix
    the scale at several binades (subnormal, tie and saturation cases)."""
    b = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    b = b[((b >> 7) & 0xFF) != 0xFF]
    rows = [np.pad(b[:, None], ((0, 0), (0, 31)))]
    vals = np.abs(synth.bf16_bits_to_f32(b).astype(np.float64))
    for anchor in (6.0, 448.0, 2.0 ** -120, 2.0 ** -126, 1.5 * 2.0 ** 100, 2.0 ** 127):
        ab = int(synth.f32_to_bf16_bits(np.array([anchor], dtype=np.float32))[0])
        sel = b[vals <= anchor]
        rows.append(_anchored_blocks(ab, sel))
    x = np.concatenate(rows)
    op = _mxg().mx_quantize_rowwise(bf16_to_dev(x), elem)
    torch.cuda.synchronize()
    d, s = oracle.quantize_mx_rowwise(x, elem)
    gd, gs = op.data.cpu().numpy(), op.scale.cpu().numpy()
    assert np.array_equal(gs, s)
    if not np.array_equal(gd, d):
        bad = np.argwhere(gd != d)[:5]
        raise AssertionError(f"code mismatch at {bad.tolist()}: gpu {gd[tuple(bad[0])]:#x} "
                             f"oracle {d[tuple(bad[0])]:#x} input row {x[bad[0][0], :4]}")


def test_rowwise_zero_rows_is_a_noop():
    x = torch.empty((0, 64), dtype=torch.bfloat16, device="cuda:0")
    op = _mxg().mx_quantize_rowwise(x, "e2m1")
    torch.cuda.synchronize()
    assert op.data.shape == (0, 32)


COL_CASES = [
    ([37, 0, 5, 64, 33], 32, 64),
    ([0, 0, 1], 32, 96),
    ([300, 17, 0, 129], 128, 160),
    ([512], 32, 32),
    ([1, 2, 3, 4, 5, 6, 7, 8], 64, 256),
]


@pytest.mark.parametrize("elem", ["e2m1", "e4m3"])
@pytest.mark.parametrize("splits,pad,cols", COL_CASES)
def test_colwise_segment_padded(elem, splits, pad, cols):
    rng = np.random.default_rng(len(splits) * 31 + pad + cols)
    splits = np.array(splits, dtype=np.int32)
    S = int(splits.sum())
    x = synth.normal_bf16(rng, (S, cols), std=3.0, outlier_frac=0.03)
    mxg = _mxg()
    st = torch.zeros(1, dtype=torch.int32, device="cuda:0")
    op, poff = mxg.mx_quantize_colwise_segment_padded(bf16_to_dev(x), i32_to_dev(splits), pad, elem,
                                                      status=st, check=True)
    d, s, p = oracle.quantize_mx_colwise_segment_padded(x, splits, pad, elem)
    spad = int(p[-1])
    assert np.array_equal(poff.cpu().numpy(), p)
    gd = op.data.cpu().numpy()
    cb = spad // 2 if elem == "e2m1" else spad
    assert np.array_equal(gd[:, :cb], d)
    assert np.array_equal(op.scale.cpu().numpy()[:, : spad // 32], s)


@pytest.mark.parametrize("bad,code", [([10, -1, 5], 4), ([5, 5, 5], 4), ([14, 0, 0], 10)])
def test_colwise_rejects_bad_splits_on_device(bad, code):
    """Invalid splits are detected on the device: status is set and no output
    byte is written."""
    mxg = _mxg()
    x = bf16_to_dev(synth.normal_bf16(np.random.default_rng(1), (14, 64)))
    st = torch.zeros(1, dtype=torch.int32, device="cuda:0")
    cap, pad = (32, 64) if code == 10 else (96, 32)   # [14,0,0] pads to 64 > capacity 32
    q = torch.full((64, cap), 0xAB, dtype=torch.uint8, device="cuda:0")
    sc = torch.full((64, cap // 32), 0xCD, dtype=torch.uint8, device="cuda:0")
    poff = torch.full((4,), -7, dtype=torch.int64, device="cuda:0")
    rc = mxg._lib.load().mx_quantize_colwise_segment_padded(
        mxg._ptr(x), 14, 64, 64, mxg._ptr(i32_to_dev(bad)), 3, pad, 2, mxg._ptr(q), q.stride(0),
        mxg._ptr(sc), sc.stride(0), cap, mxg._ptr(poff), mxg._ptr(st), mxg._stream(x.device))
    assert rc == 0
    with pytest.raises(mxg.MXGError) as ei:
        mxg.check_status(st)
    assert ei.value.code == code
    assert (q == 0xAB).all() and (sc == 0xCD).all() and (poff == -7).all()


# ------------------------------------------------------------------ fused dual quantizer

DUAL_CASES = COL_CASES + [([2000, 0, 1, 700, 129], 32, 4128)]   # > one column tile, ragged


@pytest.mark.parametrize("elem", ["e2m1", "e4m3"])
@pytest.mark.parametrize("splits,pad,cols", DUAL_CASES)
def test_dual_matches_rowwise_and_colwise_oracles(elem, splits, pad, cols):
    """One read of x: the row-wise operand and the column-wise segment-padded
    operand, each bit-exact against its own oracle."""
    rng = np.random.default_rng(len(splits) * 17 + pad + cols)
    splits = np.array(splits, dtype=np.int32)
    S = int(splits.sum())
    x = synth.normal_bf16(rng, (S, cols), std=3.0, outlier_frac=0.03)
    mxg = _mxg()
    st = torch.zeros(1, dtype=torch.int32, device="cuda:0")
    row, col, poff = mxg.mx_quantize_dual_segment_padded(bf16_to_dev(x), i32_to_dev(splits), pad, elem,
                                                         status=st, check=True)
    rd, rs = oracle.quantize_mx_rowwise(x, elem)
    assert np.array_equal(row.data.cpu().numpy(), rd)
    assert np.array_equal(row.scale.cpu().numpy(), rs)
    d, s, p = oracle.quantize_mx_colwise_segment_padded(x, splits, pad, elem)
    spad = int(p[-1])
    assert np.array_equal(poff.cpu().numpy(), p)
    cb = spad // 2 if elem == "e2m1" else spad
    assert np.array_equal(col.data.cpu().numpy()[:, :cb], d)
    assert np.array_equal(col.scale.cpu().numpy()[:, : spad // 32], s)


def test_dual_rejects_bad_splits_and_writes_nothing():
    mxg = _mxg()
    x = bf16_to_dev(synth.normal_bf16(np.random.default_rng(2), (14, 64)))
    st = torch.zeros(1, dtype=torch.int32, device="cuda:0")
    q = torch.full((14, 32), 0xAB, dtype=torch.uint8, device="cuda:0")
    s = torch.full((14, 2), 0xCD, dtype=torch.uint8, device="cuda:0")
    qT = torch.full((64, 48), 0xAB, dtype=torch.uint8, device="cuda:0")
    sT = torch.full((64, 3), 0xCD, dtype=torch.uint8, device="cuda:0")
    poff = torch.full((4,), -7, dtype=torch.int64, device="cuda:0")
    rc = mxg._lib.load().mx_quantize_dual_segment_padded(
        mxg._ptr(x), 14, 64, 64, mxg._ptr(i32_to_dev([10, -1, 5])), 3, 32, 1, mxg._ptr(q), 32,
        mxg._ptr(s), 2, mxg._ptr(qT), 48, mxg._ptr(sT), 3, 96, mxg._ptr(poff), mxg._ptr(st),
        mxg._stream(x.device))
    assert rc == 0
    with pytest.raises(mxg.MXGError) as ei:
        mxg.check_status(st)
    assert ei.value.code == 4
    assert (q == 0xAB).all() and (s == 0xCD).all() and (qT == 0xAB).all() and (sT == 0xCD).all()
    assert (poff == -7).all()


@pytest.mark.parametrize("elem", ["e2m1", "e4m3"])
def test_colwise_and_dual_with_512_experts(elem):
    """G = 512, the most the library accepts (the prefix tables' last entry is
    the one no scan pair reaches): a few ragged experts among empty ones."""
    splits = np.zeros(512, dtype=np.int32)
    splits[[0, 3, 200, 511]] = [33, 64, 1, 90]
    rng = np.random.default_rng(77)
    x = synth.normal_bf16(rng, (int(splits.sum()), 64), std=2.0, outlier_frac=0.02)
    mxg = _mxg()
    op, poff = mxg.mx_quantize_colwise_segment_padded(bf16_to_dev(x), i32_to_dev(splits), 32, elem, check=True)
    d, s, p = oracle.quantize_mx_colwise_segment_padded(x, splits, 32, elem)
    spad = int(p[-1])
    cb = spad // 2 if elem == "e2m1" else spad
    assert np.array_equal(poff.cpu().numpy(), p)
    assert np.array_equal(op.data.cpu().numpy()[:, :cb], d)
    assert np.array_equal(op.scale.cpu().numpy()[:, : spad // 32], s)
    row, col, poff2 = mxg.mx_quantize_dual_segment_padded(bf16_to_dev(x), i32_to_dev(splits), 32, elem, check=True)
    rd, rs = oracle.quantize_mx_rowwise(x, elem)
    assert np.array_equal(row.data.cpu().numpy(), rd) and np.array_equal(row.scale.cpu().numpy(), rs)
    assert np.array_equal(col.data.cpu().numpy()[:, :cb], d)
