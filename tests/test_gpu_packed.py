"""Row-wise quantization with the scales in the tensor-core staging order, and
grouped GEMMs that read them without a repacking pass.

* The packed quantizer is bit-exact against the oracle: codes against the
  oracle's row-wise quantizer, scale bytes against ``oracle.pack_scales_mma``
  of the oracle's plain scales (every byte, zero padding included).
* GEMMs fed ORACLE-packed scales match the oracle's plain grouped GEMM within
  the bound -- this pins the packed layout to the tensor cores' reading of it.
* GEMMs fed library-packed operands equal, bit for bit, the same GEMMs fed the
  plain operands (the arithmetic is identical)."""

import ctypes

import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu

from gpu_util import bf16_to_dev, i32_to_dev, oracle_operand_rowwise, u8_to_dev  # noqa: E402

KINDS = {"mxfp4": ("e2m1", "e2m1"), "mxfp8": ("e4m3", "e4m3"), "a8w4": ("e4m3", "e2m1")}


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()


def _mxg():
    import fp8_bf16_mxfp4_gb300 as mxg
    return mxg


def _check_packed(op, x, elem, segments):
    d, s = oracle.quantize_mx_rowwise(x, elem)
    assert np.array_equal(op.data.cpu().numpy(), d)
    ref = oracle.pack_scales_mma(s, segments)
    got = op.scale.cpu().numpy()
    assert got.size >= ref.size
    assert np.array_equal(got[: ref.size], ref)


@pytest.mark.parametrize("elem", ["e2m1", "e4m3"])
@pytest.mark.parametrize("splits,cols", [([0, 1, 127, 129, 300, 0], 160), ([5], 32), ([128, 128], 4096),
                                          ([0, 0, 0, 3], 96)])
def test_packed_quantize_with_splits(elem, splits, cols):
    rng = np.random.default_rng(sum(splits) + cols)
    x = synth.normal_bf16(rng, (sum(splits), cols), std=2.0, outlier_frac=0.02)
    op = _mxg().mx_quantize_rowwise_packed(bf16_to_dev(x), elem, m_splits=i32_to_dev(splits), check=True)
    _check_packed(op, x, elem, splits)


@pytest.mark.parametrize("elem", ["e2m1", "e4m3"])
@pytest.mark.parametrize("G,N,cols", [(3, 288, 256), (1, 128, 96), (4, 96, 4128)])
def test_packed_quantize_equal_segments(elem, G, N, cols):
    rng = np.random.default_rng(G * N + cols)
    x = synth.normal_bf16(rng, (G * N, cols), outlier_frac=0.01)
    op = _mxg().mx_quantize_rowwise_packed(bf16_to_dev(x), elem, groups=G)
    torch.cuda.synchronize()
    _check_packed(op, x, elem, [N] * G)


def test_packed_quantize_max_experts():
    rng = np.random.default_rng(512)
    splits = rng.integers(0, 40, size=512)
    splits[rng.random(512) < 0.3] = 0
    x = synth.normal_bf16(rng, (int(splits.sum()), 64))
    op = _mxg().mx_quantize_rowwise_packed(bf16_to_dev(x), "e2m1", m_splits=i32_to_dev(splits), check=True)
    _check_packed(op, x, "e2m1", splits)


@pytest.mark.parametrize("bad", [[100, -1, 29], [100, 20, 20]])
def test_packed_quantize_bad_splits_write_nothing(bad):
    mxg = _mxg()
    from fp8_bf16_mxfp4_gb300 import _lib
    lib = _lib.load()
    rows, cols = 128, 64
    x = bf16_to_dev(synth.normal_bf16(np.random.default_rng(1), (rows, cols)))
    q = torch.full((rows, cols // 2), 0xA5, dtype=torch.uint8, device="cuda:0")
    nbytes = mxg.mx_packed_scale_bytes(rows, cols, 3)
    s = torch.full((nbytes,), 0x5A, dtype=torch.uint8, device="cuda:0")
    st = torch.zeros(1, dtype=torch.int32, device="cuda:0")
    vp = ctypes.c_void_p
    rc = lib.mx_quantize_rowwise_packed(vp(x.data_ptr()), rows, cols, cols, 1, vp(q.data_ptr()), cols // 2,
                                        vp(s.data_ptr()), nbytes, vp(i32_to_dev(bad).data_ptr()), 3,
                                        vp(st.data_ptr()), vp(torch.cuda.current_stream().cuda_stream))
    assert rc == 0
    assert int(st.item()) == 4          # MXG_ERR_SPLITS
    assert (q == 0xA5).all() and (s == 0x5A).all()


def _oracle_packed_operand(bits, elem, segments, G):
    """Oracle-quantized operand whose scales are packed by the oracle, in a
    buffer of the library's bound size with junk beyond the packed bytes."""
    mxg = _mxg()
    op, deq = oracle_operand_rowwise(bits, elem)
    _, s = oracle.quantize_mx_rowwise(bits, elem)
    packed = oracle.pack_scales_mma(s, segments)
    nbytes = mxg.mx_packed_scale_bytes(bits.shape[0], bits.shape[1], G)
    buf = np.full(max(nbytes, 16), 0xFF, dtype=np.uint8)       # NaN scales: must never be read
    buf[: packed.size] = packed
    return mxg.MXOperand(op.data, u8_to_dev(buf), elem, bits.shape[1], "packed"), deq


@pytest.mark.parametrize("kind", ["mxfp4", "mxfp8", "a8w4"])
@pytest.mark.parametrize("which", ["A", "W", "both"])
def test_fwd_with_oracle_packed_scales(kind, which):
    ea, eb = KINDS[kind]
    splits = np.array([0, 1, 127, 129, 300, 0], dtype=np.int32)
    G, S = len(splits), int(splits.sum())
    N, K = 288, (256 if kind == "a8w4" else 160)
    rng = np.random.default_rng(11)
    x = synth.normal_bf16(rng, (S, K), outlier_frac=0.01)
    w = synth.normal_bf16(rng, (G * N, K), outlier_frac=0.01)
    if which in ("A", "both"):
        A, Ad = _oracle_packed_operand(x, ea, splits, G)
    else:
        A, Ad = oracle_operand_rowwise(x, ea)
    if which in ("W", "both"):
        W, Wd = _oracle_packed_operand(w, eb, [N] * G, G)
    else:
        W, Wd = oracle_operand_rowwise(w, eb)
    Y = _mxg().grouped_gemm_fwd(A, W, i32_to_dev(splits), N, check=True)
    oracle.assert_gemm_close(Y.float().cpu().numpy(), oracle.grouped_fwd(Ad, Wd, splits, N),
                             f"fwd {kind} packed {which}")


@pytest.mark.parametrize("kind", ["mxfp4", "a8w4"])
def test_fwd_library_packed_equals_plain(kind):
    mxg = _mxg()
    ea, eb = KINDS[kind]
    splits = np.array([300, 0, 77, 1025, 2, 640, 129, 3000], dtype=np.int32)
    G, S, N, K = len(splits), int(splits.sum()), 640, 512
    rng = np.random.default_rng(21)
    x = bf16_to_dev(synth.normal_bf16(rng, (S, K), outlier_frac=0.01))
    w = bf16_to_dev(synth.normal_bf16(rng, (G * N, K), outlier_frac=0.01))
    d_splits = i32_to_dev(splits)
    Yp = mxg.grouped_gemm_fwd(mxg.mx_quantize_rowwise_packed(x, ea, m_splits=d_splits),
                              mxg.mx_quantize_rowwise_packed(w, eb, groups=G), d_splits, N, check=True)
    Y = mxg.grouped_gemm_fwd(mxg.mx_quantize_rowwise(x, ea), mxg.mx_quantize_rowwise(w, eb), d_splits, N,
                             check=True)
    assert torch.equal(Yp, Y)


def test_dgrad_with_packed_gradient():
    mxg = _mxg()
    splits = np.array([0, 50, 131, 7], dtype=np.int32)
    G, S, N, K = len(splits), int(splits.sum()), 96, 288
    rng = np.random.default_rng(31)
    dy = synth.normal_bf16(rng, (S, N), outlier_frac=0.01)
    w = synth.normal_bf16(rng, (G * N, K), outlier_frac=0.01)
    dY, dYd = _oracle_packed_operand(dy, "e2m1", splits, G)
    from gpu_util import oracle_operand_colwise
    Wt, Wtd, _ = oracle_operand_colwise(w, [N] * G, 32, "e2m1")
    d_splits = i32_to_dev(splits)
    dX = mxg.grouped_gemm_dgrad(dY, Wt, d_splits, check=True)
    oracle.assert_gemm_close(dX.float().cpu().numpy(), oracle.grouped_dgrad(dYd, Wtd, splits), "dgrad packed dY")
    dYl = mxg.mx_quantize_rowwise_packed(bf16_to_dev(dy), "e2m1", m_splits=d_splits)
    assert torch.equal(mxg.grouped_gemm_dgrad(dYl, Wt, d_splits, check=True), dX)


# ------------------------------------------------------------------ k-segmented (column-wise) operands

@pytest.mark.parametrize("elem", ["e2m1", "e4m3"])
@pytest.mark.parametrize("splits,pad,cols", [([37, 0, 5, 300, 64], 32, 160), ([200, 1, 0, 129], 128, 256),
                                             ([256, 256, 256], 32, 96)])
def test_colwise_packed_quantize(elem, splits, pad, cols):
    mxg = _mxg()
    splits = np.array(splits, dtype=np.int32)
    x = synth.normal_bf16(np.random.default_rng(cols + pad), (int(splits.sum()), cols), std=2.0,
                          outlier_frac=0.02)
    op, poff = mxg.mx_quantize_colwise_segment_padded(bf16_to_dev(x), i32_to_dev(splits), pad, elem,
                                                      check=True, packed=True)
    d, s, p = oracle.quantize_mx_colwise_segment_padded(x, splits, pad, elem)
    spad = int(p[-1])
    assert np.array_equal(poff.cpu().numpy(), p)
    cb = spad // 2 if elem == "e2m1" else spad
    assert np.array_equal(op.data.cpu().numpy()[:, :cb], d)
    ref = oracle.pack_scales_mma_kseg(s, p)
    got = op.scale.cpu().numpy()
    assert np.array_equal(got[: ref.size], ref)
    bound = mxg.mx_packed_colwise_scale_bytes(cols, op.cols, len(splits))
    assert (got[ref.size: bound] == 0).all()     # zeroed slack up to the bound


def _kseg_oracle_operand(bits, splits, pad, elem, capacity):
    """Oracle column-wise operand with oracle-packed scales (junk NaN scale
    bytes past the packed ones: they must never be read)."""
    mxg = _mxg()
    from gpu_util import oracle_operand_colwise
    op, deq, poff = oracle_operand_colwise(bits, splits, pad, elem, capacity=capacity)
    _, s, _ = oracle.quantize_mx_colwise_segment_padded(bits, splits, pad, elem)
    packed = oracle.pack_scales_mma_kseg(s, poff)
    nbytes = mxg.mx_packed_colwise_scale_bytes(bits.shape[1], capacity, len(splits))
    buf = np.full(nbytes, 0xFF, dtype=np.uint8)
    buf[: packed.size] = packed
    return mxg.MXOperand(op.data, u8_to_dev(buf), elem, capacity, "packed"), deq, poff


@pytest.mark.parametrize("kind", ["mxfp4", "mxfp8"])
def test_wgrad_with_oracle_packed_operands(kind):
    """Segments of odd multiples of 32 (a half-filled MXFP4 step at every
    expert's end, whose second block must carry the zero slack scale)."""
    e = KINDS[kind][0]
    splits = np.array([37, 0, 5, 300, 64, 33], dtype=np.int32)
    G, S = len(splits), int(splits.sum())
    N, K, pad = 160, 288, 32
    rng = np.random.default_rng(61)
    dy = synth.normal_bf16(rng, (S, N), outlier_frac=0.01)
    x = synth.normal_bf16(rng, (S, K), outlier_frac=0.01)
    cap = synth.padded_rows_capacity(S, G, pad)
    dYt, dYtd, poff = _kseg_oracle_operand(dy, splits, pad, e, cap)
    Xt, Xtd, _ = _kseg_oracle_operand(x, splits, pad, e, cap)
    init = rng.standard_normal((G, N, K)).astype(np.float32) * np.float32(1e-3)
    out = torch.from_numpy(init.copy()).to("cuda:0")
    _mxg().grouped_gemm_wgrad(dYt, Xt, i32_to_dev(splits), S, pad, out=out, accumulate=True, check=True)
    ref = oracle.grouped_wgrad(dYtd, Xtd, poff, out_init=init)
    oracle.assert_gemm_close(out.cpu().numpy(), ref, f"wgrad {kind} oracle-packed")


@pytest.mark.parametrize("kind", ["mxfp4", "mxfp8"])
def test_dgrad_and_wgrad_library_packed_equal_plain(kind):
    mxg = _mxg()
    e = KINDS[kind][0]
    splits = np.array([300, 0, 77, 513, 1, 129], dtype=np.int32)
    G, S, N, K, pad = len(splits), int(splits.sum()), 256, 384, 32
    rng = np.random.default_rng(71)
    dy = bf16_to_dev(synth.normal_bf16(rng, (S, N), outlier_frac=0.01))
    x = bf16_to_dev(synth.normal_bf16(rng, (S, K), outlier_frac=0.01))
    w = bf16_to_dev(synth.normal_bf16(rng, (G * N, K), outlier_frac=0.01))
    ds, ws = i32_to_dev(splits), i32_to_dev([N] * G)
    dYq = mxg.mx_quantize_rowwise_packed(dy, e, m_splits=ds)
    Wt, _ = mxg.mx_quantize_colwise_segment_padded(w, ws, 32, e, capacity=G * N, check=True)
    Wtp, _ = mxg.mx_quantize_colwise_segment_padded(w, ws, 32, e, capacity=G * N, check=True, packed=True)
    assert torch.equal(mxg.grouped_gemm_dgrad(dYq, Wtp, ds, check=True), mxg.grouped_gemm_dgrad(dYq, Wt, ds, check=True))
    cap = mxg.mx_padded_rows_capacity(S, G, pad)
    outs = []
    for packed in (False, True):
        dYt, _ = mxg.mx_quantize_colwise_segment_padded(dy, ds, pad, e, capacity=cap, check=True, packed=packed)
        Xt, _ = mxg.mx_quantize_colwise_segment_padded(x, ds, pad, e, capacity=cap, check=True, packed=packed)
        o = torch.full((G, N, K), 0.5, dtype=torch.float32, device="cuda:0")
        mxg.grouped_gemm_wgrad(dYt, Xt, ds, S, pad, out=o, accumulate=True, check=True)
        outs.append(o)
    assert torch.equal(outs[0], outs[1])
