"""Blockwise FP8 on the GPU vs the oracle: quantizers bit-exact (codes and
fp32 scales), grouped GEMMs within |gpu - ref| <= 2^-8 |ref| + 1e-4 rms(ref)
on oracle-quantized operands.

Layout notes: the library stores activation-type scales block-column-major
([cols/128, rows]); the oracle returns them [rows, cols/128], so the tests
transpose.  The dgrad weight copy is [K, G*N] (experts side by side)."""

import numpy as np
import pytest
import torch

import oracle
from oracle.blockwise import transpose_bw_128x128
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


@pytest.fixture(params=[2, 1], ids=["pair", "onesm"])
def cta_group(request):
    """GEMM cases run on the CTA-pair kernel (256 x 256 tiles, 2-SM MMA, the
    default) and on the one-SM kernel (128 x 128 tiles)."""
    prev = _mxg().set_gemm_cta_group(request.param)
    yield request.param
    _mxg().set_gemm_cta_group(prev)


def _f32_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to("cuda:0")


def _u8_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint8)).to("cuda:0")


@pytest.mark.parametrize("shape", [(1, 128), (37, 384), (1000, 4096)])
def test_bw_1x128_bit_exact(shape):
    rng = np.random.default_rng(shape[0])
    x = synth.normal_bf16(rng, shape, std=2.0, outlier_frac=0.02)
    if shape[0] > 4:
        v = synth.bf16_bits_to_f32(x)
        x[1] = synth.f32_to_bf16_bits(v[1] * np.float32(1e-7))   # below the 1e-4 amax floor
        x[2, :128] = 0                                           # a zero block
        x[3, :128] = synth.f32_to_bf16_bits(np.full(128, -2.0, np.float32))
    op = _mxg().bw_quantize_1x128(bf16_to_dev(x))
    torch.cuda.synchronize()
    codes, s = oracle.quantize_bw_1x128(x)
    assert np.array_equal(op.data.cpu().numpy(), codes)
    assert np.array_equal(op.scale.cpu().numpy(), s.T)


def test_bw_128x128_and_dgrad_copy_bit_exact():
    rng = np.random.default_rng(3)
    G, N, K = 2, 256, 384
    w = synth.normal_bf16(rng, (G * N, K), outlier_frac=0.02)
    op, opT = _mxg().bw_quantize_128x128(bf16_to_dev(w))
    torch.cuda.synchronize()
    codes, s = oracle.quantize_bw_128x128(w.reshape(G, N, K))
    assert np.array_equal(op.data.cpu().numpy(), codes.reshape(G * N, K))
    assert np.array_equal(op.scale.cpu().numpy(), s.reshape(G * N // 128, K // 128))
    ct, st = transpose_bw_128x128(codes, s)
    assert np.array_equal(opT.data.cpu().numpy(), np.concatenate(list(ct), axis=1))
    assert np.array_equal(opT.scale.cpu().numpy(), np.concatenate(list(st), axis=1))


@pytest.mark.parametrize("splits,cols", [([200, 0, 1, 128, 55], 128), ([0, 0, 300], 256),
                                         ([1, 2, 3, 4], 160)])
def test_bw_colwise_padded_bit_exact(splits, cols):
    rng = np.random.default_rng(len(splits) + cols)
    splits = np.array(splits, dtype=np.int32)
    x = synth.normal_bf16(rng, (int(splits.sum()), cols), std=3.0, outlier_frac=0.02)
    op, poff = _mxg().bw_quantize_colwise_padded(bf16_to_dev(x), i32_to_dev(splits), check=True)
    codes, s, p = oracle.quantize_bw_colwise_padded(x, splits)
    spad = int(p[-1])
    assert np.array_equal(poff.cpu().numpy(), p)
    assert np.array_equal(op.data.cpu().numpy()[:, :spad], codes)
    assert np.array_equal(op.scale.cpu().numpy()[: spad // 128], s.T)


# ------------------------------------------------------------------------------ GEMMs

def _act_operand(bits):
    """Oracle 1x128 quantization -> (device operand, dequantized float64)."""
    codes, s = oracle.quantize_bw_1x128(bits)
    return _mxg().BWOperand(_u8_dev(codes), _f32_dev(s.T)), oracle.dequantize_bw_1x128(codes, s)


@pytest.mark.parametrize("splits,N,K", [([0, 130, 1, 300], 256, 384), ([512], 128, 128),
                                        ([64, 64], 384, 1024)])
def test_bw_fwd_parity(splits, N, K, cta_group):
    mxg = _mxg()
    splits = np.asarray(splits, dtype=np.int32)
    G, S = len(splits), int(splits.sum())
    rng = np.random.default_rng(N + K)
    x = synth.normal_bf16(rng, (S, K), outlier_frac=0.01)
    w = synth.normal_bf16(rng, (G * N, K), outlier_frac=0.01)
    A, Ad = _act_operand(x)
    wc, ws = oracle.quantize_bw_128x128(w.reshape(G, N, K))
    W = mxg.BWOperand(_u8_dev(wc.reshape(G * N, K)), _f32_dev(ws.reshape(G * N // 128, K // 128)))
    Wd = oracle.dequantize_bw_128x128(wc, ws).reshape(G * N, K)
    Y = mxg.bw_grouped_gemm_fwd(A, W, i32_to_dev(splits), N, check=True)
    oracle.assert_gemm_close(Y.float().cpu().numpy(), oracle.grouped_fwd(Ad, Wd, splits, N), "bw fwd")


def test_bw_fwd_many_tiles(cta_group):
    """More tiles than CTA pairs (the persistent loop wraps several times),
    ragged experts whose last 256-row pair has its odd CTA past the rows, and
    N with a half-wide last column tile."""
    rng = np.random.default_rng(77)
    splits = rng.integers(100, 700, size=40).astype(np.int32)
    splits[[3, 17]] = 0
    splits[5] = 129
    test_bw_fwd_parity(splits.tolist(), 640, 256, cta_group)


def test_bw_fwd_max_experts(cta_group):
    """G = 512 (the largest supported), most experts empty, a few with rows:
    the plan's totals entry and the tile walk at the largest G."""
    rng = np.random.default_rng(512)
    splits = np.zeros(512, dtype=np.int32)
    live = rng.choice(512, size=24, replace=False)
    splits[live] = rng.integers(1, 200, size=24)
    splits[511] = 130                                   # the last expert non-empty
    test_bw_fwd_parity(splits.tolist(), 128, 128, cta_group)


@pytest.mark.parametrize("splits,N,K", [([0, 77, 300], 256, 384), ([128], 128, 256),
                                        ([400, 3, 0, 260], 384, 640)])
def test_bw_dgrad_parity(splits, N, K, cta_group):
    mxg = _mxg()
    splits = np.asarray(splits, dtype=np.int32)
    G, S = len(splits), int(splits.sum())
    rng = np.random.default_rng(N * 3 + K)
    dy = synth.normal_bf16(rng, (S, N), outlier_frac=0.01)
    w = synth.normal_bf16(rng, (G * N, K), outlier_frac=0.01)
    dY, dYd = _act_operand(dy)
    wc, ws = oracle.quantize_bw_128x128(w.reshape(G, N, K))
    ct, st = transpose_bw_128x128(wc, ws)
    Wt = mxg.BWOperand(_u8_dev(np.concatenate(list(ct), axis=1)), _f32_dev(np.concatenate(list(st), axis=1)))
    Wtd = np.concatenate(list(oracle.dequantize_bw_128x128(ct, st)), axis=1)
    dX = mxg.bw_grouped_gemm_dgrad(dY, Wt, i32_to_dev(splits), check=True)
    oracle.assert_gemm_close(dX.float().cpu().numpy(), oracle.grouped_dgrad(dYd, Wtd, splits), "bw dgrad")


def _col_operand(bits, splits, capacity):
    codes, s, poff = oracle.quantize_bw_colwise_padded(bits, splits)
    C, spad = codes.shape
    rng = np.random.default_rng(5)
    full = rng.integers(0, 0x77, size=(C, capacity)).astype(np.uint8)   # finite junk slack
    full[:, :spad] = codes
    fs = np.full((capacity // 128, C), 7.0, dtype=np.float32)
    fs[: spad // 128] = s.T
    deq = codes.astype(np.float64)
    deq = oracle.dequantize_bw_1x128(codes, s)
    return _mxg().BWOperand(_u8_dev(full), _f32_dev(fs)), deq, poff


@pytest.mark.parametrize("accumulate", [False, True])
@pytest.mark.parametrize("N,K", [(256, 384), (384, 640)])
def test_bw_wgrad_parity(accumulate, N, K, cta_group):
    mxg = _mxg()
    splits = np.array([200, 0, 1, 300, 129], dtype=np.int32)
    G, S = len(splits), int(splits.sum())
    rng = np.random.default_rng(11 + accumulate + N)
    dy = synth.normal_bf16(rng, (S, N), outlier_frac=0.01)
    x = synth.normal_bf16(rng, (S, K), outlier_frac=0.01)
    cap = synth.padded_rows_capacity(S, G, 128)
    dYt, dYtd, poff = _col_operand(dy, splits, cap)
    Xt, Xtd, _ = _col_operand(x, splits, cap)
    init = (rng.standard_normal((G, N, K)) * 1e-3).astype(np.float32)
    out = torch.from_numpy(init.copy()).to("cuda:0")
    mxg.bw_grouped_gemm_wgrad(dYt, Xt, i32_to_dev(splits), S, out=out, accumulate=accumulate, check=True)
    ref = oracle.grouped_wgrad(dYtd, Xtd, poff, out_init=init if accumulate else None)
    got = out.cpu().numpy()
    oracle.assert_gemm_close(got, ref, f"bw wgrad acc={accumulate}")
    assert np.array_equal(got[1], init[1] if accumulate else np.zeros_like(init[1]))


def test_bw_gemm_rejects_bad_splits(cta_group):
    mxg = _mxg()
    rng = np.random.default_rng(2)
    A, _ = _act_operand(synth.normal_bf16(rng, (128, 128)))
    wc, ws = oracle.quantize_bw_128x128(synth.normal_bf16(rng, (256, 128)).reshape(2, 128, 128))
    W = mxg.BWOperand(_u8_dev(wc.reshape(256, 128)), _f32_dev(ws.reshape(2, 1)))
    out = torch.full((128, 128), 5.0, dtype=torch.bfloat16, device="cuda:0")
    st = torch.zeros(1, dtype=torch.int32, device="cuda:0")
    mxg.bw_grouped_gemm_fwd(A, W, i32_to_dev([130, -2]), 128, out=out, status=st)
    with pytest.raises(mxg.MXGError) as ei:
        mxg.check_status(st)
    assert ei.value.code == 4 and (out == 5.0).all()


# ------------------------------------------------------------- power-of-two scales (MX operands)

def _ue8m0(s, rep_rows=1, rep_cols=4):
    """UE8M0 bytes of power-of-two fp32 scales, each repeated over its rows and
    its four 32-blocks (the MX layout the pow2 quantizers write)."""
    k = np.frexp(np.asarray(s, dtype=np.float64))[1] - 1
    b = (k + 127).astype(np.uint8)
    return np.repeat(np.repeat(b, rep_rows, axis=-2), rep_cols, axis=-1)


@pytest.mark.parametrize("shape", [(1, 128), (37, 384), (1000, 4096)])
def test_bw_1x128_pow2_bit_exact(shape):
    rng = np.random.default_rng(shape[0] + 7)
    x = synth.normal_bf16(rng, shape, std=4.0, outlier_frac=0.02)
    if shape[0] > 4:
        v = synth.bf16_bits_to_f32(x)
        x[1] = synth.f32_to_bf16_bits(v[1] * np.float32(1e-7))   # below the 1e-4 floor
        x[2, :128] = 0
        x[3, :128] = synth.f32_to_bf16_bits(np.full(128, -448.0, np.float32))   # exact fit, s = 1
    op = _mxg().bw_quantize_1x128_pow2(bf16_to_dev(x))
    torch.cuda.synchronize()
    codes, s = oracle.quantize_bw_1x128(x, pow2=True)
    assert np.array_equal(op.data.cpu().numpy(), codes)
    assert np.array_equal(op.scale.cpu().numpy(), _ue8m0(s))


def test_bw_128x128_pow2_and_dgrad_copy_bit_exact():
    rng = np.random.default_rng(4)
    G, N, K = 2, 256, 384
    w = synth.normal_bf16(rng, (G * N, K), std=3.0, outlier_frac=0.02)
    op, opT = _mxg().bw_quantize_128x128_pow2(bf16_to_dev(w))
    torch.cuda.synchronize()
    codes, s = oracle.quantize_bw_128x128(w.reshape(G, N, K), pow2=True)
    assert np.array_equal(op.data.cpu().numpy(), codes.reshape(G * N, K))
    assert np.array_equal(op.scale.cpu().numpy(), _ue8m0(s.reshape(G * N // 128, K // 128), 128, 4))
    ct, st = transpose_bw_128x128(codes, s)
    assert np.array_equal(opT.data.cpu().numpy(), np.concatenate(list(ct), axis=1))
    assert np.array_equal(opT.scale.cpu().numpy(), _ue8m0(np.concatenate(list(st), axis=1), 128, 4))


@pytest.mark.parametrize("splits,cols", [([200, 0, 1, 128, 55], 128), ([0, 0, 300], 256)])
def test_bw_colwise_padded_pow2_bit_exact(splits, cols):
    rng = np.random.default_rng(len(splits) + cols + 1)
    splits = np.array(splits, dtype=np.int32)
    x = synth.normal_bf16(rng, (int(splits.sum()), cols), std=3.0, outlier_frac=0.02)
    op, poff = _mxg().bw_quantize_colwise_padded_pow2(bf16_to_dev(x), i32_to_dev(splits), check=True)
    codes, s, p = oracle.quantize_bw_colwise_padded(x, splits, pow2=True)
    spad = int(p[-1])
    assert np.array_equal(poff.cpu().numpy(), p)
    assert np.array_equal(op.data.cpu().numpy()[:, :spad], codes)
    assert np.array_equal(op.scale.cpu().numpy()[:, : spad // 32], _ue8m0(s))


def _mx_dev(codes, ue8m0, cols):
    return _mxg().MXOperand(_u8_dev(codes), _u8_dev(ue8m0), "e4m3", cols)


def test_pow2_blockwise_step_on_the_mx_gemms():
    """The pow2 blockwise recipe runs on the MXFP8 GEMMs: fwd, dgrad and wgrad
    against the oracle's per-expert contraction of the dequantized blockwise
    operands."""
    mxg = _mxg()
    splits = np.array([200, 0, 77, 300, 129], dtype=np.int32)
    G, S, N, K = len(splits), int(splits.sum()), 256, 384
    rng = np.random.default_rng(31)
    x = synth.normal_bf16(rng, (S, K), outlier_frac=0.01)
    dy = synth.normal_bf16(rng, (S, N), outlier_frac=0.01)
    w = synth.normal_bf16(rng, (G * N, K), outlier_frac=0.01)
    d_splits = i32_to_dev(splits)
    # operands quantized by the oracle
    xc, xs = oracle.quantize_bw_1x128(x, pow2=True)
    dyc, dys = oracle.quantize_bw_1x128(dy, pow2=True)
    wc, ws = oracle.quantize_bw_128x128(w.reshape(G, N, K), pow2=True)
    ct, st = transpose_bw_128x128(wc, ws)
    Xd, dYd = oracle.dequantize_bw_1x128(xc, xs), oracle.dequantize_bw_1x128(dyc, dys)
    Wd = oracle.dequantize_bw_128x128(wc, ws).reshape(G * N, K)
    Wtd = np.concatenate(list(oracle.dequantize_bw_128x128(ct, st)), axis=1)
    A = _mx_dev(xc, _ue8m0(xs), K)
    Wm = _mx_dev(wc.reshape(G * N, K), _ue8m0(ws.reshape(G * N // 128, K // 128), 128, 4), K)
    dYm = _mx_dev(dyc, _ue8m0(dys), N)
    Wt = _mx_dev(np.concatenate(list(ct), axis=1), _ue8m0(np.concatenate(list(st), axis=1), 128, 4), G * N)
    Y = mxg.grouped_gemm_fwd(A, Wm, d_splits, N, check=True)
    oracle.assert_gemm_close(Y.float().cpu().numpy(), oracle.grouped_fwd(Xd, Wd, splits, N), "pow2 fwd")
    dX = mxg.grouped_gemm_dgrad(dYm, Wt, d_splits, check=True)
    oracle.assert_gemm_close(dX.float().cpu().numpy(), oracle.grouped_dgrad(dYd, Wtd, splits), "pow2 dgrad")
    # wgrad on the column-wise operands (segments padded to 128)
    cap = synth.padded_rows_capacity(S, G, 128)
    dytc, dyts, poff = oracle.quantize_bw_colwise_padded(dy, splits, pow2=True)
    xtc, xts, _ = oracle.quantize_bw_colwise_padded(x, splits, pow2=True)
    spad = int(poff[-1])

    def full(codes, s, C):
        fc = np.zeros((C, cap), dtype=np.uint8)
        fc[:, :spad] = codes
        fs = np.full((C, cap // 32), 127, dtype=np.uint8)
        fs[:, : spad // 32] = _ue8m0(s)
        return _mx_dev(fc, fs, cap)

    out = torch.zeros((G, N, K), dtype=torch.float32, device="cuda:0")
    mxg.grouped_gemm_wgrad(full(dytc, dyts, N), full(xtc, xts, K), d_splits, S, 128, out=out, check=True)
    ref = oracle.grouped_wgrad(oracle.dequantize_bw_1x128(dytc, dyts), oracle.dequantize_bw_1x128(xtc, xts), poff)
    oracle.assert_gemm_close(out.cpu().numpy(), ref, "pow2 wgrad")


# ------------------------------------------------------------------ dual blockwise quantizer

@pytest.mark.parametrize("pow2", [False, True])
@pytest.mark.parametrize("splits,cols", [([200, 0, 1, 128, 55], 128), ([0, 0, 300], 256),
                                         ([1000, 7, 0, 450], 512)])
def test_bw_dual_matches_both_oracles(pow2, splits, cols):
    """One read of x: the 1x128 row-wise and the padded column-wise operands,
    each bit-exact against its own oracle (codes and scales), with a block
    below the amax floor, an all-zero block and an exact-fit block."""
    rng = np.random.default_rng(len(splits) + cols + pow2)
    splits = np.array(splits, dtype=np.int32)
    S = int(splits.sum())
    x = synth.normal_bf16(rng, (S, cols), std=3.0, outlier_frac=0.02)
    if S > 4:
        v = synth.bf16_bits_to_f32(x)
        x[1] = synth.f32_to_bf16_bits(v[1] * np.float32(1e-7))
        x[2, :128] = 0
        x[3, :128] = synth.f32_to_bf16_bits(np.full(128, -448.0, np.float32))
    row, col, poff = _mxg().bw_quantize_dual_padded(bf16_to_dev(x), i32_to_dev(splits), pow2=pow2, check=True)
    rc, rs = oracle.quantize_bw_1x128(x, pow2=pow2)
    assert np.array_equal(row.data.cpu().numpy(), rc)
    assert np.array_equal(row.scale.cpu().numpy(), _ue8m0(rs) if pow2 else rs.T)
    cc, cs, p = oracle.quantize_bw_colwise_padded(x, splits, pow2=pow2)
    spad = int(p[-1])
    assert np.array_equal(poff.cpu().numpy(), p)
    assert np.array_equal(col.data.cpu().numpy()[:, :spad], cc)
    if pow2:
        assert np.array_equal(col.scale.cpu().numpy()[:, : spad // 32], _ue8m0(cs))
    else:
        assert np.array_equal(col.scale.cpu().numpy()[: spad // 128], cs.T)


def test_bw_dual_rejects_bad_splits_and_writes_nothing():
    mxg = _mxg()
    x = bf16_to_dev(synth.normal_bf16(np.random.default_rng(2), (14, 128)))
    st = torch.zeros(1, dtype=torch.int32, device="cuda:0")
    q = torch.full((14, 128), 0xAB, dtype=torch.uint8, device="cuda:0")
    s = torch.full((14, 4), 0xCD, dtype=torch.uint8, device="cuda:0")
    qT = torch.full((128, 384), 0xAB, dtype=torch.uint8, device="cuda:0")
    sT = torch.full((128, 12), 0xCD, dtype=torch.uint8, device="cuda:0")
    rc = mxg._lib.load().bw_quantize_dual_padded_pow2(
        mxg._ptr(x), 14, 128, 128, mxg._ptr(i32_to_dev([10, -1, 5])), 3, mxg._ptr(q), 128, mxg._ptr(s), 4,
        mxg._ptr(qT), 384, mxg._ptr(sT), 12, 384, None, mxg._ptr(st), mxg._stream(x.device))
    assert rc == 0
    assert int(st.item()) == 4
    assert (q == 0xAB).all() and (s == 0xCD).all() and (qT == 0xAB).all() and (sT == 0xCD).all()


def test_bw_bounded_wait_gives_up_cleanly(cta_group):
    """The blockwise GEMM with an absurdly short wait limit either finishes or
    reports a timeout (its epilogue's bulk stores drained); the next normal
    call is correct."""
    mxg = _mxg()
    lib = mxg._lib.load()
    old = lib.mxg_get_wait_timeout_ns()
    try:
        lib.mxg_set_wait_timeout_ns(1)
        try:
            test_bw_fwd_parity([0, 130, 1, 300], 256, 384, cta_group)
        except mxg.MXGError as e:
            assert e.code == 8
    finally:
        lib.mxg_set_wait_timeout_ns(old)
    test_bw_fwd_parity([0, 130, 1, 300], 256, 384, cta_group)
