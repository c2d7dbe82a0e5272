"""Grouped MX GEMMs on the GPU vs the oracle.

Operands are quantized by the ORACLE and uploaded, so the GEMM is checked on
its own; the reference is the oracle's per-expert float64 contraction of the
same dequantized operands.  Bound per element (products exact, fp32
accumulation, BF16 output rounding):
    |gpu - ref| <= 2^-8 * |ref| + 1e-4 * rms(ref)."""

import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu

from gpu_util import bf16_to_dev, i32_to_dev, oracle_operand_colwise, oracle_operand_rowwise  # noqa: E402

KINDS = {"mxfp4": ("e2m1", "e2m1"), "mxfp8": ("e4m3", "e4m3"), "a8w4": ("e4m3", "e2m1")}


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()


def _mxg():
    import fp8_bf16_mxfp4_gb300 as mxg
    return mxg


@pytest.fixture(params=[2, 1], ids=["pair", "onesm"], autouse=True)
def cta_group(request):
    """Every case runs on the CTA-pair kernel (256 x 256 tiles over two SMs,
    the default) and on the one-SM kernel (128 x 256 tiles)."""
    prev = _mxg().set_gemm_cta_group(request.param)
    yield request.param
    _mxg().set_gemm_cta_group(prev)


def _run_fwd(kind, splits, N, K, out_dtype=torch.bfloat16, seed=0, std=1.0, outliers=0.01):
    ea, eb = KINDS[kind]
    splits = np.asarray(splits, dtype=np.int32)
    G, S = len(splits), int(splits.sum())
    rng = np.random.default_rng(seed)
    x = synth.normal_bf16(rng, (S, K), std=std, outlier_frac=outliers)
    w = synth.normal_bf16(rng, (G * N, K), std=std, outlier_frac=outliers)
    A, Ad = oracle_operand_rowwise(x, ea)
    W, Wd = oracle_operand_rowwise(w, eb)
    st = torch.zeros(1, dtype=torch.int32, device="cuda:0")
    Y = _mxg().grouped_gemm_fwd(A, W, i32_to_dev(splits), N, out_dtype=out_dtype, status=st, check=True)
    ref = oracle.grouped_fwd(Ad, Wd, splits, N)
    return Y.float().cpu().numpy(), ref


FWD_CASES = [
    # splits, N, K
    (None, 256, 512),                           # the tiny configuration (seeded splits)
    ([0, 1, 127, 129, 300, 0], 288, 256),       # ragged experts, N tail (256 + 32)
    ([64, 0, 200], 32, 128),                    # N smaller than a tile, K = one stage (fp8)
    ([5], 512, 1024),                           # G = 1, tiny M
    ([130, 70], 256, 4096),                     # long K
]


@pytest.mark.parametrize("kind", ["mxfp4", "mxfp8", "a8w4"])
@pytest.mark.parametrize("case", range(len(FWD_CASES)))
def test_fwd_parity(kind, case):
    splits, N, K = FWD_CASES[case]
    if splits is None:
        splits = synth.WORKLOADS["tiny_mxfp4_fwd"].splits()
    got, ref = _run_fwd(kind, splits, N, K, seed=case)
    oracle.assert_gemm_close(got, ref, f"fwd {kind} case {case}")


@pytest.mark.parametrize("kind", ["mxfp4", "mxfp8"])
@pytest.mark.parametrize("K", [96, 160, 32])
def test_fwd_k_tails(kind, K):
    """K not a multiple of the stage depth: partial stages, and for MXFP4 a
    half-filled 64-element MMA step (K % 64 == 32)."""
    got, ref = _run_fwd(kind, [3, 200, 0, 61], 256, K, seed=K)
    oracle.assert_gemm_close(got, ref, f"fwd {kind} K={K}")


def test_fwd_fp32_output():
    got, ref = _run_fwd("mxfp4", [100, 29, 3], 256, 384, out_dtype=torch.float32, seed=3)
    oracle.assert_gemm_close(got, ref, "fwd fp32 out")


def test_fwd_empty_batch():
    got, ref = _run_fwd("mxfp4", [0, 0, 0], 256, 256)
    assert got.shape == (0, 256)


@pytest.mark.parametrize("kind", ["mxfp4", "mxfp8"])
@pytest.mark.parametrize("splits,N,K", [([0, 50, 131, 7], 96, 288), ([256, 256], 256, 512),
                                        ([1, 0, 300], 160, 64)])
def test_dgrad_parity(kind, splits, N, K):
    """dX = dY @ W_g with W^T quantized along N per expert (G segments of N)."""
    e = KINDS[kind][0]
    splits = np.asarray(splits, dtype=np.int32)
    G, S = len(splits), int(splits.sum())
    rng = np.random.default_rng(N + K)
    dy = synth.normal_bf16(rng, (S, N), outlier_frac=0.01)
    w = synth.normal_bf16(rng, (G * N, K), outlier_frac=0.01)
    dY, dYd = oracle_operand_rowwise(dy, e)
    Wt, Wtd, _ = oracle_operand_colwise(w, [N] * G, 32, e)
    st = torch.zeros(1, dtype=torch.int32, device="cuda:0")
    dX = _mxg().grouped_gemm_dgrad(dY, Wt, i32_to_dev(splits), status=st, check=True)
    ref = oracle.grouped_dgrad(dYd, Wtd, splits)
    oracle.assert_gemm_close(dX.float().cpu().numpy(), ref, f"dgrad {kind}")


@pytest.mark.parametrize("kind", ["mxfp4", "mxfp8"])
@pytest.mark.parametrize("pad", [32, 128])
@pytest.mark.parametrize("accumulate", [False, True])
def test_wgrad_parity(kind, pad, accumulate):
    """Variable-K wgrad over segment-padded operands, with junk in the
    capacity slack, empty experts and odd 32-multiples of padded length."""
    e = KINDS[kind][0]
    splits = np.array([37, 0, 5, 300, 64, 0, 129], dtype=np.int32)
    G, S = len(splits), int(splits.sum())
    N, K = 160, 288
    rng = np.random.default_rng(pad + accumulate)
    dy = synth.normal_bf16(rng, (S, N), outlier_frac=0.01)
    x = synth.normal_bf16(rng, (S, K), outlier_frac=0.01)
    cap = synth.padded_rows_capacity(S, G, pad)
    dYt, dYtd, poff = oracle_operand_colwise(dy, splits, pad, e, capacity=cap)
    Xt, Xtd, _ = oracle_operand_colwise(x, splits, pad, e, capacity=cap)
    init = rng.standard_normal((G, N, K)).astype(np.float32) * np.float32(1e-3)
    out = torch.from_numpy(init.copy()).to("cuda:0")
    st = torch.zeros(1, dtype=torch.int32, device="cuda:0")
    _mxg().grouped_gemm_wgrad(dYt, Xt, i32_to_dev(splits), S, pad, out=out, accumulate=accumulate,
                              status=st, check=True)
    ref = oracle.grouped_wgrad(dYtd, Xtd, poff, out_init=init if accumulate else None)
    got = out.cpu().numpy()
    oracle.assert_gemm_close(got, ref, f"wgrad {kind} pad={pad} acc={accumulate}")
    if not accumulate:
        assert (got[1] == 0).all() and (got[5] == 0).all()   # empty experts store zeros
    else:
        assert np.array_equal(got[1], init[1]) and np.array_equal(got[5], init[5])


@pytest.mark.parametrize("kind", ["mxfp4", "mxfp8"])
def test_fp32_forward_many_tiles_per_cta(kind):
    """FP32 output over more tiles than SMs (49 m-tiles x 4 n-tiles, the last
    one ragged), so that every CTA reuses its accumulator and scale slots
    across tiles of different experts."""
    splits = [1500, 0, 1, 2047, 129, 2300]
    got, ref = _run_fwd(kind, splits, 896, 320, out_dtype=torch.float32, seed=41)
    oracle.assert_gemm_close(got, ref, f"fwd fp32 {kind} N=896")


@pytest.mark.parametrize("kind", ["mxfp4", "mxfp8"])
@pytest.mark.parametrize("N", [416, 480])
def test_fp32_output_column_tail_past_half_tile(kind, N):
    """FP32 output whose last n-tile holds 160 or 224 columns: the second half
    of that tile's accumulator is only partly used (5 or 7 of 8 column
    chunks), on top of full tiles that use all of it."""
    got, ref = _run_fwd(kind, [300, 5, 0, 129], N, 256, out_dtype=torch.float32, seed=N)
    oracle.assert_gemm_close(got, ref, f"fwd fp32 {kind} N={N}")


@pytest.mark.parametrize("kind", ["mxfp4", "mxfp8"])
def test_wgrad_accumulate_column_tail_past_half_tile(kind):
    """wgrad += with K = 448 output columns (a full n-tile and one of 192
    columns) over experts of different contraction lengths."""
    e = KINDS[kind][0]
    splits = np.array([70, 0, 200, 33], dtype=np.int32)
    G, S = len(splits), int(splits.sum())
    N, K, pad = 192, 448, 32
    rng = np.random.default_rng(448)
    dy = synth.normal_bf16(rng, (S, N), outlier_frac=0.01)
    x = synth.normal_bf16(rng, (S, K), outlier_frac=0.01)
    cap = synth.padded_rows_capacity(S, G, pad)
    dYt, dYtd, poff = oracle_operand_colwise(dy, splits, pad, e, capacity=cap)
    Xt, Xtd, _ = oracle_operand_colwise(x, splits, pad, e, capacity=cap)
    init = rng.standard_normal((G, N, K)).astype(np.float32) * np.float32(1e-3)
    out = torch.from_numpy(init.copy()).to("cuda:0")
    _mxg().grouped_gemm_wgrad(dYt, Xt, i32_to_dev(splits), S, pad, out=out, accumulate=True, check=True)
    ref = oracle.grouped_wgrad(dYtd, Xtd, poff, out_init=init)
    got = out.cpu().numpy()
    oracle.assert_gemm_close(got, ref, f"wgrad {kind} K={K} acc")
    assert np.array_equal(got[1], init[1])


@pytest.mark.parametrize("kind", ["mxfp4", "mxfp8"])
@pytest.mark.parametrize("accumulate", [False, True])
def test_wgrad_many_tiles_per_cta(kind, accumulate):
    """Variable-K wgrad with more tiles than SMs (8 experts x 4 x 5 tiles, the
    last n-tile ragged): the accumulator and every scale slot are reused
    across experts of different contraction lengths."""
    e = KINDS[kind][0]
    splits = np.array([300, 0, 77, 513, 200, 31, 1, 640], dtype=np.int32)
    G, S = len(splits), int(splits.sum())
    N, K, pad = 512, 1120, 32
    rng = np.random.default_rng(90 + accumulate)
    dy = synth.normal_bf16(rng, (S, N), outlier_frac=0.01)
    x = synth.normal_bf16(rng, (S, K), outlier_frac=0.01)
    cap = synth.padded_rows_capacity(S, G, pad)
    dYt, dYtd, poff = oracle_operand_colwise(dy, splits, pad, e, capacity=cap)
    Xt, Xtd, _ = oracle_operand_colwise(x, splits, pad, e, capacity=cap)
    init = rng.standard_normal((G, N, K)).astype(np.float32) * np.float32(1e-3)
    out = torch.from_numpy(init.copy()).to("cuda:0")
    _mxg().grouped_gemm_wgrad(dYt, Xt, i32_to_dev(splits), S, pad, out=out, accumulate=accumulate, check=True)
    ref = oracle.grouped_wgrad(dYtd, Xtd, poff, out_init=init if accumulate else None)
    got = out.cpu().numpy()
    oracle.assert_gemm_close(got, ref, f"wgrad {kind} many tiles acc={accumulate}")
    if accumulate:
        assert np.array_equal(got[1], init[1])


@pytest.mark.parametrize("kind", ["mxfp4", "mxfp8", "a8w4"])
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_dense_gemm(kind, out_dtype):
    """mx_gemm_dense (no experts, no m_splits) against the oracle, and equal bit
    for bit to the one-expert grouped forward; also with packed scales."""
    mxg = _mxg()
    ea, eb = KINDS[kind]
    M, N, K = 333, 320, 256
    rng = np.random.default_rng(7)
    x = synth.normal_bf16(rng, (M, K), outlier_frac=0.01)
    w = synth.normal_bf16(rng, (N, K), outlier_frac=0.01)
    A, Ad = oracle_operand_rowwise(x, ea)
    B, Bd = oracle_operand_rowwise(w, eb)
    C = mxg.mx_gemm_dense(A, B, out_dtype=out_dtype, check=True)
    oracle.assert_gemm_close(C.float().cpu().numpy(), Ad @ Bd.T, f"dense {kind}")
    Cg = mxg.grouped_gemm_fwd(A, B, i32_to_dev([M]), N, out_dtype=out_dtype, check=True)
    assert torch.equal(C, Cg)
    Ap = mxg.mx_quantize_rowwise_packed(bf16_to_dev(x), ea, groups=1)
    Bp = mxg.mx_quantize_rowwise_packed(bf16_to_dev(w), eb, groups=1)
    assert torch.equal(mxg.mx_gemm_dense(Ap, Bp, out_dtype=out_dtype, check=True), C)


def test_dense_gemm_empty_rows():
    mxg = _mxg()
    B, _ = oracle_operand_rowwise(synth.normal_bf16(np.random.default_rng(1), (64, 128)), "e2m1")
    A = mxg.MXOperand(torch.empty((0, 64), dtype=torch.uint8, device="cuda:0"),
                      torch.empty((0, 4), dtype=torch.uint8, device="cuda:0"), "e2m1", 128)
    C = mxg.mx_gemm_dense(A, B, check=True)
    assert C.shape == (0, 64)


def test_wgrad_bf16_output():
    splits = np.array([70, 33], dtype=np.int32)
    S, N, K = 103, 256, 256
    rng = np.random.default_rng(77)
    dy = synth.normal_bf16(rng, (S, N))
    x = synth.normal_bf16(rng, (S, K))
    dYt, dYtd, poff = oracle_operand_colwise(dy, splits, 32, "e2m1")
    Xt, Xtd, _ = oracle_operand_colwise(x, splits, 32, "e2m1")
    out = _mxg().grouped_gemm_wgrad(dYt, Xt, i32_to_dev(splits), S, 32, out_dtype=torch.bfloat16, check=True)
    ref = oracle.grouped_wgrad(dYtd, Xtd, poff)
    oracle.assert_gemm_close(out.float().cpu().numpy(), ref, "wgrad bf16")


@pytest.mark.parametrize("bad", [[100, -1, 29], [100, 20, 20]])
def test_gemm_rejects_bad_splits_on_device(bad):
    mxg = _mxg()
    rng = np.random.default_rng(4)
    x = synth.normal_bf16(rng, (128, 256))
    w = synth.normal_bf16(rng, (3 * 256, 256))
    A, _ = oracle_operand_rowwise(x, "e2m1")
    W, _ = oracle_operand_rowwise(w, "e2m1")
    out = torch.full((128, 256), 7.0, dtype=torch.bfloat16, device="cuda:0")
    st = torch.zeros(1, dtype=torch.int32, device="cuda:0")
    mxg.grouped_gemm_fwd(A, W, i32_to_dev(bad), 256, out=out, status=st)
    with pytest.raises(mxg.MXGError) as ei:
        mxg.check_status(st)
    assert ei.value.code == 4
    assert (out == 7.0).all()


def test_bounded_wait_reports_timeout_and_context_survives():
    mxg = _mxg()
    lib = mxg._lib.load()
    st = torch.zeros(1, dtype=torch.int32, device="cuda:0")
    assert lib.mxg_diag_bounded_wait(mxg._ptr(st), 50_000_000, mxg._stream(st.device)) == 0
    with pytest.raises(mxg.MXGError) as ei:
        mxg.check_status(st)
    assert ei.value.code == 8
    # a GEMM with an absurdly short wait limit either finishes or gives up
    # cleanly; either way the next normal call is correct
    old = lib.mxg_get_wait_timeout_ns()
    try:
        lib.mxg_set_wait_timeout_ns(1)
        try:
            _run_fwd("mxfp4", [300, 200], 512, 2048)
        except mxg.MXGError as e:
            assert e.code == 8
    finally:
        lib.mxg_set_wait_timeout_ns(old)
    got, ref = _run_fwd("mxfp4", [300, 200], 512, 2048)
    oracle.assert_gemm_close(got, ref, "after timeout")


@pytest.mark.parametrize("accumulate", [False, True])
def test_wgrad_empty_batch(accumulate):
    """No tokens at all: zero capacity operands; the output is zeroed (or left
    as it was when accumulating) after the splits are validated."""
    mxg = _mxg()
    G, N, K = 3, 64, 96
    empty = lambda rows: mxg.MXOperand(torch.empty((rows, 0), dtype=torch.uint8, device="cuda:0"),
                                       torch.empty((rows, 0), dtype=torch.uint8, device="cuda:0"), "e2m1", 0)
    init = torch.full((G, N, K), 3.0, dtype=torch.float32, device="cuda:0")
    mxg.grouped_gemm_wgrad(empty(N), empty(K), i32_to_dev([0, 0, 0]), 0, 32, out=init,
                           accumulate=accumulate, check=True)
    assert (init == (3.0 if accumulate else 0.0)).all()


@pytest.mark.parametrize("kind", ["mxfp4", "a8w4"])
def test_fwd_maximum_expert_count(kind):
    """G = 512 (the most the library accepts): almost every expert empty, a
    few ragged ones scattered through the table (prefix search and tile
    enumeration over the full expert table)."""
    splits = np.zeros(512, dtype=np.int32)
    splits[[0, 7, 255, 256, 400, 511]] = [1, 129, 64, 3, 200, 31]
    got, ref = _run_fwd(kind, splits, 64, 256, seed=9)
    oracle.assert_gemm_close(got, ref, f"fwd G=512 {kind}")


@pytest.mark.parametrize("kind", ["mxfp4", "mxfp8"])
def test_fwd_wide_dynamic_range(kind):
    """Rows and weight rows scaled by powers of two from 2^-40 to 2^40, so the
    block scales span ~160 binades (products stay inside fp32)."""
    ea, eb = KINDS[kind]
    rng = np.random.default_rng(12)
    splits = np.array([70, 0, 130], dtype=np.int32)
    G, S, N, K = 3, 200, 96, 256
    xs = synth.bf16_bits_to_f32(synth.normal_bf16(rng, (S, K)))
    ws = synth.bf16_bits_to_f32(synth.normal_bf16(rng, (G * N, K)))
    xs *= np.float32(2.0) ** rng.integers(-40, 41, size=(S, 1)).astype(np.float32)
    ws *= np.float32(2.0) ** rng.integers(-40, 41, size=(G * N, 1)).astype(np.float32)
    x, w = synth.f32_to_bf16_bits(xs), synth.f32_to_bf16_bits(ws)
    A, Ad = oracle_operand_rowwise(x, ea)
    W, Wd = oracle_operand_rowwise(w, eb)
    Y = _mxg().grouped_gemm_fwd(A, W, i32_to_dev(splits), N, out_dtype=torch.float32, check=True)
    ref = oracle.grouped_fwd(Ad, Wd, splits, N)
    # per output row the magnitude is set by its own scales: check row by row
    got = Y.cpu().numpy()
    for r in range(S):
        if np.abs(ref[r]).max() > 0:
            oracle.assert_gemm_close(got[r:r + 1], ref[r:r + 1], f"wide range {kind} row {r}")


@pytest.mark.parametrize("kind", ["mxfp4", "a8w4"])
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_fwd_into_a_strided_output_leaves_the_padding_alone(kind, out_dtype):
    """out is a view [S, N] of a wider buffer (ld_out = N + 64): the tiled
    stores clip at column N, so the 64 padding columns keep their sentinel;
    ragged experts exercise the partial-row boxes."""
    mxg = _mxg()
    ea, eb = KINDS[kind]
    splits = np.array([0, 1, 127, 129, 300, 17], dtype=np.int32)
    G, S, N, K = len(splits), int(splits.sum()), 288, 256
    rng = np.random.default_rng(33)
    x = synth.normal_bf16(rng, (S, K), outlier_frac=0.01)
    w = synth.normal_bf16(rng, (G * N, K), outlier_frac=0.01)
    A, Ad = oracle_operand_rowwise(x, ea)
    W, Wd = oracle_operand_rowwise(w, eb)
    big = torch.full((S, N + 64), 7.0, dtype=out_dtype, device="cuda:0")
    out = big[:, :N]
    mxg.grouped_gemm_fwd(A, W, i32_to_dev(splits), N, out=out, check=True)
    oracle.assert_gemm_close(out.float().cpu().numpy(), oracle.grouped_fwd(Ad, Wd, splits, N), f"fwd {kind} strided")
    assert (big[:, N:] == 7.0).all()


def test_dgrad_into_a_strided_output_leaves_the_padding_alone():
    mxg = _mxg()
    splits = np.array([0, 50, 131, 7], dtype=np.int32)
    G, S, N, K = len(splits), int(splits.sum()), 96, 288
    rng = np.random.default_rng(34)
    dy = synth.normal_bf16(rng, (S, N), outlier_frac=0.01)
    w = synth.normal_bf16(rng, (G * N, K), outlier_frac=0.01)
    dY, dYd = oracle_operand_rowwise(dy, "e2m1")
    from gpu_util import oracle_operand_colwise
    Wt, Wtd, _ = oracle_operand_colwise(w, [N] * G, 32, "e2m1")
    big = torch.full((S, K + 32), -3.0, dtype=torch.bfloat16, device="cuda:0")
    out = big[:, :K]
    mxg.grouped_gemm_dgrad(dY, Wt, i32_to_dev(splits), out=out, check=True)
    oracle.assert_gemm_close(out.float().cpu().numpy(), oracle.grouped_dgrad(dYd, Wtd, splits), "dgrad strided")
    assert (big[:, K:] == -3.0).all()
