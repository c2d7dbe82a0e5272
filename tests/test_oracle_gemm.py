"""Pins for the grouped GEMM oracle (CPU only).

* exact rational brute force (``fractions.Fraction`` triple loops over
  scalar-decoded codes) on tiny grouped problems for all three passes;
* the adjoint identity <dY, X W^T> = <dY^T X, W> = <X, dY W> through the full
  quantize -> grouped-pass chain on losslessly quantizable matrices, which
  fails if any pass contracts the wrong dimension or transposes an operand;
* structural invariants: per-expert concatenation, expert permutation,
  empty experts, wgrad padding invariance, accumulation, split validation;
* the comparison bound itself."""

from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle import scalar
import synth


def _rand_operand(rng, rows, cols, elem, s_lo=120, s_hi=130):
    codes = rng.integers(0, 16 if elem == "e2m1" else 0x7F, size=(rows, cols)).astype(np.uint8)
    if elem == "e4m3":
        codes |= (rng.integers(0, 2, size=codes.shape) << 7).astype(np.uint8)
    scale = rng.integers(s_lo, s_hi, size=(rows, cols // 32)).astype(np.uint8)
    return codes, scale


def _exact(codes, scale, elem):
    R, C = codes.shape
    return [[scalar.decode_code(int(codes[r, c]), elem) * Fraction(2) ** (int(scale[r, c // 32]) - 127)
             for c in range(C)] for r in range(R)]


@pytest.mark.parametrize("ea,eb", [("e2m1", "e2m1"), ("e4m3", "e2m1"), ("e4m3", "e4m3")])
def test_fwd_dgrad_exact_brute_force(ea, eb):
    rng = np.random.default_rng(31)
    splits = np.array([3, 0, 5, 1], dtype=np.int32)
    G, S, N, K = 4, 9, 32, 64
    Ac, As = _rand_operand(rng, S, K, ea)
    Wc, Ws = _rand_operand(rng, G * N, K, eb)
    A = oracle.dequantize_mx(Ac, As, ea)
    W = oracle.dequantize_mx(Wc, Ws, eb)
    Y = oracle.grouped_fwd(A, W, splits, N)
    Ax, Wx = _exact(Ac, As, ea), _exact(Wc, Ws, eb)
    off = np.concatenate([[0], np.cumsum(splits)])
    for g in range(G):
        for i in range(off[g], off[g + 1]):
            for n in range(N):
                want = sum(Ax[i][k] * Wx[g * N + n][k] for k in range(K))
                assert Fraction(Y[i, n]) == want
    # dgrad: dY [S, N'] against Wt [K', G*N'] contracting N'
    Np, Kp = 32, 32
    dYc, dYs = _rand_operand(rng, S, Np, ea)
    Wtc, Wts = _rand_operand(rng, Kp, G * Np, eb)
    dX = oracle.grouped_dgrad(oracle.dequantize_mx(dYc, dYs, ea), oracle.dequantize_mx(Wtc, Wts, eb), splits)
    dYx, Wtx = _exact(dYc, dYs, ea), _exact(Wtc, Wts, eb)
    for g in range(G):
        for i in range(off[g], off[g + 1]):
            for k in range(Kp):
                want = sum(dYx[i][n] * Wtx[k][g * Np + n] for n in range(Np))
                assert Fraction(dX[i, k]) == want


def test_wgrad_exact_brute_force():
    rng = np.random.default_rng(32)
    poff = np.array([0, 32, 32, 96], dtype=np.int64)     # experts: 32, 0, 64 padded tokens
    N, K = 8, 6
    dYc, dYs = _rand_operand(rng, N, 96, "e2m1")
    Xc, Xs = _rand_operand(rng, K, 96, "e2m1")
    init = rng.standard_normal((3, N, K))
    dW = oracle.grouped_wgrad(oracle.dequantize_mx(dYc, dYs, "e2m1"),
                              oracle.dequantize_mx(Xc, Xs, "e2m1"), poff, out_init=init)
    dYx, Xx = _exact(dYc, dYs, "e2m1"), _exact(Xc, Xs, "e2m1")
    for g in range(3):
        for n in range(N):
            for k in range(K):
                want = sum(dYx[n][j] * Xx[k][j] for j in range(poff[g], poff[g + 1]))
                assert abs(float(Fraction(dW[g, n, k]) - Fraction(init[g, n, k]) - want)) <= 1e-12 * (1 + abs(init[g, n, k]))
    assert np.array_equal(dW[1], init[1])                 # empty expert leaves the init


def _lossless_matrix(rng, rows, cols, elem):
    """Values on the element grid with unit scale, and a full-range element in
    every 32-block along both axes, so quantizing along either axis is exact.
    Blocks cut short at an expert's end may miss the anchor and get a smaller
    scale; E4M3 values with mantissa 7 would then rescale past 448, so they
    are left out (E2M1's grid is closed under that rescaling)."""
    if elem == "e2m1":
        grid = oracle.E2M1_MAGNITUDES
    else:
        codes = np.arange(0x78)
        grid = oracle.e4m3_magnitudes()[codes[(codes & 7) != 7]]
    v = rng.choice(grid, size=(rows, cols)) * rng.choice([-1.0, 1.0], size=(rows, cols))
    top = 6.0 if elem == "e2m1" else 448.0
    i, j = np.indices((rows, cols))
    v[(i + j) % 32 == 0] = top
    return synth.f32_to_bf16_bits(v.astype(np.float32)), v


@pytest.mark.parametrize("elem", ["e2m1", "e4m3"])
def test_adjoint_identity_through_quantizers(elem):
    rng = np.random.default_rng(33)
    splits = np.array([40, 0, 96, 7, 25], dtype=np.int32)
    G, S, N, K = len(splits), int(splits.sum()), 64, 96
    Xb, Xv = _lossless_matrix(rng, S, K, elem)
    dYb, dYv = _lossless_matrix(rng, S, N, elem)
    Wb, Wv = _lossless_matrix(rng, G * N, K, elem)

    def deq_row(b):
        d, s = oracle.quantize_mx_rowwise(b, elem)
        return oracle.dequantize_mx(oracle.unpack_e2m1(d) if elem == "e2m1" else d, s, elem)

    X, dY, W = deq_row(Xb), deq_row(dYb), deq_row(Wb)
    assert np.array_equal(X, Xv) and np.array_equal(W, Wv) and np.array_equal(dY, dYv)
    # dgrad operand: W^T quantized along N within each expert (G segments of N)
    wt_d, wt_s, _ = oracle.quantize_mx_colwise_segment_padded(Wb, [N] * G, 32, elem)
    Wt = oracle.dequantize_mx(oracle.unpack_e2m1(wt_d) if elem == "e2m1" else wt_d, wt_s, elem)
    assert np.array_equal(Wt, Wv.T)
    # wgrad operands: colwise, segment padded
    outs = []
    for pad in (32, 128):
        dyt_d, dyt_s, poff = oracle.quantize_mx_colwise_segment_padded(dYb, splits, pad, elem)
        xt_d, xt_s, _ = oracle.quantize_mx_colwise_segment_padded(Xb, splits, pad, elem)
        unp = (lambda d: oracle.unpack_e2m1(d)) if elem == "e2m1" else (lambda d: d)
        dYt = oracle.dequantize_mx(unp(dyt_d), dyt_s, elem)
        Xt = oracle.dequantize_mx(unp(xt_d), xt_s, elem)
        for g in range(G):
            j0 = int(poff[g])
            rows = slice(int(np.sum(splits[:g])), int(np.sum(splits[:g + 1])))
            assert np.array_equal(Xt[:, j0: j0 + splits[g]], Xv[rows].T)
            assert np.array_equal(dYt[:, j0: j0 + splits[g]], dYv[rows].T)
        outs.append(oracle.grouped_wgrad(dYt, Xt, poff))
    assert np.array_equal(outs[0], outs[1])          # pad 32 and pad 128 agree
    Y = oracle.grouped_fwd(X, W, splits, N)
    dX = oracle.grouped_dgrad(dY, Wt, splits)
    dW = outs[0]
    lhs = float(np.sum(dY * Y))
    mid = float(np.sum(dW * W.reshape(G, N, K)))
    rhs = float(np.sum(X * dX))
    # E2M1 terms are exact in float64; E4M3 subnormal-to-448 products span more
    # than 53 bits in these final inner products, so compare to 1e-12 there.
    scale = float(np.sum(np.abs(dY) * np.abs(Y))) + 1.0
    tol = 0.0 if elem == "e2m1" else 1e-12 * scale
    assert abs(lhs - mid) <= tol and abs(lhs - rhs) <= tol
    # and the identity is not vacuous: a transposed operand breaks it
    wrong = float(np.sum(X * oracle.grouped_dgrad(dY, np.ascontiguousarray(Wt[::-1]), splits)))
    assert abs(wrong - lhs) > 1e-6 * scale


def test_structural_invariants():
    rng = np.random.default_rng(34)
    splits = np.array([5, 0, 12, 3], dtype=np.int32)
    G, S, N, K = 4, 20, 16, 64
    A = rng.standard_normal((S, K))
    W = rng.standard_normal((G * N, K))
    Y = oracle.grouped_fwd(A, W, splits, N)
    off = np.concatenate([[0], np.cumsum(splits)])
    for g in range(G):
        assert np.array_equal(Y[off[g]: off[g + 1]], A[off[g]: off[g + 1]] @ W[g * N: (g + 1) * N].T)
    # G = 1 is the dense GEMM
    assert np.array_equal(oracle.grouped_fwd(A, W[:N], [S], N), A @ W[:N].T)
    # permuting experts permutes the row blocks
    perm = [2, 0, 3, 1]
    A_p = np.concatenate([A[off[g]: off[g + 1]] for g in perm])
    W_p = np.concatenate([W[g * N: (g + 1) * N] for g in perm])
    Y_p = oracle.grouped_fwd(A_p, W_p, splits[perm], N)
    assert np.array_equal(Y_p, np.concatenate([Y[off[g]: off[g + 1]] for g in perm]))
    # empty experts: dropping them (and their weights) changes nothing
    keep = [0, 2, 3]
    Y_k = oracle.grouped_fwd(A, np.concatenate([W[g * N: (g + 1) * N] for g in keep]), splits[keep], N)
    assert np.array_equal(Y_k, Y)


def test_split_validation():
    A = np.zeros((10, 32))
    W = np.zeros((2 * 8, 32))
    with pytest.raises(ValueError):
        oracle.grouped_fwd(A, W, [5, 4], 8)          # sum != rows
    with pytest.raises(ValueError):
        oracle.grouped_fwd(A, W, [11, -1], 8)        # negative
    with pytest.raises(ValueError):
        oracle.grouped_fwd(A, W, [10], 8)            # len != G


def test_tolerance_bound():
    rng = np.random.default_rng(35)
    ref = rng.standard_normal((64, 64))
    assert oracle.tolerance_violation(ref, ref) == 0.0
    bf = synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(ref.astype(np.float32))).astype(np.float64)
    assert oracle.tolerance_violation(bf, ref) <= 1.0     # BF16 rounding: half an ulp <= 2^-8 relative
    bad = bf.copy()
    bad[3, 4] *= 1.02
    with pytest.raises(AssertionError):
        oracle.assert_gemm_close(bad, ref, "planted")
    nan = bf.copy()
    nan[0, 0] = np.nan
    with pytest.raises(AssertionError):
        oracle.assert_gemm_close(nan, ref, "nan")


def test_fp64_exactness_bound():
    s = np.full((4, 2), 127, dtype=np.uint8)
    nz = np.ones_like(s, dtype=bool)
    assert oracle.fp64_sum_is_exact(s, nz, s, nz, "e4m3", "e2m1", 4096)
    s2 = s.copy()
    s2[0, 0] = 127 + 40
    assert not oracle.fp64_sum_is_exact(s2, nz, s, nz, "e4m3", "e4m3", 4096)


# --------------------------------------------------------------------------
# The fp64 reference on every configuration's operands.
# --------------------------------------------------------------------------
def _pass_shapes():
    """(config, pass, A format, B format, contraction length, std, outliers)
    for every pass of every configuration.  The wgrad contracts the largest
    expert's padded token count."""
    W = synth.WORKLOADS
    out = [("tiny_mxfp4_fwd", "fwd", "e2m1", "e2m1", W["tiny_mxfp4_fwd"].K, 1.0, 0.0),
           ("a8w4_fwd", "fwd", "e4m3", "e2m1", W["a8w4_fwd"].K, 1.0, 0.01)]
    for cfg, fmt in (("mxfp4_moe_train", "e2m1"), ("mxfp8_moe_train", "e4m3"),
                     ("blockwise_fp8", "bw"), ("blockwise_fp8_pow2", "bw_pow2"),
                     ("dense_mxfp4_m2048", "e2m1"), ("dense_mxfp4_m4096", "e2m1"),
                     ("dense_mxfp4_m8192", "e2m1")):
        w = W[{"mxfp8_moe_train": "mxfp4_moe_train", "blockwise_fp8_pow2": "blockwise_fp8"}.get(cfg, cfg)]
        m = w.splits().astype(np.int64)
        pad = 128 if fmt.startswith("bw") else w.pad
        tokens = int(((m.max() + pad - 1) // pad) * pad)
        for p, L in (("fwd", w.K), ("dgrad", w.N), ("wgrad", tokens)):
            out.append((cfg, p, fmt, fmt, L, w.std, 0.0))
    return out


def _sample_operand(rng, rows, L, fmt, std, outliers, weight):
    """`rows` rows of length L drawn as the configuration draws them,
    quantized along L; returns (dequantized float64, scale bytes or None,
    nonzero-block mask or None)."""
    x = synth.normal_bf16(rng, (rows, L), std=std, outlier_frac=outliers)
    if fmt in ("bw", "bw_pow2"):
        p2 = fmt == "bw_pow2"
        if weight:     # 128x128 tiles
            c, s = oracle.quantize_bw_128x128(x.reshape(1, rows, L), pow2=p2)
            d = oracle.dequantize_bw_128x128(c, s)[0]
            s = np.repeat(np.repeat(s[0], 128, axis=0), 4, axis=1)
        else:
            c, s = oracle.quantize_bw_1x128(x, pow2=p2)
            d = oracle.dequantize_bw_1x128(c, s)
            s = np.repeat(s, 4, axis=1)
        if not p2:
            return d, None, None
        sb = (np.log2(s.astype(np.float64)) + 127).astype(np.uint8)     # exact powers of two
        nz = np.abs(d).reshape(rows, L // 32, 32).max(axis=-1) > 0
        return d, sb, nz
    codes, scale = oracle.quantize_mx(x, fmt)
    d = oracle.dequantize_mx(codes, scale, fmt)
    nz = (codes & (0x7 if fmt == "e2m1" else 0x7F)).reshape(rows, L // 32, 32).max(axis=-1) > 0
    return d, scale, nz


# configurations whose fp64 sums are provably exact on the sampled operands
# (sufficient condition of oracle.fp64_sum_is_exact); the others are held to
# the rounding bound below.  MXFP8 (E4M3 x E4M3 with 32-element scales):
# products span more than 52 bits over a 2048- to 7168-long sum; fp32
# blockwise scales give 28-bit operand significands, so even single products
# round in fp64.  Power-of-two blockwise scales vary little within a row
# (one per 128 elements) and stay exact.
EXACT = {"tiny_mxfp4_fwd", "a8w4_fwd", "mxfp4_moe_train", "blockwise_fp8_pow2", "dense_mxfp4_m2048",
         "dense_mxfp4_m4096", "dense_mxfp4_m8192"}


def test_fp64_reference_exact_or_bounded_per_config():
    """For every pass of every configuration, on 64 x 64 sampled dot products
    of the pass's full contraction length: either the sufficient exactness
    condition holds, or the fp64 rounding bound gamma_{L+1} * sum|a_k b_k|
    is below 0.1% of the smallest per-element allowance of the GEMM
    comparison (1e-4 * rms(ref)).  Either way the oracle's own error cannot
    decide a parity test."""
    rng = np.random.default_rng(77)
    seen = {}
    for cfg, p, fa, fb, L, std, outl in _pass_shapes():
        A, sa, nza = _sample_operand(rng, 64, L, fa, std, outl, weight=False)
        B, sb, nzb = _sample_operand(rng, 64 if not fb.startswith("bw") or p == "wgrad" else 128, L, fb,
                                     std, outl, weight=p != "wgrad")
        exact = False
        if sa is not None and sb is not None:
            ea = "e2m1" if fa == "e2m1" else "e4m3"
            eb = "e2m1" if fb == "e2m1" else "e4m3"
            exact = oracle.fp64_sum_is_exact(sa, nza, sb, nzb, ea, eb, L)
        seen.setdefault(cfg, []).append(exact)
        ref = A @ B.T
        mag = np.abs(A) @ np.abs(B).T
        u = 2.0 ** -53
        gamma = (L + 1) * u / (1 - (L + 1) * u)
        floor = 1e-4 * float(np.sqrt(np.mean(ref * ref)))
        assert float(gamma * mag.max()) <= 1e-3 * floor, (cfg, p, gamma * mag.max(), floor)
    got_exact = {c for c, v in seen.items() if all(v)}
    assert got_exact == EXACT, got_exact ^ EXACT
