"""Grouped GEMM oracle: per-expert float64 contraction of dequantized operands.

TEST INFRASTRUCTURE ONLY (see the package docstring).

The three passes of an MoE expert layer, as stated in "Triton mxfp4 (and a8w4)
grouped GEMM kernel" (PR #723: forward, input-gradient and weight-gradient
entry points over prefix-summed group offsets) and in the per-pass shapes of
"Integrate MXFP4 hipblaslt GEMM support" (PR #697, benchmark section: forward
contracts hidden, dgrad contracts out, wgrad contracts tokens).  Experts'
rows are concatenated in order; off = exclusive prefix sum of m_splits.

* forward (TN): Y[off_g+i, n]  = sum_k A[off_g+i, k] * W[g*N+n, k]
* dgrad   (NN): dX[off_g+i, k] = sum_n dY[off_g+i, n] * Wt[k, g*N+n]
* wgrad   (NT): dW[g, n, k]    = sum_{j in expert g's padded token segment}
                                 dYt[n, j] * Xt[k, j]      (+= when accumulating)

Operands arrive dequantized (float64); each expert is one library matmul in
float64.  Products of MX element values times power-of-two scales are exact in
float64, and so is their sum whenever the exponent spread of the terms plus
log2(K) stays below 53 bits (``fp64_sum_is_exact`` checks that bound).

The comparison bound used against the GPU is per element
    |gpu - ref| <= 2^-8 * |ref| + 1e-4 * rms(ref):
products are exact on both sides, so only fp32 summation order and the BF16
output rounding (relative 2^-9) separate them.
"""

from __future__ import annotations

import numpy as np


def check_splits(m_splits, rows: int, G: int) -> np.ndarray:
    """The split validation the pages ask for (PR #723 review): len == G,
    non-negative, and summing to the operand's row count."""
    m = np.asarray(m_splits, dtype=np.int64)
    if m.ndim != 1 or m.shape[0] != G:
        raise ValueError("len(m_splits) != G")
    if (m < 0).any():
        raise ValueError("negative split")
    if int(m.sum()) != rows:
        raise ValueError("sum(m_splits) != rows")
    return np.concatenate([[0], np.cumsum(m)]).astype(np.int64)


def grouped_fwd(A: np.ndarray, W: np.ndarray, m_splits, N: int) -> np.ndarray:
    """A [S, K], W [G*N, K] (float64) -> Y [S, N]."""
    S, K = A.shape
    G = W.shape[0] // N
    off = check_splits(m_splits, S, G)
    Y = np.zeros((S, N), dtype=np.float64)
    for g in range(G):
        a = A[off[g]: off[g + 1]]
        if a.shape[0]:
            Y[off[g]: off[g + 1]] = a @ W[g * N: (g + 1) * N].T
    return Y


def grouped_dgrad(dY: np.ndarray, Wt: np.ndarray, m_splits) -> np.ndarray:
    """dY [S, N], Wt [K, G*N] (float64) -> dX [S, K]."""
    S, N = dY.shape
    K = Wt.shape[0]
    G = Wt.shape[1] // N
    off = check_splits(m_splits, S, G)
    dX = np.zeros((S, K), dtype=np.float64)
    for g in range(G):
        d = dY[off[g]: off[g + 1]]
        if d.shape[0]:
            dX[off[g]: off[g + 1]] = d @ Wt[:, g * N: (g + 1) * N].T
    return dX


def grouped_wgrad(dYt: np.ndarray, Xt: np.ndarray, pad_offsets,
                  out_init: np.ndarray | None = None) -> np.ndarray:
    """dYt [N, Spad], Xt [K, Spad] (float64), pad_offsets [G+1] -> dW [G, N, K].

    An empty expert contributes zero (so the output is zero, or unchanged
    when accumulating)."""
    poff = np.asarray(pad_offsets, dtype=np.int64)
    G = poff.shape[0] - 1
    N, K = dYt.shape[0], Xt.shape[0]
    dW = np.zeros((G, N, K), dtype=np.float64)
    for g in range(G):
        j0, j1 = poff[g], poff[g + 1]
        if j1 > j0:
            dW[g] = dYt[:, j0:j1] @ Xt[:, j0:j1].T
    if out_init is not None:
        dW = dW + np.asarray(out_init, dtype=np.float64)
    return dW


def tolerance_violation(gpu: np.ndarray, ref: np.ndarray,
                        rel: float = 2.0 ** -8, rms_frac: float = 1e-4) -> float:
    """max over elements of |gpu - ref| / (rel*|ref| + rms_frac*rms(ref)).
    A value <= 1 means every element is inside the bound."""
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if ref.size == 0:
        return 0.0
    rms = float(np.sqrt(np.mean(ref * ref)))
    bound = rel * np.abs(ref) + rms_frac * rms
    err = np.abs(gpu - ref)
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.where(bound > 0, err / np.where(bound > 0, bound, 1.0), np.where(err > 0, np.inf, 0.0))
    return float(r.max())


def assert_gemm_close(gpu, ref, what: str = "", rms_ref: float | None = None):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if rms_ref is None:
        v = tolerance_violation(gpu, ref)
    else:
        bound = 2.0 ** -8 * np.abs(ref) + 1e-4 * rms_ref
        v = float((np.abs(gpu - ref) / bound).max()) if ref.size else 0.0
    if not np.isfinite(gpu).all():
        raise AssertionError(f"{what}: non-finite GPU output")
    if v > 1.0:
        idx = np.unravel_index(np.argmax(np.abs(gpu - ref)), ref.shape)
        raise AssertionError(
            f"{what}: tolerance exceeded by x{v:.3g}; worst |diff| at {idx}: "
            f"gpu={gpu[idx]!r} ref={ref[idx]!r}")
    return v


def fp64_sum_is_exact(scale_bytes_a: np.ndarray, codes_nonzero_a: np.ndarray,
                      scale_bytes_b: np.ndarray, codes_nonzero_b: np.ndarray,
                      elem_a: str, elem_b: str, K: int) -> bool:
    """Sufficient condition for the float64 per-expert matmul to be exact:
    every product is an integer multiple of 2^lo and bounded by 2^hi, so the
    running sum is exact when hi - lo + log2(K) <= 52.

    Block scales of all-zero blocks are ignored (those blocks add nothing).
    ``codes_nonzero_*`` are boolean arrays with one entry per scale byte."""
    def span(scale, nz, elem):
        s = scale[nz].astype(np.int64) - 127
        if s.size == 0:
            return None
        # element magnitudes: E2M1 in [0.5, 6] with 1 mantissa bit -> quantum 2^-1,
        # max < 2^3; E4M3 in [2^-9, 448] -> quantum 2^-9, max < 2^9.
        q, top = (-1, 3) if elem == "e2m1" else (-9, 9)
        return int(s.min()) + q, int(s.max()) + top
    a = span(scale_bytes_a, codes_nonzero_a, elem_a)
    b = span(scale_bytes_b, codes_nonzero_b, elem_b)
    if a is None or b is None:
        return True
    lo = a[0] + b[0]
    hi = a[1] + b[1]
    return (hi - lo) + int(np.ceil(np.log2(max(K, 1)))) <= 52
