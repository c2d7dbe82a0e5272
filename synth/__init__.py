"""Seeded synthetic inputs shared by the tests, the bench and the smoke check.

This module only draws random numbers and lays them out: BF16 activations and
weights, per-expert row counts (``m_splits``) from MoE-style routing, and the
workload table.  It contains none of the quantization or GEMM arithmetic; the
oracle (``oracle/``) and the CUDA library each implement that on their own.

BF16 values are produced from fp32 draws by round-to-nearest-even on the bit
pattern (the usual fp32 -> bf16 conversion), and are handed around as
``uint16`` bit arrays so that neither side depends on a framework's dtype.

The workloads follow the five configurations of the grouped MX GEMM study
(tiny MXFP4 forward, a8w4 forward, MXFP4 MoE training step, blockwise-FP8
grouped GEMM, dense MXFP4 per-pass sweep).  The pages measure on no public
dataset, so these seeded recipes stand in for real routing and activations.
"""

from __future__ import annotations

import dataclasses
import numpy as np

__all__ = [
    "Workload",
    "WORKLOADS",
    "f32_to_bf16_bits",
    "bf16_bits_to_f32",
    "normal_bf16",
    "splits_tiny",
    "splits_topk",
    "splits_uniform_rows",
    "padded_rows_capacity",
]


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit pattern, round-to-nearest-even (finite inputs only)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    u = u + 0x7FFF + ((u >> 16) & 1)
    return (u >> 16).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """bf16 bit pattern -> fp32 (exact)."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def normal_bf16(rng: np.random.Generator, shape, std: float = 1.0,
                outlier_frac: float = 0.0, outlier_mult: float = 50.0,
                chunk_rows: int = 4096) -> np.ndarray:
    """N(0, std^2) values as bf16 bits; optionally a Bernoulli(outlier_frac)
    subset multiplied by ``outlier_mult``.  Drawn in row chunks to bound the
    host memory used for large tensors."""
    shape = tuple(int(s) for s in shape)
    out = np.empty(shape, dtype=np.uint16)
    if out.size == 0:
        return out
    rows = shape[0] if shape else 1
    flat = out.reshape(rows, -1) if shape else out.reshape(1, 1)
    cols = flat.shape[1]
    for r0 in range(0, rows, chunk_rows):
        r1 = min(rows, r0 + chunk_rows)
        v = rng.standard_normal((r1 - r0, cols), dtype=np.float32)
        if std != 1.0:
            v *= np.float32(std)
        if outlier_frac > 0.0:
            m = rng.random((r1 - r0, cols), dtype=np.float32) < outlier_frac
            v[m] *= np.float32(outlier_mult)
        flat[r0:r1] = f32_to_bf16_bits(v)
    return out


def _largest_remainder(total: int, p: np.ndarray) -> np.ndarray:
    raw = p * total
    base = np.floor(raw).astype(np.int64)
    rem = total - int(base.sum())
    order = np.argsort(-(raw - base), kind="stable")
    base[order[:rem]] += 1
    return base


def splits_tiny(rng: np.random.Generator, G: int = 4, S: int = 512) -> np.ndarray:
    """G-1 experts share S rows by largest-remainder rounding of
    S * Dirichlet(1,...,1); a zero split is inserted at a random index."""
    p = rng.dirichlet(np.ones(G - 1))
    s = _largest_remainder(S, p)
    at = int(rng.integers(G))
    return np.insert(s, at, 0).astype(np.int32)


def _gumbel_topk_counts(rng, p: np.ndarray, tokens: int, k: int) -> np.ndarray:
    """Each token picks k distinct experts with probability proportional to p
    (Gumbel-top-k sampling); returns the per-expert row count."""
    G = p.shape[0]
    counts = np.zeros(G, dtype=np.int64)
    logp = np.log(p)
    for t0 in range(0, tokens, 8192):
        t1 = min(tokens, t0 + 8192)
        g = rng.gumbel(size=(t1 - t0, G))
        pick = np.argpartition(-(logp[None, :] + g), k - 1, axis=1)[:, :k]
        counts += np.bincount(pick.ravel(), minlength=G)
    return counts


def splits_topk(rng: np.random.Generator, G: int, tokens: int, k: int,
                skew: str, alpha: float = 0.5, zipf_s: float = 1.1) -> np.ndarray:
    """MoE routing counts: ``skew='dirichlet'`` draws expert probabilities from
    Dirichlet(alpha); ``skew='zipf'`` makes them proportional to rank^-s over a
    seeded permutation of ranks.  The result sums to tokens * k."""
    if skew == "dirichlet":
        p = rng.dirichlet(np.full(G, alpha))
    elif skew == "zipf":
        ranks = rng.permutation(G) + 1
        p = ranks.astype(np.float64) ** (-zipf_s)
        p /= p.sum()
    else:
        raise ValueError(skew)
    p = np.maximum(p, 1e-12)
    p /= p.sum()
    return _gumbel_topk_counts(rng, p, tokens, k).astype(np.int32)


def splits_uniform_rows(rng: np.random.Generator, G: int, rows: int) -> np.ndarray:
    """Each row independently routed to a uniformly random expert."""
    e = rng.integers(G, size=rows)
    return np.bincount(e, minlength=G).astype(np.int32)


def padded_rows_capacity(rows: int, G: int, pad: int) -> int:
    """Upper bound on sum_g ceil(m_g/pad)*pad over all splits of ``rows``
    (at most min(G, rows) experts are non-empty and each adds < pad)."""
    k = min(G, rows)
    return ((rows + k * (pad - 1)) // pad) * pad


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    G: int
    N: int
    K: int
    kind: str                 # "mxfp4", "a8w4", "blockwise_fp8", "dense_mxfp4"
    passes: tuple             # subset of ("fwd", "dgrad", "wgrad")
    seed: int
    std: float = 1.0
    outlier_frac: float = 0.0
    pad: int = 32
    splits_recipe: str = ""
    M: int = 0                # dense sweep only

    def splits(self) -> np.ndarray:
        rng = np.random.default_rng(self.seed)
        r = self.splits_recipe
        if r == "tiny":
            return splits_tiny(rng, self.G, 512)
        if r == "top2_dirichlet":
            return splits_topk(rng, self.G, 4096, 2, "dirichlet", alpha=0.5)
        if r == "top8_zipf":
            return splits_topk(rng, self.G, 16384, 8, "zipf", zipf_s=1.1)
        if r == "uniform":
            return splits_uniform_rows(rng, self.G, 32768)
        if r == "dense":
            return np.array([self.M], dtype=np.int32)
        raise ValueError(r)

    def act_rng(self, which: int = 0) -> np.random.Generator:
        return np.random.default_rng(1000 + 10 * self.seed + which)

    def weight_rng(self) -> np.random.Generator:
        return np.random.default_rng(100 + self.seed)


WORKLOADS = {
    "tiny_mxfp4_fwd": Workload("tiny_mxfp4_fwd", G=4, N=256, K=512, kind="mxfp4",
                               passes=("fwd",), seed=0, splits_recipe="tiny"),
    "a8w4_fwd": Workload("a8w4_fwd", G=8, N=14336, K=4096, kind="a8w4",
                         passes=("fwd",), seed=1, outlier_frac=0.01,
                         splits_recipe="top2_dirichlet"),
    "mxfp4_moe_train": Workload("mxfp4_moe_train", G=32, N=2048, K=7168, kind="mxfp4",
                                passes=("fwd", "dgrad", "wgrad"), seed=2, pad=32,
                                splits_recipe="top8_zipf"),
    "blockwise_fp8": Workload("blockwise_fp8", G=16, N=4096, K=7168, kind="blockwise_fp8",
                              passes=("fwd", "dgrad", "wgrad"), seed=3, pad=128,
                              splits_recipe="uniform"),
    "dense_mxfp4_m2048": Workload("dense_mxfp4_m2048", G=1, N=28672, K=8192,
                                  kind="dense_mxfp4", passes=("fwd", "dgrad", "wgrad"),
                                  seed=4, std=0.02, splits_recipe="dense", M=2048),
    "dense_mxfp4_m4096": Workload("dense_mxfp4_m4096", G=1, N=28672, K=8192,
                                  kind="dense_mxfp4", passes=("fwd", "dgrad", "wgrad"),
                                  seed=4, std=0.02, splits_recipe="dense", M=4096),
    "dense_mxfp4_m8192": Workload("dense_mxfp4_m8192", G=1, N=28672, K=8192,
                                  kind="dense_mxfp4", passes=("fwd", "dgrad", "wgrad"),
                                  seed=4, std=0.02, splits_recipe="dense", M=8192),
}
