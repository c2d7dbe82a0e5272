"""The host-side size functions return upper bounds that must hold for every
routing the device may see, because the caller sizes its buffers before the
splits are known on the host.  Each bound is checked here against the exact
size the oracle computes for random and adversarial splits (CPU only, no
device calls)."""

import numpy as np
import pytest

import oracle


@pytest.fixture(scope="module")
def lib():
    from fp8_bf16_mxfp4_gb300 import build, _lib
    build.build()
    return _lib.load()


def _routings(rng, rows, G, count):
    """Random splits of `rows` over G experts (Dirichlet and with empty
    experts), plus the adversarial ones: as many experts as possible one row
    past a 128-row (and 32-row) boundary, all rows in one expert, and every
    expert empty but one."""
    out = []
    for _ in range(count):
        p = rng.dirichlet(np.full(G, rng.choice([0.1, 0.5, 2.0])))
        m = np.floor(p * rows).astype(np.int64)
        m[rng.integers(G)] += rows - m.sum()
        out.append(m)
    for step in (129, 33, 1):
        m = np.zeros(G, dtype=np.int64)
        left = rows
        for g in range(G):
            take = min(step, left)
            m[g] = take
            left -= take
        m[0] += left
        out.append(m)
    one = np.zeros(G, dtype=np.int64)
    one[-1] = rows
    out.append(one)
    return out


CASES = [(0, 1), (1, 1), (5, 8), (129, 1), (1000, 4), (4096, 32), (8192, 8), (3 * 129, 3), (20000, 512)]


@pytest.mark.parametrize("rows,G", CASES)
def test_padded_capacity_covers_every_routing(lib, rows, G):
    rng = np.random.default_rng(rows * 7 + G)
    for pad in (32, 64, 128):
        cap = lib.mx_padded_rows_capacity(rows, G, pad)
        assert cap % pad == 0
        for m in _routings(rng, rows, G, 20):
            assert m.sum() == rows and (m >= 0).all()
            assert int(((m + pad - 1) // pad * pad).sum()) <= cap


@pytest.mark.parametrize("rows,G", CASES)
def test_packed_rowwise_bound_covers_every_routing(lib, rows, G):
    rng = np.random.default_rng(rows * 11 + G)
    for cols in (32, 160, 4096):
        bound = lib.mx_packed_scale_bytes(rows, cols, G)
        worst = 0
        for m in _routings(rng, rows, G, 20):
            exact = oracle.packed_scale_bytes(m, cols // 32)
            assert exact <= bound, (m.tolist(), cols)
            worst = max(worst, exact)
        if rows == G * 129 or (G == 1 and rows % 128 == 1):
            assert worst == bound  # attained: every expert one row past a tile


@pytest.mark.parametrize("rows,G", CASES)
def test_packed_colwise_bound_covers_every_routing(lib, rows, G):
    rng = np.random.default_rng(rows * 13 + G)
    for pad in (32, 128):
        cap = lib.mx_padded_rows_capacity(rows, G, pad)
        for C in (32, 160, 2048):
            bound = lib.mx_packed_colwise_scale_bytes(C, cap, G)
            for m in _routings(rng, rows, G, 20):
                p = (m + pad - 1) // pad * pad
                poff = np.concatenate([[0], np.cumsum(p)])
                exact = int(oracle.kseg_chunk_prefix(poff)[-1]) * ((C + 127) // 128) * 512
                assert exact <= bound, (m.tolist(), pad, C)


def test_packed_colwise_bound_covers_the_dgrad_weights(lib):
    # the dgrad Wt operand: G segments of N rows each, padded to 32, capacity G * N
    for G, N, K in [(1, 32, 64), (8, 160, 256), (32, 2048, 7168), (16, 4096, 7168)]:
        poff = np.arange(G + 1) * ((N + 31) // 32 * 32)
        exact = int(oracle.kseg_chunk_prefix(poff)[-1]) * ((K + 127) // 128) * 512
        assert exact <= lib.mx_packed_colwise_scale_bytes(K, G * N, G)


@pytest.mark.parametrize("rows,G", [(1, 1), (1000, 4), (4096, 32), (3 * 129, 3), (20000, 512)])
def test_gemm_workspace_covers_every_routing(lib, rows, G):
    """The GEMM scratch holds the plan tables and, for operands with plain
    scales, both operands' scales re-laid out in the MMA order; its size is
    fixed before the splits are known."""
    rng = np.random.default_rng(rows * 17 + G)
    N, K, pad = 160, 288, 32
    kseg = lambda poff, C: int(oracle.kseg_chunk_prefix(poff)[-1]) * ((C + 127) // 128) * 512
    plan = 5 * (G + 1) * 4
    ws_f = lib.mxg_gemm_workspace_size(0, G, rows, N, K, pad)
    ws_d = lib.mxg_gemm_workspace_size(1, G, rows, N, K, pad)
    cap = lib.mx_padded_rows_capacity(rows, G, pad)
    ws_w = lib.mxg_gemm_workspace_size(2, G, cap, N, K, pad)
    w_rows = oracle.packed_scale_bytes([N] * G, K // 32)
    wt = kseg(np.arange(G + 1) * N, K)
    for m in _routings(rng, rows, G, 10):
        assert plan + oracle.packed_scale_bytes(m, K // 32) + w_rows <= ws_f
        assert plan + oracle.packed_scale_bytes(m, N // 32) + wt <= ws_d
        poff = np.concatenate([[0], np.cumsum((m + pad - 1) // pad * pad)])
        assert plan + kseg(poff, N) + kseg(poff, K) <= ws_w
