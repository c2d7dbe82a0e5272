"""Full-size parity at the benchmark's workloads, through the very step the
benchmark times: each test builds bench.py's workload object (same seeded
inputs, same library calls -- the quantizers writing scales in the MMA staging
order, then the GEMM passes), runs one step on the GPU and checks sampled
outputs against the oracle.  The oracle cannot redo a whole problem in a
test, so it recomputes sampled outputs one by one: the first and last row of
every expert, rows spread over the largest expert (whose m-tiles span
several tile groups of the GEMM's L2-friendly order), random rows, against
random columns, quantizing only the operand rows and columns those samples
need.  Code bytes of the sampled rows of the row-wise operands are compared
bit for bit.  Bound per element, with rms over the sampled references:
    |gpu - ref| <= 2^-8 * |ref| + 1e-4 * rms(ref)."""

import os
import sys

import numpy as np
import pytest
import torch

import oracle
from oracle.blockwise import transpose_bw_128x128

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()


def _mxg():
    import fp8_bf16_mxfp4_gb300 as mxg
    return mxg


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _rows(t: torch.Tensor, idx) -> np.ndarray:
    return _bits(t[torch.as_tensor(np.asarray(idx, dtype=np.int64), device=t.device)])


def _pick(rng, splits, per_expert):
    """(expert, sorted global rows): first, last and random rows of every
    expert, plus 24 rows spread evenly over the largest expert."""
    off = np.concatenate([[0], np.cumsum(splits)])
    big = int(np.argmax(splits))
    out = []
    for g, m in enumerate(splits):
        if m == 0:
            continue
        pick = {0, int(m) - 1} | set(rng.integers(0, m, size=per_expert).tolist())
        if g == big:
            pick |= set(np.linspace(0, m - 1, 24).astype(int).tolist())
        out.append((g, off[g] + np.array(sorted(pick), dtype=np.int64)))
    return off, out


def _gather(t: torch.Tensor, rows, cols) -> np.ndarray:
    r = torch.as_tensor(np.asarray(rows, dtype=np.int64), device=t.device)
    c = torch.as_tensor(np.asarray(cols, dtype=np.int64), device=t.device)
    return t[r][:, c].float().cpu().numpy()


def _check(items, what):
    rms = float(np.sqrt(np.mean(np.concatenate([r.ravel() for _, r, _ in items]) ** 2)))
    for got, ref, g in items:
        oracle.assert_gemm_close(got, ref, f"{what} expert {g}", rms_ref=rms)


def _mx_deq_rows(bits, elem):
    d, s = oracle.quantize_mx_rowwise(bits, elem)
    return oracle.dequantize_mx(oracle.unpack_e2m1(d) if elem == "e2m1" else d, s, elem), d


def _mx_deq_cols(seg_bits, m, pad, elem):
    d, s, _ = oracle.quantize_mx_colwise_segment_padded(seg_bits, [m], pad, elem)
    return oracle.dequantize_mx(oracle.unpack_e2m1(d) if elem == "e2m1" else d, s, elem)


def _workload(name):
    import bench
    wl = bench.build_workload(name, torch.device("cuda:0"))
    return wl


# ---------------------------------------------------------------- MX steps
def _mx_fwd_items(wl, rng, ea, eb, y, picks, n_cols=16):
    """Sampled forward outputs; also checks the sampled A rows' code bytes
    from the library's packed row-wise quantizer (the bench's call)."""
    mxg = _mxg()
    Aq = mxg.mx_quantize_rowwise_packed(wl.x, ea, m_splits=wl.d_splits, check=True)
    x = wl.x
    w = getattr(wl, "w", None)
    if w is None:
        w = wl.wt
    items = []
    for g, rows in picks:
        cols = np.unique(np.concatenate([[0, wl.N - 1], rng.integers(0, wl.N, size=n_cols)]))
        Ad, ad = _mx_deq_rows(_rows(x, rows), ea)
        assert np.array_equal(Aq.data[torch.as_tensor(rows)].cpu().numpy(), ad), f"A codes, expert {g}"
        Wd, _ = _mx_deq_rows(_rows(w, g * wl.N + cols), eb)
        items.append((_gather(y, rows, cols), Ad @ Wd.T, g))
    return items


def _mx_dgrad_items(wl, rng, e, dx, picks, n_cols=16):
    items = []
    for g, rows in picks:
        ks = np.unique(np.concatenate([[0, wl.K - 1], rng.integers(0, wl.K, size=n_cols)]))
        dYd, _ = _mx_deq_rows(_rows(wl.dy, rows), e)
        wband = _bits(wl.w[g * wl.N:(g + 1) * wl.N][:, torch.as_tensor(ks, device=wl.w.device)])
        Wtd, _ = _mx_deq_rows(np.ascontiguousarray(wband.T), e)        # W^T rows k, along N
        items.append((_gather(dx, rows, ks), dYd @ Wtd.T, g))
    return items


def _mx_wgrad_items(wl, rng, e, dw, init, experts, n=8):
    off = np.concatenate([[0], np.cumsum(wl.splits)])
    items = []
    for g in experts:
        m = int(wl.splits[g])
        ns = np.unique(np.concatenate([[0, wl.N - 1], rng.integers(0, wl.N, size=n)]))
        ks = np.unique(np.concatenate([[0, wl.K - 1], rng.integers(0, wl.K, size=n)]))
        dyseg = _bits(wl.dy[off[g]: off[g] + m][:, torch.as_tensor(ns, device=wl.dy.device)])
        xseg = _bits(wl.x[off[g]: off[g] + m][:, torch.as_tensor(ks, device=wl.x.device)])
        if m:
            ref = _mx_deq_cols(dyseg, m, wl.pad, e) @ _mx_deq_cols(xseg, m, wl.pad, e).T
        else:
            ref = np.zeros((len(ns), len(ks)))
        if init is not None:
            ref = ref + init[g][torch.as_tensor(ns)][:, torch.as_tensor(ks)].cpu().numpy()
        items.append((dw[g][torch.as_tensor(ns)][:, torch.as_tensor(ks)].float().cpu().numpy(), ref, g))
    return items


def _wgrad_experts(splits):
    nz = np.where(splits > 0)[0]
    pick = {int(np.argmax(splits)), int(nz[np.argmin(splits[nz])]), int(nz[0]), int(nz[-1])}
    return sorted(pick | set(range(0, len(splits), max(1, len(splits) // 6))))


def test_a8w4_forward_full_size():
    wl = _workload("a8w4_fwd")
    wl.step()
    wl.check()
    rng = np.random.default_rng(7)
    _, picks = _pick(rng, wl.splits, 6)
    _check(_mx_fwd_items(wl, rng, "e4m3", "e2m1", wl.y, picks, 30), "a8w4 fwd")


@pytest.mark.parametrize("name,elem", [("mxfp4_moe_train", "e2m1"), ("mxfp8_moe_train", "e4m3")])
def test_mx_training_step_full_size(name, elem):
    wl = _workload(name)
    init = wl.main_grad.clone()
    wl.step()
    wl.check()
    rng = np.random.default_rng(8)
    _, picks = _pick(rng, wl.splits, 2)
    _check(_mx_fwd_items(wl, rng, elem, elem, wl.y, picks), f"{name} fwd")
    _check(_mx_dgrad_items(wl, rng, elem, wl.dx, picks), f"{name} dgrad")
    _check(_mx_wgrad_items(wl, rng, elem, wl.main_grad, init, _wgrad_experts(wl.splits)), f"{name} wgrad")


def test_dense_mxfp4_m8192_full_size():
    """G = 1 at M = 8192: the forward's and dgrad's m-tiles span several tile
    groups (tile_mn), with both output dtypes of every pass."""
    wl = _workload("dense_mxfp4_m8192")
    wl.step()
    wl.check()
    rng = np.random.default_rng(10)
    _, picks = _pick(rng, wl.splits, 24)
    _check(_mx_fwd_items(wl, rng, "e2m1", "e2m1", wl.y, picks, 24), "dense fwd bf16")
    _check(_mx_fwd_items(wl, rng, "e2m1", "e2m1", wl.y32, picks, 24), "dense fwd f32")
    _check(_mx_dgrad_items(wl, rng, "e2m1", wl.dx, picks, 24), "dense dgrad bf16")
    _check(_mx_dgrad_items(wl, rng, "e2m1", wl.dx32, picks, 24), "dense dgrad f32")
    _check(_mx_wgrad_items(wl, rng, "e2m1", wl.dw, None, [0], 24), "dense wgrad f32")
    _check(_mx_wgrad_items(wl, rng, "e2m1", wl.dw16, None, [0], 24), "dense wgrad bf16")


# ---------------------------------------------------------------- blockwise steps
def _bw_items(wl, rng, pow2, picks, experts):
    off = np.concatenate([[0], np.cumsum(wl.splits)])
    N, K = wl.N, wl.K
    items = {"fwd": [], "dgrad": [], "wgrad": []}
    for g, rows in picks:
        nb = int(rng.integers(0, N // 128))
        cols = nb * 128 + np.unique(np.concatenate([[0, 127], rng.integers(0, 128, size=8)]))
        wblk = _bits(wl.w[g * N + nb * 128: g * N + nb * 128 + 128])           # one 128 x K band
        wc, ws = oracle.quantize_bw_128x128(wblk.reshape(1, 128, K), pow2=pow2)
        Wd = oracle.dequantize_bw_128x128(wc, ws)[0]
        xc, xs = oracle.quantize_bw_1x128(_rows(wl.x, rows), pow2=pow2)
        Ad = oracle.dequantize_bw_1x128(xc, xs)
        items["fwd"].append((_gather(wl.y, rows, cols), Ad @ Wd[cols - nb * 128].T, g))
        kb = int(rng.integers(0, K // 128))
        ks = kb * 128 + np.unique(np.concatenate([[0, 127], rng.integers(0, 128, size=8)]))
        wband = _bits(wl.w[g * N:(g + 1) * N][:, kb * 128: kb * 128 + 128])      # N x 128 band
        wc2, ws2 = oracle.quantize_bw_128x128(np.ascontiguousarray(wband).reshape(1, N, 128), pow2=pow2)
        ct, st = transpose_bw_128x128(wc2, ws2)
        Wtd = oracle.dequantize_bw_128x128(ct, st)[0]                            # [128, N]
        dc, dsc = oracle.quantize_bw_1x128(_rows(wl.dy, rows), pow2=pow2)
        items["dgrad"].append((_gather(wl.dx, rows, ks), oracle.dequantize_bw_1x128(dc, dsc) @ Wtd[ks - kb * 128].T,
                               g))
    for g in experts:
        m = int(wl.splits[g])
        ns = np.unique(np.concatenate([[0, N - 1], rng.integers(0, N, size=6)]))
        kk = np.unique(np.concatenate([[0, K - 1], rng.integers(0, K, size=6)]))
        dyseg = _bits(wl.dy[off[g]: off[g] + m][:, torch.as_tensor(ns, device=wl.dy.device)])
        xseg = _bits(wl.x[off[g]: off[g] + m][:, torch.as_tensor(kk, device=wl.x.device)])
        dc_, ds_, _ = oracle.quantize_bw_colwise_padded(dyseg, [m], pow2=pow2)
        xc_, xs_, _ = oracle.quantize_bw_colwise_padded(xseg, [m], pow2=pow2)
        ref = oracle.dequantize_bw_1x128(dc_, ds_) @ oracle.dequantize_bw_1x128(xc_, xs_).T
        items["wgrad"].append((wl.dw[g][torch.as_tensor(ns)][:, torch.as_tensor(kk)].float().cpu().numpy(), ref, g))
    return items


@pytest.mark.parametrize("name,pow2", [("blockwise_fp8", False), ("blockwise_fp8_pow2", True)])
def test_blockwise_step_full_size(name, pow2):
    wl = _workload(name)
    wl.step()
    wl.check()
    rng = np.random.default_rng(9)
    _, picks = _pick(rng, wl.splits, 2)
    for p, its in _bw_items(wl, rng, pow2, picks, _wgrad_experts(wl.splits)).items():
        _check(its, f"{name} {p}")
