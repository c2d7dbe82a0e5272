"""Full-size parity at the benchmark's workloads, in the launch configuration
bench.py times (library quantizers feeding the library GEMMs).  The oracle
cannot redo the whole problem in a test, so it recomputes sampled outputs one
by one: every expert's first and last row plus random rows, against random
columns, quantizing only the operand rows and columns those samples need.
Quantized bytes of the sampled rows are compared bit for bit."""

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


def _sample_rows(rng, splits, per_expert):
    off = np.concatenate([[0], np.cumsum(splits)])
    out = []
    for g, m in enumerate(splits):
        if m == 0:
            continue
        pick = {0, m - 1} | set(rng.integers(0, m, size=per_expert).tolist())
        out.append((g, sorted(off[g] + np.array(sorted(pick)))))
    return off, out


def _deq(bits, elem):
    d, s = oracle.quantize_mx_rowwise(bits, elem)
    return oracle.dequantize_mx(oracle.unpack_e2m1(d) if elem == "e2m1" else d, s, elem), d, s


def test_a8w4_forward_full_size():
    mxg = _mxg()
    w = synth.WORKLOADS["a8w4_fwd"]
    splits = w.splits()
    G, N, K, S = w.G, w.N, w.K, int(splits.sum())
    x = synth.normal_bf16(w.act_rng(), (S, K), outlier_frac=w.outlier_frac)
    wt = synth.normal_bf16(w.weight_rng(), (G * N, K), outlier_frac=w.outlier_frac)
    A = mxg.mx_quantize_rowwise(bf16_to_dev(x), "e4m3")
    W = mxg.mx_quantize_rowwise(bf16_to_dev(wt), "e2m1")
    Y = mxg.grouped_gemm_fwd(A, W, i32_to_dev(splits), N, check=True)
    rng = np.random.default_rng(7)
    _, picks = _sample_rows(rng, splits, 6)
    rms_ref = []
    checks = []
    for g, rows in picks:
        cols = np.unique(np.concatenate([[0, N - 1], rng.integers(0, N, size=30)]))
        Ad, ad, asc = _deq(x[rows], "e4m3")
        Wd, wd, wsc = _deq(wt[g * N + cols], "e2m1")
        assert np.array_equal(A.data[torch.as_tensor(rows)].cpu().numpy(), ad)
        assert np.array_equal(A.scale[torch.as_tensor(rows)].cpu().numpy(), asc)
        assert np.array_equal(W.data[torch.as_tensor(g * N + cols)].cpu().numpy(), wd)
        ref = Ad @ Wd.T
        got = Y[torch.as_tensor(rows)][:, torch.as_tensor(cols)].float().cpu().numpy()
        checks.append((got, ref, g))
        rms_ref.append(ref.ravel())
    rms = float(np.sqrt(np.mean(np.concatenate(rms_ref) ** 2)))
    for got, ref, g in checks:
        oracle.assert_gemm_close(got, ref, f"a8w4 full-size expert {g}", rms_ref=rms)


def test_mxfp4_training_step_full_size():
    mxg = _mxg()
    w = synth.WORKLOADS["mxfp4_moe_train"]
    splits = w.splits()
    G, N, K, S, pad = w.G, w.N, w.K, int(splits.sum()), w.pad
    x = synth.normal_bf16(w.act_rng(0), (S, K))
    dy = synth.normal_bf16(w.act_rng(1), (S, N))
    wt = synth.normal_bf16(w.weight_rng(), (G * N, K))
    d_splits = i32_to_dev(splits)
    xd, dyd, wd = bf16_to_dev(x), bf16_to_dev(dy), bf16_to_dev(wt)
    Xq = mxg.mx_quantize_rowwise(xd, "e2m1")
    Wq = mxg.mx_quantize_rowwise(wd, "e2m1")
    Y = mxg.grouped_gemm_fwd(Xq, Wq, d_splits, N, check=True)
    dYq = mxg.mx_quantize_rowwise(dyd, "e2m1")
    Wt, _ = mxg.mx_quantize_colwise_segment_padded(wd, i32_to_dev([N] * G), 32, "e2m1", capacity=G * N, check=True)
    dX = mxg.grouped_gemm_dgrad(dYq, Wt, d_splits, check=True)
    cap = mxg.mx_padded_rows_capacity(S, G, pad)
    dYt, _ = mxg.mx_quantize_colwise_segment_padded(dyd, d_splits, pad, "e2m1", capacity=cap, check=True)
    Xt, poff_d = mxg.mx_quantize_colwise_segment_padded(xd, d_splits, pad, "e2m1", capacity=cap, check=True)
    init = torch.randn((G, N, K), device="cuda:0", dtype=torch.float32) * 1e-3
    main_grad = init.clone()
    mxg.grouped_gemm_wgrad(dYt, Xt, d_splits, S, pad, out=main_grad, accumulate=True, check=True)
    del xd, dyd, wd
    rng = np.random.default_rng(8)
    off, picks = _sample_rows(rng, splits, 2)
    poff = oracle.padded_offsets(splits, pad)
    assert np.array_equal(poff_d.cpu().numpy(), poff)
    fwd, dgr = [], []
    for g, rows in picks[::3]:           # every third expert keeps the host work bounded
        cols = rng.integers(0, N, size=16)
        ks = rng.integers(0, K, size=16)
        Ad, _, _ = _deq(x[rows], "e2m1")
        Wd, _, _ = _deq(wt[g * N + cols], "e2m1")
        fwd.append((Y[torch.as_tensor(rows)][:, torch.as_tensor(cols)].float().cpu().numpy(), Ad @ Wd.T, g))
        dYd, _, _ = _deq(dy[rows], "e2m1")
        wcol = np.ascontiguousarray(wt[g * N:(g + 1) * N][:, ks].T)       # W^T rows k, quantized along N
        Wtd, _, _ = _deq(wcol, "e2m1")
        dgr.append((dX[torch.as_tensor(rows)][:, torch.as_tensor(ks)].float().cpu().numpy(), dYd @ Wtd.T, g))
    for name, items in (("fwd", fwd), ("dgrad", dgr)):
        rms = float(np.sqrt(np.mean(np.concatenate([r.ravel() for _, r, _ in items]) ** 2)))
        for got, ref, g in items:
            oracle.assert_gemm_close(got, ref, f"train {name} expert {g}", rms_ref=rms)
    # wgrad: sampled (n, k) of a few experts, accumulated onto the initial main_grad
    wg = []
    for g in [int(np.argmax(splits)), int(np.argmin(np.where(splits > 0, splits, 1 << 30))), 5]:
        m = int(splits[g])
        ns = rng.integers(0, N, size=8)
        ks = rng.integers(0, K, size=8)
        seg_dy = dy[off[g]: off[g] + m][:, ns]
        seg_x = x[off[g]: off[g] + m][:, ks]
        dd, ds, _ = oracle.quantize_mx_colwise_segment_padded(seg_dy, [m], pad, "e2m1")
        xd_, xs_, _ = oracle.quantize_mx_colwise_segment_padded(seg_x, [m], pad, "e2m1")
        dT = oracle.dequantize_mx(oracle.unpack_e2m1(dd), ds, "e2m1")
        xT = oracle.dequantize_mx(oracle.unpack_e2m1(xd_), xs_, "e2m1")
        ref = dT @ xT.T + init[g][torch.as_tensor(ns)][:, torch.as_tensor(ks)].cpu().numpy()
        got = main_grad[g][torch.as_tensor(ns)][:, torch.as_tensor(ks)].cpu().numpy()
        wg.append((got, ref, g))
    rms = float(np.sqrt(np.mean(np.concatenate([r.ravel() for _, r, _ in wg]) ** 2)))
    for got, ref, g in wg:
        oracle.assert_gemm_close(got, ref, f"train wgrad expert {g}", rms_ref=rms)


def test_blockwise_step_full_size():
    mxg = _mxg()
    from oracle.blockwise import transpose_bw_128x128
    w = synth.WORKLOADS["blockwise_fp8"]
    splits = w.splits()
    G, N, K, S = w.G, w.N, w.K, int(splits.sum())
    x = synth.normal_bf16(w.act_rng(0), (S, K))
    dy = synth.normal_bf16(w.act_rng(1), (S, N))
    wt = synth.normal_bf16(w.weight_rng(), (G * N, K))
    d_splits = i32_to_dev(splits)
    xd, dyd, wd = bf16_to_dev(x), bf16_to_dev(dy), bf16_to_dev(wt)
    Xq = mxg.bw_quantize_1x128(xd)
    Wq, WtQ = mxg.bw_quantize_128x128(wd)
    Y = mxg.bw_grouped_gemm_fwd(Xq, Wq, d_splits, N, check=True)
    dYq = mxg.bw_quantize_1x128(dyd)
    dX = mxg.bw_grouped_gemm_dgrad(dYq, WtQ, d_splits, check=True)
    dYt, _ = mxg.bw_quantize_colwise_padded(dyd, d_splits, check=True)
    Xt, _ = mxg.bw_quantize_colwise_padded(xd, d_splits, check=True)
    dW = mxg.bw_grouped_gemm_wgrad(dYt, Xt, d_splits, S, out_dtype=torch.bfloat16, check=True)
    del xd, dyd, wd
    rng = np.random.default_rng(9)
    off, picks = _sample_rows(rng, splits, 2)
    items = {"fwd": [], "dgrad": [], "wgrad": []}
    for g, rows in picks[::4]:
        # weight blocks needed: the 128-row block of each sampled column, all K
        nb = rng.integers(0, N // 128)
        cols = nb * 128 + rng.integers(0, 128, size=8)
        wblk = wt[g * N + nb * 128: g * N + nb * 128 + 128]             # one 128 x K row band
        wc, ws = oracle.quantize_bw_128x128(wblk.reshape(1, 128, K))
        Wd = oracle.dequantize_bw_128x128(wc, ws)[0]
        xc, xs = oracle.quantize_bw_1x128(x[rows])
        Ad = oracle.dequantize_bw_1x128(xc, xs)
        items["fwd"].append((Y[torch.as_tensor(rows)][:, torch.as_tensor(cols)].float().cpu().numpy(),
                             Ad @ Wd[cols - nb * 128].T, g))
        # dgrad: dX[row, k] needs W^T rows k over expert g's N columns (128x128 blocks)
        kb = rng.integers(0, K // 128)
        ks = kb * 128 + rng.integers(0, 128, size=8)
        wband = wt[g * N:(g + 1) * N][:, kb * 128: kb * 128 + 128]      # N x 128 column band
        wc2, ws2 = oracle.quantize_bw_128x128(np.ascontiguousarray(wband).reshape(1, N, 128))
        ct, st = transpose_bw_128x128(wc2, ws2)
        Wtd = oracle.dequantize_bw_128x128(ct, st)[0]                    # [128, N]
        dc, dsc = oracle.quantize_bw_1x128(dy[rows])
        dYd = oracle.dequantize_bw_1x128(dc, dsc)
        items["dgrad"].append((dX[torch.as_tensor(rows)][:, torch.as_tensor(ks)].float().cpu().numpy(),
                               dYd @ Wtd[ks - kb * 128].T, g))
        # wgrad: dW[g][n, k] over the expert's tokens, column-wise blocks of 128
        m = int(splits[g])
        ns = rng.integers(0, N, size=6)
        kk = rng.integers(0, K, size=6)
        dc_, ds_, _ = oracle.quantize_bw_colwise_padded(dy[off[g]: off[g] + m][:, ns], [m])
        xc_, xs_, _ = oracle.quantize_bw_colwise_padded(x[off[g]: off[g] + m][:, kk], [m])
        ref = oracle.dequantize_bw_1x128(dc_, ds_) @ oracle.dequantize_bw_1x128(xc_, xs_).T
        items["wgrad"].append((dW[g][torch.as_tensor(ns)][:, torch.as_tensor(kk)].float().cpu().numpy(), ref, g))
    for name, its in items.items():
        rms = float(np.sqrt(np.mean(np.concatenate([r.ravel() for _, r, _ in its]) ** 2)))
        for got, ref, g in its:
            oracle.assert_gemm_close(got, ref, f"blockwise {name} expert {g}", rms_ref=rms)
