"""The allocation-free forward entry point (grouped_gemm_fwd_noalloc).

It is for callers that may not allocate device memory when the GEMM runs
(plugins whose device memory is budgeted by their host framework,
latency-critical paths that never enter an allocator); its scratch is a fixed
32 MiB array inside the library.  Checked through the C ABI against the
regular grouped_gemm_fwd on calls in a row: a small problem, a larger one,
then the small one again, so that stale plan or packed-scale bytes left by a
different problem in the shared scratch would show.  The tolerance is the one
the GEMM parity tests use.  This file is collected last so that a
stop-at-first-failure run has already run every other test; it also passes
alone in a fresh process."""

import ctypes

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


def _problem(seed, splits, N, K, ea, eb):
    import fp8_bf16_mxfp4_gb300 as mxg
    rng = np.random.default_rng(seed)
    S, G = int(sum(splits)), len(splits)
    A = mxg.mx_quantize_rowwise(bf16_to_dev(synth.normal_bf16(rng, (S, K), outlier_frac=0.01)), ea)
    W = mxg.mx_quantize_rowwise(bf16_to_dev(synth.normal_bf16(rng, (G * N, K), outlier_frac=0.01)), eb)
    return A, W, i32_to_dev(splits)


def _noalloc(A, W, d_splits, N, out, status):
    import fp8_bf16_mxfp4_gb300 as mxg
    lib = mxg._lib.load()
    a, w = A.c(), W.c()
    return lib.grouped_gemm_fwd_noalloc(ctypes.byref(a), ctypes.byref(w), mxg._ptr(d_splits),
                                        d_splits.numel(), N, mxg._ptr(out), out.stride(0), 1,
                                        mxg._ptr(status), mxg._stream(out.device))


def test_noalloc_matches_regular_forward_twice():
    import fp8_bf16_mxfp4_gb300 as mxg
    small = (1, [300, 0, 129, 77], 512, 1024, "e2m1", "e2m1")
    cases = [small, (2, [1218, 854, 819, 5], 1024, 4096, "e4m3", "e2m1"), small]
    for seed, splits, N, K, ea, eb in cases:
        A, W, d_splits = _problem(seed, splits, N, K, ea, eb)
        st = torch.zeros(1, dtype=torch.int32, device="cuda:0")
        ref = mxg.grouped_gemm_fwd(A, W, d_splits, N, status=st, check=True)
        out = torch.full_like(ref, float("nan"))
        assert _noalloc(A, W, d_splits, N, out, st) == 0
        mxg.check_status(st)
        oracle.assert_gemm_close(out.float().cpu().numpy(), ref.float().cpu().numpy(),
                                 f"noalloc vs grouped_gemm_fwd (seed {seed})")


def _operand_c(buf, rows, cols):
    """A well-formed E2M1 operand description (plain scales) whose pointers
    lie in a small real buffer: the calls below reject the problem on the
    host before anything could read it."""
    import fp8_bf16_mxfp4_gb300 as mxg
    return mxg._lib.MxOperandC(buf.data_ptr(), buf.data_ptr(), rows, cols, cols // 2, cols // 32, 1, 0)


def test_noalloc_rejects_problems_beyond_its_scratch():
    import fp8_bf16_mxfp4_gb300 as mxg
    lib = mxg._lib.load()
    G, N, K, S = 64, 4096, 8192, 1024      # packed weight scales alone need 64 MiB
    assert mxg.gemm_workspace_size("fwd", G, S, N, K) > 32 << 20
    buf = torch.zeros(1 << 16, dtype=torch.uint8, device="cuda:0")
    a, w = _operand_c(buf, S, K), _operand_c(buf, G * N, K)
    out = torch.empty((S, N), dtype=torch.bfloat16, device="cuda:0")
    st = torch.zeros(1, dtype=torch.int32, device="cuda:0")
    d_splits = i32_to_dev([S // G] * G)
    stream = mxg._stream(out.device)
    assert lib.grouped_gemm_fwd_noalloc(ctypes.byref(a), ctypes.byref(w), mxg._ptr(d_splits), G, N, mxg._ptr(out),
                                        N, 1, mxg._ptr(st), stream) == 9    # MXG_ERR_WORKSPACE
    # a malformed problem gets the status the regular forward gives it, before the size test
    ws = torch.empty(256, dtype=torch.uint8, device="cuda:0")
    bad_N = N - 16                                                   # N % 32 != 0
    reg = lib.grouped_gemm_fwd(ctypes.byref(a), ctypes.byref(w), mxg._ptr(d_splits), G, bad_N, mxg._ptr(out),
                               N, 1, mxg._ptr(ws), ws.numel(), mxg._ptr(st), stream)
    assert reg == 2                                                  # MXG_ERR_SHAPE
    assert lib.grouped_gemm_fwd_noalloc(ctypes.byref(a), ctypes.byref(w), mxg._ptr(d_splits), G, bad_N,
                                        mxg._ptr(out), N, 1, mxg._ptr(st), stream) == reg
    mxg.check_status(st)                                             # nothing was enqueued
