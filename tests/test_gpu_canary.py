"""Guard bands around every output of every entry point (a stand-in for a
memory sanitizer).  Each output and each workspace is placed, through the C
ABI, between 4 KB bands of a sentinel byte inside a larger buffer, and
strided outputs get padding between their rows; after the call (and the
status check) every band and every padding byte must still hold the
sentinel.  Small cases with ragged and empty experts, all passes, element
kinds and output types, both GEMM kernels (CTA pairs and one SM)."""

import ctypes

import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu

from gpu_util import bf16_to_dev, i32_to_dev  # noqa: E402

BAND = 4096
SENT = 0xA5
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()


def _mxg():
    import fp8_bf16_mxfp4_gb300 as mxg
    return mxg


def _lib():
    return _mxg()._lib.load()


class Guard:
    """`rows` rows of `width` bytes at a stride of `ld` bytes, between bands."""

    def __init__(self, rows, width, ld=None):
        self.rows, self.width = int(rows), int(width)
        self.ld = int(ld if ld is not None else width)
        self.n = max(self.rows * self.ld, 1)
        total = BAND + ((self.n + 255) // 256) * 256 + BAND
        self.buf = torch.full((total,), SENT, dtype=torch.uint8, device=DEV)

    @property
    def p(self):
        return ctypes.c_void_p(self.buf.data_ptr() + BAND)

    def tensor(self, dtype, shape):
        return self.buf[BAND: BAND + self.n].view(dtype).view(shape)

    def check(self, what):
        torch.cuda.synchronize()
        b = self.buf.cpu().numpy()
        head, tail = b[:BAND], b[BAND + self.n:]
        assert (head == SENT).all(), f"{what}: bytes written before the output"
        assert (tail == SENT).all(), f"{what}: byte {self.n + int(np.argmax(tail != SENT))} past the output written"
        if self.ld > self.width and self.rows > 0:
            pad = b[BAND: BAND + self.n].reshape(self.rows, self.ld)[:, self.width:]
            assert (pad == SENT).all(), f"{what}: padding between rows written"


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _st():
    return torch.zeros(1, dtype=torch.int32, device=DEV)


def _ok(code, st, what):
    assert code == 0, f"{what}: status {code}"
    _mxg().check_status(st)


SPLITS = [37, 0, 130, 93, 1]
S = sum(SPLITS)


def _x(cols, seed=0):
    return bf16_to_dev(synth.normal_bf16(np.random.default_rng(seed), (S, cols), outlier_frac=0.01))


def _cw(elem, n):
    return n // 2 if elem == "e2m1" else n


ELEMS = {"e2m1": 1, "e4m3": 2}


@pytest.mark.parametrize("elem", ["e2m1", "e4m3"])
def test_mx_quantizers_stay_inside_their_outputs(elem):
    lib, C, G, pad = _lib(), 256, len(SPLITS), 32
    x, sp = _x(C), i32_to_dev(SPLITS)
    e = ELEMS[elem]
    # row-wise, plain scales, strided outputs
    q = Guard(S, _cw(elem, C), _cw(elem, C) + 16)
    s = Guard(S, C // 32, C // 32 + 3)
    assert lib.mx_quantize_rowwise(x.data_ptr(), S, C, C, e, q.p, q.ld, s.p, s.ld, _stream()) == 0
    q.check("rowwise q"), s.check("rowwise s")
    # row-wise, packed scales
    nb = lib.mx_packed_scale_bytes(S, C, G)
    q, sp_ = Guard(S, _cw(elem, C), _cw(elem, C) + 32), Guard(1, nb)
    st = _st()
    _ok(lib.mx_quantize_rowwise_packed(x.data_ptr(), S, C, C, e, q.p, q.ld, sp_.p, nb, sp.data_ptr(), G,
                                       st.data_ptr(), _stream()), st, "rowwise packed")
    q.check("rowwise packed q"), sp_.check("rowwise packed scales")
    # column-wise segment padded, plain and packed, and the dual quantizer
    cap = lib.mx_padded_rows_capacity(S, G, pad)
    qT = Guard(C, _cw(elem, cap), _cw(elem, cap) + 16)
    sT = Guard(C, cap // 32, cap // 32 + 5)
    po = Guard(1, 8 * (G + 1))
    st = _st()
    _ok(lib.mx_quantize_colwise_segment_padded(x.data_ptr(), S, C, C, sp.data_ptr(), G, pad, e, qT.p, qT.ld,
                                               sT.p, sT.ld, cap, po.p, st.data_ptr(), _stream()), st, "colwise")
    qT.check("colwise qT"), sT.check("colwise sT"), po.check("colwise pad offsets")
    nbc = lib.mx_packed_colwise_scale_bytes(C, cap, G)
    qT, sTp, po = Guard(C, _cw(elem, cap), _cw(elem, cap) + 16), Guard(1, nbc), Guard(1, 8 * (G + 1))
    st = _st()
    _ok(lib.mx_quantize_colwise_segment_padded_packed(x.data_ptr(), S, C, C, sp.data_ptr(), G, pad, e, qT.p,
                                                      qT.ld, sTp.p, nbc, cap, po.p, st.data_ptr(), _stream()),
        st, "colwise packed")
    qT.check("colwise packed qT"), sTp.check("colwise packed scales"), po.check("colwise packed pad offsets")
    q, s = Guard(S, _cw(elem, C), _cw(elem, C) + 16), Guard(S, C // 32, C // 32 + 1)
    qT, sT, po = Guard(C, _cw(elem, cap), _cw(elem, cap) + 16), Guard(C, cap // 32, cap // 32 + 2), Guard(1, 8 * (G + 1))
    st = _st()
    _ok(lib.mx_quantize_dual_segment_padded(x.data_ptr(), S, C, C, sp.data_ptr(), G, pad, e, q.p, q.ld, s.p, s.ld,
                                            qT.p, qT.ld, sT.p, sT.ld, cap, po.p, st.data_ptr(), _stream()),
        st, "dual")
    for g_, n_ in ((q, "q"), (s, "s"), (qT, "qT"), (sT, "sT"), (po, "pad offsets")):
        g_.check(f"dual {n_}")


def test_blockwise_quantizers_stay_inside_their_outputs():
    lib, C, G = _lib(), 256, len(SPLITS)
    x, sp = _x(C, 1), i32_to_dev(SPLITS)
    w = bf16_to_dev(synth.normal_bf16(np.random.default_rng(2), (256, 384)))
    cap = lib.mx_padded_rows_capacity(S, G, 128)
    # fp32 scales
    q, s = Guard(S, C, C + 8), Guard(C // 128, 4 * S, 4 * (S + 3))
    assert lib.bw_quantize_1x128(x.data_ptr(), S, C, C, q.p, q.ld, s.p, S + 3, _stream()) == 0
    q.check("1x128 q"), s.check("1x128 s")
    q, s = Guard(256, 384, 384 + 16), Guard(1, 4 * 2 * 3)
    qT, sT = Guard(384, 256, 256 + 16), Guard(1, 4 * 3 * 2)
    assert lib.bw_quantize_128x128(w.data_ptr(), 256, 384, 384, q.p, q.ld, s.p, qT.p, qT.ld, sT.p, _stream()) == 0
    for g_, n_ in ((q, "q"), (s, "s"), (qT, "qT"), (sT, "sT")):
        g_.check(f"128x128 {n_}")
    qT, sT, po = Guard(C, cap, cap + 16), Guard(cap // 128, 4 * C, 4 * (C + 5)), Guard(1, 8 * (G + 1))
    st = _st()
    _ok(lib.bw_quantize_colwise_padded(x.data_ptr(), S, C, C, sp.data_ptr(), G, qT.p, qT.ld, sT.p, C + 5, cap,
                                       po.p, st.data_ptr(), _stream()), st, "bw colwise")
    qT.check("bw colwise qT"), sT.check("bw colwise sT"), po.check("bw colwise pad offsets")
    q, s = Guard(S, C, C + 8), Guard(C // 128, 4 * S, 4 * (S + 1))
    qT, sT, po = Guard(C, cap, cap + 16), Guard(cap // 128, 4 * C, 4 * (C + 1)), Guard(1, 8 * (G + 1))
    st = _st()
    _ok(lib.bw_quantize_dual_padded(x.data_ptr(), S, C, C, sp.data_ptr(), G, q.p, q.ld, s.p, S + 1, qT.p, qT.ld,
                                    sT.p, C + 1, cap, po.p, st.data_ptr(), _stream()), st, "bw dual")
    for g_, n_ in ((q, "q"), (s, "s"), (qT, "qT"), (sT, "sT"), (po, "pad offsets")):
        g_.check(f"bw dual {n_}")
    # power-of-two scales (UE8M0 bytes)
    q, s = Guard(S, C, C + 8), Guard(S, C // 32, C // 32 + 4)
    assert lib.bw_quantize_1x128_pow2(x.data_ptr(), S, C, C, q.p, q.ld, s.p, s.ld, _stream()) == 0
    q.check("1x128 pow2 q"), s.check("1x128 pow2 s")
    q, s = Guard(256, 384, 384 + 16), Guard(256, 12, 16)
    qT, sT = Guard(384, 256, 256 + 16), Guard(384, 8, 12)
    assert lib.bw_quantize_128x128_pow2(w.data_ptr(), 256, 384, 384, q.p, q.ld, s.p, s.ld, qT.p, qT.ld, sT.p,
                                        sT.ld, _stream()) == 0
    for g_, n_ in ((q, "q"), (s, "s"), (qT, "qT"), (sT, "sT")):
        g_.check(f"128x128 pow2 {n_}")
    qT, sT, po = Guard(C, cap, cap + 16), Guard(C, cap // 32, cap // 32 + 4), Guard(1, 8 * (G + 1))
    st = _st()
    _ok(lib.bw_quantize_colwise_padded_pow2(x.data_ptr(), S, C, C, sp.data_ptr(), G, qT.p, qT.ld, sT.p, sT.ld,
                                            cap, po.p, st.data_ptr(), _stream()), st, "bw colwise pow2")
    qT.check("bw colwise pow2 qT"), sT.check("bw colwise pow2 sT"), po.check("bw colwise pow2 pad offsets")


@pytest.fixture(params=[2, 1], ids=["pair", "onesm"])
def cta_group(request):
    prev = _mxg().set_gemm_cta_group(request.param)
    yield request.param
    _mxg().set_gemm_cta_group(prev)


def _mx_operands(kind, N, K, packed):
    mxg = _mxg()
    ea, eb = {"mxfp4": ("e2m1", "e2m1"), "mxfp8": ("e4m3", "e4m3"), "a8w4": ("e4m3", "e2m1")}[kind]
    G = len(SPLITS)
    sp = i32_to_dev(SPLITS)
    x, dy = _x(K, 3), _x(N, 4)
    w = bf16_to_dev(synth.normal_bf16(np.random.default_rng(5), (G * N, K)))
    if packed:
        A = mxg.mx_quantize_rowwise_packed(x, ea, m_splits=sp, check=True)
        W = mxg.mx_quantize_rowwise_packed(w, eb, groups=G)
        dY = mxg.mx_quantize_rowwise_packed(dy, ea, m_splits=sp, check=True)
    else:
        A, W, dY = mxg.mx_quantize_rowwise(x, ea), mxg.mx_quantize_rowwise(w, eb), mxg.mx_quantize_rowwise(dy, ea)
    Wt, _ = mxg.mx_quantize_colwise_segment_padded(w, i32_to_dev([N] * G), 32, ea, capacity=G * N, check=True,
                                                   packed=packed)
    dYt, _ = mxg.mx_quantize_colwise_segment_padded(dy, sp, 32, ea, check=True, packed=packed)
    Xt, _ = mxg.mx_quantize_colwise_segment_padded(x, sp, 32, ea, check=True, packed=packed)
    return sp, A, W, dY, Wt, dYt, Xt


@pytest.mark.parametrize("kind", ["mxfp4", "mxfp8", "a8w4"])
@pytest.mark.parametrize("packed", [False, True], ids=["plain", "packed"])
def test_mx_gemms_stay_inside_their_outputs(cta_group, kind, packed):
    lib, mxg = _lib(), _mxg()
    N, K, G = 160, 256, len(SPLITS)
    sp, A, W, dY, Wt, dYt, Xt = _mx_operands(kind, N, K, packed)
    for dt, esz in ((1, 2), (2, 4)):
        out = Guard(S, N * esz, (N + 32) * esz)
        need = lib.mxg_gemm_workspace_size(0, G, S, N, K, 32)
        ws, st = Guard(1, need), _st()
        a, w = A.c(), W.c()
        _ok(lib.grouped_gemm_fwd(ctypes.byref(a), ctypes.byref(w), sp.data_ptr(), G, N, out.p, N + 32, dt, ws.p, need,
                                 st.data_ptr(), _stream()), st, f"fwd {kind}")
        out.check(f"fwd {kind} out"), ws.check(f"fwd {kind} workspace")
        if kind == "a8w4":
            continue
        out = Guard(S, K * esz, (K + 32) * esz)
        need = lib.mxg_gemm_workspace_size(1, G, S, N, K, 32)
        ws, st = Guard(1, need), _st()
        d, wt = dY.c(), Wt.c()
        _ok(lib.grouped_gemm_dgrad(ctypes.byref(d), ctypes.byref(wt), sp.data_ptr(), G, out.p, K + 32, dt, ws.p,
                                   need, st.data_ptr(), _stream()), st, f"dgrad {kind}")
        out.check(f"dgrad {kind} out"), ws.check(f"dgrad {kind} workspace")
        for acc in ((0, 1) if dt == 2 else (0,)):
            out = Guard(G, N * K * esz)
            if acc:
                out.tensor(torch.float32, (G, N, K)).zero_()
            cap = dYt.cols
            need = lib.mxg_gemm_workspace_size(2, G, cap, N, K, 32)
            ws, st = Guard(1, need), _st()
            d, xt = dYt.c(), Xt.c()
            _ok(lib.grouped_gemm_wgrad(ctypes.byref(d), ctypes.byref(xt), sp.data_ptr(), G, S, 32, out.p, dt, acc,
                                       ws.p, need, st.data_ptr(), _stream()), st, f"wgrad {kind}")
            out.check(f"wgrad {kind} out (acc {acc})"), ws.check(f"wgrad {kind} workspace")
    if kind != "a8w4":   # the dense entry point: one expert of all rows
        out = Guard(S, N * 2, (N + 32) * 2)
        need = lib.mxg_gemm_workspace_size(0, 1, S, N, K, 32)
        ws, st = Guard(1, need), _st()
        Wd = mxg.mx_quantize_rowwise_packed(bf16_to_dev(synth.normal_bf16(np.random.default_rng(6), (N, K))),
                                            A.elem, groups=1) if packed else \
            mxg.mx_quantize_rowwise(bf16_to_dev(synth.normal_bf16(np.random.default_rng(6), (N, K))), A.elem)
        Ad = mxg.mx_quantize_rowwise_packed(_x(K, 3), A.elem, m_splits=i32_to_dev([S]), check=True) if packed \
            else A
        a, b = Ad.c(), Wd.c()
        _ok(lib.mx_gemm_dense(ctypes.byref(a), ctypes.byref(b), out.p, N + 32, 1, ws.p, need, st.data_ptr(),
                              _stream()), st, "dense")
        out.check("dense out"), ws.check("dense workspace")


def test_blockwise_gemms_stay_inside_their_outputs(cta_group):
    lib, mxg = _lib(), _mxg()
    N, K, G = 256, 384, len(SPLITS)
    sp = i32_to_dev(SPLITS)
    x, dy = _x(K, 7), _x(N, 8)
    w = bf16_to_dev(synth.normal_bf16(np.random.default_rng(9), (G * N, K)))
    A, dY = mxg.bw_quantize_1x128(x), mxg.bw_quantize_1x128(dy)
    W, Wt = mxg.bw_quantize_128x128(w)
    dYt, _ = mxg.bw_quantize_colwise_padded(dy, sp, check=True)
    Xt, _ = mxg.bw_quantize_colwise_padded(x, sp, check=True)
    need = lib.bw_gemm_workspace_size(G)
    for dt, esz in ((1, 2), (2, 4)):
        out, ws, st = Guard(S, N * esz, (N + 32) * esz), Guard(1, need), _st()
        a, w_ = A.c(), W.c()
        _ok(lib.bw_grouped_gemm_fwd(ctypes.byref(a), ctypes.byref(w_), sp.data_ptr(), G, N, out.p, N + 32, dt, ws.p,
                                    need, st.data_ptr(), _stream()), st, "bw fwd")
        out.check("bw fwd out"), ws.check("bw fwd workspace")
        out, ws, st = Guard(S, K * esz, (K + 32) * esz), Guard(1, need), _st()
        d, wt = dY.c(), Wt.c()
        _ok(lib.bw_grouped_gemm_dgrad(ctypes.byref(d), ctypes.byref(wt), sp.data_ptr(), G, out.p, K + 32, dt, ws.p,
                                      need, st.data_ptr(), _stream()), st, "bw dgrad")
        out.check("bw dgrad out"), ws.check("bw dgrad workspace")
        for acc in ((0, 1) if dt == 2 else (0,)):
            out, ws, st = Guard(G, N * K * esz), Guard(1, need), _st()
            if acc:
                out.tensor(torch.float32, (G, N, K)).zero_()
            d, xt = dYt.c(), Xt.c()
            _ok(lib.bw_grouped_gemm_wgrad(ctypes.byref(d), ctypes.byref(xt), sp.data_ptr(), G, S, out.p, dt, acc,
                                          ws.p, need, st.data_ptr(), _stream()), st, "bw wgrad")
            out.check(f"bw wgrad out (acc {acc})"), ws.check("bw wgrad workspace")
