"""C-ABI checks that need no GPU: the library loads, exports every function
declared in include/*.h, and its host-side argument checks return the
documented codes without touching the device (fake, never dereferenced
pointers are used; every call here fails before any CUDA call)."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from fp8_bf16_mxfp4_gb300 import build, _lib
    build.build()
    return _lib.load()


def header_functions():
    names = []
    inc = os.path.join(ROOT, "include")
    for f in sorted(os.listdir(inc)):
        if not f.endswith(".h"):
            continue
        txt = open(os.path.join(inc, f)).read()
        txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
        txt = re.sub(r"//[^\n]*", "", txt)
        for m in re.finditer(r"^[A-Za-z_][\w \*]*?\b([a-z_][a-z0-9_]*)\s*\(", txt, flags=re.M):
            name = m.group(1)
            if name not in ("if", "sizeof"):
                names.append(name)
    return sorted(set(names))


def test_header_declares_the_documented_entry_points():
    names = header_functions()
    for must in ("mx_quantize_rowwise", "mx_quantize_colwise_segment_padded", "grouped_gemm_fwd",
                 "grouped_gemm_dgrad", "grouped_gemm_wgrad", "mxg_check_status"):
        assert must in names


def test_every_declared_symbol_is_exported(lib):
    from fp8_bf16_mxfp4_gb300 import _lib
    names = header_functions()
    for n in names:
        assert hasattr(lib, n), f"{n} declared but not exported"
    assert set(names) == set(_lib.SIGNATURES), "binding signatures out of sync with the header"


def test_pure_host_functions(lib):
    assert lib.mxg_version() == 200
    assert lib.mx_padded_rows_capacity(131072, 32, 32) == ((131072 + 32 * 31) // 32) * 32
    assert lib.mx_padded_rows_capacity(3, 8, 32) == 96
    assert lib.mx_padded_rows_capacity(0, 4, 128) == 0
    assert lib.mx_padded_rows_capacity(-1, 4, 32) == -1
    assert lib.mxg_status_string(0) == b"ok"
    assert b"m_splits" in lib.mxg_status_string(4)
    old = lib.mxg_get_wait_timeout_ns()
    lib.mxg_set_wait_timeout_ns(12345)
    assert lib.mxg_get_wait_timeout_ns() == 12345
    lib.mxg_set_wait_timeout_ns(old)
    prev = lib.mxg_get_gemm_cta_group()
    assert prev == 2                                      # CTA pairs by default
    assert lib.mxg_set_gemm_cta_group(1) == 0 and lib.mxg_get_gemm_cta_group() == 1
    assert lib.mxg_set_gemm_cta_group(3) == 2 and lib.mxg_get_gemm_cta_group() == 1  # rejected, unchanged
    assert lib.mxg_set_gemm_cta_group(0) == 2
    assert lib.mxg_set_gemm_cta_group(prev) == 0
    assert lib.mxg_gemm_workspace_size(0, 0, 10, 32, 32, 32) == 0      # G < 1
    assert lib.mxg_gemm_workspace_size(2, 4, 1024, 256, 512, 48) == 0  # pad % 32
    assert lib.mxg_gemm_workspace_size(0, 4, 512, 256, 512, 32) > 0


FAKE = 0x10000  # 16-byte aligned, never dereferenced


def test_quantize_host_checks(lib):
    vp = ctypes.c_void_p
    q = lib.mx_quantize_rowwise
    assert q(None, 4, 64, 64, 1, vp(FAKE), 32, vp(FAKE), 2, None) == 1           # NULL x
    assert q(vp(FAKE), 4, 48, 64, 1, vp(FAKE), 32, vp(FAKE), 2, None) == 2       # cols % 32
    assert q(vp(FAKE), 4, 64, 32, 1, vp(FAKE), 32, vp(FAKE), 2, None) == 2       # ld_x < cols
    assert q(vp(FAKE), 4, 64, 64, 3, vp(FAKE), 32, vp(FAKE), 2, None) == 5       # bad elem
    assert q(vp(FAKE), 4, 64, 64, 3 | 0x100, vp(FAKE), 32, vp(FAKE), 2, None) == 5  # bad elem with the rule flag
    assert q(vp(FAKE), 4, 64, 64, 1 | 0x200, vp(FAKE), 32, vp(FAKE), 2, None) == 5  # unknown flag
    assert q(vp(FAKE + 2), 4, 64, 64, 1 | 0x100, vp(FAKE), 32, vp(FAKE), 2, None) == 3  # flag accepted, x misaligned
    assert q(vp(FAKE + 2), 4, 64, 64, 1, vp(FAKE), 32, vp(FAKE), 2, None) == 3   # x misaligned
    assert q(vp(FAKE), 4, 64, 68, 1, vp(FAKE), 32, vp(FAKE), 2, None) == 3       # ld_x % 8
    assert q(vp(FAKE), 4, 64, 64, 1, vp(FAKE + 4), 32, vp(FAKE), 2, None) == 3   # q not 16-B aligned
    assert q(vp(FAKE), 4, 64, 64, 1, vp(FAKE), 36, vp(FAKE), 2, None) == 3       # ld_q % 16
    c = lib.mx_quantize_colwise_segment_padded
    args = [vp(FAKE), 64, 64, 64, vp(FAKE), 4, 32, 1, vp(FAKE), 96, vp(FAKE), 4, 192, vp(FAKE),
            vp(FAKE), None]
    bad = list(args); bad[14] = None
    assert c(*bad) == 1                                                           # NULL status
    bad = list(args); bad[5] = 0
    assert c(*bad) == 2                                                           # G < 1
    bad = list(args); bad[5] = 513
    assert c(*bad) == 2                                                           # G > 512
    bad = list(args); bad[6] = 48
    assert c(*bad) == 2                                                           # pad % 32
    bad = list(args); bad[12] = 100
    assert c(*bad) == 2                                                           # capacity % 32
    d = lib.mx_quantize_dual_segment_padded
    #        x        rows cols ld_x splits    G  pad elem q        ld_q s        ld_s qT       ld_qT sT
    dargs = [vp(FAKE), 64, 64, 64, vp(FAKE), 4, 32, 1, vp(FAKE), 32, vp(FAKE), 2, vp(FAKE), 96, vp(FAKE),
             6, 192, vp(FAKE), vp(FAKE), None]
    bad = list(dargs); bad[18] = None
    assert d(*bad) == 1                                                           # NULL status
    bad = list(dargs); bad[8] = None
    assert d(*bad) == 1                                                           # NULL row-wise codes
    bad = list(dargs); bad[9] = 16
    assert d(*bad) == 2                                                           # ld_q < cols/2
    bad = list(dargs); bad[9] = 36
    assert d(*bad) == 3                                                           # ld_q % 16
    bad = list(dargs); bad[8] = vp(FAKE + 4)
    assert d(*bad) == 3                                                           # q misaligned
    bad = list(dargs); bad[15] = 4
    assert d(*bad) == 2                                                           # ld_sT < capacity/32
    bad = list(dargs); bad[7] = 3
    assert d(*bad) == 5                                                           # bad elem


def _op(rows, cols, elem, data=FAKE, ld=None, scale_ld=None):
    from fp8_bf16_mxfp4_gb300 import _lib
    cb = cols // 2 if elem == 1 else cols
    return _lib.MxOperandC(data, FAKE, rows, cols, ld if ld is not None else cb,
                           scale_ld if scale_ld is not None else cols // 32, elem, 0)


def test_gemm_host_checks(lib):
    vp = ctypes.c_void_p
    f = lib.grouped_gemm_fwd
    ws = 1 << 30
    A, W = _op(512, 512, 1), _op(4 * 256, 512, 1)
    call = lambda A, W, G=4, N=256, ldo=256, dt=1, ws_bytes=ws, status=vp(FAKE): f(
        ctypes.byref(A), ctypes.byref(W), vp(FAKE), G, N, vp(FAKE), ldo, dt, vp(FAKE), ws_bytes, status, None)
    assert call(A, W, status=None) == 1                       # NULL status
    assert call(A, _op(4 * 256, 480, 1)) == 2                  # K mismatch
    assert call(A, _op(3 * 256, 512, 1)) == 2                  # W rows != G*N
    assert call(A, W, G=0) == 2 and call(A, W, G=513) == 2     # G range
    assert call(A, W, N=250, ldo=256) == 2                     # N % 32
    assert call(A, W, ldo=200) == 2                            # ld_out < N
    assert call(A, W, dt=3) == 5                               # bad out dtype
    assert call(_op(512, 512, 1, data=FAKE + 8), W) == 3       # misaligned data
    assert call(A, W, ws_bytes=16) == 9                        # workspace too small
    assert call(_op(512, 512, 1), _op(1024, 512, 2)) == 5      # E2M1 x E4M3 not provided
    assert call(_op(512, 96, 2), _op(1024, 96, 1)) == 2        # a8w4 needs K % 128
    assert call(_op(512, 512, 1 | 0x100), W) == 5                # the rule flag is not an operand format
    bad = _op(512, 512, 1); bad.scale_layout = 7
    assert call(bad, W) == 5                                   # unknown scale layout
    pk = _op(512, 512, 1); pk.scale_layout = 1; pk.scale = FAKE + 4
    assert call(pk, W) == 3                                    # packed scales not 16-byte aligned
    dense = lib.mx_gemm_dense
    assert dense(ctypes.byref(A), None, vp(FAKE), 256, 1, vp(FAKE), ws, vp(FAKE), None) == 1   # NULL B
    assert dense(ctypes.byref(A), ctypes.byref(_op(256, 512, 1)), vp(FAKE), 256, 1, vp(FAKE), ws, None,
                 None) == 1                                    # NULL status
    assert dense(ctypes.byref(A), ctypes.byref(_op(256, 480, 1)), vp(FAKE), 256, 1, vp(FAKE), ws, vp(FAKE),
                 None) == 2                                    # K mismatch
    assert dense(ctypes.byref(A), ctypes.byref(_op(250, 512, 1)), vp(FAKE), 256, 1, vp(FAKE), ws, vp(FAKE),
                 None) == 2                                    # N % 32
    assert dense(ctypes.byref(A), ctypes.byref(_op(256, 512, 1)), vp(FAKE), 256, 1, vp(FAKE), 16, vp(FAKE),
                 None) == 9                                    # workspace too small
    d = lib.grouped_gemm_dgrad
    dY, Wt = _op(512, 256, 2), _op(512, 4 * 256, 1)
    assert d(ctypes.byref(dY), ctypes.byref(Wt), vp(FAKE), 4, vp(FAKE), 512, 1, vp(FAKE), ws,
             vp(FAKE), None) == 5                              # a8w4 is forward-only
    w = lib.grouped_gemm_wgrad
    dYt, Xt = _op(256, 1024, 1), _op(512, 1024, 1)
    assert w(ctypes.byref(dYt), ctypes.byref(Xt), vp(FAKE), 4, 900, 32, vp(FAKE), 1, 1, vp(FAKE),
             ws, vp(FAKE), None) == 5                          # accumulate needs FP32
    assert w(ctypes.byref(dYt), ctypes.byref(Xt), vp(FAKE), 4, 900, 48, vp(FAKE), 2, 1, vp(FAKE),
             ws, vp(FAKE), None) == 2                          # pad % 32
    dYtp = _op(256, 1024, 1); dYtp.scale_layout = 1; dYtp.scale = FAKE + 8
    assert w(ctypes.byref(dYtp), ctypes.byref(Xt), vp(FAKE), 4, 900, 32, vp(FAKE), 2, 1, vp(FAKE),
             ws, vp(FAKE), None) == 3                          # packed wgrad scales must be 16-byte aligned


def test_packed_colwise_host_checks(lib):
    vp = ctypes.c_void_p
    assert lib.mx_packed_colwise_scale_bytes(2048, 4096, 8) == (32 + 8) * 16 * 512
    assert lib.mx_packed_colwise_scale_bytes(160, 0, 1) == 1 * 2 * 512
    assert lib.mx_packed_colwise_scale_bytes(100, 64, 1) == -1 and lib.mx_packed_colwise_scale_bytes(64, 64, 0) == -1
    f = lib.mx_quantize_colwise_segment_padded_packed
    need = lib.mx_packed_colwise_scale_bytes(64, 96, 4)
    #       x        rows cols ld_x splits    G  pad elem q        ld_q s        bytes cap poff      status
    args = [vp(FAKE), 64, 64, 64, vp(FAKE), 4, 32, 1, vp(FAKE), 48, vp(FAKE), need, 96, vp(FAKE), vp(FAKE), None]
    bad = list(args); bad[11] = need - 1
    assert f(*bad) == 2                                                   # packed buffer too small
    bad = list(args); bad[10] = vp(FAKE + 4)
    assert f(*bad) == 3                                                   # packed scales misaligned
    bad = list(args); bad[14] = None
    assert f(*bad) == 1                                                   # NULL status
    bad = list(args); bad[6] = 48
    assert f(*bad) == 2                                                   # pad % 32
    bad = list(args); bad[7] = 4
    assert f(*bad) == 5                                                   # bad elem


def test_packed_quantize_host_checks(lib):
    vp = ctypes.c_void_p
    assert lib.mx_packed_scale_bytes(1000, 160, 4) == 2 * ((1000 + 4 * 127) // 128) * 512
    assert lib.mx_packed_scale_bytes(3 * 256, 512, 3) == 4 * 8 * 512       # bound, not the 6 exact tiles
    assert lib.mx_packed_scale_bytes(2, 64, 8) == 1 * ((2 + 2 * 127) // 128) * 512
    assert lib.mx_packed_scale_bytes(0, 64, 8) == 0
    assert lib.mx_packed_scale_bytes(10, 48, 8) == -1 and lib.mx_packed_scale_bytes(10, 64, 0) == -1
    f = lib.mx_quantize_rowwise_packed
    need = lib.mx_packed_scale_bytes(768, 512, 3)
    #        x         rows cols ld_x elem q        ld_q s         bytes splits G  status     stream
    args = [vp(FAKE), 768, 512, 512, 1, vp(FAKE), 256, vp(FAKE), need, None, 3, vp(FAKE), None]
    bad = list(args); bad[8] = need - 1
    assert f(*bad) == 2                                                   # packed buffer too small
    bad = list(args); bad[10] = 5
    assert f(*bad) == 2                                                   # rows % G with equal segments
    bad = list(args); bad[9] = vp(FAKE); bad[11] = None
    assert f(*bad) == 1                                                   # splits without a status word
    bad = list(args); bad[7] = vp(FAKE + 8)
    assert f(*bad) == 3                                                   # packed scales misaligned
    bad = list(args); bad[4] = 3
    assert f(*bad) == 5                                                   # bad elem
    bad = list(args); bad[10] = 513
    assert f(*bad) == 2                                                   # G > 512


def test_binding_refuses_cpu_tensors():
    import torch
    import fp8_bf16_mxfp4_gb300 as mxg
    with pytest.raises(ValueError):
        mxg.mx_quantize_rowwise(torch.zeros((4, 64), dtype=torch.bfloat16), "e2m1")
