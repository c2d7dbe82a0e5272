"""GB300 grouped microscaled (MX) GEMM library -- Python binding.

Argument marshalling only: every computation runs in libmxg.so (CUDA kernels
for sm_103a) through its C ABI (include/mxg.h).  PyTorch provides device
memory and the current stream.  There is no CPU fallback: without the built
library or a GPU these functions raise.

Layouts (row-major, K-major operands):
  * E2M1 codes: uint8 [rows, cols/2], element 2j in the low nibble.
  * E4M3 codes: uint8 [rows, cols].
  * UE8M0 scales: uint8 [rows, cols/32] (one per 32 elements along cols).
"""

from __future__ import annotations

import ctypes
from dataclasses import dataclass

import torch

from . import _lib

__all__ = [
    "MXOperand", "MXGError", "mx_quantize_rowwise", "mx_quantize_colwise_segment_padded",
    "mx_quantize_rowwise_packed", "mx_packed_scale_bytes", "mx_packed_colwise_scale_bytes",
    "mx_quantize_dual_segment_padded",
    "grouped_gemm_fwd", "grouped_gemm_dgrad", "grouped_gemm_wgrad", "gemm_workspace_size", "mx_gemm_dense",
    "mx_padded_rows_capacity", "check_status", "status_tensor", "set_wait_timeout_ns", "set_gemm_cta_group",
    "library_path", "BWOperand", "bw_quantize_1x128", "bw_quantize_128x128",
    "bw_quantize_colwise_padded", "bw_grouped_gemm_fwd", "bw_grouped_gemm_dgrad",
    "bw_grouped_gemm_wgrad", "bw_quantize_1x128_pow2", "bw_quantize_128x128_pow2",
    "bw_quantize_colwise_padded_pow2", "bw_quantize_dual_padded",
]

ELEM = {"e2m1": 1, "e4m3": 2}
SCALE_LAYOUT = {"plain": 0, "packed": 1}
PASS = {"fwd": 0, "dgrad": 1, "wgrad": 2}
_OUT = {torch.bfloat16: 1, torch.float32: 2}

library_path = _lib.LIB_PATH


class MXGError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        msg = _lib.load().mxg_status_string(code).decode()
        super().__init__(f"{what}: {msg} (status {code})")


def _ok(code: int, what: str):
    if code != 0:
        raise MXGError(code, what)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _stream(dev) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)


def _need_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("libmxg operates on CUDA tensors only")


@dataclass
class MXOperand:
    """A quantized K-major operand: codes, UE8M0 scales, element format and
    logical column count (the contraction length).  ``scale_layout`` "plain"
    means scales [rows, cols/32]; "packed" means the tensor-core staging order
    of ``mx_quantize_rowwise_packed`` (a flat uint8 tensor)."""
    data: torch.Tensor
    scale: torch.Tensor
    elem: str
    cols: int
    scale_layout: str = "plain"

    @property
    def rows(self) -> int:
        return self.data.shape[0]

    def c(self) -> _lib.MxOperandC:
        packed = self.scale_layout == "packed"
        return _lib.MxOperandC(self.data.data_ptr(), self.scale.data_ptr(), self.rows, self.cols,
                               _ld(self.data, _codes_cols(self.elem, self.cols)),
                               0 if packed else _ld(self.scale, self.cols // 32), ELEM[self.elem],
                               SCALE_LAYOUT[self.scale_layout])


def _ld(t: torch.Tensor, row_elems: int) -> int:
    """Row stride in elements.  Zero-size tensors and tensors with a single
    row report arbitrary strides (the stride is never used for them), so their
    logical contiguous stride is passed instead."""
    if t.numel() == 0 or t.shape[0] <= 1:
        return max(row_elems, 16)
    return t.stride(0)


_status = {}


def status_tensor(device) -> torch.Tensor:
    """Per-device int32 status word used when the caller passes none."""
    d = torch.device(device)
    idx = d.index if d.index is not None else torch.cuda.current_device()
    if idx not in _status:
        _status[idx] = torch.zeros(1, dtype=torch.int32, device=f"cuda:{idx}")
    return _status[idx]


def check_status(status: torch.Tensor | None = None, device=None) -> int:
    """Synchronise, read and clear the device status word; raise on error."""
    st = status if status is not None else status_tensor(device or torch.cuda.current_device())
    code = _lib.load().mxg_check_status(_ptr(st), _stream(st.device))
    _ok(code, "device-side check")
    return code


def set_wait_timeout_ns(ns: int):
    _lib.load().mxg_set_wait_timeout_ns(int(ns))


def set_gemm_cta_group(n: int) -> int:
    """Choose the MX GEMM kernel: 2 = CTA pairs sharing each 256x256 tile
    (the default), 1 = the one-SM kernel.  Returns the previous choice."""
    lib = _lib.load()
    prev = int(lib.mxg_get_gemm_cta_group())
    _ok(lib.mxg_set_gemm_cta_group(int(n)), "set_gemm_cta_group")
    return prev


def mx_padded_rows_capacity(rows: int, G: int, pad: int) -> int:
    return int(_lib.load().mx_padded_rows_capacity(rows, G, pad))


def _codes_cols(elem: str, cols: int) -> int:
    return cols // 2 if elem == "e2m1" else cols


SCALE_RULES = {"ocp": 0, "round_up": 0x100}  # MXG_SCALE_ROUND_UP


def _quant_elem(elem: str, rule: str) -> int:
    """The quantizers' elem argument: format code with the scale-rule flag."""
    if rule not in SCALE_RULES:
        raise ValueError(f"unknown scale rule {rule!r} (ocp or round_up)")
    return ELEM[elem] | SCALE_RULES[rule]


def mx_quantize_rowwise(x: torch.Tensor, elem: str, q: torch.Tensor | None = None,
                        s: torch.Tensor | None = None, rule: str = "ocp") -> MXOperand:
    """BF16 [rows, cols] -> MX operand quantized along cols."""
    _need_cuda(x)
    if x.dtype != torch.bfloat16 or x.dim() != 2:
        raise ValueError("x must be a 2-D bfloat16 tensor")
    rows, cols = x.shape
    if q is None:
        q = torch.empty((rows, _codes_cols(elem, cols)), dtype=torch.uint8, device=x.device)
    if s is None:
        s = torch.empty((rows, cols // 32), dtype=torch.uint8, device=x.device)
    lib = _lib.load()
    _ok(lib.mx_quantize_rowwise(_ptr(x), rows, cols, _ld(x, cols), _quant_elem(elem, rule), _ptr(q),
                                _ld(q, _codes_cols(elem, cols)), _ptr(s), _ld(s, cols // 32),
                                _stream(x.device)), "mx_quantize_rowwise")
    return MXOperand(q, s, elem, cols)


def mx_packed_scale_bytes(rows: int, cols: int, G: int) -> int:
    """Bytes of packed scales for `rows` x `cols` cut into G segments (an upper
    bound over every split)."""
    return int(_lib.load().mx_packed_scale_bytes(rows, cols, G))


def mx_packed_colwise_scale_bytes(cols: int, capacity: int, G: int) -> int:
    """Bytes of packed scales of a column-wise operand with `cols` channels and
    `capacity` padded positions over G experts (an upper bound over splits)."""
    return int(_lib.load().mx_packed_colwise_scale_bytes(cols, capacity, G))


def mx_quantize_rowwise_packed(x: torch.Tensor, elem: str, m_splits: torch.Tensor | None = None,
                               groups: int | None = None, status: torch.Tensor | None = None,
                               check: bool = False, rule: str = "ocp") -> MXOperand:
    """BF16 [rows, cols] -> MX operand whose scales are already in the grouped
    GEMM's tensor-core staging order (no repacking pass in the GEMM).  Rows
    are cut into segments by the device ``m_splits`` (activations and
    gradients), or into ``groups`` equal segments (forward weights: G experts
    of N rows).  The GEMM call must use the same segments."""
    _need_cuda(x, m_splits)
    if x.dtype != torch.bfloat16 or x.dim() != 2:
        raise ValueError("x must be a 2-D bfloat16 tensor")
    if (m_splits is None) == (groups is None):
        raise ValueError("give exactly one of m_splits and groups")
    rows, cols = x.shape
    G = m_splits.numel() if m_splits is not None else int(groups)
    if m_splits is not None and m_splits.dtype != torch.int32:
        raise ValueError("m_splits must be int32")
    nbytes = mx_packed_scale_bytes(rows, cols, G)
    if nbytes < 0:
        raise ValueError("invalid shape for packed scales")
    q = torch.empty((rows, _codes_cols(elem, cols)), dtype=torch.uint8, device=x.device)
    s = torch.empty((max(nbytes, 16),), dtype=torch.uint8, device=x.device)
    st = status if status is not None else status_tensor(x.device)
    lib = _lib.load()
    _ok(lib.mx_quantize_rowwise_packed(_ptr(x), rows, cols, _ld(x, cols), _quant_elem(elem, rule), _ptr(q),
                                       _ld(q, _codes_cols(elem, cols)), _ptr(s), s.numel(),
                                       _ptr(m_splits), G, _ptr(st),
                                       _stream(x.device)), "mx_quantize_rowwise_packed")
    if check:
        check_status(st)
    return MXOperand(q, s, elem, cols, "packed")


def mx_quantize_colwise_segment_padded(x: torch.Tensor, m_splits: torch.Tensor, pad_multiple: int,
                                       elem: str, capacity: int | None = None,
                                       status: torch.Tensor | None = None, check: bool = False,
                                       rule: str = "ocp", packed: bool = False):
    """BF16 [S, C] with experts' rows concatenated -> (operand [C, capacity],
    int64 padded offsets [G+1]).  Columns beyond the last expert's padded end
    are left uninitialised.  With ``packed`` the scales are written in the
    grouped GEMM's staging order (a flat uint8 tensor; the GEMM call must use
    the same splits and pad)."""
    _need_cuda(x, m_splits)
    S, C = x.shape
    G = m_splits.numel()
    if capacity is None:
        capacity = mx_padded_rows_capacity(S, G, pad_multiple)
    qT = torch.empty((C, _codes_cols(elem, capacity)), dtype=torch.uint8, device=x.device)
    poff = torch.empty(G + 1, dtype=torch.int64, device=x.device)
    st = status if status is not None else status_tensor(x.device)
    lib = _lib.load()
    if packed:
        nbytes = mx_packed_colwise_scale_bytes(C, capacity, G)
        if nbytes < 0:
            raise ValueError("invalid shape for packed scales")
        sp = torch.empty((max(nbytes, 16),), dtype=torch.uint8, device=x.device)
        _ok(lib.mx_quantize_colwise_segment_padded_packed(
            _ptr(x), S, C, _ld(x, C), _ptr(m_splits), G, pad_multiple, _quant_elem(elem, rule), _ptr(qT),
            _ld(qT, _codes_cols(elem, capacity)), _ptr(sp), sp.numel(), capacity, _ptr(poff), _ptr(st),
            _stream(x.device)), "mx_quantize_colwise_segment_padded_packed")
        if check:
            check_status(st)
        return MXOperand(qT, sp, elem, capacity, "packed"), poff
    sT = torch.empty((C, capacity // 32), dtype=torch.uint8, device=x.device)
    _ok(lib.mx_quantize_colwise_segment_padded(
        _ptr(x), S, C, _ld(x, C), _ptr(m_splits), G, pad_multiple, _quant_elem(elem, rule), _ptr(qT),
        _ld(qT, _codes_cols(elem, capacity)), _ptr(sT), _ld(sT, capacity // 32), capacity,
        _ptr(poff), _ptr(st), _stream(x.device)),
        "mx_quantize_colwise_segment_padded")
    if check:
        check_status(st)
    return MXOperand(qT, sT, elem, capacity), poff


def mx_quantize_dual_segment_padded(x: torch.Tensor, m_splits: torch.Tensor, pad_multiple: int,
                                    elem: str, capacity: int | None = None,
                                    q: torch.Tensor | None = None, s: torch.Tensor | None = None,
                                    status: torch.Tensor | None = None, check: bool = False,
                                    rule: str = "ocp"):
    """BF16 [S, C] -> (row-wise operand [S, C], column-wise operand
    [C, capacity], int64 padded offsets [G+1]) from one read of x; the same
    bytes as mx_quantize_rowwise plus mx_quantize_colwise_segment_padded."""
    _need_cuda(x, m_splits)
    if x.dtype != torch.bfloat16 or x.dim() != 2:
        raise ValueError("x must be a 2-D bfloat16 tensor")
    S, C = x.shape
    G = m_splits.numel()
    if capacity is None:
        capacity = mx_padded_rows_capacity(S, G, pad_multiple)
    if q is None:
        q = torch.empty((S, _codes_cols(elem, C)), dtype=torch.uint8, device=x.device)
    if s is None:
        s = torch.empty((S, C // 32), dtype=torch.uint8, device=x.device)
    qT = torch.empty((C, _codes_cols(elem, capacity)), dtype=torch.uint8, device=x.device)
    sT = torch.empty((C, capacity // 32), dtype=torch.uint8, device=x.device)
    poff = torch.empty(G + 1, dtype=torch.int64, device=x.device)
    st = status if status is not None else status_tensor(x.device)
    lib = _lib.load()
    _ok(lib.mx_quantize_dual_segment_padded(
        _ptr(x), S, C, _ld(x, C), _ptr(m_splits), G, pad_multiple, _quant_elem(elem, rule), _ptr(q),
        _ld(q, _codes_cols(elem, C)), _ptr(s), _ld(s, C // 32), _ptr(qT),
        _ld(qT, _codes_cols(elem, capacity)), _ptr(sT), _ld(sT, capacity // 32), capacity,
        _ptr(poff), _ptr(st), _stream(x.device)),
        "mx_quantize_dual_segment_padded")
    if check:
        check_status(st)
    return MXOperand(q, s, elem, C), MXOperand(qT, sT, elem, capacity), poff


def gemm_workspace_size(pass_: str, G: int, S: int, N: int, K: int, pad: int = 32) -> int:
    return int(_lib.load().mxg_gemm_workspace_size(PASS[pass_], G, S, N, K, pad))


def _workspace(nbytes: int, device, ws: torch.Tensor | None):
    if ws is not None:
        return ws
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)


def grouped_gemm_fwd(A: MXOperand, W: MXOperand, m_splits: torch.Tensor, N: int,
                     out_dtype=torch.bfloat16, out: torch.Tensor | None = None,
                     workspace: torch.Tensor | None = None, status: torch.Tensor | None = None,
                     check: bool = False) -> torch.Tensor:
    """Y[off_g+i, :] = A[off_g+i, :] @ W[g*N:(g+1)*N, :]^T for every expert g."""
    _need_cuda(A.data, W.data, m_splits)
    G = m_splits.numel()
    dev = A.data.device
    if out is None:
        out = torch.empty((A.rows, N), dtype=out_dtype, device=dev)
    need = gemm_workspace_size("fwd", G, A.rows, N, A.cols)
    ws = _workspace(need, dev, workspace)
    st = status if status is not None else status_tensor(dev)
    a, w = A.c(), W.c()
    _ok(_lib.load().grouped_gemm_fwd(ctypes.byref(a), ctypes.byref(w), _ptr(m_splits), G, N,
                                     _ptr(out), _ld(out, N), _OUT[out.dtype], _ptr(ws),
                                     ws.numel(), _ptr(st), _stream(dev)), "grouped_gemm_fwd")
    if check:
        check_status(st)
    return out


def mx_gemm_dense(A: MXOperand, B: MXOperand, out_dtype=torch.bfloat16, out: torch.Tensor | None = None,
                  workspace: torch.Tensor | None = None, status: torch.Tensor | None = None,
                  check: bool = False) -> torch.Tensor:
    """C[M, N] = A[M, K] @ B[N, K]^T, both MX operands quantized along K (no
    experts, no m_splits)."""
    _need_cuda(A.data, B.data)
    dev = A.data.device
    N = B.rows
    if out is None:
        out = torch.empty((A.rows, N), dtype=out_dtype, device=dev)
    need = gemm_workspace_size("fwd", 1, A.rows, N, A.cols)
    ws = _workspace(need, dev, workspace)
    st = status if status is not None else status_tensor(dev)
    a, b = A.c(), B.c()
    _ok(_lib.load().mx_gemm_dense(ctypes.byref(a), ctypes.byref(b), _ptr(out), _ld(out, N), _OUT[out.dtype],
                                  _ptr(ws), ws.numel(), _ptr(st), _stream(dev)), "mx_gemm_dense")
    if check:
        check_status(st)
    return out


def grouped_gemm_dgrad(dY: MXOperand, Wt: MXOperand, m_splits: torch.Tensor,
                       out_dtype=torch.bfloat16, out: torch.Tensor | None = None,
                       workspace: torch.Tensor | None = None, status: torch.Tensor | None = None,
                       check: bool = False) -> torch.Tensor:
    """dX[off_g+i, :] = dY[off_g+i, :] @ Wt[:, g*N:(g+1)*N]^T (Wt = W^T quantized along N)."""
    _need_cuda(dY.data, Wt.data, m_splits)
    G = m_splits.numel()
    dev = dY.data.device
    K = Wt.rows
    if out is None:
        out = torch.empty((dY.rows, K), dtype=out_dtype, device=dev)
    need = gemm_workspace_size("dgrad", G, dY.rows, dY.cols, K)
    ws = _workspace(need, dev, workspace)
    st = status if status is not None else status_tensor(dev)
    a, b = dY.c(), Wt.c()
    _ok(_lib.load().grouped_gemm_dgrad(ctypes.byref(a), ctypes.byref(b), _ptr(m_splits), G,
                                       _ptr(out), _ld(out, K), _OUT[out.dtype], _ptr(ws),
                                       ws.numel(), _ptr(st), _stream(dev)), "grouped_gemm_dgrad")
    if check:
        check_status(st)
    return out


def grouped_gemm_wgrad(dYt: MXOperand, Xt: MXOperand, m_splits: torch.Tensor, total_rows: int,
                       pad_multiple: int, out: torch.Tensor | None = None,
                       out_dtype=torch.float32, accumulate: bool = False,
                       workspace: torch.Tensor | None = None, status: torch.Tensor | None = None,
                       check: bool = False) -> torch.Tensor:
    """dW[g] (+)= dYt[:, seg_g] @ Xt[:, seg_g]^T over expert g's padded token
    segment; out is [G, N, K]."""
    _need_cuda(dYt.data, Xt.data, m_splits)
    G = m_splits.numel()
    dev = dYt.data.device
    N, K = dYt.rows, Xt.rows
    if out is None:
        if accumulate:
            raise ValueError("accumulate needs an existing out tensor")
        out = torch.empty((G, N, K), dtype=out_dtype, device=dev)
    need = gemm_workspace_size("wgrad", G, dYt.cols, N, K, pad_multiple)
    ws = _workspace(need, dev, workspace)
    st = status if status is not None else status_tensor(dev)
    a, b = dYt.c(), Xt.c()
    _ok(_lib.load().grouped_gemm_wgrad(ctypes.byref(a), ctypes.byref(b), _ptr(m_splits), G,
                                       total_rows, pad_multiple, _ptr(out), _OUT[out.dtype],
                                       1 if accumulate else 0, _ptr(ws), ws.numel(), _ptr(st),
                                       _stream(dev)), "grouped_gemm_wgrad")
    if check:
        check_status(st)
    return out


# ----------------------------------------------------------------------------- blockwise FP8


@dataclass
class BWOperand:
    """Blockwise-FP8 K-major operand: E4M3 codes [rows, cols] and fp32 scales
    (activation-type [cols/128, >= rows] or weight-type [rows/128, cols/128])."""
    data: torch.Tensor
    scale: torch.Tensor

    @property
    def rows(self) -> int:
        return self.data.shape[0]

    @property
    def cols(self) -> int:
        return self.data.shape[1]

    def c(self) -> _lib.BwOperandC:
        return _lib.BwOperandC(self.data.data_ptr(), self.scale.data_ptr(), self.rows, self.cols,
                               _ld(self.data, self.cols), _ld(self.scale, self.scale.shape[-1]),
                               0, 0)


def bw_quantize_1x128(x: torch.Tensor) -> BWOperand:
    """BF16 [rows, cols] -> E4M3 [rows, cols] + activation-type scales [cols/128, rows]."""
    _need_cuda(x)
    R, C = x.shape
    q = torch.empty((R, C), dtype=torch.uint8, device=x.device)
    s = torch.empty((C // 128, R), dtype=torch.float32, device=x.device)
    _ok(_lib.load().bw_quantize_1x128(_ptr(x), R, C, _ld(x, C), _ptr(q), _ld(q, C), _ptr(s),
                                      _ld(s, R), _stream(x.device)), "bw_quantize_1x128")
    return BWOperand(q, s)


def bw_quantize_128x128(w: torch.Tensor, transposed: bool = True):
    """BF16 weights [rows, cols] -> (operand with weight-type scales, and when
    `transposed` the dgrad copy [cols, rows] with its scales)."""
    _need_cuda(w)
    R, C = w.shape
    dev = w.device
    q = torch.empty((R, C), dtype=torch.uint8, device=dev)
    s = torch.empty((R // 128, C // 128), dtype=torch.float32, device=dev)
    qT = torch.empty((C, R), dtype=torch.uint8, device=dev) if transposed else None
    sT = torch.empty((C // 128, R // 128), dtype=torch.float32, device=dev) if transposed else None
    _ok(_lib.load().bw_quantize_128x128(_ptr(w), R, C, _ld(w, C), _ptr(q), _ld(q, C), _ptr(s),
                                        _ptr(qT), _ld(qT, R) if transposed else 0, _ptr(sT),
                                        _stream(dev)), "bw_quantize_128x128")
    return BWOperand(q, s), (BWOperand(qT, sT) if transposed else None)


def bw_quantize_colwise_padded(x: torch.Tensor, m_splits: torch.Tensor, capacity: int | None = None,
                               status: torch.Tensor | None = None, check: bool = False):
    """BF16 [S, C] -> (operand [C, capacity] with activation-type scales
    [capacity/128, C], int64 padded offsets [G+1]); segments padded to 128."""
    _need_cuda(x, m_splits)
    S, C = x.shape
    G = m_splits.numel()
    if capacity is None:
        capacity = mx_padded_rows_capacity(S, G, 128)
    qT = torch.empty((C, capacity), dtype=torch.uint8, device=x.device)
    sT = torch.empty((capacity // 128, C), dtype=torch.float32, device=x.device)
    poff = torch.empty(G + 1, dtype=torch.int64, device=x.device)
    st = status if status is not None else status_tensor(x.device)
    _ok(_lib.load().bw_quantize_colwise_padded(
        _ptr(x), S, C, _ld(x, C), _ptr(m_splits), G, _ptr(qT), _ld(qT, capacity), _ptr(sT),
        _ld(sT, C), capacity, _ptr(poff), _ptr(st), _stream(x.device)), "bw_quantize_colwise_padded")
    if check:
        check_status(st)
    return BWOperand(qT, sT), poff


def bw_quantize_1x128_pow2(x: torch.Tensor) -> MXOperand:
    """BF16 [rows, cols] -> blockwise FP8 (1x128, power-of-two scales) as an
    MXFP8 operand: E4M3 [rows, cols] + UE8M0 [rows, cols/32]."""
    _need_cuda(x)
    R, C = x.shape
    q = torch.empty((R, C), dtype=torch.uint8, device=x.device)
    s = torch.empty((R, C // 32), dtype=torch.uint8, device=x.device)
    _ok(_lib.load().bw_quantize_1x128_pow2(_ptr(x), R, C, _ld(x, C), _ptr(q), _ld(q, C), _ptr(s),
                                           _ld(s, C // 32), _stream(x.device)), "bw_quantize_1x128_pow2")
    return MXOperand(q, s, "e4m3", C)


def bw_quantize_128x128_pow2(w: torch.Tensor, transposed: bool = True):
    """BF16 weights [rows, cols] -> (MXFP8 operand with 128x128 power-of-two
    scales, and when `transposed` the dgrad copy [cols, rows])."""
    _need_cuda(w)
    R, C = w.shape
    dev = w.device
    q = torch.empty((R, C), dtype=torch.uint8, device=dev)
    s = torch.empty((R, C // 32), dtype=torch.uint8, device=dev)
    qT = torch.empty((C, R), dtype=torch.uint8, device=dev) if transposed else None
    sT = torch.empty((C, R // 32), dtype=torch.uint8, device=dev) if transposed else None
    _ok(_lib.load().bw_quantize_128x128_pow2(
        _ptr(w), R, C, _ld(w, C), _ptr(q), _ld(q, C), _ptr(s), _ld(s, C // 32), _ptr(qT),
        _ld(qT, R) if transposed else 0, _ptr(sT), _ld(sT, R // 32) if transposed else 0, _stream(dev)),
        "bw_quantize_128x128_pow2")
    return MXOperand(q, s, "e4m3", C), (MXOperand(qT, sT, "e4m3", R) if transposed else None)


def bw_quantize_colwise_padded_pow2(x: torch.Tensor, m_splits: torch.Tensor, capacity: int | None = None,
                                    status: torch.Tensor | None = None, check: bool = False):
    """BF16 [S, C] -> (MXFP8 operand [C, capacity], segments padded to 128,
    power-of-two 1x128 scales as UE8M0 [C, capacity/32]; int64 padded offsets)."""
    _need_cuda(x, m_splits)
    S, C = x.shape
    G = m_splits.numel()
    if capacity is None:
        capacity = mx_padded_rows_capacity(S, G, 128)
    qT = torch.empty((C, capacity), dtype=torch.uint8, device=x.device)
    sT = torch.empty((C, capacity // 32), dtype=torch.uint8, device=x.device)
    poff = torch.empty(G + 1, dtype=torch.int64, device=x.device)
    st = status if status is not None else status_tensor(x.device)
    _ok(_lib.load().bw_quantize_colwise_padded_pow2(
        _ptr(x), S, C, _ld(x, C), _ptr(m_splits), G, _ptr(qT), _ld(qT, capacity), _ptr(sT),
        _ld(sT, capacity // 32), capacity, _ptr(poff), _ptr(st), _stream(x.device)),
        "bw_quantize_colwise_padded_pow2")
    if check:
        check_status(st)
    return MXOperand(qT, sT, "e4m3", capacity), poff


def bw_quantize_dual_padded(x: torch.Tensor, m_splits: torch.Tensor, capacity: int | None = None,
                            pow2: bool = False, status: torch.Tensor | None = None, check: bool = False):
    """One read of BF16 x [S, C] -> (row-wise 1x128 operand, column-wise
    operand [C, capacity] with segments padded to 128, int64 padded offsets):
    the same bytes as the separate row-wise and column-wise quantizers.  With
    pow2 both are MXFP8 operands (UE8M0 power-of-two scales); otherwise
    BWOperands with fp32 activation-type scales."""
    _need_cuda(x, m_splits)
    S, C = x.shape
    G = m_splits.numel()
    dev = x.device
    if capacity is None:
        capacity = mx_padded_rows_capacity(S, G, 128)
    q = torch.empty((S, C), dtype=torch.uint8, device=dev)
    qT = torch.empty((C, capacity), dtype=torch.uint8, device=dev)
    if pow2:
        s = torch.empty((S, C // 32), dtype=torch.uint8, device=dev)
        sT = torch.empty((C, capacity // 32), dtype=torch.uint8, device=dev)
        ld_s, ld_sT = _ld(s, C // 32), _ld(sT, capacity // 32)
    else:
        s = torch.empty((C // 128, S), dtype=torch.float32, device=dev)
        sT = torch.empty((capacity // 128, C), dtype=torch.float32, device=dev)
        ld_s, ld_sT = _ld(s, S), _ld(sT, C)
    poff = torch.empty(G + 1, dtype=torch.int64, device=dev)
    st = status if status is not None else status_tensor(dev)
    fn = _lib.load().bw_quantize_dual_padded_pow2 if pow2 else _lib.load().bw_quantize_dual_padded
    _ok(fn(_ptr(x), S, C, _ld(x, C), _ptr(m_splits), G, _ptr(q), _ld(q, C), _ptr(s), ld_s, _ptr(qT),
           _ld(qT, capacity), _ptr(sT), ld_sT, capacity, _ptr(poff), _ptr(st), _stream(dev)),
        "bw_quantize_dual_padded")
    if check:
        check_status(st)
    if pow2:
        return MXOperand(q, s, "e4m3", C), MXOperand(qT, sT, "e4m3", capacity), poff
    return BWOperand(q, s), BWOperand(qT, sT), poff


def _bw_ws(G, device, ws):
    if ws is not None:
        return ws
    return torch.empty(max(int(_lib.load().bw_gemm_workspace_size(G)), 256), dtype=torch.uint8,
                       device=device)


def bw_grouped_gemm_fwd(A: BWOperand, W: BWOperand, m_splits: torch.Tensor, N: int,
                        out_dtype=torch.bfloat16, out: torch.Tensor | None = None,
                        workspace: torch.Tensor | None = None, status: torch.Tensor | None = None,
                        check: bool = False) -> torch.Tensor:
    _need_cuda(A.data, W.data, m_splits)
    G = m_splits.numel()
    dev = A.data.device
    if out is None:
        out = torch.empty((A.rows, N), dtype=out_dtype, device=dev)
    ws = _bw_ws(G, dev, workspace)
    st = status if status is not None else status_tensor(dev)
    a, w = A.c(), W.c()
    _ok(_lib.load().bw_grouped_gemm_fwd(ctypes.byref(a), ctypes.byref(w), _ptr(m_splits), G, N,
                                        _ptr(out), _ld(out, N), _OUT[out.dtype], _ptr(ws),
                                        ws.numel(), _ptr(st), _stream(dev)), "bw_grouped_gemm_fwd")
    if check:
        check_status(st)
    return out


def bw_grouped_gemm_dgrad(dY: BWOperand, Wt: BWOperand, m_splits: torch.Tensor,
                          out_dtype=torch.bfloat16, out: torch.Tensor | None = None,
                          workspace: torch.Tensor | None = None, status: torch.Tensor | None = None,
                          check: bool = False) -> torch.Tensor:
    _need_cuda(dY.data, Wt.data, m_splits)
    G = m_splits.numel()
    dev = dY.data.device
    K = Wt.rows
    if out is None:
        out = torch.empty((dY.rows, K), dtype=out_dtype, device=dev)
    ws = _bw_ws(G, dev, workspace)
    st = status if status is not None else status_tensor(dev)
    a, b = dY.c(), Wt.c()
    _ok(_lib.load().bw_grouped_gemm_dgrad(ctypes.byref(a), ctypes.byref(b), _ptr(m_splits), G,
                                          _ptr(out), _ld(out, K), _OUT[out.dtype], _ptr(ws),
                                          ws.numel(), _ptr(st), _stream(dev)), "bw_grouped_gemm_dgrad")
    if check:
        check_status(st)
    return out


def bw_grouped_gemm_wgrad(dYt: BWOperand, Xt: BWOperand, m_splits: torch.Tensor, total_rows: int,
                          out: torch.Tensor | None = None, out_dtype=torch.float32,
                          accumulate: bool = False, workspace: torch.Tensor | None = None,
                          status: torch.Tensor | None = None, check: bool = False) -> torch.Tensor:
    _need_cuda(dYt.data, Xt.data, m_splits)
    G = m_splits.numel()
    dev = dYt.data.device
    N, K = dYt.rows, Xt.rows
    if out is None:
        if accumulate:
            raise ValueError("accumulate needs an existing out tensor")
        out = torch.empty((G, N, K), dtype=out_dtype, device=dev)
    ws = _bw_ws(G, dev, workspace)
    st = status if status is not None else status_tensor(dev)
    a, b = dYt.c(), Xt.c()
    _ok(_lib.load().bw_grouped_gemm_wgrad(ctypes.byref(a), ctypes.byref(b), _ptr(m_splits), G,
                                          total_rows, _ptr(out), _OUT[out.dtype],
                                          1 if accumulate else 0, _ptr(ws), ws.numel(), _ptr(st),
                                          _stream(dev)), "bw_grouped_gemm_wgrad")
    if check:
        check_status(st)
    return out
