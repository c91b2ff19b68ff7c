"""Python binding of the h32 C-ABI library (the Hadamard-route prompt path).

The functions below carry the names of the C entry points declared in
``include/h32.h`` and only marshal arguments: they take CUDA torch tensors,
allocate outputs with torch when none are given, pass raw device pointers and
the current CUDA stream to the library, and raise ``H32Error`` on a non-OK
status.  Every step of the path runs in the library's CUDA kernels; there is
no CPU fallback, and calling any function without the built library raises.

Build the library with ``python -m hadamard_rotated_bit_gb300._build`` (or
``__graft_entry__.build()``).
"""
from __future__ import annotations

import ctypes
import os
import threading

__all__ = [
    "H32Error", "lib", "library_path", "EXPORTED_SYMBOLS",
    "h32_quantize_act_q4", "h32_quantize_act_q8", "h32_rotate_quantize_weights_q4_0",
    "q4_0_x_q4_gemm", "q4_0_x_q8_gemm", "q4_0_x_q4_gemm_experts",
    "h32_device_status", "h32_status_string", "h32_set_wait_limit", "h32_version",
    "h32_last_cuda_error", "h32_quantize_act_q4_tc", "h32_prepack_weights_q4_0_tc",
    "q4_0_x_q4_gemm_tc", "h32_quantize_act_q4_tc_gather", "q4_0_x_q4_gemm_tc_experts",
    "h32_quantize_act_q8_tc", "q4_0_x_q8_gemm_tc", "q4_0_x_q4_gemm_tc_quant_next",
    "h32_moe_route", "h32_moe_combine",
]


def h32_last_cuda_error() -> str:
    return lib().h32_last_cuda_error().decode()

_PKG = os.path.dirname(os.path.abspath(__file__))
library_path = os.path.join(_PKG, "lib", "libh32.so")

H32_OK, H32_ERR_INVALID_ARG, H32_ERR_ALIGNMENT, H32_ERR_UNSUPPORTED = 0, 1, 2, 3
H32_ERR_CUDA, H32_ERR_TIMEOUT, H32_ERR_DEVICE_GUARD = 4, 5, 6
H32_IN_F32, H32_IN_BF16 = 0, 1

_P, _I64, _I32, _INT = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_int

# name -> (restype, argtypes); mirrors include/h32.h
_SIGS = {
    "h32_quantize_act_q4": (_INT, [_P, _INT, _I64, _I64, _I64, _P, _P, _INT, _P]),
    "h32_quantize_act_q8": (_INT, [_P, _INT, _I64, _I64, _I64, _P, _P, _INT, _P]),
    "h32_rotate_quantize_weights_q4_0": (_INT, [_P, _I64, _I64, _INT, _P, _P, _P]),
    "q4_0_x_q4_gemm": (_INT, [_P, _P, _P, _P, _I64, _I64, _I64, _P, _I64, _P, _P]),
    "q4_0_x_q8_gemm": (_INT, [_P, _P, _P, _P, _I64, _I64, _I64, _P, _I64, _P, _P]),
    "q4_0_x_q4_gemm_experts": (_INT, [_P, _P, _I32, _P, _P, _P, _I64, _P, _I64, _I64, _I64,
                                      _P, _I64, _P, _P]),
    "h32_device_status": (_INT, [_P]),
    "h32_status_string": (ctypes.c_char_p, [_INT]),
    "h32_set_wait_limit": (None, [ctypes.c_uint64]),
    "h32_version": (_INT, []),
    "h32_last_cuda_error": (ctypes.c_char_p, []),
    "h32_quantize_act_q4_tc": (_INT, [_P, _INT, _I64, _I64, _I64, _P, _P, _I64, _INT, _P]),
    "h32_prepack_weights_q4_0_tc": (_INT, [_P, _P, _I64, _I64, _P, _P, _I64, _P]),
    "q4_0_x_q4_gemm_tc": (_INT, [_P, _P, _I64, _P, _P, _I64, _I64, _I64, _I64, _P, _I64, _P, _P]),
    "q4_0_x_q4_gemm_tc_quant_next": (_INT, [_P, _P, _I64, _P, _P, _I64, _I64, _I64, _I64, _P,
                                            _I64, _P, _P, _I64, _INT, _P]),
    "h32_quantize_act_q8_tc": (_INT, [_P, _INT, _I64, _I64, _I64, _P, _P, _I64, _INT, _P]),
    "q4_0_x_q8_gemm_tc": (_INT, [_P, _P, _I64, _P, _P, _I64, _I64, _I64, _I64, _P, _I64, _P, _P]),
    "h32_quantize_act_q4_tc_gather": (_INT, [_P, _INT, _I64, _I64, _I64, _P, _I64, _P, _P, _I64,
                                             _INT, _P]),
    "q4_0_x_q4_gemm_tc_experts": (_INT, [_P, _P, _I64, ctypes.c_int32, _P, _P, _I64, _P, _I64, _I64,
                                         _I64, _P, _I64, _P, _P]),
    "h32_moe_route": (_INT, [_P, _I64, _I32, _I64, _I32, _P, _P, _P, _P, _P, _P]),
    "h32_moe_combine": (_INT, [_P, _I64, _I64, _P, _P, _I64, _I32, _I64, _P, _I64, _P]),
}
EXPORTED_SYMBOLS = tuple(_SIGS)

_lib = None
_lock = threading.Lock()


class H32Error(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        msg = f"{fn}: {h32_status_string(status)} (status {status})"
        if status == H32_ERR_CUDA:
            msg += f": {lib().h32_last_cuda_error().decode()}"
        super().__init__(msg)


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(library_path):
                raise ImportError(
                    f"h32 CUDA library not built ({library_path} missing); run "
                    "`python -m hadamard_rotated_bit_gb300._build` first")
            L = ctypes.CDLL(library_path)
            for name, (res, args) in _SIGS.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


def h32_status_string(status: int) -> str:
    return lib().h32_status_string(int(status)).decode()


def h32_version() -> int:
    return int(lib().h32_version())


def h32_set_wait_limit(polls: int) -> None:
    lib().h32_set_wait_limit(int(polls))


# --------------------------------------------------------------------------
# marshalling helpers
# --------------------------------------------------------------------------
def _torch():
    import torch
    return torch


def _stream(stream):
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _rot_arg(rotate) -> int:
    """rotate: False/0 (none), True/1/32 (32 points), 64 or 128 points."""
    if rotate is True:
        return 1
    if rotate is False or rotate is None:
        return 0
    return int(rotate)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _check(fn: str, st: int):
    if st != H32_OK:
        raise H32Error(fn, st)


def _cuda(t, name):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    return t


def _rows(t, name):
    """2-D tensor with unit stride in its last dimension; returns its row pitch."""
    if t.dim() != 2 or (t.shape[1] > 1 and t.stride(1) != 1):
        raise ValueError(f"{name} must be 2-D with a contiguous last dimension")
    return t.stride(0) if t.shape[0] > 1 else t.shape[1]


# --------------------------------------------------------------------------
# quantizers
# --------------------------------------------------------------------------
def _quantize_act(fn_name, bits, x, rotate, xq, xd, stream):
    torch = _torch()
    _cuda(x, "x")
    if x.dtype == torch.bfloat16:
        dt = H32_IN_BF16
    elif x.dtype == torch.float32:
        dt = H32_IN_F32
    else:
        raise ValueError("x must be bf16 or fp32")
    ldx = _rows(x, "x")
    M, K = x.shape
    if xq is None:
        xq = torch.empty((M, K // 2 if bits == 4 else K),
                         dtype=torch.uint8 if bits == 4 else torch.int8, device=x.device)
    if xd is None:
        xd = torch.empty((M, K // 32), dtype=torch.float32, device=x.device)
    st = getattr(lib(), fn_name)(_ptr(x), dt, M, K, ldx, _ptr(xq), _ptr(xd), _rot_arg(rotate),
                                 _stream(stream))
    _check(fn_name, st)
    return xq, xd


def h32_quantize_act_q4(x, rotate=True, xq=None, xd=None, stream=None):
    """x [M][K] bf16/fp32 -> (xq [M][K/2] uint8, xd [M][K/32] fp32)."""
    return _quantize_act("h32_quantize_act_q4", 4, x, rotate, xq, xd, stream)


def h32_quantize_act_q8(x, rotate=True, xq=None, xd=None, stream=None):
    """x [M][K] bf16/fp32 -> (xq [M][K] int8, xd [M][K/32] fp32)."""
    return _quantize_act("h32_quantize_act_q8", 8, x, rotate, xq, xd, stream)


def h32_rotate_quantize_weights_q4_0(w, rotate=True, wq=None, wd=None, stream=None):
    """w [N][K] fp32 (contiguous) -> (wq [N][K/2] uint8, wd [N][K/32] int16 holding fp16 bits)."""
    torch = _torch()
    _cuda(w, "w")
    if w.dtype != torch.float32 or not w.is_contiguous() or w.dim() != 2:
        raise ValueError("w must be a contiguous 2-D fp32 tensor")
    N, K = w.shape
    if wq is None:
        wq = torch.empty((N, K // 2), dtype=torch.uint8, device=w.device)
    if wd is None:
        wd = torch.empty((N, K // 32), dtype=torch.int16, device=w.device)
    st = lib().h32_rotate_quantize_weights_q4_0(_ptr(w), N, K, _rot_arg(rotate), _ptr(wq),
                                                _ptr(wd), _stream(stream))
    _check("h32_rotate_quantize_weights_q4_0", st)
    return wq, wd


# --------------------------------------------------------------------------
# GEMMs
# --------------------------------------------------------------------------
def _gemm(fn_name, wq, wd, xq, xd, y, block_sums, stream):
    torch = _torch()
    for t, n in ((wq, "wq"), (wd, "wd"), (xq, "xq"), (xd, "xd")):
        _cuda(t, n)
        if not t.is_contiguous():
            raise ValueError(f"{n} must be contiguous")
    N = wq.shape[0]
    K = wq.shape[1] * 2
    M = xq.shape[0]
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=wq.device)
    ldy = _rows(y, "y")
    S = None
    if block_sums is True:
        S = torch.empty((M, N, K // 32), dtype=torch.int32, device=wq.device)
    elif block_sums is not None and block_sums is not False:
        S = block_sums
    st = getattr(lib(), fn_name)(_ptr(wq), _ptr(wd), _ptr(xq), _ptr(xd), M, N, K, _ptr(y), ldy,
                                 _ptr(S), _stream(stream))
    _check(fn_name, st)
    return (y, S) if S is not None else y


def q4_0_x_q4_gemm(wq, wd, xq, xd, y=None, block_sums=None, stream=None):
    """y [M][N] = block-scaled product of Q4_0 weights and 4-bit activations.

    block_sums=True also returns the exact per-block sums int32 [M][N][K/32]."""
    return _gemm("q4_0_x_q4_gemm", wq, wd, xq, xd, y, block_sums, stream)


def q4_0_x_q8_gemm(wq, wd, xq, xd, y=None, block_sums=None, stream=None):
    """The exact route: Q4_0 weights against 8-bit activation codes."""
    return _gemm("q4_0_x_q8_gemm", wq, wd, xq, xd, y, block_sums, stream)


def q4_0_x_q4_gemm_experts(wq, wd, xq, xd, row_idx, expert_off, R, y=None, block_sums=None,
                           stream=None):
    """Expert-batched product: wq [E][N][K/2], wd [E][N][K/32]; rows grouped by expert."""
    torch = _torch()
    for t, n in ((wq, "wq"), (wd, "wd"), (xq, "xq"), (xd, "xd"), (expert_off, "expert_off")):
        _cuda(t, n)
        if not t.is_contiguous():
            raise ValueError(f"{n} must be contiguous")
    E, N, K = wq.shape[0], wq.shape[1], wq.shape[2] * 2
    if y is None:
        y = torch.empty((R, N), dtype=torch.float32, device=wq.device)
    ldy = _rows(y, "y")
    S = None
    if block_sums is True:
        S = torch.empty((R, N, K // 32), dtype=torch.int32, device=wq.device)
    elif block_sums is not None and block_sums is not False:
        S = block_sums
    st = lib().q4_0_x_q4_gemm_experts(_ptr(wq), _ptr(wd), E, _ptr(xq), _ptr(xd), _ptr(row_idx),
                                      xq.shape[0], _ptr(expert_off), R, N, K, _ptr(y), ldy,
                                      _ptr(S), _stream(stream))
    _check("q4_0_x_q4_gemm_experts", st)
    return (y, S) if S is not None else y


def h32_device_status(stream=None) -> int:
    """Synchronize the stream and return (and clear) the library's device status."""
    return int(lib().h32_device_status(_stream(stream)))


# --------------------------------------------------------------------------
# tensor-core form (one byte per code: the e4m3 encoding of the integer code)
# --------------------------------------------------------------------------
def _round4(n: int) -> int:
    return (n + 3) // 4 * 4


def h32_quantize_act_q4_tc(x, rotate=True, xw=None, xdt=None, stream=None):
    """x [M][K] bf16/fp32 -> (xw [M][K] uint8 tc-form codes, xdt [K/32][ldxd] fp32 scales,
    block-major, ldxd = M rounded up to a multiple of 4)."""
    return _quantize_tc("h32_quantize_act_q4_tc", 1, x, rotate, xw, xdt, stream)


def h32_quantize_act_q8_tc(x, rotate=True, xw=None, xdt=None, stream=None):
    """x [M][K] bf16/fp32 -> (xw8 [M][2K] uint8: per 32-block the e4m3 bytes of 16 h
    then of l, code = 16 h + l; xdt [K/32][ldxd] fp32 scales)."""
    return _quantize_tc("h32_quantize_act_q8_tc", 2, x, rotate, xw, xdt, stream)


def _quantize_tc(fn, bytes_per_code, x, rotate, xw, xdt, stream):
    torch = _torch()
    _cuda(x, "x")
    if x.dtype == torch.bfloat16:
        dt = H32_IN_BF16
    elif x.dtype == torch.float32:
        dt = H32_IN_F32
    else:
        raise ValueError("x must be bf16 or fp32")
    ldx = _rows(x, "x")
    M, K = x.shape
    if xw is None:
        xw = torch.empty((M, K * bytes_per_code), dtype=torch.uint8, device=x.device)
    if xdt is None:
        xdt = torch.zeros((K // 32, _round4(M)), dtype=torch.float32, device=x.device)
    st = getattr(lib(), fn)(_ptr(x), dt, M, K, ldx, _ptr(xw), _ptr(xdt), xdt.shape[1],
                            _rot_arg(rotate), _stream(stream))
    _check(fn, st)
    return xw, xdt


def h32_prepack_weights_q4_0_tc(wq, wd, wp=None, wsc=None, stream=None):
    """Q4_0 planes (wq [N][K/2], wd [N][K/32] fp16 bits) -> tc form
    (wp [N][K] uint8, wsc [N][ldws] fp32 = d, ldws = K/32 rounded up to 4)."""
    torch = _torch()
    _cuda(wq, "wq")
    _cuda(wd, "wd")
    N, K = wq.shape[0], wq.shape[1] * 2
    if wp is None:
        wp = torch.empty((N, K), dtype=torch.uint8, device=wq.device)
    if wsc is None:
        wsc = torch.empty((N, _round4(K // 32)), dtype=torch.float32, device=wq.device)
    st = lib().h32_prepack_weights_q4_0_tc(_ptr(wq), _ptr(wd), N, K, _ptr(wp), _ptr(wsc),
                                           wsc.shape[1], _stream(stream))
    _check("h32_prepack_weights_q4_0_tc", st)
    return wp, wsc


def q4_0_x_q4_gemm_tc(wp, wsc, xw, xdt, M=None, y=None, block_sums=None, stream=None):
    """The W4A4 product on tc-form operands (bit-identical to q4_0_x_q4_gemm)."""
    return _gemm_tc("q4_0_x_q4_gemm_tc", wp, wsc, xw, xdt, M, y, block_sums, stream)


def q4_0_x_q8_gemm_tc(wp, wsc, xw8, xdt, M=None, y=None, block_sums=None, stream=None):
    """The W4A8 product on tc-form operands (bit-identical to q4_0_x_q8_gemm)."""
    return _gemm_tc("q4_0_x_q8_gemm_tc", wp, wsc, xw8, xdt, M, y, block_sums, stream)


def _gemm_tc(fn, wp, wsc, xw, xdt, M, y, block_sums, stream):
    torch = _torch()
    N, K = wp.shape
    if M is None:
        M = xw.shape[0]
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=wp.device)
    ldy = _rows(y, "y")
    S = None
    if block_sums is True:
        S = torch.empty((M, N, K // 32), dtype=torch.int32, device=wp.device)
    elif block_sums is not None and block_sums is not False:
        S = block_sums
    st = getattr(lib(), fn)(_ptr(wp), _ptr(wsc), wsc.shape[1], _ptr(xw), _ptr(xdt), xdt.shape[1],
                            M, N, K, _ptr(y), ldy, _ptr(S), _stream(stream))
    _check(fn, st)
    return (y, S) if S is not None else y


def h32_quantize_act_q4_tc_gather(x, row_idx, rotate=True, xw=None, xdt=None, stream=None):
    """x [T][K] bf16/fp32, row_idx [R] int32 -> (xw [R][K] uint8, xdt [K/32][ldxd] fp32):
    output row r is the tc-form quantization of x[row_idx[r]]."""
    torch = _torch()
    _cuda(x, "x")
    _cuda(row_idx, "row_idx")
    if x.dtype == torch.bfloat16:
        dt = H32_IN_BF16
    elif x.dtype == torch.float32:
        dt = H32_IN_F32
    else:
        raise ValueError("x must be bf16 or fp32")
    if row_idx.dtype != torch.int32 or not row_idx.is_contiguous():
        raise ValueError("row_idx must be a contiguous int32 tensor")
    ldx = _rows(x, "x")
    T, K = x.shape
    R = row_idx.shape[0]
    if xw is None:
        xw = torch.empty((R, K), dtype=torch.uint8, device=x.device)
    if xdt is None:
        xdt = torch.zeros((K // 32, _round4(R)), dtype=torch.float32, device=x.device)
    st = lib().h32_quantize_act_q4_tc_gather(_ptr(x), dt, T, K, ldx, _ptr(row_idx), R, _ptr(xw),
                                             _ptr(xdt), xdt.shape[1], _rot_arg(rotate),
                                             _stream(stream))
    _check("h32_quantize_act_q4_tc_gather", st)
    return xw, xdt


def q4_0_x_q4_gemm_tc_experts(wp, wsc, xw, xdt, expert_off, N, R=None, y=None, block_sums=None,
                              stream=None):
    """Expert-batched tc GEMM.  wp [E*N][K] uint8, wsc [E*N][ldws] fp32 (the experts'
    repacked planes stacked), xw [R][K] / xdt [K/32][ldxd] in grouped order,
    expert_off [E+1] int32 -> y [R][N] fp32 in grouped order."""
    torch = _torch()
    EN, K = wp.shape
    if EN % N != 0:
        raise ValueError("wp rows must be E * N")
    E = EN // N
    if R is None:
        R = xw.shape[0]
    if y is None:
        y = torch.empty((R, N), dtype=torch.float32, device=wp.device)
    ldy = _rows(y, "y") if R > 0 else N
    S = None
    if block_sums is True:
        S = torch.empty((R, N, K // 32), dtype=torch.int32, device=wp.device)
    elif block_sums is not None and block_sums is not False:
        S = block_sums
    st = lib().q4_0_x_q4_gemm_tc_experts(_ptr(wp), _ptr(wsc), wsc.shape[1], E, _ptr(xw), _ptr(xdt),
                                         xdt.shape[1], _ptr(expert_off), R, N, K, _ptr(y), ldy,
                                         _ptr(S), _stream(stream))
    _check("q4_0_x_q4_gemm_tc_experts", st)
    return (y, S) if S is not None else y


def q4_0_x_q4_gemm_tc_quant_next(wp, wsc, xw, xdt, M=None, y=None, want_y=True, rotate_next=True,
                                 xw_next=None, xdt_next=None, stream=None):
    """The tc W4A4 product with its output also quantized for the next projection
    in the same kernel.  Returns (y or None, xw_next [M][N] uint8, xdt_next
    [N/32][ldxd] fp32)."""
    torch = _torch()
    N, K = wp.shape
    if M is None:
        M = xw.shape[0]
    if y is None and want_y:
        y = torch.empty((M, N), dtype=torch.float32, device=wp.device)
    ldy = _rows(y, "y") if y is not None else N
    if xw_next is None:
        xw_next = torch.empty((M, N), dtype=torch.uint8, device=wp.device)
    if xdt_next is None:
        xdt_next = torch.zeros((N // 32, _round4(M)), dtype=torch.float32, device=wp.device)
    st = lib().q4_0_x_q4_gemm_tc_quant_next(_ptr(wp), _ptr(wsc), wsc.shape[1], _ptr(xw), _ptr(xdt),
                                            xdt.shape[1], M, N, K, _ptr(y), ldy, _ptr(xw_next),
                                            _ptr(xdt_next), xdt_next.shape[1],
                                            _rot_arg(rotate_next), _stream(stream))
    _check("q4_0_x_q4_gemm_tc_quant_next", st)
    return y, xw_next, xdt_next


def h32_moe_route(logits, k, topk_id=None, topk_w=None, expert_off=None, row_idx=None,
                  row_of=None, stream=None):
    """Router: logits [T][E] fp32 -> (topk_id [T][k] int32, topk_w [T][k] fp32,
    expert_off [E+1] int32, row_idx [T*k] int32, row_of [T][k] int32).  The k
    largest logits (ties: lower id), softmax weights over them, rows grouped by
    expert then token."""
    torch = _torch()
    _cuda(logits, "logits")
    if logits.dtype != torch.float32:
        raise ValueError("logits must be fp32")
    T, E = logits.shape
    ldl = _rows(logits, "logits") if T > 0 else E
    dev = logits.device
    if topk_id is None:
        topk_id = torch.empty((T, k), dtype=torch.int32, device=dev)
    if topk_w is None:
        topk_w = torch.empty((T, k), dtype=torch.float32, device=dev)
    if expert_off is None:
        expert_off = torch.empty(E + 1, dtype=torch.int32, device=dev)
    if row_idx is None:
        row_idx = torch.empty(T * k, dtype=torch.int32, device=dev)
    if row_of is None:
        row_of = torch.empty((T, k), dtype=torch.int32, device=dev)
    st = lib().h32_moe_route(_ptr(logits), T, E, ldl, k, _ptr(topk_id), _ptr(topk_w),
                             _ptr(expert_off), _ptr(row_idx), _ptr(row_of), _stream(stream))
    _check("h32_moe_route", st)
    return topk_id, topk_w, expert_off, row_idx, row_of


def h32_moe_combine(y, row_of, topk_w, out=None, stream=None):
    """Weighted combine: y [R][H] fp32 (grouped rows), row_of [T][k], topk_w [T][k]
    -> out [T][H] fp32, the token's k rows added in choice order (fp32 fma from 0)."""
    torch = _torch()
    _cuda(y, "y")
    R, H = y.shape
    T, k = row_of.shape
    if row_of.dtype != torch.int32 or topk_w.dtype != torch.float32:
        raise ValueError("row_of must be int32 and topk_w fp32")
    if not (row_of.is_contiguous() and topk_w.is_contiguous()):
        raise ValueError("row_of and topk_w must be contiguous")
    if out is None:
        out = torch.empty((T, H), dtype=torch.float32, device=y.device)
    ldy = _rows(y, "y") if R > 0 else H
    ldo = _rows(out, "out") if T > 0 else H
    st = lib().h32_moe_combine(_ptr(y), R, ldy, _ptr(row_of), _ptr(topk_w), T, k, H, _ptr(out),
                               ldo, _stream(stream))
    _check("h32_moe_combine", st)
    return out


# --------------------------------------------------------------------------
# optional per-call tracing (H32_TRACE=1: device time per call; H32_TRACE=hash:
# also a hash of every output), off by default; see trace.py
# --------------------------------------------------------------------------
from . import trace as _trace  # noqa: E402

_COMPUTE_CALLS = (
    "h32_quantize_act_q4", "h32_quantize_act_q8", "h32_rotate_quantize_weights_q4_0",
    "q4_0_x_q4_gemm", "q4_0_x_q8_gemm", "q4_0_x_q4_gemm_experts", "h32_quantize_act_q4_tc",
    "h32_quantize_act_q8_tc", "h32_prepack_weights_q4_0_tc", "q4_0_x_q4_gemm_tc",
    "q4_0_x_q8_gemm_tc", "h32_quantize_act_q4_tc_gather", "q4_0_x_q4_gemm_tc_experts",
    "q4_0_x_q4_gemm_tc_quant_next", "h32_moe_route", "h32_moe_combine",
)
for _name in _COMPUTE_CALLS:
    globals()[_name] = _trace.traced(_name)(globals()[_name])
del _name
