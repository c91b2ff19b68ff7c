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
    "h32_quantize_act_q4_tc_e5m2", "h32_quantize_act_q4_tc_e5m2_gather",
    "q4_0_x_q4_gemm_tc_widen", "q4_0_x_q4_gemm_tc_widen_experts",
    "h32_q4_0_blocks_to_planes", "h32_q4_0_planes_to_blocks",
    "h32_gemm_tc_workspace_bytes", "h32_gemm_tc_schedule",
    "q4_0_x_q4_gemm_tc_noalloc", "q4_0_x_q8_gemm_tc_noalloc",
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
    "h32_gemm_tc_workspace_bytes": (_INT, [_I64, _I64, _I64, ctypes.POINTER(ctypes.c_size_t)]),
    "h32_gemm_tc_schedule": (_INT, [_I64, _I64, _I64, _I32, _I32, ctypes.POINTER(ctypes.c_int64)]),
    "q4_0_x_q4_gemm_tc_quant_next_ws": (_INT, [_P, _P, _I64, _P, _P, _I64, _I64, _I64, _I64, _P,
                                               _I64, _P, _P, _I64, _INT, _P, ctypes.c_size_t, _P]),
    "q4_0_x_q4_gemm_tc_noalloc": (_INT, [_P, _P, _I64, _P, _P, _I64, _I64, _I64, _I64, _P, _I64,
                                         _P, _P]),
    "q4_0_x_q8_gemm_tc_noalloc": (_INT, [_P, _P, _I64, _P, _P, _I64, _I64, _I64, _I64, _P, _I64,
                                         _P, _P]),
    "q4_0_x_q4_gemm_tc_ws": (_INT, [_P, _P, _I64, _P, _P, _I64, _I64, _I64, _I64, _P, _I64, _P,
                                    _P, ctypes.c_size_t, _P]),
    "q4_0_x_q8_gemm_tc_ws": (_INT, [_P, _P, _I64, _P, _P, _I64, _I64, _I64, _I64, _P, _I64, _P,
                                    _P, ctypes.c_size_t, _P]),
    "h32_q4_0_blocks_to_planes": (_INT, [_P, _I64, _I64, _P, _P, _P]),
    "h32_q4_0_planes_to_blocks": (_INT, [_P, _P, _I64, _I64, _P, _P]),
    "h32_quantize_act_q4_tc_e5m2": (_INT, [_P, _INT, _I64, _I64, _I64, _P, _P, _I64, _INT, _P]),
    "h32_quantize_act_q4_tc_e5m2_gather": (_INT, [_P, _INT, _I64, _I64, _I64, _P, _I64, _P, _P,
                                                  _I64, _INT, _P]),
    "q4_0_x_q4_gemm_tc_widen": (_INT, [_P, _P, _P, _P, _I64, _I64, _I64, _I64, _P, _I64, _P, _P]),
    "q4_0_x_q4_gemm_tc_widen_experts": (_INT, [_P, _P, ctypes.c_int32, _P, _P, _I64, _P, _I64,
                                               _I64, _I64, _P, _I64, _P, _P]),
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


def _rows(t, name):
    """2-D tensor with unit stride in its last dimension; returns its row pitch."""
    if t.dim() != 2 or (t.shape[1] > 1 and t.stride(1) != 1):
        raise ValueError(f"{name} must be 2-D with a contiguous last dimension")
    return t.stride(0) if t.shape[0] > 1 else t.shape[1]


class _AtLeast(int):
    """A shape entry the tensor may exceed (rows beyond those used, a row pitch)."""


def _ge(n) -> _AtLeast:
    return _AtLeast(int(n))


def _fp16_bits():
    torch = _torch()
    return tuple(d for d in (torch.int16, getattr(torch, "uint16", None), torch.float16) if d)


def _need(t, name, dtypes, shape, pitched=False):
    """Check a tensor the library reaches only through a raw pointer, so that no
    kernel reads or writes past it: dtype, shape (entries made with _ge may be
    exceeded, the others must match) and layout (contiguous, or with `pitched`
    2-D rows of unit stride that do not overlap).  Returns the tensor; the
    device is checked by _same_gpu once all of a call's tensors are."""
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch tensor")
    if t.dtype not in dtypes:
        raise ValueError(f"{name}: dtype {t.dtype}, expected " + " or ".join(map(str, dtypes)))
    want = "(" + ", ".join((">=" if isinstance(d, _AtLeast) else "") + str(int(d))
                           for d in shape) + ")"
    if t.dim() != len(shape) or any(h < d or (not isinstance(d, _AtLeast) and h != d)
                                    for h, d in zip(t.shape, shape)):
        raise ValueError(f"{name}: shape {tuple(t.shape)}, expected {want}")
    if pitched:
        if t.dim() != 2 or (t.shape[1] > 1 and t.stride(1) != 1) or \
                (t.shape[0] > 1 and t.stride(0) < t.shape[1]):
            raise ValueError(f"{name} must be 2-D with contiguous, non-overlapping rows")
    elif not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _same_gpu(*named):
    """Every (name, tensor) given (None skipped) is on one CUDA device."""
    dev = None
    for name, t in named:
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if dev is None:
            dev = t.device
        elif t.device != dev:
            raise ValueError(f"{name} is on {t.device}, the call's other tensors on {dev}")


def _act_dtype(x, name="x"):
    torch = _torch()
    if x.dtype == torch.bfloat16:
        return H32_IN_BF16
    if x.dtype == torch.float32:
        return H32_IN_F32
    raise ValueError(f"{name} must be bf16 or fp32")


def _sums(block_sums, rows, N, nb, dev):
    """The optional block-sum output: True allocates it, a tensor is checked."""
    torch = _torch()
    if block_sums is True:
        return torch.empty((rows, N, nb), dtype=torch.int32, device=dev)
    if block_sums is None or block_sums is False:
        return None
    return _need(block_sums, "block_sums", (torch.int32,), (_ge(rows), N, nb))


# --------------------------------------------------------------------------
# quantizers
# --------------------------------------------------------------------------
def _quantize_act(fn_name, bits, x, rotate, xq, xd, stream):
    torch = _torch()
    dt = _act_dtype(x)
    _need(x, "x", (x.dtype,), (_ge(0), _ge(0)), pitched=True)
    ldx = _rows(x, "x")
    M, K = x.shape
    dev = x.device
    qcols, qtype = (K // 2, torch.uint8) if bits == 4 else (K, torch.int8)
    if xq is None:
        xq = torch.empty((M, qcols), dtype=qtype, device=dev)
    # code buffers are raw bytes: 8-bit codes may sit in an int8 or a uint8 tensor
    _need(xq, "xq", (qtype,) if bits == 4 else (torch.int8, torch.uint8), (_ge(M), qcols))
    if xd is None:
        xd = torch.empty((M, K // 32), dtype=torch.float32, device=dev)
    _need(xd, "xd", (torch.float32,), (_ge(M), K // 32))
    _same_gpu(("x", x), ("xq", xq), ("xd", xd))
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
    if not isinstance(w, torch.Tensor) or w.dim() != 2:
        raise ValueError("w must be a contiguous 2-D fp32 tensor")
    N, K = w.shape
    _need(w, "w", (torch.float32,), (N, K))
    if wq is None:
        wq = torch.empty((N, K // 2), dtype=torch.uint8, device=w.device)
    _need(wq, "wq", (torch.uint8,), (_ge(N), K // 2))
    if wd is None:
        wd = torch.empty((N, K // 32), dtype=torch.int16, device=w.device)
    _need(wd, "wd", _fp16_bits(), (_ge(N), K // 32))
    _same_gpu(("w", w), ("wq", wq), ("wd", wd))
    st = lib().h32_rotate_quantize_weights_q4_0(_ptr(w), N, K, _rot_arg(rotate), _ptr(wq),
                                                _ptr(wd), _stream(stream))
    _check("h32_rotate_quantize_weights_q4_0", st)
    return wq, wd


# --------------------------------------------------------------------------
# GEMMs
# --------------------------------------------------------------------------
def h32_q4_0_blocks_to_planes(blocks, wq=None, wd=None, stream=None):
    """Q4_0 file blocks uint8 [N][K/32][18] (fp16 d, then 16 code bytes) -> the planes
    (wq [N][K/2] uint8, wd [N][K/32] int16 fp16 bits)."""
    torch = _torch()
    if blocks.dim() != 3 or blocks.shape[2] != 18:
        raise ValueError("blocks must be [N][K/32][18]")
    N, nb = blocks.shape[0], blocks.shape[1]
    K = nb * 32
    dev = blocks.device
    _need(blocks, "blocks", (torch.uint8,), (N, nb, 18))
    if wq is None:
        wq = torch.empty((N, K // 2), dtype=torch.uint8, device=dev)
    if wd is None:
        wd = torch.empty((N, nb), dtype=torch.int16, device=dev)
    _need(wq, "wq", (torch.uint8,), (N, K // 2))
    _need(wd, "wd", _fp16_bits(), (N, nb))
    _same_gpu(("blocks", blocks), ("wq", wq), ("wd", wd))
    st = lib().h32_q4_0_blocks_to_planes(_ptr(blocks), N, K, _ptr(wq), _ptr(wd), _stream(stream))
    _check("h32_q4_0_blocks_to_planes", st)
    return wq, wd


def h32_q4_0_planes_to_blocks(wq, wd, blocks=None, stream=None):
    """The planes (wq [N][K/2], wd [N][K/32]) -> Q4_0 file blocks uint8 [N][K/32][18]."""
    torch = _torch()
    if wq.dim() != 2:
        raise ValueError("wq must be 2-D [N][K/2]")
    N, K = wq.shape[0], wq.shape[1] * 2
    dev = wq.device
    _need(wq, "wq", (torch.uint8,), (N, K // 2))
    _need(wd, "wd", _fp16_bits(), (N, K // 32))
    if blocks is None:
        blocks = torch.empty((N, K // 32, 18), dtype=torch.uint8, device=dev)
    _need(blocks, "blocks", (torch.uint8,), (N, K // 32, 18))
    _same_gpu(("wq", wq), ("wd", wd), ("blocks", blocks))
    st = lib().h32_q4_0_planes_to_blocks(_ptr(wq), _ptr(wd), N, K, _ptr(blocks), _stream(stream))
    _check("h32_q4_0_planes_to_blocks", st)
    return blocks


def _gemm(fn_name, wq, wd, xq, xd, y, block_sums, stream):
    torch = _torch()
    if wq.dim() != 2 or xq.dim() != 2:
        raise ValueError("wq and xq must be 2-D")
    N, K = wq.shape[0], wq.shape[1] * 2
    M = xq.shape[0]
    dev = wq.device
    _need(wq, "wq", (torch.uint8,), (N, K // 2))
    _need(wd, "wd", _fp16_bits(), (_ge(N), K // 32))
    if fn_name == "q4_0_x_q8_gemm":
        _need(xq, "xq", (torch.int8, torch.uint8), (M, K))
    else:
        _need(xq, "xq", (torch.uint8,), (M, K // 2))
    _need(xd, "xd", (torch.float32,), (_ge(M), K // 32))
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=dev)
    _need(y, "y", (torch.float32,), (_ge(M), _ge(N)), pitched=True)
    ldy = _rows(y, "y")
    S = _sums(block_sums, M, N, K // 32, dev)
    _same_gpu(("wq", wq), ("wd", wd), ("xq", xq), ("xd", xd), ("y", y), ("S", S))
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
    if wq.dim() != 3 or xq.dim() != 2:
        raise ValueError("wq must be 3-D [E][N][K/2] and xq 2-D")
    E, N, K = wq.shape[0], wq.shape[1], wq.shape[2] * 2
    T = xq.shape[0]
    dev = wq.device
    _need(wq, "wq", (torch.uint8,), (E, N, K // 2))
    _need(wd, "wd", _fp16_bits(), (E, N, K // 32))
    _need(xq, "xq", (torch.uint8,), (T, K // 2))
    _need(xd, "xd", (torch.float32,), (_ge(T), K // 32))
    if row_idx is not None:
        _need(row_idx, "row_idx", (torch.int32,), (_ge(R),))
    elif T < R:
        raise ValueError("without row_idx, xq must have at least R rows")
    _need(expert_off, "expert_off", (torch.int32,), (_ge(E + 1),))
    if y is None:
        y = torch.empty((R, N), dtype=torch.float32, device=dev)
    _need(y, "y", (torch.float32,), (_ge(R), _ge(N)), pitched=True)
    ldy = _rows(y, "y")
    S = _sums(block_sums, R, N, K // 32, dev)
    _same_gpu(("wq", wq), ("wd", wd), ("xq", xq), ("xd", xd),
              ("row_idx", row_idx), ("expert_off", expert_off), ("y", y), ("S", S))
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


def h32_quantize_act_q4_tc_e5m2(x, rotate=True, xw=None, xdt=None, stream=None):
    """As h32_quantize_act_q4_tc with each code c stored as the e5m2 byte of 512 c
    (the activations of the widening GEMMs)."""
    return _quantize_tc("h32_quantize_act_q4_tc_e5m2", 1, x, rotate, xw, xdt, stream)


def h32_quantize_act_q8_tc(x, rotate=True, xw=None, xdt=None, stream=None):
    """x [M][K] bf16/fp32 -> (xw8 [M][2K] uint8: per 32-block the e4m3 bytes of 16 h
    then of l, code = 16 h + l; xdt [K/32][ldxd] fp32 scales)."""
    return _quantize_tc("h32_quantize_act_q8_tc", 2, x, rotate, xw, xdt, stream)


def _quantize_tc(fn, bytes_per_code, x, rotate, xw, xdt, stream):
    torch = _torch()
    dt = _act_dtype(x)
    _need(x, "x", (x.dtype,), (_ge(0), _ge(0)), pitched=True)
    ldx = _rows(x, "x")
    M, K = x.shape
    dev = x.device
    if xw is None:
        xw = torch.empty((M, K * bytes_per_code), dtype=torch.uint8, device=dev)
    _need(xw, "xw", (torch.uint8,), (_ge(M), K * bytes_per_code))
    if xdt is None:
        xdt = torch.zeros((K // 32, _round4(M)), dtype=torch.float32, device=dev)
    _need(xdt, "xdt", (torch.float32,), (_ge(K // 32), _ge(M)))
    _same_gpu(("x", x), ("xw", xw), ("xdt", xdt))
    st = getattr(lib(), fn)(_ptr(x), dt, M, K, ldx, _ptr(xw), _ptr(xdt), xdt.shape[1],
                            _rot_arg(rotate), _stream(stream))
    _check(fn, st)
    return xw, xdt


def h32_prepack_weights_q4_0_tc(wq, wd, wp=None, wsc=None, stream=None):
    """Q4_0 planes (wq [N][K/2], wd [N][K/32] fp16 bits) -> tc form
    (wp [N][K] uint8, wsc [N][ldws] fp32 = d, ldws = K/32 rounded up to 4)."""
    torch = _torch()
    if wq.dim() != 2:
        raise ValueError("wq must be 2-D [N][K/2]")
    N, K = wq.shape[0], wq.shape[1] * 2
    dev = wq.device
    _need(wq, "wq", (torch.uint8,), (N, K // 2))
    _need(wd, "wd", _fp16_bits(), (_ge(N), K // 32))
    if wp is None:
        wp = torch.empty((N, K), dtype=torch.uint8, device=dev)
    _need(wp, "wp", (torch.uint8,), (_ge(N), K))
    if wsc is None:
        wsc = torch.empty((N, _round4(K // 32)), dtype=torch.float32, device=dev)
    _need(wsc, "wsc", (torch.float32,), (_ge(N), _ge(K // 32)))
    _same_gpu(("wq", wq), ("wd", wd), ("wp", wp), ("wsc", wsc))
    st = lib().h32_prepack_weights_q4_0_tc(_ptr(wq), _ptr(wd), N, K, _ptr(wp), _ptr(wsc),
                                           wsc.shape[1], _stream(stream))
    _check("h32_prepack_weights_q4_0_tc", st)
    return wp, wsc


def q4_0_x_q4_gemm_tc(wp, wsc, xw, xdt, M=None, y=None, block_sums=None, stream=None,
                      workspace=None):
    """The W4A4 product on tc-form operands (bit-identical to q4_0_x_q4_gemm).

    workspace: None (default) lets shapes whose schedule splits the last wave's
    pieces along K use a workspace the binding keeps per device and stream; False
    calls q4_0_x_q4_gemm_tc (no split); a uint8 CUDA tensor (zero-filled before
    its first use, used by one call at a time) is passed as given."""
    return _gemm_tc("q4_0_x_q4_gemm_tc", wp, wsc, xw, xdt, M, y, block_sums, stream, workspace)


def q4_0_x_q8_gemm_tc(wp, wsc, xw8, xdt, M=None, y=None, block_sums=None, stream=None,
                      workspace=None):
    """The W4A8 product on tc-form operands (bit-identical to q4_0_x_q8_gemm);
    workspace as for q4_0_x_q4_gemm_tc."""
    return _gemm_tc("q4_0_x_q8_gemm_tc", wp, wsc, xw8, xdt, M, y, block_sums, stream, workspace)


def q4_0_x_q4_gemm_tc_noalloc(wp, wsc, xw, xdt, M=None, y=None, block_sums=None, stream=None):
    """q4_0_x_q4_gemm_tc with the K split on the library's static per-device
    workspace: no allocation by the call (calls sharing a device are ordered)."""
    return _gemm_tc("q4_0_x_q4_gemm_tc", wp, wsc, xw, xdt, M, y, block_sums, stream, "noalloc")


def q4_0_x_q8_gemm_tc_noalloc(wp, wsc, xw8, xdt, M=None, y=None, block_sums=None, stream=None):
    """q4_0_x_q8_gemm_tc on the library's static workspace (as the 4-bit form)."""
    return _gemm_tc("q4_0_x_q8_gemm_tc", wp, wsc, xw8, xdt, M, y, block_sums, stream, "noalloc")


def h32_gemm_tc_workspace_bytes(M: int, N: int, K: int) -> int:
    """Workspace bytes q4_0_x_q4_gemm_tc_ws / q4_0_x_q8_gemm_tc_ws use for an
    M x N x K product on the current device (0: the schedule does not split)."""
    n = ctypes.c_size_t(0)
    _check("h32_gemm_tc_workspace_bytes",
           lib().h32_gemm_tc_workspace_bytes(int(M), int(N), int(K), ctypes.byref(n)))
    return int(n.value)


TC_SCHEDULE_KEYS = ("bn", "tail_k", "tail_first", "total", "grid", "split_p", "split_kh",
                    "ws_ld", "ws_bytes")


def h32_gemm_tc_schedule(M: int, N: int, K: int, sms: int, with_workspace: bool = True) -> dict:
    """The dense tc GEMM's schedule for an M x N x K product on `sms` SMs (host
    arithmetic, no device): tile width, the cut and the K split of the last wave."""
    out = (ctypes.c_int64 * 9)()
    _check("h32_gemm_tc_schedule", lib().h32_gemm_tc_schedule(int(M), int(N), int(K), int(sms),
                                                             int(bool(with_workspace)), out))
    return dict(zip(TC_SCHEDULE_KEYS, (int(v) for v in out)))


# workspaces kept per (device, stream); a grown workspace keeps the old one
# alive, since a captured CUDA graph may still use it
_workspaces = {}
_retired_workspaces = []


def _workspace_for(M, N, K, dev, stream):
    torch = _torch()
    need = h32_gemm_tc_workspace_bytes(M, N, K)
    if need == 0:
        return None
    if torch.cuda.is_current_stream_capturing():
        # inside a capture: a workspace of the graph's own, zeroed on every replay
        return torch.zeros(need, dtype=torch.uint8, device=dev)
    key = (dev.index, _stream(stream).value)
    ws = _workspaces.get(key)
    if ws is None or ws.numel() < need:
        if ws is not None:
            _retired_workspaces.append(ws)
        ws = torch.zeros(need, dtype=torch.uint8, device=dev)
        _workspaces[key] = ws
    return ws


def _tc_operands(wp, wsc, xw, xdt, rows, bytes_per_code, weight_rows=None):
    """Check the tc-form operands of a GEMM over `rows` activation rows; returns (N, K)."""
    torch = _torch()
    if wp.dim() != 2:
        raise ValueError("wp must be 2-D [N][K]")
    N, K = wp.shape
    dev = wp.device
    _need(wp, "wp", (torch.uint8,), (N, K))
    _need(wsc, "wsc", (torch.float32,), (N, _ge(K // 32)))
    _need(xw, "xw", (torch.uint8,), (_ge(rows), K * bytes_per_code))
    _need(xdt, "xdt", (torch.float32,), (_ge(K // 32), _ge(rows)))
    return N, K


def _gemm_tc(fn, wp, wsc, xw, xdt, M, y, block_sums, stream, workspace=False):
    torch = _torch()
    if M is None:
        M = xw.shape[0]
    N, K = _tc_operands(wp, wsc, xw, xdt, M, 2 if fn == "q4_0_x_q8_gemm_tc" else 1)
    dev = wp.device
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=dev)
    _need(y, "y", (torch.float32,), (_ge(M), _ge(N)), pitched=True)
    ldy = _rows(y, "y")
    S = _sums(block_sums, M, N, K // 32, dev)
    explicit_ws = workspace is not None and workspace is not False and not isinstance(workspace, str)
    if explicit_ws:
        _need(workspace, "workspace", (torch.uint8,), (_ge(0),))
    _same_gpu(("wp", wp), ("wsc", wsc), ("xw", xw), ("xdt", xdt), ("y", y), ("S", S),
              ("workspace", workspace if explicit_ws else None))
    if isinstance(workspace, str) and workspace == "noalloc":
        fn = fn + "_noalloc"
        st = getattr(lib(), fn)(_ptr(wp), _ptr(wsc), wsc.shape[1], _ptr(xw), _ptr(xdt),
                                xdt.shape[1], M, N, K, _ptr(y), ldy, _ptr(S), _stream(stream))
        _check(fn, st)
        return (y, S) if S is not None else y
    ws = None
    if workspace is None and S is None and M > 0:
        ws = _workspace_for(M, N, K, dev, stream)
    elif explicit_ws:
        ws = workspace
    if ws is None:
        st = getattr(lib(), fn)(_ptr(wp), _ptr(wsc), wsc.shape[1], _ptr(xw), _ptr(xdt),
                                xdt.shape[1], M, N, K, _ptr(y), ldy, _ptr(S), _stream(stream))
    else:
        fn = fn + "_ws"
        st = getattr(lib(), fn)(_ptr(wp), _ptr(wsc), wsc.shape[1], _ptr(xw), _ptr(xdt),
                                xdt.shape[1], M, N, K, _ptr(y), ldy, _ptr(S), _ptr(ws),
                                ws.numel(), _stream(stream))
    _check(fn, st)
    return (y, S) if S is not None else y


def _widen_operands(wq, wd, xw, xdt, rows):
    """Check Q4_0 weight planes and tc-form activations over `rows` rows; returns (N, K)."""
    torch = _torch()
    if wq.dim() != 2:
        raise ValueError("wq must be 2-D [N][K/2]")
    N, K = wq.shape[0], wq.shape[1] * 2
    _need(wq, "wq", (torch.uint8,), (N, K // 2))
    _need(wd, "wd", _fp16_bits(), (N, K // 32))
    _need(xw, "xw", (torch.uint8,), (_ge(rows), K))
    _need(xdt, "xdt", (torch.float32,), (_ge(K // 32), _ge(rows)))
    return N, K


def q4_0_x_q4_gemm_tc_widen(wq, wd, xw, xdt, M=None, y=None, block_sums=None, stream=None):
    """The W4A4 product on the Q4_0 planes (wq [N][K/2], wd [N][K/32] fp16 bits),
    widened in shared memory, against activations from
    h32_quantize_act_q4_tc_e5m2; bit-identical to q4_0_x_q4_gemm_tc."""
    torch = _torch()
    if M is None:
        M = xw.shape[0]
    N, K = _widen_operands(wq, wd, xw, xdt, M)
    dev = wq.device
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=dev)
    _need(y, "y", (torch.float32,), (_ge(M), _ge(N)), pitched=True)
    ldy = _rows(y, "y")
    S = _sums(block_sums, M, N, K // 32, dev)
    _same_gpu(("wq", wq), ("wd", wd), ("xw", xw), ("xdt", xdt), ("y", y), ("S", S))
    st = lib().q4_0_x_q4_gemm_tc_widen(_ptr(wq), _ptr(wd), _ptr(xw), _ptr(xdt), xdt.shape[1], M, N,
                                       K, _ptr(y), ldy, _ptr(S), _stream(stream))
    _check("q4_0_x_q4_gemm_tc_widen", st)
    return (y, S) if S is not None else y


def q4_0_x_q4_gemm_tc_widen_experts(wq, wd, xw, xdt, expert_off, N, R=None, y=None,
                                    block_sums=None, stream=None):
    """Expert-batched product on the experts' Q4_0 planes stacked as E * N rows
    (wq [E*N][K/2], wd [E*N][K/32]), widened in shared memory; xw / xdt in grouped
    order from h32_quantize_act_q4_tc_e5m2_gather, expert_off [E+1] int32 -> y [R][N]
    fp32 in grouped order."""
    torch = _torch()
    if wq.dim() != 2 or N <= 0 or wq.shape[0] % N != 0:
        raise ValueError("wq must be 2-D with E * N rows")
    E = wq.shape[0] // N
    if R is None:
        R = xw.shape[0]
    EN, K = _widen_operands(wq, wd, xw, xdt, R)
    dev = wq.device
    _need(expert_off, "expert_off", (torch.int32,), (_ge(E + 1),))
    if y is None:
        y = torch.empty((R, N), dtype=torch.float32, device=dev)
    _need(y, "y", (torch.float32,), (_ge(R), _ge(N)), pitched=True)
    ldy = _rows(y, "y") if R > 0 else N
    S = _sums(block_sums, R, N, K // 32, dev)
    _same_gpu(("wq", wq), ("wd", wd), ("xw", xw), ("xdt", xdt),
              ("expert_off", expert_off), ("y", y), ("S", S))
    st = lib().q4_0_x_q4_gemm_tc_widen_experts(_ptr(wq), _ptr(wd), E, _ptr(xw), _ptr(xdt),
                                               xdt.shape[1], _ptr(expert_off), R, N, K, _ptr(y),
                                               ldy, _ptr(S), _stream(stream))
    _check("q4_0_x_q4_gemm_tc_widen_experts", st)
    return (y, S) if S is not None else y


def h32_quantize_act_q4_tc_gather(x, row_idx, rotate=True, xw=None, xdt=None, stream=None):
    """x [T][K] bf16/fp32, row_idx [R] int32 -> (xw [R][K] uint8, xdt [K/32][ldxd] fp32):
    output row r is the tc-form quantization of x[row_idx[r]]."""
    return _quantize_tc_gather("h32_quantize_act_q4_tc_gather", x, row_idx, rotate, xw, xdt,
                               stream)


def h32_quantize_act_q4_tc_e5m2_gather(x, row_idx, rotate=True, xw=None, xdt=None, stream=None):
    """The row gather of h32_quantize_act_q4_tc_e5m2 (activations of the widening
    expert GEMM in grouped order)."""
    return _quantize_tc_gather("h32_quantize_act_q4_tc_e5m2_gather", x, row_idx, rotate, xw, xdt,
                               stream)


def _quantize_tc_gather(fn, x, row_idx, rotate, xw, xdt, stream):
    torch = _torch()
    dt = _act_dtype(x)
    _need(x, "x", (x.dtype,), (_ge(0), _ge(0)), pitched=True)
    ldx = _rows(x, "x")
    T, K = x.shape
    dev = x.device
    if row_idx.dim() != 1:
        raise ValueError("row_idx must be 1-D")
    R = row_idx.shape[0]
    _need(row_idx, "row_idx", (torch.int32,), (R,))
    if xw is None:
        xw = torch.empty((R, K), dtype=torch.uint8, device=dev)
    _need(xw, "xw", (torch.uint8,), (_ge(R), K))
    if xdt is None:
        xdt = torch.zeros((K // 32, _round4(R)), dtype=torch.float32, device=dev)
    _need(xdt, "xdt", (torch.float32,), (_ge(K // 32), _ge(R)))
    _same_gpu(("x", x), ("row_idx", row_idx), ("xw", xw), ("xdt", xdt))
    st = getattr(lib(), fn)(_ptr(x), dt, T, K, ldx, _ptr(row_idx), R, _ptr(xw), _ptr(xdt),
                            xdt.shape[1], _rot_arg(rotate), _stream(stream))
    _check(fn, st)
    return xw, xdt


def q4_0_x_q4_gemm_tc_experts(wp, wsc, xw, xdt, expert_off, N, R=None, y=None, block_sums=None,
                              stream=None):
    """Expert-batched tc GEMM.  wp [E*N][K] uint8, wsc [E*N][ldws] fp32 (the experts'
    repacked planes stacked), xw [R][K] / xdt [K/32][ldxd] in grouped order,
    expert_off [E+1] int32 -> y [R][N] fp32 in grouped order."""
    torch = _torch()
    if wp.dim() != 2 or N <= 0 or wp.shape[0] % N != 0:
        raise ValueError("wp must be 2-D with E * N rows")
    E = wp.shape[0] // N
    if R is None:
        R = xw.shape[0]
    EN, K = _tc_operands(wp, wsc, xw, xdt, R, 1)
    dev = wp.device
    _need(expert_off, "expert_off", (torch.int32,), (_ge(E + 1),))
    if y is None:
        y = torch.empty((R, N), dtype=torch.float32, device=dev)
    _need(y, "y", (torch.float32,), (_ge(R), _ge(N)), pitched=True)
    ldy = _rows(y, "y") if R > 0 else N
    S = _sums(block_sums, R, N, K // 32, dev)
    _same_gpu(("wp", wp), ("wsc", wsc), ("xw", xw), ("xdt", xdt),
              ("expert_off", expert_off), ("y", y), ("S", S))
    st = lib().q4_0_x_q4_gemm_tc_experts(_ptr(wp), _ptr(wsc), wsc.shape[1], E, _ptr(xw), _ptr(xdt),
                                         xdt.shape[1], _ptr(expert_off), R, N, K, _ptr(y), ldy,
                                         _ptr(S), _stream(stream))
    _check("q4_0_x_q4_gemm_tc_experts", st)
    return (y, S) if S is not None else y


def q4_0_x_q4_gemm_tc_quant_next(wp, wsc, xw, xdt, M=None, y=None, want_y=True, rotate_next=True,
                                 xw_next=None, xdt_next=None, stream=None, workspace=None):
    """The tc W4A4 product with its output also quantized for the next projection
    in the same kernel.  Returns (y or None, xw_next [M][N] uint8, xdt_next
    [N/32][ldxd] fp32).  workspace as for q4_0_x_q4_gemm_tc (the K split)."""
    torch = _torch()
    if M is None:
        M = xw.shape[0]
    N, K = _tc_operands(wp, wsc, xw, xdt, M, 1)
    dev = wp.device
    if y is None and want_y:
        y = torch.empty((M, N), dtype=torch.float32, device=dev)
    if y is not None:
        _need(y, "y", (torch.float32,), (_ge(M), _ge(N)), pitched=True)
    ldy = _rows(y, "y") if y is not None else N
    if xw_next is None:
        xw_next = torch.empty((M, N), dtype=torch.uint8, device=dev)
    _need(xw_next, "xw_next", (torch.uint8,), (_ge(M), N))
    if xdt_next is None:
        xdt_next = torch.zeros((N // 32, _round4(M)), dtype=torch.float32, device=dev)
    _need(xdt_next, "xdt_next", (torch.float32,), (_ge(N // 32), _ge(M)))
    explicit_ws = workspace is not None and workspace is not False
    if explicit_ws:
        _need(workspace, "workspace", (torch.uint8,), (_ge(0),))
    _same_gpu(("wp", wp), ("wsc", wsc), ("xw", xw), ("xdt", xdt),
              ("y", y), ("xw_next", xw_next), ("xdt_next", xdt_next),
              ("workspace", workspace if explicit_ws else None))
    ws = None
    if workspace is None and M > 0:
        ws = _workspace_for(M, N, K, dev, stream)
    elif explicit_ws:
        ws = workspace
    if ws is None:
        st = lib().q4_0_x_q4_gemm_tc_quant_next(
            _ptr(wp), _ptr(wsc), wsc.shape[1], _ptr(xw), _ptr(xdt), xdt.shape[1], M, N, K, _ptr(y),
            ldy, _ptr(xw_next), _ptr(xdt_next), xdt_next.shape[1], _rot_arg(rotate_next),
            _stream(stream))
        _check("q4_0_x_q4_gemm_tc_quant_next", st)
    else:
        st = lib().q4_0_x_q4_gemm_tc_quant_next_ws(
            _ptr(wp), _ptr(wsc), wsc.shape[1], _ptr(xw), _ptr(xdt), xdt.shape[1], M, N, K, _ptr(y),
            ldy, _ptr(xw_next), _ptr(xdt_next), xdt_next.shape[1], _rot_arg(rotate_next),
            _ptr(ws), ws.numel(), _stream(stream))
        _check("q4_0_x_q4_gemm_tc_quant_next_ws", st)
    return y, xw_next, xdt_next


def h32_moe_route(logits, k, topk_id=None, topk_w=None, expert_off=None, row_idx=None,
                  row_of=None, stream=None):
    """Router: logits [T][E] fp32 -> (topk_id [T][k] int32, topk_w [T][k] fp32,
    expert_off [E+1] int32, row_idx [T*k] int32, row_of [T][k] int32).  The k
    largest logits (ties: lower id), softmax weights over them, rows grouped by
    expert then token."""
    torch = _torch()
    _need(logits, "logits", (torch.float32,), (_ge(0), _ge(0)), pitched=True)
    T, E = logits.shape
    ldl = _rows(logits, "logits") if T > 0 else E
    dev = logits.device
    i32 = (torch.int32,)
    if topk_id is None:
        topk_id = torch.empty((T, k), dtype=torch.int32, device=dev)
    _need(topk_id, "topk_id", i32, (_ge(T), k))
    if topk_w is None:
        topk_w = torch.empty((T, k), dtype=torch.float32, device=dev)
    _need(topk_w, "topk_w", (torch.float32,), (_ge(T), k))
    if expert_off is None:
        expert_off = torch.empty(E + 1, dtype=torch.int32, device=dev)
    _need(expert_off, "expert_off", i32, (_ge(E + 1),))
    if row_idx is None:
        row_idx = torch.empty(T * k, dtype=torch.int32, device=dev)
    _need(row_idx, "row_idx", i32, (_ge(T * k),))
    if row_of is None:
        row_of = torch.empty((T, k), dtype=torch.int32, device=dev)
    _need(row_of, "row_of", i32, (_ge(T), k))
    _same_gpu(("logits", logits), ("topk_id", topk_id), ("topk_w", topk_w), ("expert_off", expert_off),
              ("row_idx", row_idx), ("row_of", row_of))
    st = lib().h32_moe_route(_ptr(logits), T, E, ldl, k, _ptr(topk_id), _ptr(topk_w),
                             _ptr(expert_off), _ptr(row_idx), _ptr(row_of), _stream(stream))
    _check("h32_moe_route", st)
    return topk_id, topk_w, expert_off, row_idx, row_of


def h32_moe_combine(y, row_of, topk_w, out=None, stream=None):
    """Weighted combine: y [R][H] fp32 (grouped rows), row_of [T][k], topk_w [T][k]
    -> out [T][H] fp32, the token's k rows added in choice order (fp32 fma from 0)."""
    torch = _torch()
    _need(y, "y", (torch.float32,), (_ge(0), _ge(0)), pitched=True)
    R, H = y.shape
    dev = y.device
    if row_of.dim() != 2:
        raise ValueError("row_of must be 2-D [T][k]")
    T, k = row_of.shape
    _need(row_of, "row_of", (torch.int32,), (T, k))
    _need(topk_w, "topk_w", (torch.float32,), (T, k))
    if out is None:
        out = torch.empty((T, H), dtype=torch.float32, device=dev)
    _need(out, "out", (torch.float32,), (_ge(T), _ge(H)), pitched=True)
    ldy = _rows(y, "y") if R > 0 else H
    ldo = _rows(out, "out") if T > 0 else H
    _same_gpu(("y", y), ("row_of", row_of), ("topk_w", topk_w), ("out", out))
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
    "h32_quantize_act_q4_tc_e5m2", "h32_quantize_act_q4_tc_e5m2_gather",
    "q4_0_x_q4_gemm_tc_widen", "q4_0_x_q4_gemm_tc_widen_experts",
    "h32_q4_0_blocks_to_planes", "h32_q4_0_planes_to_blocks",
    "q4_0_x_q4_gemm_tc_noalloc", "q4_0_x_q8_gemm_tc_noalloc",
)
for _name in _COMPUTE_CALLS:
    globals()[_name] = _trace.traced(_name)(globals()[_name])
del _name
