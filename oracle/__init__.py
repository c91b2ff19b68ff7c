"""Plain CPU oracle for the Hadamard route (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never imports it, and it shares no code with them.

The arithmetic lives in ``h32_oracle.c`` (plain C99, single threaded, built
with ``-O2 -ffp-contract=off``); this module compiles it on first use and wraps
each entry point for numpy arrays.  Each function's docstring names the
section of the pages it follows; the C file's header lists the readings taken
where the pages leave a step open.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "h32_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle_h32.so")

_lib = None
_lock = threading.Lock()

_P = ctypes.c_void_p
_I64 = ctypes.c_int64


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math, no FP contraction)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)) or (
        os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-std=gnu11", "-O2", "-ffp-contract=off", "-fno-fast-math",
               "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            sigs = {
                "o_bf16_to_f32": [_P, _P, _I64],
                "o_f32_to_f16": [_P, _P, _I64],
                "o_f16_to_f32": [_P, _P, _I64],
                "o_fwht32_f32": [_P, _P, _I64],
                "o_fwht32_f64": [_P, _P, _I64],
                "o_fwht_n_f32": [_P, _P, _I64, ctypes.c_int],
                "o_fwht_n_f64": [_P, _P, _I64, ctypes.c_int],
                "o_quantize_act": [_P, _I64, _I64, ctypes.c_int, ctypes.c_int, _P, _P],
                "o_quantize_weights_q4_0": [_P, _I64, _I64, ctypes.c_int, _P, _P],
                "o_decode_act4": [_P, _I64, _I64, _P],
                "o_decode_w4": [_P, _I64, _I64, _P],
                "o_gemm": [_P, _P, _P, _P, ctypes.c_int, _I64, _I64, _I64, _P, _P, _P],
                "o_gemm_sampled": [_P, _P, _P, _P, ctypes.c_int, _I64, _I64, _P, _P, _P, _P, _P],
                "o_gemm_experts_sampled": [_P, _P, _I64, _P, _P, _P, _P, _I64, _I64, _I64,
                                           _P, _P, _P, _P, _P],
                "o_moe_route": [_P, _I64, _I64, _I64, _P, _P, _P, _P, _P],
                "o_moe_combine": [_P, _I64, _P, _P, _I64, _I64, _I64, _P],
            }
            for name, args in sigs.items():
                fn = getattr(lib, name)
                fn.argtypes = args
                fn.restype = None
            lib.o_h32_scale.argtypes = []
            lib.o_h32_scale.restype = ctypes.c_float
            lib.o_rot_scale.argtypes = [ctypes.c_int]
            lib.o_rot_scale.restype = ctypes.c_float
            _lib = lib
    return _lib


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# --------------------------------------------------------------------------
# conversions
# --------------------------------------------------------------------------
def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 (given as uint16 bits) to fp32 exactly (step 1 of the path)."""
    bits = _c(bits, np.uint16)
    out = np.empty(bits.shape, np.float32)
    _load().o_bf16_to_f32(_ptr(bits), _ptr(out), bits.size)
    return out


def f32_to_f16(x: np.ndarray) -> np.ndarray:
    """fp32 -> fp16 bits, round to nearest even (the Q4_0 scale format)."""
    x = _c(x, np.float32)
    out = np.empty(x.shape, np.uint16)
    _load().o_f32_to_f16(_ptr(x), _ptr(out), x.size)
    return out


def f16_to_f32(bits: np.ndarray) -> np.ndarray:
    bits = _c(bits, np.uint16)
    out = np.empty(bits.shape, np.float32)
    _load().o_f16_to_f32(_ptr(bits), _ptr(out), bits.size)
    return out


# --------------------------------------------------------------------------
# the rotation ("The rotation"; "Prompt processing: 4-bit activations, rotated first")
# --------------------------------------------------------------------------
def h32_scale() -> float:
    """The fp32 constant the rotation multiplies by (nearest to 1/sqrt(32))."""
    return float(_load().o_h32_scale())


def fwht32(x: np.ndarray) -> np.ndarray:
    """Rotate every consecutive 32-block of ``x`` (fp32, size % 32 == 0)."""
    x = _c(x, np.float32)
    assert x.size % 32 == 0
    out = np.empty_like(x)
    _load().o_fwht32_f32(_ptr(x), _ptr(out), x.size // 32)
    return out


def fwht32_f64(x: np.ndarray) -> np.ndarray:
    """Same butterfly in fp64 (for the x.w = (Hx).(Hw) check)."""
    x = _c(x, np.float64)
    assert x.size % 32 == 0
    out = np.empty_like(x)
    _load().o_fwht32_f64(_ptr(x), _ptr(out), x.size // 32)
    return out


# the larger rotations (the pages' next step: 64 and 128 points, scales per 32)
ROTATIONS = (32, 64, 128)


def rot_points(rotate) -> int:
    """The quantizers' `rotate` argument -> points of the transform (0 = none):
    False/0 -> 0, True/1/32 -> 32, 64 -> 64, 128 -> 128."""
    if rotate is True or rotate == 1:
        return 32
    if rotate is False or rotate == 0 or rotate is None:
        return 0
    n = int(rotate)
    assert n in ROTATIONS, f"rotation of {n} points is not supported"
    return n


def rot_scale(n: int) -> float:
    """The fp32 constant an n-point rotation multiplies by (nearest 1/sqrt(n))."""
    return float(_load().o_rot_scale(int(n)))


def fwht_n(x: np.ndarray, n: int) -> np.ndarray:
    """Rotate every consecutive n-block of ``x`` (fp32, size % n == 0)."""
    x = _c(x, np.float32)
    assert x.size % n == 0 and n in ROTATIONS
    out = np.empty_like(x)
    _load().o_fwht_n_f32(_ptr(x), _ptr(out), x.size, n)
    return out


def fwht_n_f64(x: np.ndarray, n: int) -> np.ndarray:
    x = _c(x, np.float64)
    assert x.size % n == 0 and n in ROTATIONS
    out = np.empty_like(x)
    _load().o_fwht_n_f64(_ptr(x), _ptr(out), x.size, n)
    return out


# --------------------------------------------------------------------------
# activation quantizers (4-bit route and the exact 8-bit route)
# --------------------------------------------------------------------------
def _widen(x: np.ndarray) -> np.ndarray:
    if x.dtype == np.uint16:  # bf16 bits
        return bf16_to_f32(x)
    return _c(x, np.float32)


def quantize_act_q4(x: np.ndarray, rotate=True):
    """x [M][K] (fp32, or bf16 as uint16 bits) -> (xq [M][K/2] u8, xd [M][K/32] f32).
    rotate: False / True (32 points) / 64 / 128."""
    xf = _widen(x)
    M, K = xf.shape
    n = rot_points(rotate)
    assert K % 32 == 0 and K % max(n, 1) == 0
    xq = np.empty((M, K // 2), np.uint8)
    xd = np.empty((M, K // 32), np.float32)
    _load().o_quantize_act(_ptr(xf), M, K, 4, n, _ptr(xq), _ptr(xd))
    return xq, xd


def quantize_act_q8(x: np.ndarray, rotate=True):
    """x [M][K] -> (xq [M][K] int8, xd [M][K/32] f32).  rotate as for quantize_act_q4."""
    xf = _widen(x)
    M, K = xf.shape
    n = rot_points(rotate)
    assert K % 32 == 0 and K % max(n, 1) == 0
    xq = np.empty((M, K), np.int8)
    xd = np.empty((M, K // 32), np.float32)
    _load().o_quantize_act(_ptr(xf), M, K, 8, n, _ptr(xq), _ptr(xd))
    return xq, xd


def quantize_weights_q4_0(w: np.ndarray, rotate=True):
    """w [N][K] fp32 -> (wq [N][K/2] u8 codes 0..15, wd [N][K/32] fp16 bits as u16).
    rotate as for quantize_act_q4."""
    w = _c(w, np.float32)
    N, K = w.shape
    n = rot_points(rotate)
    assert K % 32 == 0 and K % max(n, 1) == 0
    wq = np.empty((N, K // 2), np.uint8)
    wd = np.empty((N, K // 32), np.uint16)
    _load().o_quantize_weights_q4_0(_ptr(w), N, K, n, _ptr(wq), _ptr(wd))
    return wq, wd


def decode_act4(xq: np.ndarray, K: int) -> np.ndarray:
    xq = _c(xq, np.uint8)
    M = xq.shape[0]
    out = np.empty((M, K), np.int8)
    _load().o_decode_act4(_ptr(xq), M, K, _ptr(out))
    return out


def decode_w4(wq: np.ndarray, K: int) -> np.ndarray:
    wq = _c(wq, np.uint8)
    N = wq.shape[0]
    out = np.empty((N, K), np.int8)
    _load().o_decode_w4(_ptr(wq), N, K, _ptr(out))
    return out


# --------------------------------------------------------------------------
# block-scaled integer GEMM
# --------------------------------------------------------------------------
def _xbits(xq: np.ndarray) -> int:
    return 8 if xq.dtype == np.int8 else 4


def gemm(wq, wd, xq, xd, K: int, want_block_sums: bool = False):
    """All outputs: returns (y32 [M][N] fp32, y64 [M][N] fp64, S [M][N][K/32] int64 or None)."""
    wq, wd, xd = _c(wq, np.uint8), _c(wd, np.uint16), _c(xd, np.float32)
    xbits = _xbits(xq)
    xq = np.ascontiguousarray(xq)
    M, N = xq.shape[0], wq.shape[0]
    y32 = np.empty((M, N), np.float32)
    y64 = np.empty((M, N), np.float64)
    S = np.empty((M, N, K // 32), np.int64) if want_block_sums else None
    _load().o_gemm(_ptr(wq), _ptr(wd), _ptr(xq), _ptr(xd), xbits, M, N, K,
                   _ptr(y32), _ptr(y64), _ptr(S))
    return y32, y64, S


def gemm_sampled(wq, wd, xq, xd, K: int, m_idx, n_idx, want_block_sums: bool = False):
    """Outputs (m_idx[i], n_idx[i]) only: returns (y32 [P], y64 [P], S [P][K/32] or None)."""
    wq, wd, xd = _c(wq, np.uint8), _c(wd, np.uint16), _c(xd, np.float32)
    xbits = _xbits(xq)
    xq = np.ascontiguousarray(xq)
    m_idx, n_idx = _c(m_idx, np.int64), _c(n_idx, np.int64)
    P = m_idx.size
    y32 = np.empty(P, np.float32)
    y64 = np.empty(P, np.float64)
    S = np.empty((P, K // 32), np.int64) if want_block_sums else None
    _load().o_gemm_sampled(_ptr(wq), _ptr(wd), _ptr(xq), _ptr(xd), xbits, K, P,
                           _ptr(m_idx), _ptr(n_idx), _ptr(y32), _ptr(y64), _ptr(S))
    return y32, y64, S


def gemm_experts_sampled(wq, wd, xq, xd, row_idx, expert_off, N: int, K: int,
                         r_idx, n_idx, want_block_sums: bool = False):
    """Expert-batched GEMM at sampled (row, n) outputs; 4-bit activations.

    wq [E][N][K/2], wd [E][N][K/32]; row r of the grouped output uses expert e
    with expert_off[e] <= r < expert_off[e+1] and activation row row_idx[r]."""
    wq, wd, xq, xd = _c(wq, np.uint8), _c(wd, np.uint16), _c(xq, np.uint8), _c(xd, np.float32)
    E = wq.shape[0]
    ri = None if row_idx is None else _c(row_idx, np.int32)
    off = _c(expert_off, np.int32)
    r_idx, n_idx = _c(r_idx, np.int64), _c(n_idx, np.int64)
    P = r_idx.size
    y32 = np.empty(P, np.float32)
    y64 = np.empty(P, np.float64)
    S = np.empty((P, K // 32), np.int64) if want_block_sums else None
    _load().o_gemm_experts_sampled(_ptr(wq), _ptr(wd), E, _ptr(xq), _ptr(xd), _ptr(ri),
                                   _ptr(off), N, K, P, _ptr(r_idx), _ptr(n_idx),
                                   _ptr(y32), _ptr(y64), _ptr(S))
    return y32, y64, S


# --------------------------------------------------------------------------
# routing and the weighted combine around the expert GEMM ("Where the engine
# is going: HRX and the NPU", section "4-bit activations reach the MoE experts")
# --------------------------------------------------------------------------
def moe_route(logits: np.ndarray, k: int):
    """logits [T][E] fp32 -> (topk_id [T][k] int32, topk_w [T][k] fp32,
    expert_off [E+1] int32, row_idx [T*k] int32, row_of [T][k] int32).

    Top k by logit (ties: lower id), weights = softmax over the k chosen
    logits (fp32, sum in choice order), rows grouped by expert then token."""
    logits = _c(logits, np.float32)
    T, E = logits.shape
    assert 1 <= k <= E
    topk_id = np.empty((T, k), np.int32)
    topk_w = np.empty((T, k), np.float32)
    off = np.empty(E + 1, np.int32)
    row_idx = np.empty(T * k, np.int32)
    row_of = np.empty((T, k), np.int32)
    _load().o_moe_route(_ptr(logits), T, E, k, _ptr(topk_id), _ptr(topk_w), _ptr(off),
                        _ptr(row_idx), _ptr(row_of))
    return topk_id, topk_w, off, row_idx, row_of


def moe_combine(y: np.ndarray, row_of: np.ndarray, topk_w: np.ndarray) -> np.ndarray:
    """y [R][H] fp32 (grouped rows) -> out [T][H]: sum over the token's k
    choices in order of w_j * y[row_of[t][j]], fp32 fma from +0."""
    y = _c(y, np.float32)
    row_of, topk_w = _c(row_of, np.int32), _c(topk_w, np.float32)
    T, k = row_of.shape
    H = y.shape[1]
    assert row_of.size == 0 or (row_of.min() >= 0 and row_of.max() < y.shape[0])
    out = np.empty((T, H), np.float32)
    _load().o_moe_combine(_ptr(y), H, _ptr(row_of), _ptr(topk_w), T, k, H, _ptr(out))
    return out


# --------------------------------------------------------------------------
# Q4_0 interchange: the file format's blocks <-> the two planes of the path
# ("Qwen3.8-27B at 45.7 tok/s ...", section "Prompt processing: 4-bit
# activations, rotated first": the route reads plain Q4_0 files).  Reading
# taken: a block is 18 bytes, the fp16 scale d (little endian) and then the 16
# code bytes in Q4_0 nibble order, the layout of a Q4_0 block in those files.
# --------------------------------------------------------------------------
def q4_0_planes_from_blocks(blocks: np.ndarray, N: int, K: int):
    """blocks u8 [N][K/32][18] -> (wq [N][K/2] u8, wd [N][K/32] fp16 bits as u16)."""
    b = np.asarray(blocks, np.uint8).reshape(N, K // 32, 18)
    wd = b[:, :, 0].astype(np.uint16) | (b[:, :, 1].astype(np.uint16) << 8)
    wq = np.ascontiguousarray(b[:, :, 2:]).reshape(N, K // 2)
    return wq, wd


def q4_0_blocks_from_planes(wq: np.ndarray, wd: np.ndarray) -> np.ndarray:
    """(wq [N][K/2], wd [N][K/32] u16) -> blocks u8 [N][K/32][18]."""
    wq = np.asarray(wq, np.uint8)
    wd = np.asarray(wd, np.uint16)
    N, nb = wd.shape
    out = np.empty((N, nb, 18), np.uint8)
    out[:, :, 0] = (wd & 0xFF).astype(np.uint8)
    out[:, :, 1] = (wd >> 8).astype(np.uint8)
    out[:, :, 2:] = wq.reshape(N, nb, 16)
    return out
