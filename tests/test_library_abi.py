"""The C-ABI library loads without a GPU, exports every entry point that
include/h32.h declares, and rejects bad arguments before touching the device."""
import ctypes
import os
import re

import pytest

import hadamard_rotated_bit_gb300 as h32
from hadamard_rotated_bit_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return h32.lib()


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "h32.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(h32_\w+|q4_0_\w+)\s*\(", text)))


def test_header_declares_the_path(lib):
    names = _declared_functions()
    for n in ("h32_quantize_act_q4", "h32_quantize_act_q8", "h32_rotate_quantize_weights_q4_0",
              "q4_0_x_q4_gemm", "q4_0_x_q8_gemm", "q4_0_x_q4_gemm_experts", "h32_device_status"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for n in _declared_functions():
        assert hasattr(lib, n), n
        assert n in h32.EXPORTED_SYMBOLS, n


def test_status_strings(lib):
    assert h32.h32_status_string(0) == "ok"
    assert "aligned" in h32.h32_status_string(2)
    assert h32.h32_version() >= 100


def _call(fn, *args):
    return getattr(h32.lib(), fn)(*args)


def test_bad_arguments_rejected_before_launch(lib):
    p = ctypes.c_void_p(256)   # never dereferenced: validation fails first
    bad = ctypes.c_void_p(258)  # not 16-byte aligned
    s = ctypes.c_void_p(0)
    # K not a multiple of 32
    assert _call("h32_quantize_act_q4", p, 1, 4, 33, 33, p, p, 1, s) == h32.H32_ERR_INVALID_ARG
    # ldx < K
    assert _call("h32_quantize_act_q8", p, 1, 4, 64, 32, p, p, 1, s) == h32.H32_ERR_INVALID_ARG
    # bad dtype
    assert _call("h32_quantize_act_q4", p, 7, 4, 64, 64, p, p, 1, s) == h32.H32_ERR_INVALID_ARG
    # null pointer
    assert _call("h32_quantize_act_q4", None, 1, 4, 64, 64, p, p, 1, s) == h32.H32_ERR_INVALID_ARG
    # misaligned pointer / pitch
    assert _call("h32_quantize_act_q4", bad, 1, 4, 64, 64, p, p, 1, s) == h32.H32_ERR_ALIGNMENT
    assert _call("h32_quantize_act_q4", p, 1, 4, 64, 68, p, p, 1, s) == h32.H32_ERR_ALIGNMENT
    assert _call("h32_rotate_quantize_weights_q4_0", p, 4, 48, 1, p, p, s) == h32.H32_ERR_INVALID_ARG
    # empty input is valid and enqueues nothing
    assert _call("h32_quantize_act_q4", p, 1, 0, 64, 64, p, p, 1, s) == h32.H32_OK


def test_gemm_bad_arguments(lib):
    p = ctypes.c_void_p(256)
    s = ctypes.c_void_p(0)
    # K not a multiple of 32, N not a multiple of 16, ldy < N
    assert _call("q4_0_x_q4_gemm", p, p, p, p, 4, 16, 48, p, 16, None, s) == h32.H32_ERR_INVALID_ARG
    assert _call("q4_0_x_q4_gemm", p, p, p, p, 4, 20, 64, p, 20, None, s) == h32.H32_ERR_INVALID_ARG
    assert _call("q4_0_x_q8_gemm", p, p, p, p, 4, 16, 64, p, 8, None, s) == h32.H32_ERR_INVALID_ARG
    assert _call("q4_0_x_q4_gemm_experts", p, p, 0, p, p, None, 4, p, 4, 16, 64, p, 16, None,
                 s) == h32.H32_ERR_INVALID_ARG
    assert _call("q4_0_x_q4_gemm_experts", p, p, 2, p, p, None, 4, None, 4, 16, 64, p, 16, None,
                 s) == h32.H32_ERR_INVALID_ARG
    assert _call("q4_0_x_q4_gemm", p, p, p, p, 0, 16, 64, p, 16, None, s) == h32.H32_OK


def test_no_device_is_reported_not_hidden(lib):
    """On a machine without a GPU a valid call reports 'unsupported': there is no CPU fallback."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    p = ctypes.c_void_p(256)
    s = ctypes.c_void_p(0)
    assert _call("h32_quantize_act_q4", p, 1, 4, 64, 64, p, p, 1, s) == h32.H32_ERR_UNSUPPORTED


def test_tc_form_bad_arguments(lib):
    p = ctypes.c_void_p(256)
    bad = ctypes.c_void_p(260)
    s = ctypes.c_void_p(0)
    # quantizer: ldxd < M, ldxd not a multiple of 4
    assert _call("h32_quantize_act_q4_tc", p, 1, 8, 64, 64, p, p, 4, 1, s) == h32.H32_ERR_INVALID_ARG
    assert _call("h32_quantize_act_q4_tc", p, 1, 8, 64, 64, p, p, 10, 1, s) == h32.H32_ERR_INVALID_ARG
    assert _call("h32_quantize_act_q4_tc", p, 1, 8, 64, 64, bad, p, 8, 1, s) == h32.H32_ERR_ALIGNMENT
    # gather: null index, misaligned index
    assert _call("h32_quantize_act_q4_tc_gather", p, 1, 4, 64, 64, None, 8, p, p, 8, 1,
                 s) == h32.H32_ERR_INVALID_ARG
    assert _call("h32_quantize_act_q4_tc_gather", p, 1, 4, 64, 64, bad, 8, p, p, 8, 1,
                 s) == h32.H32_ERR_ALIGNMENT
    # repack: ldws < K/32
    assert _call("h32_prepack_weights_q4_0_tc", p, p, 16, 256, p, p, 4, s) == h32.H32_ERR_INVALID_ARG
    # GEMM: K % 128, N % 16, ldxd < M
    assert _call("q4_0_x_q4_gemm_tc", p, p, 4, p, p, 8, 8, 16, 96, p, 16, None,
                 s) == h32.H32_ERR_INVALID_ARG
    assert _call("q4_0_x_q4_gemm_tc", p, p, 4, p, p, 8, 8, 24, 128, p, 24, None,
                 s) == h32.H32_ERR_INVALID_ARG
    assert _call("q4_0_x_q4_gemm_tc", p, p, 4, p, p, 4, 8, 16, 128, p, 16, None,
                 s) == h32.H32_ERR_INVALID_ARG
    # experts: E out of range, null offsets
    assert _call("q4_0_x_q4_gemm_tc_experts", p, p, 4, 0, p, p, 8, p, 8, 16, 128, p, 16, None,
                 s) == h32.H32_ERR_INVALID_ARG
    assert _call("q4_0_x_q4_gemm_tc_experts", p, p, 4, 1025, p, p, 8, p, 8, 16, 128, p, 16, None,
                 s) == h32.H32_ERR_INVALID_ARG
    assert _call("q4_0_x_q4_gemm_tc_experts", p, p, 4, 2, p, p, 8, None, 8, 16, 128, p, 16, None,
                 s) == h32.H32_ERR_INVALID_ARG
    assert _call("q4_0_x_q4_gemm_tc", p, p, 4, p, p, 8, 0, 16, 128, p, 16, None, s) == h32.H32_OK


def test_widen_bad_arguments(lib):
    """The GEMMs on Q4_0 planes widened in shared memory: K % 256 (the fp16 scale
    rows feed a tensor copy of 16-byte units), null or misaligned scales, the
    expert count and offsets; M = 0 enqueues nothing."""
    p = ctypes.c_void_p(256)
    bad = ctypes.c_void_p(264)
    s = ctypes.c_void_p(0)
    assert _call("q4_0_x_q4_gemm_tc_widen", p, p, p, p, 8, 8, 16, 384, p, 16, None,
                 s) == h32.H32_ERR_INVALID_ARG
    assert _call("q4_0_x_q4_gemm_tc_widen", p, None, p, p, 8, 8, 16, 256, p, 16, None,
                 s) == h32.H32_ERR_INVALID_ARG
    assert _call("q4_0_x_q4_gemm_tc_widen", p, bad, p, p, 8, 8, 16, 256, p, 16, None,
                 s) == h32.H32_ERR_ALIGNMENT
    assert _call("q4_0_x_q4_gemm_tc_widen", p, p, p, p, 8, 8, 24, 256, p, 24, None,
                 s) == h32.H32_ERR_INVALID_ARG
    assert _call("q4_0_x_q4_gemm_tc_widen_experts", p, p, 0, p, p, 8, p, 8, 16, 256, p, 16, None,
                 s) == h32.H32_ERR_INVALID_ARG
    assert _call("q4_0_x_q4_gemm_tc_widen_experts", p, p, 2, p, p, 8, None, 8, 16, 256, p, 16,
                 None, s) == h32.H32_ERR_INVALID_ARG
    assert _call("q4_0_x_q4_gemm_tc_widen_experts", p, p, 2, p, p, 8, p, 8, 16, 128, p, 16, None,
                 s) == h32.H32_ERR_INVALID_ARG
    assert _call("q4_0_x_q4_gemm_tc_widen", p, p, p, p, 8, 0, 16, 256, p, 16, None,
                 s) == h32.H32_OK
    # the widening form's activation quantizers: ldxd < M, null index, misaligned index
    assert _call("h32_quantize_act_q4_tc_e5m2", p, 1, 8, 64, 64, p, p, 4, 1,
                 s) == h32.H32_ERR_INVALID_ARG
    assert _call("h32_quantize_act_q4_tc_e5m2_gather", p, 1, 4, 64, 64, None, 8, p, p, 8, 1,
                 s) == h32.H32_ERR_INVALID_ARG
    assert _call("h32_quantize_act_q4_tc_e5m2_gather", p, 1, 4, 64, 64, bad, 8, p, p, 8, 1,
                 s) == h32.H32_ERR_ALIGNMENT


def test_q4_0_layout_bad_arguments(lib):
    p = ctypes.c_void_p(256)
    bad = ctypes.c_void_p(258)
    s = ctypes.c_void_p(0)
    assert _call("h32_q4_0_blocks_to_planes", p, 4, 48, p, p, s) == h32.H32_ERR_INVALID_ARG
    assert _call("h32_q4_0_blocks_to_planes", None, 4, 64, p, p, s) == h32.H32_ERR_INVALID_ARG
    assert _call("h32_q4_0_blocks_to_planes", bad, 4, 64, p, p, s) == h32.H32_ERR_ALIGNMENT
    assert _call("h32_q4_0_planes_to_blocks", p, p, 4, 48, p, s) == h32.H32_ERR_INVALID_ARG
    assert _call("h32_q4_0_planes_to_blocks", p, None, 4, 64, p, s) == h32.H32_ERR_INVALID_ARG
    assert _call("h32_q4_0_planes_to_blocks", p, p, 0, 64, p, s) == h32.H32_OK


def test_rotation_size_validated(lib):
    p = ctypes.c_void_p(256)
    s = ctypes.c_void_p(0)
    # unsupported size, and K not a multiple of the rotation
    assert _call("h32_quantize_act_q4", p, 1, 4, 64, 64, p, p, 16, s) == h32.H32_ERR_INVALID_ARG
    assert _call("h32_quantize_act_q8", p, 1, 4, 96, 96, p, p, 64, s) == h32.H32_ERR_INVALID_ARG
    assert _call("h32_rotate_quantize_weights_q4_0", p, 4, 192, 128, p, p,
                 s) == h32.H32_ERR_INVALID_ARG
    assert _call("h32_quantize_act_q4_tc", p, 1, 8, 64, 64, p, p, 8, 128, s) == h32.H32_ERR_INVALID_ARG
    assert _call("h32_quantize_act_q4", p, 1, 0, 128, 128, p, p, 128, s) == h32.H32_OK


def test_quant_next_bad_arguments(lib):
    p = ctypes.c_void_p(256)
    s = ctypes.c_void_p(0)
    # N not a multiple of 32; no next codes; bad rotation; ldxd_next < M
    assert _call("q4_0_x_q4_gemm_tc_quant_next", p, p, 4, p, p, 8, 8, 48, 128, p, 48, p, p, 8, 1,
                 s) == h32.H32_ERR_INVALID_ARG
    assert _call("q4_0_x_q4_gemm_tc_quant_next", p, p, 4, p, p, 8, 8, 64, 128, p, 64, None, p, 8, 1,
                 s) == h32.H32_ERR_INVALID_ARG
    assert _call("q4_0_x_q4_gemm_tc_quant_next", p, p, 4, p, p, 8, 8, 64, 128, p, 64, p, p, 8, 64,
                 s) == h32.H32_ERR_INVALID_ARG
    assert _call("q4_0_x_q4_gemm_tc_quant_next", p, p, 4, p, p, 8, 8, 64, 128, None, 64, p, p, 4, 1,
                 s) == h32.H32_ERR_INVALID_ARG


def test_moe_route_and_combine_bad_arguments(lib):
    p = ctypes.c_void_p(256)
    s = ctypes.c_void_p(0)
    # route: k > E, k > 32, E > 1024, ldl < E, missing offsets
    assert _call("h32_moe_route", p, 4, 8, 8, 9, p, p, p, p, p, s) == h32.H32_ERR_INVALID_ARG
    assert _call("h32_moe_route", p, 4, 64, 64, 33, p, p, p, p, p, s) == h32.H32_ERR_INVALID_ARG
    assert _call("h32_moe_route", p, 4, 1025, 1025, 2, p, p, p, p, p, s) == h32.H32_ERR_INVALID_ARG
    assert _call("h32_moe_route", p, 4, 16, 15, 2, p, p, p, p, p, s) == h32.H32_ERR_INVALID_ARG
    assert _call("h32_moe_route", p, 4, 16, 16, 2, p, p, None, p, p, s) == h32.H32_ERR_INVALID_ARG
    assert _call("h32_moe_route", None, 4, 16, 16, 2, p, p, p, p, p, s) == h32.H32_ERR_INVALID_ARG
    assert _call("h32_moe_route", ctypes.c_void_p(258), 4, 16, 16, 2, p, p, p, p, p, s) == \
        h32.H32_ERR_ALIGNMENT
    assert _call("h32_moe_route", p, 4, 16, 16, 2, ctypes.c_void_p(264), p, p, p, p, s) == \
        h32.H32_ERR_ALIGNMENT
    # combine: H not a multiple of 4, ldy < H, misaligned y or pitch; T = 0 is a no-op
    assert _call("h32_moe_combine", p, 8, 6, p, p, 2, 4, 6, p, 6, s) == h32.H32_ERR_INVALID_ARG
    assert _call("h32_moe_combine", p, 8, 4, p, p, 2, 4, 8, p, 8, s) == h32.H32_ERR_INVALID_ARG
    assert _call("h32_moe_combine", ctypes.c_void_p(260), 8, 8, p, p, 2, 4, 8, p, 8, s) == \
        h32.H32_ERR_ALIGNMENT
    assert _call("h32_moe_combine", p, 8, 10, p, p, 2, 4, 8, p, 8, s) == h32.H32_ERR_ALIGNMENT
    assert _call("h32_moe_combine", p, 8, 8, p, p, 2, 33, 8, p, 8, s) == h32.H32_ERR_INVALID_ARG
    assert _call("h32_moe_combine", p, 8, 8, p, p, 0, 4, 8, p, 8, s) == h32.H32_OK
