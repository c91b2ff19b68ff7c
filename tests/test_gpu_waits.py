"""Bounded device waits: a wait that gives up is reported as a status, the
kernel drains its own copies and MMAs and returns, and the context stays
usable.  The failure is made on the host (a one-poll wait bound); nothing
here faults, traps or hangs the GPU."""
import numpy as np
import pytest

import oracle
from hadamard_rotated_bit_gb300 import workloads as wl
from tests._gpu import np_of, torch_of

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def h32():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import hadamard_rotated_bit_gb300 as m
    from hadamard_rotated_bit_gb300 import _build
    _build.build()
    return m


def test_one_poll_wait_bound_reports_timeout_and_recovers(h32):
    import torch
    g = torch.Generator(device="cuda").manual_seed(0)
    M, N, K = 512, 4096, 4096
    wq = torch.randint(0, 256, (N, K // 2), dtype=torch.uint8, device="cuda", generator=g)
    wd = torch.full((N, K // 32), 0x2C00, dtype=torch.int16, device="cuda")  # fp16 0.0625
    xq = torch.randint(0, 256, (M, K // 2), dtype=torch.uint8, device="cuda", generator=g)
    xd = torch.ones((M, K // 32), dtype=torch.float32, device="cuda")
    assert h32.h32_device_status() == 0
    h32.h32_set_wait_limit(1)
    try:
        for _ in range(3):
            h32.q4_0_x_q4_gemm(wq, wd, xq, xd)
        st = h32.h32_device_status()
    finally:
        h32.h32_set_wait_limit(0)
    assert st == h32.H32_ERR_TIMEOUT
    assert h32.h32_device_status() == 0
    # the same context still computes exact results
    x = wl.act_normal_outliers(64, 256, 0.01, 20.0, 0, wl.CFG_TEST, 120)
    w = wl.weights_normal(128, 256, 0.02, 0, wl.CFG_TEST, 121)
    rwq, rwd = oracle.quantize_weights_q4_0(w)
    rxq, rxd = oracle.quantize_act_q4(x)
    y = h32.q4_0_x_q4_gemm(torch_of(rwq), torch_of(rwd.view(np.int16)), torch_of(rxq),
                           torch_of(rxd))
    assert h32.h32_device_status() == 0
    r32, _, _ = oracle.gemm(rwq, rwd, rxq, rxd, 256)
    assert np.array_equal(np_of(y).view(np.uint32), r32.view(np.uint32))


def _tc_ones(h32, rows, K, scale=1.0):
    """tc-form operands whose every code is 1 (e4m3 0x38), scales `scale`."""
    import torch
    w = torch.full((rows, K), 0x38, dtype=torch.uint8, device="cuda")
    sc = torch.full((rows, (K // 32 + 3) // 4 * 4), scale, dtype=torch.float32, device="cuda")
    return w, sc


def _exact_small_case(h32):
    """A small tc product after the timeouts, against the oracle bit for bit."""
    x = wl.f32_to_bf16_bits(wl.act_normal_outliers(70, 256, 0.01, 20.0, 0, wl.CFG_TEST, 122))
    w = wl.weights_normal(160, 256, 0.02, 0, wl.CFG_TEST, 123)
    rwq, rwd = oracle.quantize_weights_q4_0(w)
    rxq, rxd = oracle.quantize_act_q4(x)
    from tests._gpu import torch_bf16
    wp, wsc = h32.h32_prepack_weights_q4_0_tc(torch_of(rwq), torch_of(rwd.view(np.int16)))
    xw, xdt = h32.h32_quantize_act_q4_tc(torch_bf16(x))
    y = h32.q4_0_x_q4_gemm_tc(wp, wsc, xw, xdt, M=70)
    assert h32.h32_device_status() == 0
    r32, _, _ = oracle.gemm(rwq, rwd, rxq, rxd, 256)
    assert np.array_equal(np_of(y).view(np.uint32), r32.view(np.uint32))


def _exact_split_case(h32):
    """A product whose last wave is split along K, through the binding's
    workspace of the stream the timed-out launches used: exact, so the
    generation the aborted launches left behind is consistent."""
    M, N, K = 64, 20480, 256
    x = wl.f32_to_bf16_bits(wl.act_normal_outliers(M, K, 0.01, 20.0, 0, wl.CFG_TEST, 124))
    w = wl.weights_normal(N, K, 0.02, 0, wl.CFG_TEST, 125)
    rwq, rwd = oracle.quantize_weights_q4_0(w)
    rxq, rxd = oracle.quantize_act_q4(x)
    from tests._gpu import torch_bf16
    wp, wsc = h32.h32_prepack_weights_q4_0_tc(torch_of(rwq), torch_of(rwd.view(np.int16)))
    xw, xdt = h32.h32_quantize_act_q4_tc(torch_bf16(x))
    y = h32.q4_0_x_q4_gemm_tc(wp, wsc, xw, xdt, M=M)
    assert h32.h32_device_status() == 0
    r32, _, _ = oracle.gemm(rwq, rwd, rxq, rxd, K)
    assert np.array_equal(np_of(y).view(np.uint32), r32.view(np.uint32))


@pytest.mark.parametrize("kind", ["q4_tc", "q8_tc", "experts_tc", "widen", "widen_experts",
                                  "q4_tc_split", "q8_tc_split"])
def test_tc_gemm_one_poll_wait_bound(h32, kind):
    """The tensor-core-form GEMM (the chain's kernel, its 8-bit and its expert
    instances, the instances that widen Q4_0 planes in shared memory, and the
    instances whose last wave is split along K, whose second parts also wait
    for the first parts' flags) under a one-poll wait bound: the TMA, MMA,
    widening and epilogue roles that give up record H32_ERR_TIMEOUT, drain
    their copies and MMAs, free TMEM and return; the status is reported once
    and the same context then computes exact results."""
    import torch
    M, N, K = 512, 4096, 2048
    if kind.endswith("_split"):
        N = 5120   # 160 tiles: a full wave and 8 tiles cut and split
        if h32.h32_gemm_tc_workspace_bytes(M, N, K) == 0:
            pytest.skip("this device's schedule does not split the case")
    wp, wsc = _tc_ones(h32, N, K, 0.0625)
    xb = 2 if kind.startswith("q8_tc") else 1
    xw = torch.full((M, K * xb), 0x38, dtype=torch.uint8, device="cuda")
    xdt = torch.ones((K // 32, M), dtype=torch.float32, device="cuda")
    E = 8
    off = torch.tensor([i * M // E for i in range(E + 1)], dtype=torch.int32, device="cuda")
    wpe, wsce = _tc_ones(h32, E * 512, K, 0.0625)
    # Q4_0 planes: every code 9 (value +1), scales fp16 0.0625
    wq = torch.full((E * 512, K // 2), 0x99, dtype=torch.uint8, device="cuda")
    wd = torch.full((E * 512, K // 32), 0x2C00, dtype=torch.int16, device="cuda")
    assert h32.h32_device_status() == 0
    h32.h32_set_wait_limit(1)
    try:
        for _ in range(3):
            if kind in ("q4_tc", "q4_tc_split"):
                h32.q4_0_x_q4_gemm_tc(wp, wsc, xw, xdt, M=M)
            elif kind in ("q8_tc", "q8_tc_split"):
                h32.q4_0_x_q8_gemm_tc(wp, wsc, xw, xdt, M=M)
            elif kind == "experts_tc":
                h32.q4_0_x_q4_gemm_tc_experts(wpe, wsce, xw, xdt, off, 512, R=M)
            elif kind == "widen":
                h32.q4_0_x_q4_gemm_tc_widen(wq, wd, xw, xdt, M=M)
            else:
                h32.q4_0_x_q4_gemm_tc_widen_experts(wq, wd, xw, xdt, off, 512, R=M)
        st = h32.h32_device_status()
    finally:
        h32.h32_set_wait_limit(0)
    assert st == h32.H32_ERR_TIMEOUT
    assert h32.h32_device_status() == 0
    torch.cuda.synchronize()
    _exact_small_case(h32)
    if kind.endswith("_split"):
        _exact_split_case(h32)
