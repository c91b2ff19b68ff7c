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
