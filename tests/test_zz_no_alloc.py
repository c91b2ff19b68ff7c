"""The no-alloc entry points of the tc GEMMs: the K split of the last wave on
the library's static per-device workspace.  Two calls in a row on one stream
(the second finds the workspace as the first left it) are each bit-exact
against the oracle, and neither changes the device's free memory ("509 tokens
a second of prompt: the Hadamard route ships", sections "Why prompts are a
matrix-unit problem" and "The rotation")."""
import numpy as np
import pytest

import oracle
from hadamard_rotated_bit_gb300 import workloads as wl
from tests._gpu import np_of, torch_bf16, torch_of

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


@pytest.mark.parametrize("bits", [4, 8])
def test_two_calls_in_a_row_no_allocation(h32, bits):
    import torch
    M, N, K = 64, 20480, 256   # a full wave and 8 tiles over: the last wave is split
    if h32.h32_gemm_tc_workspace_bytes(M, N, K) == 0:
        pytest.skip("this device's schedule does not split the case")
    gemm = h32.q4_0_x_q4_gemm_tc_noalloc if bits == 4 else h32.q4_0_x_q8_gemm_tc_noalloc
    quant = h32.h32_quantize_act_q4_tc if bits == 4 else h32.h32_quantize_act_q8_tc
    qref = oracle.quantize_act_q4 if bits == 4 else oracle.quantize_act_q8
    w = wl.weights_normal(N, K, 0.02, 0, wl.CFG_TEST, 990 + bits)
    wq, wd = oracle.quantize_weights_q4_0(w)
    wp, wsc = h32.h32_prepack_weights_q4_0_tc(torch_of(wq), torch_of(wd.view(np.int16)))
    xs = [wl.f32_to_bf16_bits(wl.act_normal_outliers(M, K, 0.01, 20.0, r, wl.CFG_TEST, 992))
          for r in range(3)]
    ops = [quant(torch_bf16(x)) for x in xs]
    ys = [torch.empty((M, N), dtype=torch.float32, device="cuda") for _ in xs]
    gemm(wp, wsc, *ops[0], M=M, y=ys[0])
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    gemm(wp, wsc, *ops[1], M=M, y=ys[1])
    gemm(wp, wsc, *ops[2], M=M, y=ys[2])
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0
    assert h32.h32_device_status() == 0
    for x, y in zip(xs, ys):
        xq, xd = qref(x)
        r32, _, _ = oracle.gemm(wq, wd, xq, xd, K)
        assert np.array_equal(np_of(y).view(np.uint32), r32.view(np.uint32))
