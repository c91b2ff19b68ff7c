"""GPU parity of the Q4_0 interchange helpers against the oracle's layout
functions: file blocks (fp16 d, then 16 code bytes) to planes and back, byte
for byte, and a product run on weights that arrive as file blocks ("Qwen3.8-27B
at 45.7 tok/s ...", section "Prompt processing: 4-bit activations, rotated
first": the route reads plain Q4_0 files)."""
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


@pytest.mark.parametrize("N,K", [(1, 32), (37, 256), (300, 5120)])
def test_blocks_planes_round_trip(h32, N, K):
    import torch
    blocks = np.random.default_rng(N).integers(0, 256, (N, K // 32, 18), dtype=np.uint8)
    wq, wd = h32.h32_q4_0_blocks_to_planes(torch_of(blocks))
    back = h32.h32_q4_0_planes_to_blocks(wq, wd)
    torch.cuda.synchronize()
    assert h32.h32_device_status() == 0
    rq, rd = oracle.q4_0_planes_from_blocks(blocks, N, K)
    assert np.array_equal(np_of(wq), rq)
    assert np.array_equal(np_of(wd).view(np.uint16), rd)
    assert np.array_equal(np_of(back), blocks)


def test_product_on_weights_from_file_blocks(h32):
    """Weights quantized by the oracle, written as file blocks, converted on the
    GPU, then the tensor-core-form and widening-form products: bit-exact."""
    import torch
    M, N, K = 70, 160, 512
    x = wl.act_normal_outliers(M, K, 0.01, 20.0, 0, wl.CFG_TEST, 710)
    w = wl.weights_normal(N, K, 0.02, 0, wl.CFG_TEST, 711)
    rwq, rwd = oracle.quantize_weights_q4_0(w)
    blocks = oracle.q4_0_blocks_from_planes(rwq, rwd)
    wq, wd = h32.h32_q4_0_blocks_to_planes(torch_of(blocks))
    wp, wsc = h32.h32_prepack_weights_q4_0_tc(wq, wd)
    xw, xdt = h32.h32_quantize_act_q4_tc(torch_of(x))
    y = h32.q4_0_x_q4_gemm_tc(wp, wsc, xw, xdt, M=M)
    xw5, xdt5 = h32.h32_quantize_act_q4_tc_e5m2(torch_of(x))
    y5 = h32.q4_0_x_q4_gemm_tc_widen(wq, wd, xw5, xdt5, M=M)
    torch.cuda.synchronize()
    assert h32.h32_device_status() == 0
    rxq, rxd = oracle.quantize_act_q4(x)
    r32, _, _ = oracle.gemm(rwq, rwd, rxq, rxd, K)
    assert np.array_equal(np_of(y).view(np.uint32), r32.view(np.uint32))
    assert np.array_equal(np_of(y5).view(np.uint32), r32.view(np.uint32))


def test_gate_up_size_round_trip(h32):
    """The pp512 FFN gate/up weights (34816 x 5120, 100 MB of blocks)."""
    import torch
    N, K = 34816, 5120
    blocks = np.random.default_rng(9).integers(0, 256, (N, K // 32, 18), dtype=np.uint8)
    tb = torch_of(blocks)
    wq, wd = h32.h32_q4_0_blocks_to_planes(tb)
    back = h32.h32_q4_0_planes_to_blocks(wq, wd)
    torch.cuda.synchronize()
    assert h32.h32_device_status() == 0
    assert torch.equal(back, tb)
    rq, rd = oracle.q4_0_planes_from_blocks(blocks, N, K)
    rows = np.random.default_rng(10).integers(0, N, 64)
    assert np.array_equal(np_of(wq)[rows], rq[rows])
    assert np.array_equal(np_of(wd).view(np.uint16)[rows], rd[rows])
