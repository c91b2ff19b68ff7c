"""GPU parity of the larger rotations (64 and 128 points, scales still per
32-block: "Qwen3.8-27B at 45.7 tok/s ...", section "What's next") against the
CPU oracle: every quantizer's codes and scales bit for bit, and the products
built on them."""
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


def e4m3_value(b):
    b = b.astype(np.int64)
    sign = np.where(b & 0x80, -1.0, 1.0)
    e = (b >> 3) & 0xF
    m = b & 7
    return sign * np.where(e == 0, m / 8.0 * 2.0 ** -6, (1 + m / 8.0) * 2.0 ** (e - 7.0))


def e5m2_value(b):
    b = b.astype(np.int64)
    sign = np.where(b & 0x80, -1.0, 1.0)
    e = (b >> 2) & 0x1F
    m = b & 3
    return sign * np.where(e == 0, m / 4.0 * 2.0 ** -14, (1 + m / 4.0) * 2.0 ** (e - 15.0))


def _acts(M, K, tid, bf16=True):
    x = wl.act_normal_outliers(M, K, 0.01, 25.0, 0, wl.CFG_TEST, tid)
    return wl.f32_to_bf16_bits(x) if bf16 else x


def _dev(x):
    return torch_bf16(x) if x.dtype == np.uint16 else torch_of(x)


@pytest.mark.parametrize("n", [64, 128])
@pytest.mark.parametrize("M,K,bf16", [(37, 512, True), (5, 256, False), (2048, 17408, True)])
def test_direct_quantizers(h32, n, M, K, bf16):
    """Q4_0-order 4-bit and int8 codes; the last shape makes every thread walk
    several blocks."""
    import torch
    x = _acts(M, K, 400 + n, bf16)
    for bits in (4, 8):
        fn = h32.h32_quantize_act_q4 if bits == 4 else h32.h32_quantize_act_q8
        xq, xd = fn(_dev(x), rotate=n)
        torch.cuda.synchronize()
        rq, rd = (oracle.quantize_act_q4 if bits == 4 else oracle.quantize_act_q8)(x, n)
        assert np.array_equal(np_of(xq).view(np.uint8), rq.view(np.uint8)), bits
        assert np.array_equal(np_of(xd).view(np.uint32), rd.view(np.uint32)), bits


@pytest.mark.parametrize("n", [64, 128])
@pytest.mark.parametrize("M,K", [(37, 512), (1, 128), (600, 5120)])
def test_tc_quantizers(h32, n, M, K):
    import torch
    if K % n:
        pytest.skip("K not a multiple of the rotation")
    x = _acts(M, K, 410 + n)
    xw, xdt = h32.h32_quantize_act_q4_tc(torch_bf16(x), rotate=n)
    xw8, xdt8 = h32.h32_quantize_act_q8_tc(torch_bf16(x), rotate=n)
    torch.cuda.synchronize()
    rq, rd = oracle.quantize_act_q4(x, n)
    assert np.array_equal(e4m3_value(np_of(xw)), oracle.decode_act4(rq, K).astype(np.float64))
    assert np.array_equal(np_of(xdt)[:, :M].T.view(np.uint32), rd.view(np.uint32))
    xw5, xdt5 = h32.h32_quantize_act_q4_tc_e5m2(torch_bf16(x), rotate=n)
    assert np.array_equal(e5m2_value(np_of(xw5)) / 512.0,
                          oracle.decode_act4(rq, K).astype(np.float64))
    assert np.array_equal(np_of(xdt5)[:, :M].T.view(np.uint32), rd.view(np.uint32))
    r8, rd8 = oracle.quantize_act_q8(x, n)
    v = e4m3_value(np_of(xw8)).reshape(M, K // 32, 2, 32)
    assert np.array_equal((v[:, :, 0] + v[:, :, 1]).reshape(M, K), r8.astype(np.float64))
    assert np.array_equal(np_of(xdt8)[:, :M].T.view(np.uint32), rd8.view(np.uint32))


@pytest.mark.parametrize("n", [64, 128])
def test_tc_gather_quantizer(h32, n):
    import torch
    T, K, R = 29, 384, 77
    x = _acts(T, K, 420 + n)
    ridx = np.random.default_rng(n).integers(0, T, R).astype(np.int32)
    xw, xdt = h32.h32_quantize_act_q4_tc_gather(torch_bf16(x), torch_of(ridx), rotate=n)
    torch.cuda.synchronize()
    assert h32.h32_device_status() == 0
    rq, rd = oracle.quantize_act_q4(x[ridx], n)
    assert np.array_equal(e4m3_value(np_of(xw)), oracle.decode_act4(rq, K).astype(np.float64))
    assert np.array_equal(np_of(xdt)[:, :R].T.view(np.uint32), rd.view(np.uint32))


@pytest.mark.parametrize("n", [64, 128])
def test_weight_quantizer(h32, n):
    import torch
    w = wl.weights_normal(300, 640, 0.02, 0, wl.CFG_TEST, 430 + n)
    w[7, 130] = 3.0   # an outlier weight
    wq, wd = h32.h32_rotate_quantize_weights_q4_0(torch_of(w), rotate=n)
    torch.cuda.synchronize()
    rq, rd = oracle.quantize_weights_q4_0(w, n)
    assert np.array_equal(np_of(wq), rq)
    assert np.array_equal(np_of(wd).view(np.uint16), rd)


@pytest.mark.parametrize("n", [64, 128])
def test_products_with_larger_rotation(h32, n):
    """The tensor-core-form W4A4 and W4A8 products, the widening-form W4A4
    product and the Q4_0-direct W4A4 product on n-point-rotated operands, bit for
    bit against the oracle."""
    import torch
    M, N, K = 70, 160, 1024
    x = _acts(M, K, 440 + n)
    w = wl.weights_normal(N, K, 0.02, 0, wl.CFG_TEST, 441 + n)
    wq, wd = h32.h32_rotate_quantize_weights_q4_0(torch_of(w), rotate=n)
    wp, wsc = h32.h32_prepack_weights_q4_0_tc(wq, wd)
    rwq, rwd = oracle.quantize_weights_q4_0(w, n)
    for bits in (4, 8):
        if bits == 4:
            xw, xdt = h32.h32_quantize_act_q4_tc(torch_bf16(x), rotate=n)
            y = h32.q4_0_x_q4_gemm_tc(wp, wsc, xw, xdt, M=M)
            rxq, rxd = oracle.quantize_act_q4(x, n)
        else:
            xw, xdt = h32.h32_quantize_act_q8_tc(torch_bf16(x), rotate=n)
            y = h32.q4_0_x_q8_gemm_tc(wp, wsc, xw, xdt, M=M)
            rxq, rxd = oracle.quantize_act_q8(x, n)
        torch.cuda.synchronize()
        assert h32.h32_device_status() == 0
        r32, _, _ = oracle.gemm(rwq, rwd, rxq, rxd, K)
        assert np.array_equal(np_of(y).view(np.uint32), r32.view(np.uint32)), bits
    xw5, xdt5 = h32.h32_quantize_act_q4_tc_e5m2(torch_bf16(x), rotate=n)
    y = h32.q4_0_x_q4_gemm_tc_widen(wq, wd, xw5, xdt5, M=M)
    torch.cuda.synchronize()
    assert h32.h32_device_status() == 0
    rxq, rxd = oracle.quantize_act_q4(x, n)
    r32, _, _ = oracle.gemm(rwq, rwd, rxq, rxd, K)
    assert np.array_equal(np_of(y).view(np.uint32), r32.view(np.uint32)), "widen"
    xq, xd = h32.h32_quantize_act_q4(torch_bf16(x), rotate=n)
    y = h32.q4_0_x_q4_gemm(wq, wd, xq, xd)
    torch.cuda.synchronize()
    rxq, rxd = oracle.quantize_act_q4(x, n)
    r32, _, _ = oracle.gemm(rwq, rwd, rxq, rxd, K)
    assert np.array_equal(np_of(y).view(np.uint32), r32.view(np.uint32))
