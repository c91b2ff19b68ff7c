"""GPU parity of the rotate+quantize kernels against the CPU oracle: codes and
scales must be bit-identical ("509 tokens a second of prompt: the Hadamard
route ships", section "The rotation"; the 8-bit route of "Prompt processing:
4-bit activations, rotated first"; the Q4_0 weight step of "Making the file is
part of the engine")."""
import numpy as np
import pytest

import oracle
from hadamard_rotated_bit_gb300 import workloads as wl
from tests._gpu import np_of, torch_bf16, torch_of, wd_bits

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


def _gpu_act(h32, x_np, bits, rotate, bf16):
    import torch
    x = torch_bf16(x_np) if bf16 else torch_of(x_np.astype(np.float32))
    fn = h32.h32_quantize_act_q4 if bits == 4 else h32.h32_quantize_act_q8
    xq, xd = fn(x, rotate=rotate)
    torch.cuda.synchronize()
    return np_of(xq), np_of(xd)


def _oracle_act(x_np, bits, rotate):
    fn = oracle.quantize_act_q4 if bits == 4 else oracle.quantize_act_q8
    return fn(x_np, rotate)


def _same(a, b):
    assert a.shape == b.shape
    assert np.array_equal(a.view(np.uint8).reshape(-1), b.view(np.uint8).reshape(-1))


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("rotate", [True, False])
def test_tiny_fp32(h32, bits, rotate):
    x = wl.TINY.chain[0].activations(64, 0, wl.CFG_TINY, bf16=False)
    q, d = _gpu_act(h32, x, bits, rotate, bf16=False)
    rq, rd = _oracle_act(x, bits, rotate)
    _same(q, rq.view(np.uint8) if bits == 8 else rq)
    _same(d, rd)


@pytest.mark.parametrize("bits", [4, 8])
def test_pp512_attention_bf16(h32, bits):
    x = wl.ATTN.activations(512, 0, wl.CFG_ATTN)
    q, d = _gpu_act(h32, x, bits, True, bf16=True)
    rq, rd = _oracle_act(x, bits, True)
    _same(q, rq.view(np.uint8) if bits == 8 else rq)
    _same(d, rd)


def test_pp512_ffn_down_input_bf16(h32):
    x = wl.FFN_DOWN.activations(512, 0, wl.CFG_FFN)
    q, d = _gpu_act(h32, x, 4, True, bf16=True)
    rq, rd = _oracle_act(x, 4, True)
    _same(q, rq)
    _same(d, rd)


@pytest.mark.parametrize("M,K", [(1, 32), (3, 96), (77, 160), (129, 1056)])
def test_ragged_shapes(h32, M, K):
    x = wl.act_normal_outliers(M, K, 0.02, 25.0, 0, wl.CFG_TEST, 20 + M)
    for bits in (4, 8):
        q, d = _gpu_act(h32, wl.f32_to_bf16_bits(x), bits, True, bf16=True)
        rq, rd = _oracle_act(wl.f32_to_bf16_bits(x), bits, True)
        _same(q, rq.view(np.uint8) if bits == 8 else rq)
        _same(d, rd)


def test_row_pitch_larger_than_k(h32):
    import torch
    x = wl.act_normal_outliers(40, 256, 0.01, 20.0, 0, wl.CFG_TEST, 31)
    wide = torch.zeros((40, 256 + 64), dtype=torch.float32, device="cuda")
    wide[:, :256] = torch.from_numpy(x).cuda()
    xq, xd = h32.h32_quantize_act_q4(wide[:, :256])
    rq, rd = oracle.quantize_act_q4(x)
    _same(np_of(xq), rq)
    _same(np_of(xd), rd)


def test_edge_blocks(h32):
    """Zero, tiny (1/d overflows), ramp, tie, constant, huge and one-hot blocks."""
    rows = [np.zeros(32), np.r_[2.0 ** -130, np.zeros(31)], np.arange(32.0),
            np.r_[7, 2.5, -0.5, 1.5, 3.5, -2.5, np.zeros(26)], np.full(32, -3.0),
            np.r_[3e38, -3e38, np.zeros(30)], np.eye(32)[5], np.r_[2.0 ** 24, 1.0, np.zeros(14),
                                                                    -(2.0 ** 24), np.zeros(15)]]
    x = np.stack(rows).astype(np.float32)
    for bits in (4, 8):
        for rotate in (True, False):
            q, d = _gpu_act(h32, x, bits, rotate, bf16=False)
            rq, rd = _oracle_act(x, bits, rotate)
            _same(q, rq.view(np.uint8) if bits == 8 else rq)
            _same(d, rd)


def test_empty_m(h32):
    import torch
    x = torch.zeros((0, 64), dtype=torch.bfloat16, device="cuda")
    xq, xd = h32.h32_quantize_act_q4(x)
    assert xq.shape == (0, 32) and xd.shape == (0, 2)


def test_bad_k_raises(h32):
    import torch
    x = torch.zeros((4, 48), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(h32.H32Error):
        h32.h32_quantize_act_q4(x)


@pytest.mark.parametrize("rotate", [True, False])
def test_weights_tiny(h32, rotate):
    w = wl.TINY.chain[0].weights(0, wl.CFG_TINY)
    wq, wd = h32.h32_rotate_quantize_weights_q4_0(torch_of(w), rotate=rotate)
    rq, rd = oracle.quantize_weights_q4_0(w, rotate)
    _same(np_of(wq), rq)
    _same(wd_bits(wd), rd)


def test_weights_edge_blocks(h32):
    rows = [np.zeros(32), np.arange(32.0) - 16, np.r_[0, 0, 0, 1.0, 0, 0, 0, -1.0, np.zeros(24)],
            np.r_[2.0 ** -140, np.zeros(31)], np.full(32, 1e5)]
    w = np.stack(rows).astype(np.float32)
    for rotate in (True, False):
        wq, wd = h32.h32_rotate_quantize_weights_q4_0(torch_of(w), rotate=rotate)
        rq, rd = oracle.quantize_weights_q4_0(w, rotate)
        _same(np_of(wq), rq)
        _same(wd_bits(wd), rd)


def test_weights_pp512_gate_up_full(h32):
    """Full-size offline step: 34816 x 5120 weights, every code and scale."""
    w = wl.FFN_GATE_UP.weights(0, wl.CFG_FFN)
    wq, wd = h32.h32_rotate_quantize_weights_q4_0(torch_of(w))
    rq, rd = oracle.quantize_weights_q4_0(w)
    _same(np_of(wq), rq)
    _same(wd_bits(wd), rd)
