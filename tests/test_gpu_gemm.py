"""GPU parity of the block-scaled integer GEMMs against the CPU oracle.

The product ("509 tokens a second of prompt: the Hadamard route ships",
sections "Why prompts are a matrix-unit problem" and "The rotation"): exact
int32 block sums of 4-bit (or 8-bit) activation codes against Q4_0 weight
codes, scaled by both blocks' scales and accumulated in block order in fp32.
Bar: block sums bit-exact; fp32 outputs equal to the oracle's same-order fp32
result (tolerance 1e-5 relative, met with 0 difference) and within 1e-3 of its
fp64 result.  The oracle computes every input from the seeded generators.
"""
import numpy as np
import pytest

import oracle
from hadamard_rotated_bit_gb300 import workloads as wl
from tests._gpu import np_of, torch_of

pytestmark = pytest.mark.gpu

REL_F32 = 1e-5   # against the oracle's same-order fp32 accumulation
REL_F64 = 1e-3   # against the oracle's fp64 accumulation


@pytest.fixture(scope="module")
def h32():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import hadamard_rotated_bit_gb300 as m
    from hadamard_rotated_bit_gb300 import _build
    _build.build()
    return m


def rel_err(got, ref):
    """|g - r| / max(|r|, 1e-6 * max|r|): relative error that tolerates exact cancellation."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    floor = 1e-6 * max(np.abs(ref).max(), 1e-30)
    return np.abs(got - ref) / np.maximum(np.abs(ref), floor)


def f64_excess(got, r64, wd, xd_rows, S):
    """Error against the fp64 result in units of its allowance,
    max(1e-3 |y64|, (nb + 1) 2^-24 sum_b |d_w d_x S_b|): 1e-3 relative, or the
    forward error bound of fp32 recursive summation for outputs that cancel.
    wd: [P][nb] fp16 bits, xd_rows: [P][nb], S: [P][nb] -> values <= 1 pass."""
    nb = S.shape[-1]
    terms = np.abs(wd.view(np.float16).astype(np.float64) * xd_rows.astype(np.float64) * S)
    allow = np.maximum(REL_F64 * np.abs(r64), (nb + 1) * 2.0 ** -24 * terms.sum(axis=-1))
    allow = np.maximum(allow, 1e-300)
    return np.abs(np.asarray(got, np.float64) - r64) / allow


def operands(M, N, K, xbits, seed_tid, outlier_frac=0.01, outlier_scale=20.0, rotate=True):
    x = wl.act_normal_outliers(M, K, outlier_frac, outlier_scale, 0, wl.CFG_TEST, seed_tid)
    w = wl.weights_normal(N, K, 0.02, 0, wl.CFG_TEST, seed_tid + 1)
    wq, wd = oracle.quantize_weights_q4_0(w, rotate)
    if xbits == 4:
        xq, xd = oracle.quantize_act_q4(x, rotate)
    else:
        xq, xd = oracle.quantize_act_q8(x, rotate)
    return wq, wd, xq, xd


def run_gpu(h32, wq, wd, xq, xd, xbits, block_sums=True):
    import torch
    fn = h32.q4_0_x_q4_gemm if xbits == 4 else h32.q4_0_x_q8_gemm
    out = fn(torch_of(wq), torch_of(wd.view(np.int16)), torch_of(xq), torch_of(xd),
             block_sums=block_sums)
    torch.cuda.synchronize()
    assert h32.h32_device_status() == 0
    if block_sums:
        y, S = out
        return np_of(y), np_of(S)
    return np_of(out), None


def check_full(h32, wq, wd, xq, xd, K, xbits):
    y, S = run_gpu(h32, wq, wd, xq, xd, xbits)
    r32, r64, rS = oracle.gemm(wq, wd, xq, xd, K, want_block_sums=True)
    assert np.array_equal(S.astype(np.int64), rS), "block sums differ"
    assert rel_err(y, r32).max() <= REL_F32
    assert np.array_equal(y.view(np.uint32), r32.view(np.uint32)), "fp32 outputs not bit-identical"
    M, N, nb = rS.shape
    ex = f64_excess(y, r64, np.broadcast_to(wd[None], (M, N, nb)),
                    np.broadcast_to(xd[:, None, :], (M, N, nb)), rS)
    assert ex.max() <= 1.0


@pytest.mark.parametrize("xbits", [4, 8])
def test_tiny_config(h32, xbits):
    proj = wl.TINY.chain[0]
    x = proj.activations(wl.TINY.M, 0, wl.CFG_TINY, bf16=False)
    w = proj.weights(0, wl.CFG_TINY)
    wq, wd = oracle.quantize_weights_q4_0(w)
    xq, xd = (oracle.quantize_act_q4 if xbits == 4 else oracle.quantize_act_q8)(x)
    check_full(h32, wq, wd, xq, xd, proj.K, xbits)


@pytest.mark.parametrize("xbits", [4, 8])
@pytest.mark.parametrize("M,N,K", [(1, 16, 32), (17, 144, 96), (100, 256, 288), (129, 128, 160),
                                   (200, 48, 544), (300, 384, 64)])
def test_ragged_shapes(h32, xbits, M, N, K):
    wq, wd, xq, xd = operands(M, N, K, xbits, 40 + M)
    check_full(h32, wq, wd, xq, xd, K, xbits)


@pytest.mark.parametrize("xbits", [4, 8])
def test_unrotated_route(h32, xbits):
    wq, wd, xq, xd = operands(70, 160, 256, xbits, 60, rotate=False)
    check_full(h32, wq, wd, xq, xd, 256, xbits)


def test_extreme_codes(h32):
    """All activation codes -8 against weight value -8 (S = 2048 per block),
    mixed with +7 and zero blocks."""
    M, N, K = 40, 32, 256
    xq = np.full((M, K // 2), 0x88, np.uint8)
    xq[::3] = 0x77
    xq[1::5] = 0x00
    wq = np.zeros((N, K // 2), np.uint8)
    wq[::2] = 0xFF
    xd = np.full((M, K // 32), 0.5, np.float32)
    wd = oracle.f32_to_f16(np.full((N, K // 32), 0.25, np.float32))
    check_full(h32, wq, wd, xq, xd, K, 4)
    xq8 = np.full((M, K), -127, np.int8)
    xq8[::2] = 127
    xq8[1::7] = 119
    check_full(h32, wq, wd, xq8, xd, K, 8)


def test_tiny_scales_take_the_exact_slow_path(h32):
    """Activation rows of magnitude ~1e-33 give d_w * d_x below the normal
    range; the result must still equal the sequential fp32 definition."""
    M, N, K = 32, 64, 128
    x = wl.act_normal_outliers(M, K, 0.0, 1.0, 0, wl.CFG_TEST, 70)
    x[::4] *= np.float32(1e-33)
    w = wl.weights_normal(N, K, 0.02, 0, wl.CFG_TEST, 71)
    wq, wd = oracle.quantize_weights_q4_0(w)
    xq, xd = oracle.quantize_act_q4(x)
    y, S = run_gpu(h32, wq, wd, xq, xd, 4)
    r32, r64, rS = oracle.gemm(wq, wd, xq, xd, K, want_block_sums=True)
    assert np.array_equal(S.astype(np.int64), rS)
    assert np.array_equal(y.view(np.uint32), r32.view(np.uint32))


def test_gpu_quantizers_feed_gemm(h32):
    """The chain on the device: rotate+quantize activations and weights, then
    the GEMM, equals the oracle's chain bit for bit."""
    import torch
    M, N, K = 96, 256, 512
    x = wl.f32_to_bf16_bits(wl.act_normal_outliers(M, K, 0.005, 30.0, 0, wl.CFG_TEST, 80))
    w = wl.weights_normal(N, K, 0.02, 0, wl.CFG_TEST, 81)
    from tests._gpu import torch_bf16
    xq, xd = h32.h32_quantize_act_q4(torch_bf16(x))
    wq, wd = h32.h32_rotate_quantize_weights_q4_0(torch_of(w))
    y = h32.q4_0_x_q4_gemm(wq, wd, xq, xd)
    torch.cuda.synchronize()
    rwq, rwd = oracle.quantize_weights_q4_0(w)
    rxq, rxd = oracle.quantize_act_q4(x)
    r32, _, _ = oracle.gemm(rwq, rwd, rxq, rxd, K)
    assert np.array_equal(np_of(y).view(np.uint32), r32.view(np.uint32))


def test_row_pitch_of_y(h32):
    import torch
    M, N, K = 33, 64, 128
    wq, wd, xq, xd = operands(M, N, K, 4, 90)
    ybig = torch.full((M, N + 32), -7.0, dtype=torch.float32, device="cuda")
    h32.q4_0_x_q4_gemm(torch_of(wq), torch_of(wd.view(np.int16)), torch_of(xq), torch_of(xd),
                       y=ybig[:, :N])
    torch.cuda.synchronize()
    r32, _, _ = oracle.gemm(wq, wd, xq, xd, K)
    yb = np_of(ybig)
    assert np.array_equal(yb[:, :N].view(np.uint32), r32.view(np.uint32))
    assert np.all(yb[:, N:] == -7.0)


# --------------------------------------------------------------------------
# full-size configurations, sampled outputs
# --------------------------------------------------------------------------
def sampled_check(h32, wq, wd, xq, xd, K, xbits, nsamp=3000, seed=0):
    y, _ = run_gpu(h32, wq, wd, xq, xd, xbits, block_sums=False)
    M, N = y.shape
    r = np.random.default_rng(seed)
    mi = np.concatenate([r.integers(0, M, nsamp), [0, M - 1, M - 1, 0]])
    ni = np.concatenate([r.integers(0, N, nsamp), [0, N - 1, 0, N - 1]])
    r32, r64, rS = oracle.gemm_sampled(wq, wd, xq, xd, K, mi, ni, want_block_sums=True)
    got = y[mi, ni]
    assert np.array_equal(got.view(np.uint32), r32.view(np.uint32))
    assert f64_excess(got, r64, wd[ni], xd[mi], rS).max() <= 1.0
    assert np.isfinite(y).all()


@pytest.mark.parametrize("xbits", [4, 8])
def test_pp512_attention_projection(h32, xbits):
    p = wl.ATTN
    x = p.activations(512, 0, wl.CFG_ATTN)
    w = p.weights(0, wl.CFG_ATTN)
    wq, wd = oracle.quantize_weights_q4_0(w)
    xq, xd = (oracle.quantize_act_q4 if xbits == 4 else oracle.quantize_act_q8)(x)
    sampled_check(h32, wq, wd, xq, xd, p.K, xbits)


@pytest.mark.parametrize("xbits", [4, 8])
@pytest.mark.parametrize("proj", ["gate_up", "down"])
def test_pp512_ffn(h32, proj, xbits):
    p = wl.FFN_GATE_UP if proj == "gate_up" else wl.FFN_DOWN
    x = p.activations(512, 0, wl.CFG_FFN)
    w = p.weights(0, wl.CFG_FFN)
    wq, wd = oracle.quantize_weights_q4_0(w)
    xq, xd = (oracle.quantize_act_q4 if xbits == 4 else oracle.quantize_act_q8)(x)
    sampled_check(h32, wq, wd, xq, xd, p.K, xbits)


# --------------------------------------------------------------------------
# expert-batched GEMM
# --------------------------------------------------------------------------
def run_experts(h32, wq, wd, xq, xd, row_idx, off, N, K, block_sums=True):
    import torch
    R = int(off[-1])
    out = h32.q4_0_x_q4_gemm_experts(
        torch_of(wq), torch_of(wd.view(np.int16)), torch_of(xq), torch_of(xd),
        None if row_idx is None else torch_of(row_idx.astype(np.int32)),
        torch_of(off.astype(np.int32)), R, block_sums=block_sums)
    torch.cuda.synchronize()
    st = h32.h32_device_status()
    if block_sums:
        return np_of(out[0]), np_of(out[1]), st
    return np_of(out), None, st


def test_experts_small_all_outputs(h32):
    r = np.random.default_rng(5)
    E, N, K, T = 6, 48, 96, 30
    counts = np.array([3, 0, 140, 1, 17, 0])
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    R = int(off[-1])
    row_idx = r.integers(0, T, R).astype(np.int32)
    x = wl.act_normal_outliers(T, K, 0.02, 25.0, 0, wl.CFG_TEST, 100)
    w = wl.weights_normal(E * N, K, 0.02, 0, wl.CFG_TEST, 101)
    wq, wd = oracle.quantize_weights_q4_0(w)
    xq, xd = oracle.quantize_act_q4(x)
    wq, wd = wq.reshape(E, N, K // 2), wd.reshape(E, N, K // 32)
    y, S, st = run_experts(h32, wq, wd, xq, xd, row_idx, off, N, K)
    assert st == 0
    ri = np.repeat(np.arange(R), N)
    ni = np.tile(np.arange(N), R)
    r32, r64, rS = oracle.gemm_experts_sampled(wq, wd, xq, xd, row_idx, off, N, K, ri, ni, True)
    assert np.array_equal(S.reshape(R * N, -1).astype(np.int64), rS)
    assert np.array_equal(y.reshape(-1).view(np.uint32), r32.view(np.uint32))


def test_experts_identity_rows(h32):
    E, N, K = 3, 32, 64
    off = np.array([0, 5, 5, 21], np.int32)
    x = wl.act_normal_outliers(21, K, 0.0, 1.0, 0, wl.CFG_TEST, 110)
    w = wl.weights_normal(E * N, K, 0.02, 0, wl.CFG_TEST, 111)
    wq, wd = oracle.quantize_weights_q4_0(w)
    xq, xd = oracle.quantize_act_q4(x)
    wq, wd = wq.reshape(E, N, K // 2), wd.reshape(E, N, K // 32)
    y, S, st = run_experts(h32, wq, wd, xq, xd, None, off, N, K)
    assert st == 0
    ri = np.repeat(np.arange(21), N)
    ni = np.tile(np.arange(N), 21)
    r32, _, _ = oracle.gemm_experts_sampled(wq, wd, xq, xd, None, off, N, K, ri, ni)
    assert np.array_equal(y.reshape(-1).view(np.uint32), r32.view(np.uint32))


def test_experts_bad_offsets_guarded(h32):
    """Offsets that are not non-decreasing from 0 to R set the guard status and
    leave y untouched."""
    import torch
    E, N, K = 2, 16, 32
    wq = torch.zeros((E, N, K // 2), dtype=torch.uint8, device="cuda")
    wd = torch.zeros((E, N, 1), dtype=torch.int16, device="cuda")
    xq = torch.zeros((8, K // 2), dtype=torch.uint8, device="cuda")
    xd = torch.zeros((8, 1), dtype=torch.float32, device="cuda")
    off = torch.tensor([0, 6, 4], dtype=torch.int32, device="cuda")
    y = torch.full((4, N), 3.0, dtype=torch.float32, device="cuda")
    h32.q4_0_x_q4_gemm_experts(wq, wd, xq, xd, None, off, 4, y=y)
    assert h32.h32_device_status() == h32.H32_ERR_DEVICE_GUARD
    assert torch.all(y == 3.0)
    assert h32.h32_device_status() == 0


def test_experts_row_index_out_of_range_guarded(h32):
    import torch
    E, N, K = 1, 16, 32
    wq = torch.zeros((E, N, K // 2), dtype=torch.uint8, device="cuda")
    wd = torch.zeros((E, N, 1), dtype=torch.int16, device="cuda")
    xq = torch.zeros((4, K // 2), dtype=torch.uint8, device="cuda")
    xd = torch.ones((4, 1), dtype=torch.float32, device="cuda")
    off = torch.tensor([0, 3], dtype=torch.int32, device="cuda")
    ridx = torch.tensor([0, 99, 2], dtype=torch.int32, device="cuda")
    y = h32.q4_0_x_q4_gemm_experts(wq, wd, xq, xd, ridx, off, 3)
    assert h32.h32_device_status() == h32.H32_ERR_DEVICE_GUARD
    assert torch.all(y[1] == 0)


def test_moe_config_sampled(h32):
    """1024-token micro-batch, 128 experts, top-8 routing: gate/up and down."""
    cfg = wl.MOE
    row_idx, off, _ = wl.moe_routing(cfg)
    x_gu, x_dn = wl.moe_inputs(cfg)
    w_gu, w_dn = wl.moe_weights(cfg)
    r = np.random.default_rng(3)
    for x, w, ridx in ((x_gu, w_gu, row_idx), (x_dn, w_dn, None)):
        E, N, K = w.shape
        wq, wd = oracle.quantize_weights_q4_0(w.reshape(E * N, K))
        wq, wd = wq.reshape(E, N, K // 2), wd.reshape(E, N, K // 32)
        xq, xd = oracle.quantize_act_q4(x)
        y, _, st = run_experts(h32, wq, wd, xq, xd, ridx, off, N, K, block_sums=False)
        assert st == 0
        R = int(off[-1])
        ri = np.concatenate([r.integers(0, R, 3000), off[1:-1].astype(np.int64), [R - 1]])
        ni = r.integers(0, N, ri.size)
        r32, r64, rS = oracle.gemm_experts_sampled(wq, wd, xq, xd, ridx, off, N, K, ri, ni, True)
        got = y[ri, ni]
        assert np.array_equal(got.view(np.uint32), r32.view(np.uint32))
        e = np.searchsorted(off, ri, side="right") - 1
        xrow = ri if ridx is None else ridx[ri]
        assert f64_excess(got, r64, wd[e, ni], xd[xrow], rS).max() <= 1.0
