"""GPU parity of the tensor-core-form path against the CPU oracle.

The tc form stores every 4-bit code v as the e4m3 byte of the integer v (the
exact operand form of the FP8 tensor cores).  The bytes are decoded here with
an independent e4m3 decoder; codes and scales must equal the oracle's, and the
tc GEMM must equal the oracle's same-order fp32 result bit for bit ("509
tokens a second of prompt: the Hadamard route ships", sections "Why prompts
are a matrix-unit problem" and "The rotation")."""
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


def e4m3_value(b: np.ndarray) -> np.ndarray:
    """IEEE-style e4m3 (bias 7, subnormals, no infinities) -> float64."""
    b = b.astype(np.int64)
    sign = np.where(b & 0x80, -1.0, 1.0)
    e = (b >> 3) & 0xF
    m = b & 7
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1 + m / 8.0) * 2.0 ** (e - 7.0))
    return sign * mag


def test_prepack_matches_q4_0(h32):
    w = wl.weights_normal(80, 384, 0.02, 0, wl.CFG_TEST, 200)
    wq, wd = oracle.quantize_weights_q4_0(w)
    wp, wsc = h32.h32_prepack_weights_q4_0_tc(torch_of(wq), torch_of(wd.view(np.int16)))
    wp, wsc = np_of(wp), np_of(wsc)
    codes = oracle.decode_w4(wq, 384).astype(np.float64)
    assert np.array_equal(e4m3_value(wp), codes)
    nb = 384 // 32
    assert wsc.shape == (80, 12)
    assert np.array_equal(wsc.astype(np.float64), wd.view(np.float16).astype(np.float64))
    w2 = wl.weights_normal(16, 160, 0.02, 0, wl.CFG_TEST, 201)   # nb = 5, padded to 8
    wq2, wd2 = oracle.quantize_weights_q4_0(w2)
    wp2, wsc2 = h32.h32_prepack_weights_q4_0_tc(torch_of(wq2), torch_of(wd2.view(np.int16)))
    wsc2 = np_of(wsc2)
    assert wsc2.shape == (16, 8) and np.all(wsc2[:, 5:] == 0)


@pytest.mark.parametrize("M,K", [(1, 128), (37, 256), (512, 5120)])
def test_quantize_tc_matches_oracle(h32, M, K):
    x = wl.f32_to_bf16_bits(wl.act_normal_outliers(M, K, 0.005, 30.0, 0, wl.CFG_TEST, 210 + M))
    xw, xdt = h32.h32_quantize_act_q4_tc(torch_bf16(x))
    xw, xdt = np_of(xw), np_of(xdt)
    rq, rd = oracle.quantize_act_q4(x)
    codes = oracle.decode_act4(rq, K).astype(np.float64)
    assert np.array_equal(e4m3_value(xw), codes)
    assert np.array_equal(xdt[:, :M].T.view(np.uint32), rd.view(np.uint32))


EDGE_ROWS = [np.zeros(32), np.r_[2.0 ** -130, np.zeros(31)], np.arange(32.0),
             np.r_[7, 2.5, -0.5, 1.5, 3.5, -2.5, np.zeros(26)], np.full(32, -3.0),
             np.r_[3e38, -3e38, np.zeros(30)], np.eye(32)[5],
             np.r_[2.0 ** 24, 1.0, np.zeros(14), -(2.0 ** 24), np.zeros(15)],
             np.r_[np.zeros(7), -(2.0 ** -131), np.zeros(12), 2.0 ** -133, np.zeros(11)]]


@pytest.mark.parametrize("rotate", [True, False])
def test_quantize_tc_edge_blocks(h32, rotate):
    """Zero, subnormal-size (1/d overflows: zeros stay code 0), ramp, tie,
    constant, overflowing, one-hot and wide-range blocks through the tc
    quantizers (4-bit, 8-bit and the gathered form) against the oracle."""
    import torch
    x = np.stack(EDGE_ROWS).astype(np.float32)
    M, K = x.shape[0], 32
    rq, rd = oracle.quantize_act_q4(x, rotate)
    xw, xdt = h32.h32_quantize_act_q4_tc(torch_of(x), rotate=rotate)
    assert np.array_equal(e4m3_value(np_of(xw)), oracle.decode_act4(rq, K).astype(np.float64))
    assert np.array_equal(np_of(xdt)[:, :M].T.view(np.uint32), rd.view(np.uint32))
    rq8, rd8 = oracle.quantize_act_q8(x, rotate)
    xw8, xdt8 = h32.h32_quantize_act_q8_tc(torch_of(x), rotate=rotate)
    assert np.array_equal(_q8_codes_from_tc(np_of(xw8), K)[0], rq8.astype(np.float64))
    assert np.array_equal(np_of(xdt8)[:, :M].T.view(np.uint32), rd8.view(np.uint32))
    idx = np.array([8, 1, 1, 5, 0, 7], np.int32)
    xg, xgd = h32.h32_quantize_act_q4_tc_gather(torch_of(x), torch_of(idx), rotate=rotate)
    torch.cuda.synchronize()
    assert h32.h32_device_status() == 0
    assert np.array_equal(e4m3_value(np_of(xg)),
                          oracle.decode_act4(rq, K).astype(np.float64)[idx])
    assert np.array_equal(np_of(xgd)[:, :idx.size].T.view(np.uint32), rd[idx].view(np.uint32))


def _tc_operands(h32, x, w, bf16=True):
    """x: bf16 bits (uint16) when bf16, else fp32."""
    wq, wd = oracle.quantize_weights_q4_0(w)
    xq, xd = oracle.quantize_act_q4(x)
    wp, wsc = h32.h32_prepack_weights_q4_0_tc(torch_of(wq), torch_of(wd.view(np.int16)))
    xw, xdt = h32.h32_quantize_act_q4_tc(torch_bf16(x) if bf16 else torch_of(x))
    return (wq, wd, xq, xd), (wp, wsc, xw, xdt)


@pytest.mark.parametrize("M,N,K", [(1, 16, 128), (17, 144, 256), (64, 256, 512), (129, 128, 384),
                                   (300, 384, 1024),
                                   # last-wave tiles cut into pieces, some of them empty
                                   (33, 1024, 256), (34, 2560, 128)])
def test_gemm_tc_bit_exact(h32, M, N, K):
    import torch
    x = wl.f32_to_bf16_bits(wl.act_normal_outliers(M, K, 0.01, 20.0, 0, wl.CFG_TEST, 220 + M))
    w = wl.weights_normal(N, K, 0.02, 0, wl.CFG_TEST, 221 + N)
    (wq, wd, xq, xd), (wp, wsc, xw, xdt) = _tc_operands(h32, x, w)
    y, S = h32.q4_0_x_q4_gemm_tc(wp, wsc, xw, xdt, M=M, block_sums=True)
    torch.cuda.synchronize()
    assert h32.h32_device_status() == 0
    r32, r64, rS = oracle.gemm(wq, wd, xq, xd, K, want_block_sums=True)
    assert np.array_equal(np_of(S).astype(np.int64), rS)
    assert np.array_equal(np_of(y).view(np.uint32), r32.view(np.uint32))
    y2 = h32.q4_0_x_q4_gemm_tc(wp, wsc, xw, xdt, M=M)
    assert np.array_equal(np_of(y2).view(np.uint32), r32.view(np.uint32))


def test_gemm_tc_tiny_scales(h32):
    """Rows of magnitude ~1e-33 put d_w * d_x below the normal fp32 range; the
    tc GEMM takes no special path and must still equal the sequential fp32
    definition bit for bit."""
    import torch
    M, N, K = 32, 64, 256
    x = wl.act_normal_outliers(M, K, 0.0, 1.0, 0, wl.CFG_TEST, 230)
    x[::4] *= np.float32(1e-33)
    x[1::4] *= np.float32(1e30)
    w = wl.weights_normal(N, K, 0.02, 0, wl.CFG_TEST, 231)
    (wq, wd, xq, xd), (wp, wsc, xw, xdt) = _tc_operands(h32, x, w, bf16=False)
    y, S = h32.q4_0_x_q4_gemm_tc(wp, wsc, xw, xdt, M=M, block_sums=True)
    torch.cuda.synchronize()
    assert h32.h32_device_status() == 0
    r32, _, rS = oracle.gemm(wq, wd, xq, xd, K, want_block_sums=True)
    assert np.array_equal(np_of(S).astype(np.int64), rS)
    assert np.array_equal(np_of(y).view(np.uint32), r32.view(np.uint32))


def test_gemm_tc_extreme_codes(h32):
    """Weight value -8 against activation code -8 (S = 2048 per block, the
    largest block sum), next to +7 and all-zero blocks; e4m3 bytes are built
    here from their definition, independently of the quantizer."""
    import torch
    M, N, K = 40, 32, 256
    xc = np.full((M, K), -8, np.int64)
    xc[::3] = 7
    xc[1::5] = 0
    wc = np.zeros((N, K), np.int64)
    wc[::2] = -8
    wc[1::4] = 7

    def e4m3_bytes(c):
        lut = {0: 0x00, 1: 0x38, 2: 0x40, 3: 0x44, 4: 0x48, 5: 0x4A, 6: 0x4C, 7: 0x4E, 8: 0x50}
        mag = np.vectorize(lut.get)(np.abs(c))
        return (mag | np.where(c < 0, 0x80, 0)).astype(np.uint8)

    assert np.array_equal(e4m3_value(e4m3_bytes(np.arange(-8, 9))), np.arange(-8, 9))
    xd = np.full((M, K // 32), 0.5, np.float32)
    xd[2::7] = 1e-30
    wd = oracle.f32_to_f16(np.full((N, K // 32), 0.25, np.float32))
    # the same operands in the oracle's nibble layout: element j < 16 of a
    # block in the low nibble of byte j, element j + 16 in its high nibble
    def pack(u):
        u = u.reshape(u.shape[0], -1, 32)
        return ((u[:, :, :16] & 15) | ((u[:, :, 16:] & 15) << 4)).reshape(u.shape[0], -1).astype(np.uint8)

    wq = pack(wc + 8)
    xq = pack(xc)
    assert np.array_equal(oracle.decode_w4(wq, K), wc)
    assert np.array_equal(oracle.decode_act4(xq, K), xc)
    wsc = np.zeros((N, 8), np.float32)
    wsc[:, :K // 32] = wd.view(np.float16).astype(np.float32)
    xdt = np.zeros((K // 32, M), np.float32)
    xdt[:, :] = xd.T
    y, S = h32.q4_0_x_q4_gemm_tc(torch_of(e4m3_bytes(wc)), torch_of(wsc), torch_of(e4m3_bytes(xc)),
                                 torch_of(xdt), M=M, block_sums=True)
    torch.cuda.synchronize()
    assert h32.h32_device_status() == 0
    r32, _, rS = oracle.gemm(wq, wd, xq, xd, K, want_block_sums=True)
    assert np.abs(rS).max() == 2048
    assert np.array_equal(np_of(S).astype(np.int64), rS)
    assert np.array_equal(np_of(y).view(np.uint32), r32.view(np.uint32))


@pytest.mark.parametrize("proj", ["attn", "ffn_gate_up", "ffn_down"])
def test_gemm_tc_pp512_sampled(h32, proj):
    import torch
    p = {q.name: q for q in (wl.ATTN, wl.FFN_GATE_UP, wl.FFN_DOWN)}[proj]
    cid = wl.CFG_ATTN if p is wl.ATTN else wl.CFG_FFN
    x = p.activations(512, 0, cid)
    w = p.weights(0, cid)
    (wq, wd, xq, xd), (wp, wsc, xw, xdt) = _tc_operands(h32, x, w)
    y = np_of(h32.q4_0_x_q4_gemm_tc(wp, wsc, xw, xdt, M=512))
    torch.cuda.synchronize()
    assert h32.h32_device_status() == 0
    r = np.random.default_rng(1)
    mi = np.concatenate([r.integers(0, 512, 3000), [0, 511]])
    ni = np.concatenate([r.integers(0, p.N, 3000), [p.N - 1, 0]])
    r32, _, _ = oracle.gemm_sampled(wq, wd, xq, xd, p.K, mi, ni)
    assert np.array_equal(y[mi, ni].view(np.uint32), r32.view(np.uint32))


# --------------------------------------------------------------------------
# expert-batched products in tc form ("Where the engine is going: HRX and the
# NPU", section "4-bit activations reach the MoE experts")
# --------------------------------------------------------------------------
def test_quantize_tc_gather_matches_oracle(h32):
    import torch
    T, K, R = 37, 256, 101
    x = wl.f32_to_bf16_bits(wl.act_normal_outliers(T, K, 0.01, 20.0, 0, wl.CFG_TEST, 240))
    ridx = np.random.default_rng(7).integers(0, T, R).astype(np.int32)
    xw, xdt = h32.h32_quantize_act_q4_tc_gather(torch_bf16(x), torch_of(ridx))
    torch.cuda.synchronize()
    assert h32.h32_device_status() == 0
    rq, rd = oracle.quantize_act_q4(x[ridx])
    assert np.array_equal(e4m3_value(np_of(xw)), oracle.decode_act4(rq, K).astype(np.float64))
    assert np.array_equal(np_of(xdt)[:, :R].T.view(np.uint32), rd.view(np.uint32))


def test_quantize_tc_gather_index_guard(h32):
    import torch
    x = torch.ones((4, 64), dtype=torch.float32, device="cuda")
    ridx = torch.tensor([0, 9, 3, -1], dtype=torch.int32, device="cuda")
    xw, xdt = h32.h32_quantize_act_q4_tc_gather(x, ridx)
    assert h32.h32_device_status() == h32.H32_ERR_DEVICE_GUARD
    xw, xdt = np_of(xw), np_of(xdt)
    assert np.all(xw[[1, 3]] == 0) and np.all(xdt[:, [1, 3]] == 0)
    assert np.all(xdt[:, [0, 2]] > 0)
    assert h32.h32_device_status() == 0


def _tc_experts(h32, x, w, E, N, ridx, off, block_sums=True):
    """oracle operands + the tc path: gather-quantize (or plain), repack, experts GEMM."""
    import torch
    K = x.shape[1]
    wq, wd = oracle.quantize_weights_q4_0(w)
    xq, xd = oracle.quantize_act_q4(x)
    wp, wsc = h32.h32_prepack_weights_q4_0_tc(torch_of(wq), torch_of(wd.view(np.int16)))
    xt = torch_bf16(x) if x.dtype == np.uint16 else torch_of(x)
    if ridx is None:
        xw, xdt = h32.h32_quantize_act_q4_tc(xt)
    else:
        xw, xdt = h32.h32_quantize_act_q4_tc_gather(xt, torch_of(ridx))
    out = h32.q4_0_x_q4_gemm_tc_experts(wp, wsc, xw, xdt, torch_of(off), N, R=int(off[-1]),
                                        block_sums=block_sums)
    torch.cuda.synchronize()
    st = h32.h32_device_status()
    if block_sums:
        y, S = out
        return (wq.reshape(E, N, K // 2), wd.reshape(E, N, K // 32), xq, xd), np_of(y), np_of(S), st
    return (wq.reshape(E, N, K // 2), wd.reshape(E, N, K // 32), xq, xd), np_of(out), None, st


def test_tc_experts_small_all_outputs(h32):
    """Ragged groups (empty ones, a 1-row one, one longer than a tile), rows
    gathered by index, group starts not multiples of 4."""
    E, N, K, T = 6, 48, 256, 30
    counts = np.array([3, 0, 140, 1, 17, 0])
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    R = int(off[-1])
    ridx = np.random.default_rng(5).integers(0, T, R).astype(np.int32)
    x = wl.act_normal_outliers(T, K, 0.02, 25.0, 0, wl.CFG_TEST, 250)
    w = wl.weights_normal(E * N, K, 0.02, 0, wl.CFG_TEST, 251)
    (wq, wd, xq, xd), y, S, st = _tc_experts(h32, x, w, E, N, ridx, off)
    assert st == 0
    ri = np.repeat(np.arange(R), N)
    ni = np.tile(np.arange(N), R)
    r32, _, rS = oracle.gemm_experts_sampled(wq, wd, xq, xd, ridx, off, N, K, ri, ni, True)
    assert np.array_equal(S.reshape(R * N, -1).astype(np.int64), rS)
    assert np.array_equal(y.reshape(-1).view(np.uint32), r32.view(np.uint32))


def test_tc_experts_identity_rows(h32):
    E, N, K = 3, 32, 128
    off = np.array([0, 5, 5, 21], np.int32)
    x = wl.act_normal_outliers(21, K, 0.0, 1.0, 0, wl.CFG_TEST, 260)
    w = wl.weights_normal(E * N, K, 0.02, 0, wl.CFG_TEST, 261)
    (wq, wd, xq, xd), y, _, st = _tc_experts(h32, x, w, E, N, None, off, block_sums=False)
    assert st == 0
    ri = np.repeat(np.arange(21), N)
    ni = np.tile(np.arange(N), 21)
    r32, _, _ = oracle.gemm_experts_sampled(wq, wd, xq, xd, None, off, N, K, ri, ni)
    assert np.array_equal(y.reshape(-1).view(np.uint32), r32.view(np.uint32))


def test_tc_experts_every_group_width(h32):
    """Plain-output expert launches over groups of 1 .. 200 rows (every count
    of 16-column chunks a 128-token chunk can have, ragged chunk widths,
    groups longer than one chunk, empty groups) with group starts at every
    residue mod 4; every output against the oracle's same-order fp32 value."""
    counts = np.array([1, 7, 8, 9, 15, 16, 17, 23, 24, 25, 31, 33, 40, 47, 48, 49, 56, 63, 64,
                       65, 72, 79, 80, 81, 88, 95, 96, 97, 104, 111, 112, 113, 120, 125, 127,
                       128, 129, 0, 3, 200, 2, 41])
    E, N, K, T = counts.size, 32, 128, 300
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    R = int(off[-1])
    assert len({int(o) % 4 for o in off[:-1]}) == 4
    ridx = np.random.default_rng(11).integers(0, T, R).astype(np.int32)
    x = wl.act_normal_outliers(T, K, 0.02, 25.0, 0, wl.CFG_TEST, 270)
    w = wl.weights_normal(E * N, K, 0.02, 0, wl.CFG_TEST, 271)
    (wq, wd, xq, xd), y, _, st = _tc_experts(h32, x, w, E, N, ridx, off, block_sums=False)
    assert st == 0
    ri = np.repeat(np.arange(R), N)
    ni = np.tile(np.arange(N), R)
    r32, _, _ = oracle.gemm_experts_sampled(wq, wd, xq, xd, ridx, off, N, K, ri, ni)
    assert np.array_equal(y.reshape(-1).view(np.uint32), r32.view(np.uint32))


def test_tc_experts_bad_offsets_guarded(h32):
    import torch
    E, N, K = 2, 16, 128
    wp = torch.zeros((E * N, K), dtype=torch.uint8, device="cuda")
    wsc = torch.zeros((E * N, 4), dtype=torch.float32, device="cuda")
    xw = torch.zeros((8, K), dtype=torch.uint8, device="cuda")
    xdt = torch.zeros((K // 32, 8), dtype=torch.float32, device="cuda")
    off = torch.tensor([0, 6, 4], dtype=torch.int32, device="cuda")
    y = torch.full((4, N), 3.0, dtype=torch.float32, device="cuda")
    h32.q4_0_x_q4_gemm_tc_experts(wp, wsc, xw, xdt, off, N, R=4, y=y)
    assert h32.h32_device_status() == h32.H32_ERR_DEVICE_GUARD
    assert torch.all(y == 3.0)
    assert h32.h32_device_status() == 0


def test_tc_moe_config_sampled(h32):
    """1024-token micro-batch, 128 experts, top-8 routing: gate/up (rows gathered)
    and down (rows already grouped)."""
    cfg = wl.MOE
    row_idx, off, _ = wl.moe_routing(cfg)
    x_gu, x_dn = wl.moe_inputs(cfg)
    w_gu, w_dn = wl.moe_weights(cfg)
    r = np.random.default_rng(3)
    for x, w, ridx in ((x_gu, w_gu, row_idx), (x_dn, w_dn, None)):
        E, N, K = w.shape
        (wq, wd, xq, xd), y, _, st = _tc_experts(h32, x, w.reshape(E * N, K), E, N, ridx, off,
                                                  block_sums=False)
        assert st == 0
        R = int(off[-1])
        ri = np.concatenate([r.integers(0, R, 3000), off[1:-1].astype(np.int64), [R - 1]])
        ni = r.integers(0, N, ri.size)
        r32, _, _ = oracle.gemm_experts_sampled(wq, wd, xq, xd, ridx, off, N, K, ri, ni)
        assert np.array_equal(y[ri, ni].view(np.uint32), r32.view(np.uint32))


# --------------------------------------------------------------------------
# the exact 8-bit route in tc form: code = 16 h + l, both parts exact in e4m3
# --------------------------------------------------------------------------
def _q8_codes_from_tc(xw8, K):
    M = xw8.shape[0]
    v = e4m3_value(xw8).reshape(M, K // 32, 2, 32)
    return (v[:, :, 0, :] + v[:, :, 1, :]).reshape(M, K), v


@pytest.mark.parametrize("M,K", [(3, 128), (45, 256), (512, 5120)])
def test_quantize_q8_tc_matches_oracle(h32, M, K):
    x = wl.f32_to_bf16_bits(wl.act_normal_outliers(M, K, 0.005, 30.0, 0, wl.CFG_TEST, 270 + M))
    xw8, xdt = h32.h32_quantize_act_q8_tc(torch_bf16(x))
    xw8, xdt = np_of(xw8), np_of(xdt)
    rq, rd = oracle.quantize_act_q8(x)
    codes, parts = _q8_codes_from_tc(xw8, K)
    assert np.array_equal(codes, rq.astype(np.float64))
    # the parts are the digits: l in 0..15, 16 h with h in -8..7
    assert parts[:, :, 1, :].min() >= 0 and parts[:, :, 1, :].max() <= 15
    assert np.all(np.mod(parts[:, :, 0, :], 16) == 0)
    assert np.array_equal(xdt[:, :M].T.view(np.uint32), rd.view(np.uint32))


@pytest.mark.parametrize("M,N,K", [(1, 16, 128), (33, 144, 256), (130, 128, 512)])
def test_gemm_q8_tc_bit_exact(h32, M, N, K):
    import torch
    x = wl.f32_to_bf16_bits(wl.act_normal_outliers(M, K, 0.01, 20.0, 0, wl.CFG_TEST, 280 + M))
    w = wl.weights_normal(N, K, 0.02, 0, wl.CFG_TEST, 281 + N)
    wq, wd = oracle.quantize_weights_q4_0(w)
    xq, xd = oracle.quantize_act_q8(x)
    wp, wsc = h32.h32_prepack_weights_q4_0_tc(torch_of(wq), torch_of(wd.view(np.int16)))
    xw8, xdt = h32.h32_quantize_act_q8_tc(torch_bf16(x))
    y, S = h32.q4_0_x_q8_gemm_tc(wp, wsc, xw8, xdt, M=M, block_sums=True)
    torch.cuda.synchronize()
    assert h32.h32_device_status() == 0
    r32, _, rS = oracle.gemm(wq, wd, xq, xd, K, want_block_sums=True)
    assert np.array_equal(np_of(S).astype(np.int64), rS)
    assert np.array_equal(np_of(y).view(np.uint32), r32.view(np.uint32))


def test_gemm_q8_tc_extreme_codes(h32):
    """Codes +-127 against weight values -8 and +7: the largest 8-bit block sums
    (|S| = 32512), built here from the byte definition."""
    import torch
    M, N, K = 24, 32, 128
    xc = np.full((M, K), -127, np.int64)
    xc[::2] = 127
    xc[1::3] = 0
    xc[2::5, ::3] = -1
    wc = np.full((N, K), -8, np.int64)
    wc[1::2] = 7

    lut = {0: 0x00, 1: 0x38, 2: 0x40, 3: 0x44, 4: 0x48, 5: 0x4A, 6: 0x4C, 7: 0x4E, 8: 0x50}

    def e4m3_int(v):   # |v| <= 15 or a multiple of 16 up to 128: exact
        a = abs(int(v))
        if a <= 8:
            b = lut[a]
        elif a < 16:
            b = 0x48 + a
        else:
            b = lut[a // 16] + 0x20
        return b | (0x80 if v < 0 else 0)

    xb = np.zeros((M, 2 * K), np.uint8)
    for m in range(M):
        for k in range(K):
            c = int(xc[m, k])
            l = c & 15
            h = (c - l) // 16
            blk, j = divmod(k, 32)
            xb[m, 64 * blk + j] = e4m3_int(16 * h)
            xb[m, 64 * blk + 32 + j] = e4m3_int(l)
    assert np.array_equal(_q8_codes_from_tc(xb, K)[0], xc.astype(np.float64))
    wb = np.vectorize(e4m3_int)(wc).astype(np.uint8)
    xd = np.full((M, K // 32), 0.25, np.float32)
    wd = oracle.f32_to_f16(np.full((N, K // 32), 0.5, np.float32))
    wsc = wd.view(np.float16).astype(np.float32)
    xdt = np.ascontiguousarray(xd.T)
    y, S = h32.q4_0_x_q8_gemm_tc(torch_of(wb), torch_of(wsc), torch_of(xb), torch_of(xdt), M=M,
                                 block_sums=True)
    torch.cuda.synchronize()
    assert h32.h32_device_status() == 0
    def pack(u):
        u = u.reshape(u.shape[0], -1, 32)
        return ((u[:, :, :16] & 15) | ((u[:, :, 16:] & 15) << 4)).reshape(u.shape[0], -1).astype(np.uint8)
    wq = pack(wc + 8)
    r32, _, rS = oracle.gemm(wq, wd, xc.astype(np.int8), xd, K, want_block_sums=True)
    assert np.abs(rS).max() == 32512
    assert np.array_equal(np_of(S).astype(np.int64), rS)
    assert np.array_equal(np_of(y).view(np.uint32), r32.view(np.uint32))


def test_gemm_q8_tc_pp512_sampled(h32):
    import torch
    p = wl.ATTN
    x = p.activations(512, 0, wl.CFG_ATTN)
    w = p.weights(0, wl.CFG_ATTN)
    wq, wd = oracle.quantize_weights_q4_0(w)
    xq, xd = oracle.quantize_act_q8(x)
    wp, wsc = h32.h32_prepack_weights_q4_0_tc(torch_of(wq), torch_of(wd.view(np.int16)))
    xw8, xdt = h32.h32_quantize_act_q8_tc(torch_bf16(x))
    y = np_of(h32.q4_0_x_q8_gemm_tc(wp, wsc, xw8, xdt, M=512))
    torch.cuda.synchronize()
    assert h32.h32_device_status() == 0
    r = np.random.default_rng(2)
    mi = np.concatenate([r.integers(0, 512, 3000), [511]])
    ni = np.concatenate([r.integers(0, p.N, 3000), [p.N - 1]])
    r32, _, _ = oracle.gemm_sampled(wq, wd, xq, xd, p.K, mi, ni)
    assert np.array_equal(y[mi, ni].view(np.uint32), r32.view(np.uint32))


@pytest.mark.parametrize("proj", ["gate_up", "down"])
def test_gemm_q8_tc_pp512_ffn_sampled(h32, proj):
    """The exact 8-bit route at the pp512 FFN shapes (gate/up 512 x 34816 x 5120,
    down 512 x 5120 x 17408), sampled outputs against the oracle bit for bit."""
    import torch
    p = wl.FFN_GATE_UP if proj == "gate_up" else wl.FFN_DOWN
    x = p.activations(512, 0, wl.CFG_FFN)
    w = p.weights(0, wl.CFG_FFN)
    wq, wd = oracle.quantize_weights_q4_0(w)
    xq, xd = oracle.quantize_act_q8(x)
    wp, wsc = h32.h32_prepack_weights_q4_0_tc(torch_of(wq), torch_of(wd.view(np.int16)))
    xw8, xdt = h32.h32_quantize_act_q8_tc(torch_bf16(x))
    # the quantizer at this size: every code and scale
    codes, _ = _q8_codes_from_tc(np_of(xw8), p.K)
    assert np.array_equal(codes, xq.astype(np.float64))
    assert np.array_equal(np_of(xdt)[:, :512].T.view(np.uint32), xd.view(np.uint32))
    y = np_of(h32.q4_0_x_q8_gemm_tc(wp, wsc, xw8, xdt, M=512))
    torch.cuda.synchronize()
    assert h32.h32_device_status() == 0
    r = np.random.default_rng(3)
    mi = np.concatenate([r.integers(0, 512, 3000), [0, 511, 511, 0]])
    ni = np.concatenate([r.integers(0, p.N, 3000), [0, p.N - 1, 0, p.N - 1]])
    r32, _, _ = oracle.gemm_sampled(wq, wd, xq, xd, p.K, mi, ni)
    assert np.array_equal(y[mi, ni].view(np.uint32), r32.view(np.uint32))
    assert np.isfinite(y).all()


# --------------------------------------------------------------------------
# the fused producer: the product quantized for the next projection in the
# GEMM's own epilogue
# --------------------------------------------------------------------------
def test_gemm_tc_quant_next_pp512_sampled_rows(h32):
    """The attention projection at pp512 (512 x 5120 x 5120): 8 whole token rows
    of the next projection's input against the oracle's quantizer applied to
    the oracle's output rows."""
    import torch
    p = wl.ATTN
    x = p.activations(512, 0, wl.CFG_ATTN)
    w = p.weights(0, wl.CFG_ATTN)
    (wq, wd, xq, xd), (wp, wsc, xw, xdt) = _tc_operands(h32, x, w)
    _, xn, xnd = h32.q4_0_x_q4_gemm_tc_quant_next(wp, wsc, xw, xdt, M=512, want_y=False)
    torch.cuda.synchronize()
    assert h32.h32_device_status() == 0
    rows = np.array([0, 1, 77, 200, 311, 400, 510, 511])
    mi = np.repeat(rows, p.N)
    ni = np.tile(np.arange(p.N), rows.size)
    r32, _, _ = oracle.gemm_sampled(wq, wd, xq, xd, p.K, mi, ni)
    nq, nd = oracle.quantize_act_q4(r32.reshape(rows.size, p.N))
    assert np.array_equal(e4m3_value(np_of(xn)[rows]),
                          oracle.decode_act4(nq, p.N).astype(np.float64))
    assert np.array_equal(np_of(xnd)[:, rows].T.view(np.uint32), nd.view(np.uint32))


@pytest.mark.parametrize("rot", [True, False])
def test_gemm_tc_quant_next_degenerate_blocks(h32, rot):
    """Output blocks of the fused producer that are all zero (a zero token row)
    or of subnormal size (token rows scaled by 2^-131 and 2^-140, so the output
    blocks' 1/d overflows): the codes must equal the oracle's quantizer on the
    oracle's output, zeros staying code 0."""
    import torch
    M, N, K = 40, 128, 256
    x = wl.act_normal_outliers(M, K, 0.01, 20.0, 0, wl.CFG_TEST, 296).astype(np.float32)
    x[3] = 0.0
    x[5] *= np.float32(2.0 ** -131)
    x[6, :128] *= np.float32(2.0 ** -131)
    x[7] *= np.float32(2.0 ** -140)
    w = wl.weights_normal(N, K, 0.02, 0, wl.CFG_TEST, 297)
    (wq, wd, xq, xd), (wp, wsc, xw, xdt) = _tc_operands(h32, x, w, bf16=False)
    y, xn, xnd = h32.q4_0_x_q4_gemm_tc_quant_next(wp, wsc, xw, xdt, M=M, rotate_next=rot)
    torch.cuda.synchronize()
    assert h32.h32_device_status() == 0
    r32, _, _ = oracle.gemm(wq, wd, xq, xd, K)
    assert np.array_equal(np_of(y).view(np.uint32), r32.view(np.uint32))
    nq, nd = oracle.quantize_act_q4(r32, rot)
    assert np.any(np.isinf(np.float32(1.0) / nd[nd > 0]))   # some block is degenerate
    assert np.array_equal(e4m3_value(np_of(xn)), oracle.decode_act4(nq, N).astype(np.float64))
    assert np.array_equal(np_of(xnd)[:, :M].T.view(np.uint32), nd.view(np.uint32))


@pytest.mark.parametrize("M,N,K,rot", [(70, 160, 256, True), (17, 96, 128, False),
                                       (130, 256, 512, True)])
def test_gemm_tc_quant_next_matches_oracle(h32, M, N, K, rot):
    import torch
    x = wl.f32_to_bf16_bits(wl.act_normal_outliers(M, K, 0.01, 20.0, 0, wl.CFG_TEST, 290 + M))
    w = wl.weights_normal(N, K, 0.02, 0, wl.CFG_TEST, 291 + N)
    (wq, wd, xq, xd), (wp, wsc, xw, xdt) = _tc_operands(h32, x, w)
    y, xn, xnd = h32.q4_0_x_q4_gemm_tc_quant_next(wp, wsc, xw, xdt, M=M, rotate_next=rot)
    torch.cuda.synchronize()
    assert h32.h32_device_status() == 0
    r32, _, _ = oracle.gemm(wq, wd, xq, xd, K)
    assert np.array_equal(np_of(y).view(np.uint32), r32.view(np.uint32))
    # the next projection's input: the oracle's quantizer on the oracle's output
    nq, nd = oracle.quantize_act_q4(r32, rot)
    assert np.array_equal(e4m3_value(np_of(xn)), oracle.decode_act4(nq, N).astype(np.float64))
    assert np.array_equal(np_of(xnd)[:, :M].T.view(np.uint32), nd.view(np.uint32))
    # without y: the same codes
    y2, xn2, xnd2 = h32.q4_0_x_q4_gemm_tc_quant_next(wp, wsc, xw, xdt, M=M, want_y=False,
                                                      rotate_next=rot)
    torch.cuda.synchronize()
    assert y2 is None
    assert np.array_equal(np_of(xn2), np_of(xn)) and np.array_equal(np_of(xnd2), np_of(xnd))


def test_gemm_tc_long_prompt_microbatch_sampled(h32):
    """The long-prompt sweep's micro-batch: 1024 tokens through FFN gate/up
    (1024 x 34816 x 5120), sampled outputs against the oracle."""
    import torch
    p = wl.LONG_GATE_UP
    x = p.activations(1024, 0, wl.CFG_LONG)
    w = p.weights(0, wl.CFG_LONG)
    (wq, wd, xq, xd), (wp, wsc, xw, xdt) = _tc_operands(h32, x, w)
    y = np_of(h32.q4_0_x_q4_gemm_tc(wp, wsc, xw, xdt, M=1024))
    torch.cuda.synchronize()
    assert h32.h32_device_status() == 0
    r = np.random.default_rng(8)
    mi = np.concatenate([r.integers(0, 1024, 3000), [1023, 0]])
    ni = np.concatenate([r.integers(0, p.N, 3000), [p.N - 1, 0]])
    r32, _, _ = oracle.gemm_sampled(wq, wd, xq, xd, p.K, mi, ni)
    assert np.array_equal(y[mi, ni].view(np.uint32), r32.view(np.uint32))


def test_gemm_tc_output_pitch_and_zero_rows(h32):
    """y written into a wider buffer (ldy > N) leaves the padding untouched; M = 0
    is a no-op."""
    import torch
    M, N, K = 33, 96, 256
    x = wl.f32_to_bf16_bits(wl.act_normal_outliers(M, K, 0.01, 20.0, 0, wl.CFG_TEST, 310))
    w = wl.weights_normal(N, K, 0.02, 0, wl.CFG_TEST, 311)
    (wq, wd, xq, xd), (wp, wsc, xw, xdt) = _tc_operands(h32, x, w)
    big = torch.full((M, N + 32), 7.0, dtype=torch.float32, device="cuda")
    h32.q4_0_x_q4_gemm_tc(wp, wsc, xw, xdt, M=M, y=big[:, :N])
    torch.cuda.synchronize()
    assert h32.h32_device_status() == 0
    r32, _, _ = oracle.gemm(wq, wd, xq, xd, K)
    got = np_of(big)
    assert np.array_equal(got[:, :N].view(np.uint32), r32.view(np.uint32))
    assert np.all(got[:, N:] == 7.0)
    y0 = torch.empty((0, N), dtype=torch.float32, device="cuda")
    h32.q4_0_x_q4_gemm_tc(wp, wsc, xw, xdt, M=0, y=y0)
    torch.cuda.synchronize()
    assert h32.h32_device_status() == 0


def test_gemm_tc_many_tiles_per_cta_sampled(h32):
    """8192 tokens through the 5120x5120 projection in one call: every CTA of
    the persistent grid walks many tiles, so the stage and TMEM-buffer rings
    wrap many times; sampled outputs against the oracle, bit for bit."""
    import torch
    p = wl.ATTN
    x = p.activations(8192, 3, wl.CFG_ATTN)
    w = p.weights(0, wl.CFG_ATTN)
    (wq, wd, xq, xd), (wp, wsc, xw, xdt) = _tc_operands(h32, x, w)
    y = np_of(h32.q4_0_x_q4_gemm_tc(wp, wsc, xw, xdt, M=8192))
    torch.cuda.synchronize()
    assert h32.h32_device_status() == 0
    r = np.random.default_rng(9)
    mi = np.concatenate([r.integers(0, 8192, 4000), [8191, 0]])
    ni = np.concatenate([r.integers(0, p.N, 4000), [p.N - 1, 0]])
    r32, _, _ = oracle.gemm_sampled(wq, wd, xq, xd, p.K, mi, ni)
    assert np.array_equal(y[mi, ni].view(np.uint32), r32.view(np.uint32))


def test_back_to_back_launches_reuse_buffers(h32):
    """Quantize, GEMM, quantize again into the same activation buffers, GEMM
    again, eight rounds on one stream with no host synchronization: each kernel
    may start under its predecessor's tail, so this fails if a kernel touched
    memory before its predecessor finished (the second quantizer overwriting
    codes the first GEMM still reads, or a GEMM reading codes not yet written)."""
    import torch
    M, N, K = 256, 1024, 2048
    w = wl.weights_normal(N, K, 0.02, 0, wl.CFG_TEST, 330)
    wq, wd = oracle.quantize_weights_q4_0(w)
    wp, wsc = h32.h32_prepack_weights_q4_0_tc(torch_of(wq), torch_of(wd.view(np.int16)))
    xs = [wl.f32_to_bf16_bits(wl.act_normal_outliers(M, K, 0.01, 20.0, r, wl.CFG_TEST, 331))
          for r in range(8)]
    xdev = [torch_bf16(x) for x in xs]
    xw = torch.empty((M, K), dtype=torch.uint8, device="cuda")
    xdt = torch.zeros((K // 32, M), dtype=torch.float32, device="cuda")
    ys = [torch.empty((M, N), dtype=torch.float32, device="cuda") for _ in xs]
    torch.cuda.synchronize()
    for x, y in zip(xdev, ys):
        h32.h32_quantize_act_q4_tc(x, xw=xw, xdt=xdt)
        h32.q4_0_x_q4_gemm_tc(wp, wsc, xw, xdt, M=M, y=y)
    torch.cuda.synchronize()
    assert h32.h32_device_status() == 0
    for x, y in zip(xs, ys):
        xq, xd = oracle.quantize_act_q4(x)
        r32, _, _ = oracle.gemm(wq, wd, xq, xd, K)
        assert np.array_equal(np_of(y).view(np.uint32), r32.view(np.uint32))


def test_chain_step_captured_in_a_cuda_graph(h32):
    """Quantize + tc GEMM captured once in a CUDA graph (the launches carry the
    programmatic-dependency attribute) and replayed on new inputs written into
    the same buffers: every replay bit-exact against the oracle."""
    import torch
    M, N, K = 64, 256, 512
    w = wl.weights_normal(N, K, 0.02, 0, wl.CFG_TEST, 700)
    rwq, rwd = oracle.quantize_weights_q4_0(w)
    wp, wsc = h32.h32_prepack_weights_q4_0_tc(torch_of(rwq), torch_of(rwd.view(np.int16)))
    x = torch.empty((M, K), dtype=torch.float32, device="cuda")
    xw = torch.empty((M, K), dtype=torch.uint8, device="cuda")
    xdt = torch.zeros((K // 32, M), dtype=torch.float32, device="cuda")
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()

    def step():
        h32.h32_quantize_act_q4_tc(x, xw=xw, xdt=xdt, stream=s)
        h32.q4_0_x_q4_gemm_tc(wp, wsc, xw, xdt, M=M, y=y, stream=s)

    x.copy_(torch_of(wl.act_normal_outliers(M, K, 0.01, 20.0, 0, wl.CFG_TEST, 701)))
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        step()
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step()
    for tid in (702, 703):
        xh = wl.act_normal_outliers(M, K, 0.01, 20.0, 0, wl.CFG_TEST, tid)
        x.copy_(torch_of(xh))
        torch.cuda.synchronize()
        with torch.cuda.stream(s):
            g.replay()
        s.synchronize()
        assert h32.h32_device_status(s) == 0
        rxq, rxd = oracle.quantize_act_q4(xh)
        r32, _, _ = oracle.gemm(rwq, rwd, rxq, rxd, K)
        assert np.array_equal(np_of(y).view(np.uint32), r32.view(np.uint32)), tid
