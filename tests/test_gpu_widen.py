"""GPU parity of the widening form against the CPU oracle: the activation
quantizer that writes each code c as the e5m2 byte of 512 c (decoded here
independently), and the GEMMs that take the Q4_0 weight planes themselves and
widen the nibbles in shared memory (q4_0_x_q4_gemm_tc_widen and its
expert-batched form): exact block sums and the oracle's same-order fp32 result
bit for bit ("509 tokens a second of prompt: the Hadamard route ships",
sections "Why prompts are a matrix-unit problem" and "The rotation"; "Where the
engine is going: HRX and the NPU", section "4-bit activations reach the MoE
experts")."""
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


def e5m2_value(b: np.ndarray) -> np.ndarray:
    """Value of e5m2 bytes (sign, 5 exponent bits with bias 15, 2 mantissa bits)."""
    b = b.astype(np.int64)
    s = np.where(b & 0x80, -1.0, 1.0)
    e = (b >> 2) & 0x1F
    m = b & 3
    mag = np.where(e == 0, m / 4.0 * 2.0 ** -14, (1 + m / 4.0) * 2.0 ** (e - 15))
    return s * mag


def e5m2_bytes_x512(c: np.ndarray) -> np.ndarray:
    """The widening form's activation byte of code c (|c| <= 8), from its definition."""
    lut = {0: 0x00, 1: 0x60, 2: 0x64, 3: 0x66, 4: 0x68, 5: 0x69, 6: 0x6A, 7: 0x6B, 8: 0x6C}
    return (np.vectorize(lut.get)(np.abs(c)) | np.where(c < 0, 0x80, 0)).astype(np.uint8)


def test_e5m2_table_is_the_encoding():
    c = np.arange(-8, 9)
    assert np.array_equal(e5m2_value(e5m2_bytes_x512(c)), 512.0 * c)


def _operands(h32, x, w):
    """Oracle Q4_0 planes and 4-bit codes; the GPU gets the same Q4_0 planes and
    the widening form's activations (x: bf16 bits as uint16, or fp32)."""
    wq, wd = oracle.quantize_weights_q4_0(w)
    xq, xd = oracle.quantize_act_q4(x)
    xw, xdt = h32.h32_quantize_act_q4_tc_e5m2(torch_bf16(x) if x.dtype == np.uint16
                                              else torch_of(x))
    return (wq, wd, xq, xd), (torch_of(wq), torch_of(wd.view(np.int16)), xw, xdt)


@pytest.mark.parametrize("M,K,rot", [(1, 256, True), (37, 512, True), (512, 5120, True),
                                     (70, 256, False)])
def test_quantize_e5m2_matches_oracle(h32, M, K, rot):
    """Codes (decoded from the e5m2 bytes, divided by 512) and scales equal the
    oracle's 4-bit quantizer; degenerate and all-zero blocks included."""
    x = wl.act_normal_outliers(M, K, 0.01, 20.0, 0, wl.CFG_TEST, 600 + M)
    if M > 3:
        x[1, :32] = 0.0
        x[2, 32:64] *= np.float32(2.0 ** -140)
    xb = wl.f32_to_bf16_bits(x)
    xq, xd = oracle.quantize_act_q4(xb, rotate=32 if rot else 0)
    xw, xdt = h32.h32_quantize_act_q4_tc_e5m2(torch_bf16(xb), rotate=rot)
    codes = e5m2_value(np_of(xw)) / 512.0
    assert np.array_equal(codes.astype(np.int64), oracle.decode_act4(xq, K))
    assert np.array_equal(np_of(xdt)[:, :M].T.view(np.uint32), xd.view(np.uint32))
    assert h32.h32_device_status() == 0


@pytest.mark.parametrize("M,N,K", [(1, 16, 256), (17, 144, 256), (64, 256, 512), (129, 128, 768),
                                   (300, 384, 1024),
                                   # last-wave tiles cut into pieces, some of them empty
                                   (33, 1024, 256), (34, 2560, 256)])
def test_widen_bit_exact(h32, M, N, K):
    import torch
    x = wl.f32_to_bf16_bits(wl.act_normal_outliers(M, K, 0.01, 20.0, 0, wl.CFG_TEST, 620 + M))
    w = wl.weights_normal(N, K, 0.02, 0, wl.CFG_TEST, 621 + N)
    (wq, wd, xq, xd), (gq, gd, xw, xdt) = _operands(h32, x, w)
    y, S = h32.q4_0_x_q4_gemm_tc_widen(gq, gd, xw, xdt, M=M, block_sums=True)
    torch.cuda.synchronize()
    assert h32.h32_device_status() == 0
    r32, _, rS = oracle.gemm(wq, wd, xq, xd, K, want_block_sums=True)
    assert np.array_equal(np_of(S).astype(np.int64), rS)
    assert np.array_equal(np_of(y).view(np.uint32), r32.view(np.uint32))
    y2 = h32.q4_0_x_q4_gemm_tc_widen(gq, gd, xw, xdt, M=M)
    assert np.array_equal(np_of(y2).view(np.uint32), r32.view(np.uint32))


def test_widen_every_weight_code(h32):
    """Every Q4_0 code 0..15 at every position of a block (rows of the weight
    matrix cycle through the codes with a different phase each), against
    activation codes of both signs up to -8; block sums exact."""
    import torch
    M, N, K = 48, 64, 256
    n = np.arange(N)[:, None]
    k = np.arange(K)[None, :]
    wc = ((n * 7 + k * 3 + (k // 32)) % 16).astype(np.int64)          # codes q
    xc = (((np.arange(M)[:, None] * 5 + k) % 16) - 8).astype(np.int64)  # -8 .. 7

    def pack(u):
        u = u.reshape(u.shape[0], -1, 32)
        return ((u[:, :, :16] & 15) | ((u[:, :, 16:] & 15) << 4)).reshape(u.shape[0], -1).astype(np.uint8)

    wq = pack(wc)
    xq = pack(xc)
    assert np.array_equal(oracle.decode_w4(wq, K), wc - 8)
    assert np.array_equal(oracle.decode_act4(xq, K), xc)
    wd = oracle.f32_to_f16(np.full((N, K // 32), 0.125, np.float32))
    xd = np.full((M, K // 32), 0.5, np.float32)
    xb = e5m2_bytes_x512(xc)     # activation bytes built here from the definition
    xdt = np.ascontiguousarray(xd.T)
    y, S = h32.q4_0_x_q4_gemm_tc_widen(torch_of(wq), torch_of(wd.view(np.int16)), torch_of(xb),
                                       torch_of(xdt), M=M, block_sums=True)
    torch.cuda.synchronize()
    assert h32.h32_device_status() == 0
    r32, _, rS = oracle.gemm(wq, wd, xq, xd, K, want_block_sums=True)
    assert np.array_equal(np_of(S).astype(np.int64), rS)
    assert np.array_equal(np_of(y).view(np.uint32), r32.view(np.uint32))


def test_widen_extreme_sums(h32):
    """Weight value -8 (code 0) against activation code -8: S = 2048, the
    largest block sum, next to +7 blocks and zero blocks."""
    import torch
    M, N, K = 40, 32, 256
    xc = np.full((M, K), -8, np.int64)
    xc[::3] = 7
    xc[1::5] = 0
    wc = np.zeros((N, K), np.int64)   # code 0: value -8
    wc[1::4] = 15                     # value +7
    wc[2::4] = 8                      # value 0

    def pack(u):
        u = u.reshape(u.shape[0], -1, 32)
        return ((u[:, :, :16] & 15) | ((u[:, :, 16:] & 15) << 4)).reshape(u.shape[0], -1).astype(np.uint8)

    wq, xq = pack(wc), pack(xc)
    wd = oracle.f32_to_f16(np.full((N, K // 32), 0.25, np.float32))
    xd = np.full((M, K // 32), 0.5, np.float32)
    xd[2::7] = 1e-30
    xb = e5m2_bytes_x512(xc)
    y, S = h32.q4_0_x_q4_gemm_tc_widen(torch_of(wq), torch_of(wd.view(np.int16)), torch_of(xb),
                                       torch_of(np.ascontiguousarray(xd.T)), M=M, block_sums=True)
    torch.cuda.synchronize()
    assert h32.h32_device_status() == 0
    r32, _, rS = oracle.gemm(wq, wd, xq, xd, K, want_block_sums=True)
    assert np.abs(rS).max() == 2048
    assert np.array_equal(np_of(S).astype(np.int64), rS)
    assert np.array_equal(np_of(y).view(np.uint32), r32.view(np.uint32))


def test_widen_tiny_scales(h32):
    """Products d_w * d_x below the normal fp32 range take no special path."""
    import torch
    M, N, K = 32, 64, 256
    x = wl.act_normal_outliers(M, K, 0.0, 1.0, 0, wl.CFG_TEST, 630)
    x[::4] *= np.float32(1e-33)
    x[1::4] *= np.float32(1e30)
    w = wl.weights_normal(N, K, 0.02, 0, wl.CFG_TEST, 631)
    (wq, wd, xq, xd), (gq, gd, xw, xdt) = _operands(h32, x, w)
    y, S = h32.q4_0_x_q4_gemm_tc_widen(gq, gd, xw, xdt, M=M, block_sums=True)
    torch.cuda.synchronize()
    assert h32.h32_device_status() == 0
    r32, _, rS = oracle.gemm(wq, wd, xq, xd, K, want_block_sums=True)
    assert np.array_equal(np_of(S).astype(np.int64), rS)
    assert np.array_equal(np_of(y).view(np.uint32), r32.view(np.uint32))


@pytest.mark.parametrize("proj", ["attn", "ffn_gate_up", "ffn_down"])
def test_widen_pp512_sampled(h32, proj):
    """The pp512 projections in the launch configuration the bench times:
    sampled outputs against the oracle, every output against the repacked-form
    GEMM (two GPU paths, same bits)."""
    import torch
    p = {q.name: q for q in (wl.ATTN, wl.FFN_GATE_UP, wl.FFN_DOWN)}[proj]
    cid = wl.CFG_ATTN if p is wl.ATTN else wl.CFG_FFN
    x = p.activations(512, 0, cid)
    w = p.weights(0, cid)
    (wq, wd, xq, xd), (gq, gd, xw, xdt) = _operands(h32, x, w)
    y = h32.q4_0_x_q4_gemm_tc_widen(gq, gd, xw, xdt, M=512)
    wp, wsc = h32.h32_prepack_weights_q4_0_tc(gq, gd)
    xw4, xdt4 = h32.h32_quantize_act_q4_tc(torch_bf16(x))
    y_tc = h32.q4_0_x_q4_gemm_tc(wp, wsc, xw4, xdt4, M=512)
    torch.cuda.synchronize()
    assert h32.h32_device_status() == 0
    y = np_of(y)
    assert np.array_equal(y.view(np.uint32), np_of(y_tc).view(np.uint32))
    r = np.random.default_rng(2)
    mi = np.concatenate([r.integers(0, 512, 3000), [0, 511]])
    ni = np.concatenate([r.integers(0, p.N, 3000), [p.N - 1, 0]])
    r32, _, _ = oracle.gemm_sampled(wq, wd, xq, xd, p.K, mi, ni)
    assert np.array_equal(y[mi, ni].view(np.uint32), r32.view(np.uint32))


# --------------------------------------------------------------------------
# expert-batched
# --------------------------------------------------------------------------
def _experts(h32, x, w, E, N, ridx, off, block_sums=False):
    import torch
    K = x.shape[1]
    wq, wd = oracle.quantize_weights_q4_0(w)
    xq, xd = oracle.quantize_act_q4(x)
    xt = torch_bf16(x) if x.dtype == np.uint16 else torch_of(x)
    if ridx is None:
        xw, xdt = h32.h32_quantize_act_q4_tc_e5m2(xt)
    else:
        xw, xdt = h32.h32_quantize_act_q4_tc_e5m2_gather(xt, torch_of(ridx))
    out = h32.q4_0_x_q4_gemm_tc_widen_experts(torch_of(wq), torch_of(wd.view(np.int16)), xw, xdt,
                                              torch_of(off), N, R=int(off[-1]),
                                              block_sums=block_sums)
    torch.cuda.synchronize()
    st = h32.h32_device_status()
    y, S = out if block_sums else (out, None)
    ops = (wq.reshape(E, N, K // 2), wd.reshape(E, N, K // 32), xq, xd)
    return ops, np_of(y), (np_of(S) if S is not None else None), st


def test_widen_experts_small_all_outputs(h32):
    """Ragged groups (empty ones, a 1-row one, one longer than a tile), rows
    gathered by index, group starts not multiples of 4; block sums too."""
    E, N, K, T = 6, 48, 256, 30
    counts = np.array([3, 0, 140, 1, 17, 0])
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    R = int(off[-1])
    ridx = np.random.default_rng(15).integers(0, T, R).astype(np.int32)
    x = wl.act_normal_outliers(T, K, 0.02, 25.0, 0, wl.CFG_TEST, 640)
    w = wl.weights_normal(E * N, K, 0.02, 0, wl.CFG_TEST, 641)
    (wq, wd, xq, xd), y, S, st = _experts(h32, x, w, E, N, ridx, off, block_sums=True)
    assert st == 0
    ri = np.repeat(np.arange(R), N)
    ni = np.tile(np.arange(N), R)
    r32, _, rS = oracle.gemm_experts_sampled(wq, wd, xq, xd, ridx, off, N, K, ri, ni, True)
    assert np.array_equal(S.reshape(R * N, -1).astype(np.int64), rS)
    assert np.array_equal(y.reshape(-1).view(np.uint32), r32.view(np.uint32))


def test_widen_experts_every_group_width(h32):
    """Groups of 1 .. 200 rows at every residue mod 4 of their start; every
    output against the oracle."""
    counts = np.array([1, 7, 8, 9, 15, 16, 17, 23, 24, 25, 31, 33, 40, 47, 48, 49, 56, 63, 64,
                       65, 72, 79, 80, 81, 88, 95, 96, 97, 104, 111, 112, 113, 120, 125, 127,
                       128, 129, 0, 3, 200, 2, 41])
    E, N, K, T = counts.size, 32, 256, 300
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    R = int(off[-1])
    assert len({int(o) % 4 for o in off[:-1]}) == 4
    ridx = np.random.default_rng(17).integers(0, T, R).astype(np.int32)
    x = wl.act_normal_outliers(T, K, 0.02, 25.0, 0, wl.CFG_TEST, 650)
    w = wl.weights_normal(E * N, K, 0.02, 0, wl.CFG_TEST, 651)
    (wq, wd, xq, xd), y, _, st = _experts(h32, x, w, E, N, ridx, off)
    assert st == 0
    ri = np.repeat(np.arange(R), N)
    ni = np.tile(np.arange(N), R)
    r32, _, _ = oracle.gemm_experts_sampled(wq, wd, xq, xd, ridx, off, N, K, ri, ni)
    assert np.array_equal(y.reshape(-1).view(np.uint32), r32.view(np.uint32))


def test_quantize_e5m2_gather_matches_oracle(h32):
    T, K, R = 50, 256, 90
    ridx = np.random.default_rng(21).integers(0, T, R).astype(np.int32)
    x = wl.act_normal_outliers(T, K, 0.02, 25.0, 0, wl.CFG_TEST, 660)
    xq, xd = oracle.quantize_act_q4(x[ridx])
    xw, xdt = h32.h32_quantize_act_q4_tc_e5m2_gather(torch_of(x), torch_of(ridx))
    codes = e5m2_value(np_of(xw)) / 512.0
    assert np.array_equal(codes.astype(np.int64), oracle.decode_act4(xq, K))
    assert np.array_equal(np_of(xdt)[:, :R].T.view(np.uint32), xd.view(np.uint32))
    assert h32.h32_device_status() == 0


def test_widen_experts_bad_offsets_guarded(h32):
    import torch
    E, N, K = 2, 16, 256
    wq = torch.zeros((E * N, K // 2), dtype=torch.uint8, device="cuda")
    wd = torch.zeros((E * N, K // 32), dtype=torch.int16, device="cuda")
    xw = torch.zeros((8, K), dtype=torch.uint8, device="cuda")
    xdt = torch.zeros((K // 32, 8), dtype=torch.float32, device="cuda")
    off = torch.tensor([0, 6, 4], dtype=torch.int32, device="cuda")
    y = torch.full((4, N), 3.0, dtype=torch.float32, device="cuda")
    h32.q4_0_x_q4_gemm_tc_widen_experts(wq, wd, xw, xdt, off, N, R=4, y=y)
    assert h32.h32_device_status() == h32.H32_ERR_DEVICE_GUARD
    assert torch.all(y == 3.0)
    assert h32.h32_device_status() == 0


def test_widen_moe_config_sampled(h32):
    """1024-token micro-batch, 128 experts, top-8 routing: gate/up (rows
    gathered) and down (rows already grouped), as the bench launches them."""
    cfg = wl.MOE
    row_idx, off, _ = wl.moe_routing(cfg)
    x_gu, x_dn = wl.moe_inputs(cfg)
    w_gu, w_dn = wl.moe_weights(cfg)
    r = np.random.default_rng(4)
    for x, w, ridx in ((x_gu, w_gu, row_idx), (x_dn, w_dn, None)):
        E, N, K = w.shape
        (wq, wd, xq, xd), y, _, st = _experts(h32, x, w.reshape(E * N, K), E, N, ridx, off)
        assert st == 0
        R = int(off[-1])
        ri = np.concatenate([r.integers(0, R, 3000), off[1:-1].astype(np.int64), [R - 1]])
        ni = r.integers(0, N, ri.size)
        r32, _, _ = oracle.gemm_experts_sampled(wq, wd, xq, xd, ridx, off, N, K, ri, ni)
        assert np.array_equal(y[ri, ni].view(np.uint32), r32.view(np.uint32))
