"""Pins for the CPU oracle: each check ties it to something other than itself.

Sources: "509 tokens a second of prompt: the Hadamard route ships" (sections
"Why prompts are a matrix-unit problem", "The rotation", "Making the file is
part of the engine") and "Prompt processing: 4-bit activations, rotated
first".  The pins are closed forms, a library Hadamard matrix, brute force on
small inputs, exhaustive decode tables and hand-derived golden blocks, chosen
so that a dropped term, a wrong sign or index, or a transposed operand in the
oracle fails at least one of them.
"""
from decimal import Decimal, getcontext

import numpy as np
import pytest
import scipy.linalg

import oracle
from hadamard_rotated_bit_gb300 import workloads as wl

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _ints(s):
    return np.array([int(t) for t in s.split()], np.int64)


def _hexbytes(s):
    return np.array([int(t, 16) for t in s.split()], np.uint8)


def _popcount(v):
    return bin(v).count("1")


# --------------------------------------------------------------------------
# the rotation
# --------------------------------------------------------------------------
def test_scale_constant_is_nearest_fp32_to_inv_sqrt32():
    getcontext().prec = 60
    exact = Decimal(1) / Decimal(32).sqrt()
    c = np.float32(oracle.h32_scale())
    up = np.nextafter(c, np.float32(1))
    dn = np.nextafter(c, np.float32(0))
    err = abs(Decimal(float(c)) - exact)
    assert err <= abs(Decimal(float(up)) - exact)
    assert err <= abs(Decimal(float(dn)) - exact)
    assert c.view(np.uint32) == 0x3E3504F3


def _materialize_h():
    """Column k of the transform is its image of the unit vector e_k."""
    eye = np.eye(32, dtype=np.float32)
    cols = oracle.fwht32(eye.reshape(-1)).reshape(32, 32)  # row k = H e_k
    return cols.T.astype(np.float64)  # H[i][k]


def test_h_entries_are_sylvester_signs_times_c():
    H = _materialize_h()
    c = np.float64(np.float32(oracle.h32_scale()))
    for i in range(32):
        for k in range(32):
            assert H[i, k] == (-1) ** _popcount(i & k) * c


def test_h_is_orthonormal():
    H = _materialize_h()
    err = np.abs(H @ H.T - np.eye(32)).max()
    assert err <= 1e-6


def test_h_matches_library_hadamard():
    H = _materialize_h()
    ref = scipy.linalg.hadamard(32).astype(np.float64) / np.sqrt(32.0)
    assert np.abs(H - ref).max() <= 1e-7


def test_fwht_random_blocks_vs_dense_matrix():
    r = np.random.default_rng(1)
    x = r.standard_normal((200, 32)).astype(np.float32)
    ref = x.astype(np.float64) @ (scipy.linalg.hadamard(32) / np.sqrt(32.0)).T
    y32 = oracle.fwht32(x.reshape(-1)).reshape(200, 32).astype(np.float64)
    y64 = oracle.fwht32_f64(x.astype(np.float64).reshape(-1)).reshape(200, 32)
    scale = np.abs(x).sum(axis=1, keepdims=True)
    assert (np.abs(y32 - ref) <= 8 * 2.0 ** -24 * scale + 1e-30).all()
    assert np.abs(y64 - ref).max() <= 1e-13 * scale.max()


def test_invariance_x_dot_w_fp64():
    """x . w = (Hx) . (Hw): the transform is orthogonal ("The rotation")."""
    r = np.random.default_rng(2)
    for K in (32, 256, 5120):
        x = r.standard_normal(K)
        w = r.standard_normal(K)
        hx, hw = oracle.fwht32_f64(x), oracle.fwht32_f64(w)
        a, b = float(x @ w), float(hx @ hw)
        denom = float(np.abs(x * w).sum())
        assert abs(a - b) <= 1e-9 * denom


def test_stage_order_golden(golden):
    g = golden("fwht_order.txt")
    x = np.zeros(32, np.float32)
    x[0], x[1], x[16] = 2.0 ** 24, 1.0, -(2.0 ** 24)
    c = np.float32(oracle.h32_scale())
    v = np.array([float(t) for t in g["v_before_scale"].split()], np.float32)
    assert np.array_equal(oracle.fwht32(x), (v * c).astype(np.float32))


def test_one_hot_block_closed_form():
    c = np.float32(oracle.h32_scale())
    for k in (0, 1, 5, 16, 31):
        x = np.zeros((1, 32), np.float32)
        x[0, k] = 1.0
        y = oracle.fwht32(x.reshape(-1))
        sign = np.array([(-1) ** _popcount(i & k) for i in range(32)], np.float32)
        assert np.array_equal(y, sign * c)
        xq, xd = oracle.quantize_act_q4(x)
        codes = oracle.decode_act4(xq, 32)[0]
        assert np.array_equal(codes, (7 * sign).astype(np.int8))
        # d is the fp32 quotient amax / 7 with amax = C
        assert xd[0, 0] == np.float32(c / np.float32(7))


def test_constant_block_closed_form():
    c = np.float32(oracle.h32_scale())
    for val in (0.75, -3.0, 1e-3):
        x = np.full((1, 32), val, np.float32)
        y = oracle.fwht32(x.reshape(-1))
        assert y[0] == np.float32(np.float32(32 * val) * c)
        assert np.all(y[1:] == 0)
        codes = oracle.decode_act4(oracle.quantize_act_q4(x)[0], 32)[0]
        expect = np.zeros(32, np.int8)
        expect[0] = 7 if val > 0 else -7
        assert np.array_equal(codes, expect)
        codes8 = oracle.quantize_act_q8(x)[0][0]
        expect[0] = 127 if val > 0 else -127
        assert np.array_equal(codes8, expect)


def test_all_zero_block():
    x = np.zeros((2, 64), np.float32)
    xq, xd = oracle.quantize_act_q4(x)
    assert np.all(xq == 0) and np.all(xd == 0)
    wq, wd = oracle.quantize_weights_q4_0(x)
    # d = 0 / -8 is -0 in IEEE arithmetic: fp16 bits 0x8000; every code is 8 (value 0)
    assert np.all(wq == 0x88) and np.all(wd == 0x8000)


# --------------------------------------------------------------------------
# activation codes and scales: golden ramp block and properties
# --------------------------------------------------------------------------
def test_ramp_block_golden(golden):
    g = golden("ramp_block_act.txt")
    x = np.arange(32, dtype=np.float32)[None, :]
    c = np.float32(oracle.h32_scale())
    y = oracle.fwht32(x.reshape(-1))
    v = np.zeros(32, np.float32)
    for tok in g["v_nonzero"].split():
        i, val = tok.split(":")
        v[int(i)] = float(val)
    assert np.array_equal(y, (v * c).astype(np.float32))
    xq, xd = oracle.quantize_act_q4(x)
    assert np.array_equal(xq[0], _hexbytes(g["q4_bytes"]))
    assert np.array_equal(oracle.decode_act4(xq, 32)[0], _ints(g["q4_codes"]))
    assert abs(float(xd[0, 0]) - 496 / (7 * np.sqrt(32))) <= 2e-6 * float(xd[0, 0])
    q8, d8 = oracle.quantize_act_q8(x)
    assert np.array_equal(q8[0].astype(np.int64), _ints(g["q8_codes"]))
    assert abs(float(d8[0, 0]) - 496 / (127 * np.sqrt(32))) <= 2e-6 * float(d8[0, 0])


def test_tie_block_golden(golden):
    g = golden("tie_block.txt")
    for bits in (4, 8):
        x = np.zeros((1, 32), np.float32)
        vals = [float(t) for t in g[f"q{bits}_input"].split()]
        x[0, :len(vals)] = vals
        expect = np.zeros(32, np.int64)
        codes = _ints(g[f"q{bits}_codes"])
        expect[:codes.size] = codes
        if bits == 4:
            xq, xd = oracle.quantize_act_q4(x, rotate=False)
            got = oracle.decode_act4(xq, 32)[0]
        else:
            xq, xd = oracle.quantize_act_q8(x, rotate=False)
            got = xq[0]
        assert xd[0, 0] == 1.0
        assert np.array_equal(got.astype(np.int64), expect)


def test_tiny_block_edge_golden(golden):
    """Blocks whose 1/d overflows: zeros stay 0, the largest element gets +-qmax."""
    g = golden("tiny_block.txt")
    u = np.float32(2.0 ** -149)
    x = np.zeros((1, 32), np.float32)
    x[0, 0] = np.float32(2.0 ** -130)
    xq, xd = oracle.quantize_act_q4(x, rotate=False)
    assert xd[0, 0] == np.float32(int(g["case_a_d_units"]) * u)
    assert np.array_equal(oracle.decode_act4(xq, 32)[0].astype(np.int64), _ints(g["case_a_q4_codes"]))
    xq, xd = oracle.quantize_act_q8(x, rotate=False)
    assert xd[0, 0] == np.float32(int(g["case_b_d_units"]) * u)
    assert np.array_equal(xq[0].astype(np.int64), _ints(g["case_b_q8_codes"]))
    xq, xd = oracle.quantize_act_q4(x, rotate=True)
    assert xd[0, 0] == np.float32(int(g["case_c_d_units"]) * u)
    assert np.array_equal(oracle.decode_act4(xq, 32)[0].astype(np.int64), _ints(g["case_c_q4_codes"]))
    w = np.zeros((1, 32), np.float32)
    w[0, 0] = np.float32(2.0 ** -140)
    wq, wd = oracle.quantize_weights_q4_0(w, rotate=False)
    assert np.array_equal(oracle.decode_w4(wq, 32)[0].astype(np.int64) + 8, _ints(g["case_d_codes"]))
    assert int(wd[0, 0]) == int(g["case_d_d16"], 16)


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("rotate", [True, False])
def test_degenerate_blocks_reconstruction_bound(bits, rotate):
    """Blocks of subnormal size (1/d overflows) keep the half-step bound of the
    ordinary blocks, |y - q d| <= d/2 up to the rounding of y / d, wherever
    y / d is inside the code range (a subnormal d can be far from amax/qmax,
    and then the clamp decides); an exact zero keeps code 0."""
    r = np.random.default_rng(11)
    x = (r.standard_normal((64, 64)) * 2.0 ** -131).astype(np.float32)
    x[:, 5] = 0.0                      # exact zeros (unrotated: they stay zero)
    x[0] = 0.0
    x[0, 7] = np.float32(2.0 ** -140)  # one nonzero element: the rest of the block is zero
    if bits == 4:
        xq, xd = oracle.quantize_act_q4(x, rotate)
        q = oracle.decode_act4(xq, 64).astype(np.float64)
        qmax = 7
    else:
        xq, xd = oracle.quantize_act_q8(x, rotate)
        q = xq.astype(np.float64)
        qmax = 127
    y = (oracle.fwht32(x.reshape(-1)).reshape(x.shape) if rotate else x).astype(np.float64)
    d = np.repeat(xd.astype(np.float64), 32, axis=1)
    assert np.all(np.isinf(np.float32(1.0) / xd[xd > 0].astype(np.float32)))   # degenerate indeed
    assert np.abs(q).max() <= qmax
    ratio = np.divide(y, d, out=np.zeros_like(y), where=d > 0)
    inside = np.abs(ratio) <= qmax + 0.5
    assert np.all((np.abs(y - q * d) <= 0.5 * d + 2.0 ** -23 * np.abs(y))[inside])
    assert np.all((q == np.sign(y) * qmax)[~inside])
    assert np.all(q[y == 0] == 0)
    # the element of largest magnitude gets the largest code magnitude
    yb, qb = y.reshape(64, 2, 32), q.reshape(64, 2, 32)
    pos = np.abs(yb).argmax(axis=2)
    top = np.take_along_axis(qb, pos[..., None], axis=2)[..., 0]
    assert np.array_equal(np.abs(top), np.abs(qb).max(axis=2))
    assert (np.abs(top) == qmax).mean() > 0.9


def test_overflowed_rotation_block():
    """A block whose rotation overflows to +-inf: finite elements get 0, the
    infinite ones +-qmax (the limit of y / d), d = inf."""
    x = np.zeros((1, 32), np.float32)
    x[0, 0], x[0, 1] = np.float32(3e38), np.float32(-3e38)
    y = oracle.fwht32(x.reshape(-1))
    assert np.isinf(y).any() and np.isfinite(y).any()
    xq, xd = oracle.quantize_act_q4(x, rotate=True)
    q = oracle.decode_act4(xq, 32)[0]
    assert np.isinf(xd[0, 0])
    assert np.array_equal(q, np.where(np.isinf(y), np.sign(y) * 7, 0).astype(q.dtype))
    xq, xd = oracle.quantize_act_q8(x, rotate=True)
    assert np.array_equal(xq[0], np.where(np.isinf(y), np.sign(y) * 127, 0).astype(xq.dtype))


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("rotate", [True, False])
def test_act_quant_properties(bits, rotate):
    x = wl.act_normal_outliers(16, 512, 0.01, 20.0, 0, wl.CFG_TEST, 1)
    if bits == 4:
        xq, xd = oracle.quantize_act_q4(x, rotate)
        q = oracle.decode_act4(xq, 512).astype(np.float64)
        qmax = 7
    else:
        xq, xd = oracle.quantize_act_q8(x, rotate)
        q = xq.astype(np.float64)
        qmax = 127
    y = oracle.fwht32(x.reshape(-1)).reshape(x.shape) if rotate else x
    yb = y.reshape(16, 16, 32).astype(np.float64)
    qb = q.reshape(16, 16, 32)
    d = xd.astype(np.float64)[..., None]
    assert np.abs(qb).max() <= qmax
    amax = np.abs(yb).max(axis=2)
    # d is amax / qmax to within one fp32 rounding
    assert np.all(np.abs(xd - amax / qmax) <= 2.0 ** -23 * amax / qmax)
    # the largest element gets the extreme code
    pos = np.abs(yb).argmax(axis=2)
    top = np.take_along_axis(qb, pos[..., None], axis=2)[..., 0]
    assert np.all(np.abs(top) == qmax)
    # reconstruction error at most half a step (plus fp32 rounding)
    assert np.all(np.abs(yb - qb * d) <= 0.5 * d * (1 + 1e-5) + 1e-30)


def test_bf16_widening_matches_bit_shift():
    r = np.random.default_rng(3)
    bits = r.integers(0, 0x7F80, size=4096, dtype=np.uint16)  # finite positives
    bits = bits | (r.integers(0, 2, size=4096, dtype=np.uint16) << 15)
    ref = (bits.astype(np.uint32) << 16).view(np.float32)
    out = oracle.bf16_to_f32(bits)
    assert np.array_equal(out.view(np.uint32), ref.view(np.uint32))


# --------------------------------------------------------------------------
# Q4_0 weights and decoding
# --------------------------------------------------------------------------
def test_q4_0_golden_blocks(golden):
    g = golden("ramp_block_q4_0.txt")
    w = (np.arange(32, dtype=np.float32) - 16)[None, :]
    wq, wd = oracle.quantize_weights_q4_0(w, rotate=False)
    codes = oracle.decode_w4(wq, 32)[0].astype(np.int64) + 8
    assert np.array_equal(codes, _ints(g["case_a_codes"]))
    assert int(wd[0, 0]) == int(g["case_a_d16"], 16)
    wq, wd = oracle.quantize_weights_q4_0(w, rotate=True)
    codes = oracle.decode_w4(wq, 32)[0].astype(np.int64) + 8
    assert np.array_equal(codes, _ints(g["case_b_codes"]))
    assert int(wd[0, 0]) == int(g["case_b_d16"], 16)
    w = np.zeros((1, 32), np.float32)
    w[0, 3], w[0, 7] = 1.0, -1.0
    wq, wd = oracle.quantize_weights_q4_0(w, rotate=False)
    codes = oracle.decode_w4(wq, 32)[0].astype(np.int64) + 8
    assert np.array_equal(codes, _ints(g["case_c_codes"]))
    assert int(wd[0, 0]) == int(g["case_c_d16"], 16)


def test_q4_0_nibble_layout_all_bytes():
    """Decode of every byte value: element j = low nibble - 8, element j+16 = high nibble - 8."""
    row = np.zeros((256, 16), np.uint8)
    row[:, 0] = np.arange(256)
    dec = oracle.decode_w4(row, 32)
    assert np.array_equal(dec[:, 0], (np.arange(256) & 15) - 8)
    assert np.array_equal(dec[:, 16], (np.arange(256) >> 4) - 8)
    a = oracle.decode_act4(row, 32)
    lo, hi = np.arange(256) & 15, np.arange(256) >> 4
    assert np.array_equal(a[:, 0], np.where(lo < 8, lo, lo - 16))
    assert np.array_equal(a[:, 16], np.where(hi < 8, hi, hi - 16))


def test_bit_flip_decode_exhaustive():
    """For every code q: flipping the top bit of q, read as a signed nibble, is q - 8."""
    for q in range(16):
        f = q ^ 8
        signed = f - 16 if f & 8 else f
        assert signed == q - 8
    row = np.zeros((16, 16), np.uint8)
    row[:, 3] = np.arange(16)
    w_dec = oracle.decode_w4(row, 32)[:, 3]
    a_dec = oracle.decode_act4((row ^ 0x08).astype(np.uint8), 32)[:, 3]
    assert np.array_equal(w_dec, a_dec)


def test_fp16_scale_matches_numpy():
    r = np.random.default_rng(4)
    x = np.concatenate([r.standard_normal(5000).astype(np.float32) * 1e-2,
                        np.float32([6.1e-5, 5.9e-8, 65504.0, 1e-9, 0.0, -0.0])])
    assert np.array_equal(oracle.f32_to_f16(x), x.astype(np.float16).view(np.uint16))
    bits = oracle.f32_to_f16(x)
    assert np.array_equal(oracle.f16_to_f32(bits), bits.view(np.float16).astype(np.float32))


@pytest.mark.parametrize("rotate", [True, False])
def test_q4_0_properties(rotate):
    w = wl.weights_normal(64, 256, 0.02, 0, wl.CFG_TEST, 2)
    wq, wd = oracle.quantize_weights_q4_0(w, rotate)
    y = oracle.fwht32(w.reshape(-1)).reshape(w.shape) if rotate else w
    yb = y.reshape(64, 8, 32).astype(np.float64)
    c = oracle.decode_w4(wq, 256).reshape(64, 8, 32).astype(np.float64) + 8
    assert c.min() >= 0 and c.max() <= 15
    pos = np.abs(yb).argmax(axis=2)
    mx = np.take_along_axis(yb, pos[..., None], axis=2)[..., 0]
    assert np.all(np.take_along_axis(c, pos[..., None], axis=2)[..., 0] == 0)
    d32 = mx / -8.0
    d16 = wd.view(np.float16).astype(np.float64)
    assert np.all(np.abs(d16 - d32) <= 2.0 ** -11 * np.abs(d32) + 1e-12)
    err = np.abs(yb - (c - 8) * d32[..., None])
    assert np.all(err <= np.abs(d32)[..., None] * (1 + 1e-5))
    inner = (c > 0) & (c < 15)
    assert np.all(err[inner] <= 0.5 * np.broadcast_to(np.abs(d32)[..., None], err.shape)[inner]
                  * (1 + 1e-5))


# --------------------------------------------------------------------------
# block sums and the epilogue
# --------------------------------------------------------------------------
def _tiny_operands(xbits=4, rotate=True, M=24, N=40, K=256):
    x = wl.act_normal_outliers(M, K, 0.01, 20.0, 0, wl.CFG_TEST, 5)
    w = wl.weights_normal(N, K, 0.02, 0, wl.CFG_TEST, 6)
    wq, wd = oracle.quantize_weights_q4_0(w, rotate)
    if xbits == 4:
        xq, xd = oracle.quantize_act_q4(x, rotate)
        xv = oracle.decode_act4(xq, K)
    else:
        xq, xd = oracle.quantize_act_q8(x, rotate)
        xv = xq
    return x, w, wq, wd, xq, xd, xv


@pytest.mark.parametrize("xbits", [4, 8])
def test_block_sums_vs_numpy_einsum(xbits):
    K = 256
    x, w, wq, wd, xq, xd, xv = _tiny_operands(xbits, K=K)
    M, N = xv.shape[0], wq.shape[0]
    y32, y64, S = oracle.gemm(wq, wd, xq, xd, K, want_block_sums=True)
    wv = oracle.decode_w4(wq, K).astype(np.int64).reshape(N, K // 32, 32)
    ref = np.einsum("mbj,nbj->mnb", xv.astype(np.int64).reshape(M, K // 32, 32), wv)
    assert np.array_equal(S, ref)
    bound = 2048 if xbits == 4 else 127 * 8 * 32
    assert np.abs(S).max() <= bound


def test_block_sum_extremes():
    # all activation codes -8 against all weight codes 0 (value -8): S = 32 * 64
    xq = np.full((1, 16), 0x88, np.uint8)
    wq = np.zeros((1, 16), np.uint8)
    wd = oracle.f32_to_f16(np.float32([1.0]))[None, :]
    xd = np.float32([[1.0]])
    y32, y64, S = oracle.gemm(wq, wd, xq, xd, 32, want_block_sums=True)
    assert S[0, 0, 0] == 2048 and y32[0, 0] == 2048.0
    # 8-bit: codes -127 against -8
    xq8 = np.full((1, 32), -127, np.int8)
    y32, y64, S = oracle.gemm(wq, wd, xq8, xd, 32, want_block_sums=True)
    assert S[0, 0, 0] == 127 * 8 * 32


def test_fp64_output_vs_numpy_and_fp32_error_bound():
    K = 256
    x, w, wq, wd, xq, xd, xv = _tiny_operands(4, K=K)
    y32, y64, S = oracle.gemm(wq, wd, xq, xd, K, want_block_sums=True)
    dw = wd.view(np.float16).astype(np.float64)
    terms = dw[None, :, :] * xd.astype(np.float64)[:, None, :] * S
    ref = terms.sum(axis=2)
    assert np.abs(y64 - ref).max() <= 1e-12 * np.abs(terms).sum(axis=2).max()
    # fp32 recursive fma summation: |y32 - exact| <= (nb + 1) u sum|terms|
    bound = (K // 32 + 1) * 2.0 ** -24 * np.abs(terms).sum(axis=2)
    assert np.all(np.abs(y32.astype(np.float64) - ref) <= bound + 1e-30)
    assert np.all(np.abs(y32 - y64) <= 1e-3 * np.maximum(np.abs(y64), 1e-6 * np.abs(y64).max()))


def test_fma_order_golden(golden):
    g = golden("fma_order.txt")
    assert g["y_exact"] == "5 * 2^-23"
    xq = np.zeros((1, 32), np.uint8)
    xq[0, 0] = np.uint8(-5 & 15)           # element 0 = -5
    xq[0, 16] = 5                          # element 32 = 5 (block 1, element 0)
    wq = np.full((1, 32), 0x88, np.uint8)  # every weight value 0 ...
    wq[0, 0] = 0x89                        # ... except element 0 = 1
    wq[0, 16] = 0x89                       # and element 32 = 1
    wd = oracle.f32_to_f16(np.float32([1.0, 1.0]))[None, :]
    xd = np.float32([[1.0, 1.0 + 2.0 ** -23]])
    y32, _, S = oracle.gemm(wq, wd, xq, xd, 64, want_block_sums=True)
    assert list(S[0, 0]) == [-5, 5]
    assert y32[0, 0] == np.float32(5 * 2.0 ** -23)


def test_sampled_gemm_matches_full():
    K = 256
    x, w, wq, wd, xq, xd, xv = _tiny_operands(8, K=K)
    y32, y64, S = oracle.gemm(wq, wd, xq, xd, K, want_block_sums=True)
    r = np.random.default_rng(7)
    mi = r.integers(0, xq.shape[0], 50)
    ni = r.integers(0, wq.shape[0], 50)
    s32, s64, sS = oracle.gemm_sampled(wq, wd, xq, xd, K, mi, ni, want_block_sums=True)
    assert np.array_equal(s32, y32[mi, ni]) and np.array_equal(sS, S[mi, ni])


@pytest.mark.parametrize("rotate", [True, False])
def test_route_approximates_exact_product(rotate):
    """Both sides rotated by the same H leave the product unchanged: the 8-bit
    route reproduces x.W^T up to rounding, with or without the rotation; a
    transform applied to one side only would not."""
    K = 512
    x, w, wq, wd, xq, xd, xv = _tiny_operands(8, rotate=rotate, M=16, N=32, K=K)
    y32, y64, _ = oracle.gemm(wq, wd, xq, xd, K)
    ref = x.astype(np.float64) @ w.astype(np.float64).T
    rel = np.linalg.norm(y64 - ref) / np.linalg.norm(ref)
    assert rel < 0.12
    # one side rotated, the other not: the product is destroyed
    wq_u, wd_u = oracle.quantize_weights_q4_0(w, rotate=not rotate)
    _, y_bad, _ = oracle.gemm(wq_u, wd_u, xq, xd, K)
    assert np.linalg.norm(y_bad - ref) / np.linalg.norm(ref) > 0.5


def test_rotation_lowers_4bit_error_on_outlier_channels():
    """The method's claim ("The rotation"): rotating spreads a block's outliers,
    so the 4-bit reconstruction error drops.  Reported as a property."""
    x = wl.act_normal_outliers(64, 1024, 0.01, 20.0, 0, wl.CFG_TEST, 8)
    errs = {}
    for rotate in (True, False):
        xq, xd = oracle.quantize_act_q4(x, rotate)
        q = oracle.decode_act4(xq, 1024).astype(np.float64).reshape(64, 32, 32)
        y = (oracle.fwht32(x.reshape(-1)).reshape(x.shape) if rotate else x)
        rec = (q * xd.astype(np.float64)[..., None]).reshape(64, 1024)
        errs[rotate] = np.linalg.norm(rec - y) / np.linalg.norm(y)
    assert errs[True] < errs[False]


def test_experts_sampled_vs_numpy():
    r = np.random.default_rng(9)
    E, N, K = 5, 24, 64
    counts = np.array([3, 0, 7, 1, 5])
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    R = int(off[-1])
    T = 9
    row_idx = r.integers(0, T, R).astype(np.int32)
    x = r.standard_normal((T, K)).astype(np.float32)
    w = (0.02 * r.standard_normal((E * N, K))).astype(np.float32)
    wq, wd = oracle.quantize_weights_q4_0(w)
    xq, xd = oracle.quantize_act_q4(x)
    wq, wd = wq.reshape(E, N, K // 2), wd.reshape(E, N, K // 32)
    ri = np.repeat(np.arange(R), N)
    ni = np.tile(np.arange(N), R)
    y32, y64, S = oracle.gemm_experts_sampled(wq, wd, xq, xd, row_idx, off, N, K, ri, ni, True)
    xv = oracle.decode_act4(xq, K).astype(np.int64)
    for i in range(ri.size):
        rr, n = ri[i], ni[i]
        e = int(np.searchsorted(off, rr, side="right") - 1)
        wv = oracle.decode_w4(wq[e], K).astype(np.int64)[n]
        xrow = xv[row_idx[rr]]
        sb = (xrow * wv).reshape(K // 32, 32).sum(axis=1)
        assert np.array_equal(S[i], sb)
        ref = (wd[e, n].view(np.float16).astype(np.float64) * xd[row_idx[rr]] * sb).sum()
        assert abs(y64[i] - ref) <= 1e-12 * max(1.0, abs(ref))


# --------------------------------------------------------------------------
# larger rotations, 64 and 128 points, scales still per 32-block ("Qwen3.8-27B
# at 45.7 tok/s ...", section "What's next")
# --------------------------------------------------------------------------
@pytest.mark.parametrize("n", [64, 128])
def test_rot_scale_is_nearest_fp32(n):
    getcontext().prec = 60
    exact = Decimal(1) / Decimal(n).sqrt()
    c = np.float32(oracle.rot_scale(n))
    for nb in (np.nextafter(c, np.float32(1)), np.nextafter(c, np.float32(0))):
        assert abs(Decimal(float(c)) - exact) <= abs(Decimal(float(nb)) - exact)
    if n == 64:
        assert c == np.float32(0.125)
    assert np.float32(oracle.rot_scale(32)) == np.float32(oracle.h32_scale())


def _materialize_hn(n):
    eye = np.eye(n, dtype=np.float32)
    return oracle.fwht_n(eye.reshape(-1), n).reshape(n, n).T.astype(np.float64)


@pytest.mark.parametrize("n", [64, 128])
def test_hn_entries_are_sylvester_signs_times_c(n):
    H = _materialize_hn(n)
    c = np.float64(np.float32(oracle.rot_scale(n)))
    ref = scipy.linalg.hadamard(n).astype(np.float64) * c
    assert np.array_equal(H, ref)
    for i in (0, 3, n - 1):
        for k in (0, 5, n // 2, n - 1):
            assert H[i, k] == (-1) ** _popcount(i & k) * c
    assert np.abs(H @ H.T - np.eye(n)).max() <= 1e-6


@pytest.mark.parametrize("n", [64, 128])
def test_fwht_n_vs_dense_matrix_and_invariance(n):
    r = np.random.default_rng(11)
    x = r.standard_normal((50, n))
    ref = x @ (scipy.linalg.hadamard(n) / np.sqrt(float(n))).T
    y64 = oracle.fwht_n_f64(x.reshape(-1), n).reshape(50, n)
    assert np.abs(y64 - ref).max() <= 1e-13 * np.abs(x).sum(axis=1).max()
    for K in (n, 4 * n, 5120):
        a, b = r.standard_normal(K), r.standard_normal(K)
        ha, hb = oracle.fwht_n_f64(a, n), oracle.fwht_n_f64(b, n)
        assert abs(float(a @ b) - float(ha @ hb)) <= 1e-9 * float(np.abs(a * b).sum())


@pytest.mark.parametrize("n", [64, 128])
def test_one_hot_closed_form_larger_rotation(n):
    """A unit vector in an n-block spreads to +-C_n at every position, so each of
    its n/32 scale blocks gets d = C_n / 7 and codes +-7 with Sylvester signs;
    the Q4_0 weight rule takes each 32-block's first element as its signed max
    s C_n, giving d = -s C_n / 8 and codes 0 where the sign is s, 15 elsewhere."""
    c = np.float32(oracle.rot_scale(n))
    K = 2 * n
    for k in (0, 1, n // 2 + 3, n - 1):
        x = np.zeros((1, K), np.float32)
        x[0, n + k] = 1.0      # second n-block; the first stays zero
        sign = np.array([(-1) ** _popcount(i & k) for i in range(n)], np.float32)
        xq, xd = oracle.quantize_act_q4(x, n)
        codes = oracle.decode_act4(xq, K)[0]
        assert np.all(codes[:n] == 0) and np.all(xd[0, : n // 32] == 0)
        assert np.array_equal(codes[n:], (7 * sign).astype(np.int8))
        assert np.all(xd[0, n // 32:] == np.float32(c / np.float32(7)))
        q8, _ = oracle.quantize_act_q8(x, n)
        assert np.array_equal(q8[0, n:], (127 * sign).astype(np.int8))
        wq, wd = oracle.quantize_weights_q4_0(x, n)
        wc = oracle.decode_w4(wq, K)[0] + 8
        dw = oracle.f16_to_f32(wd[0])
        for j in range(n // 32):
            s0 = sign[32 * j]          # the block's signed max is its first element
            blk = sign[32 * j: 32 * j + 32]
            assert np.array_equal(wc[n + 32 * j: n + 32 * j + 32], np.where(blk == s0, 0, 15))
            d = oracle.f16_to_f32(oracle.f32_to_f16(np.array([-s0 * c / 8], np.float32)))[0]
            assert dw[n // 32 + j] == d


@pytest.mark.parametrize("n", [64, 128])
def test_constant_block_larger_rotation(n):
    """A constant n-block rotates to (n c C_n, 0, ..., 0): the first 32-block
    gets code 7 at position 0, the other blocks of the n-block are all zero
    with d = 0."""
    for val in (0.75, -3.0):
        x = np.full((1, n), val, np.float32)
        y = oracle.fwht_n(x.reshape(-1), n)
        assert y[0] == np.float32(np.float32(n * val) * np.float32(oracle.rot_scale(n)))
        assert np.all(y[1:] == 0)
        xq, xd = oracle.quantize_act_q4(x, n)
        codes = oracle.decode_act4(xq, n)[0]
        expect = np.zeros(n, np.int8)
        expect[0] = 7 if val > 0 else -7
        assert np.array_equal(codes, expect)
        assert np.all(xd[0, 1:] == 0) and xd[0, 0] > 0


@pytest.mark.parametrize("n", [64, 128])
def test_larger_rotation_route_approximates_exact_product(n):
    r = np.random.default_rng(12)
    M, N, K = 8, 16, 512
    x = wl.act_normal_outliers(M, K, 0.01, 20.0, 0, wl.CFG_TEST, 300)
    w = (0.02 * r.standard_normal((N, K))).astype(np.float32)
    wq, wd = oracle.quantize_weights_q4_0(w, n)
    xq, xd = oracle.quantize_act_q4(x, n)
    _, y64, _ = oracle.gemm(wq, wd, xq, xd, K)
    ref = x.astype(np.float64) @ w.astype(np.float64).T
    assert np.linalg.norm(y64 - ref) / np.linalg.norm(ref) < 0.12
    # weights rotated with 32 points, activations with n: the product is destroyed
    wq32, wd32 = oracle.quantize_weights_q4_0(w, 32)
    _, ybad, _ = oracle.gemm(wq32, wd32, xq, xd, K)
    assert np.linalg.norm(ybad - ref) / np.linalg.norm(ref) > 0.5


@pytest.mark.parametrize("n", [64, 128])
def test_larger_rotation_stage_order(n):
    """Hand-derived: x[0] = 2^24, x[1] = 1, x[n/2] = -2^24.  With strides in
    ascending order the stride-1 stage rounds 2^24 + 1 to 2^24 first (ties to
    even); the last stage then gives y[0] = 0, y[1] = -1, y[n/2] = 2^25 and
    y[n/2 + 1] = fl(2^25 - 1) = 2^25, each times C_n.  Descending strides would
    give y[0] = C_n instead."""
    c = np.float32(oracle.rot_scale(n))
    x = np.zeros(n, np.float32)
    x[0], x[1], x[n // 2] = 2.0 ** 24, 1.0, -(2.0 ** 24)
    y = oracle.fwht_n(x, n)
    assert y[0] == 0 and y[1] == -c
    assert y[n // 2] == np.float32(2.0 ** 25) * c and y[n // 2 + 1] == np.float32(2.0 ** 25) * c


def test_q4_0_block_layout_pins():
    """A Q4_0 block built by hand from its layout (fp16 d = 0.5 as bytes 00 38,
    then byte j holding element j in its low nibble and element j + 16 in its
    high one): the planes decode to the values the layout gives, and the two
    conversions are inverse to each other."""
    blk = np.zeros((1, 1, 18), np.uint8)
    blk[0, 0, 0], blk[0, 0, 1] = 0x00, 0x38          # fp16 0.5, little endian
    for j in range(16):
        blk[0, 0, 2 + j] = j | ((15 - j) << 4)
    wq, wd = oracle.q4_0_planes_from_blocks(blk, 1, 32)
    assert oracle.f16_to_f32(wd)[0, 0] == np.float32(0.5)
    vals = oracle.decode_w4(wq, 32)[0]
    assert list(vals[:16]) == [j - 8 for j in range(16)]
    assert list(vals[16:]) == [7 - j for j in range(16)]
    rng = np.random.default_rng(5)
    blocks = rng.integers(0, 256, (7, 5, 18), dtype=np.uint8)
    wq, wd = oracle.q4_0_planes_from_blocks(blocks, 7, 160)
    assert np.array_equal(oracle.q4_0_blocks_from_planes(wq, wd), blocks)
