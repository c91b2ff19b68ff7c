"""GPU parity of the routing and weighted combine around the expert GEMMs
against the CPU oracle ("Where the engine is going: HRX and the NPU",
section "4-bit activations reach the MoE experts").

Expert ids, group offsets and row maps must equal the oracle's exactly.  The
weights use each side's fp32 exp (CUDA's expf, within 2 ulp, and the C
library's), so they are compared within a bound derived from that: the exps
differ by at most 3 ulp, the k-term sum in the same order by at most k - 1
more ulps of re-rounding, the divide by one: 2e-6 relative for k <= 8
(12 ulp), 5e-6 up to k = 32.  The combine is fed the oracle's weights and
must equal the oracle's fp32 fma sequence bit for bit."""
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


def _logits(T, E, seed, ties=True):
    r = np.random.default_rng(seed)
    l = r.standard_normal((T, E)).astype(np.float32)
    if ties and E > 1:
        for t in range(0, T, 3):
            a, b = r.integers(0, E, 2)
            l[t, b] = l[t, a]
        l[T // 2, :] = np.float32(0.75)
    return l


def _w_tol(k):
    return 2e-6 if k <= 8 else 5e-6


def _check_route(h32, l, k, ldl_pad=0):
    import torch
    T, E = l.shape
    if ldl_pad:
        lp = np.zeros((T, E + ldl_pad), np.float32)
        lp[:, :E] = l
        lt = torch_of(lp)[:, :E]
    else:
        lt = torch_of(l)
    ids, w, off, ridx, row_of = h32.h32_moe_route(lt, k)
    torch.cuda.synchronize()
    assert h32.h32_device_status() == 0
    rid, rw, roff, rridx, rrow = oracle.moe_route(l, k)
    assert np.array_equal(np_of(ids), rid)
    assert np.array_equal(np_of(off), roff)
    assert np.array_equal(np_of(ridx), rridx)
    assert np.array_equal(np_of(row_of), rrow)
    gw = np_of(w).astype(np.float64)
    # relative bound, with the smallest normal fp32 as the floor where a weight
    # underflows (subnormal or zero on both sides)
    assert np.all(np.abs(gw - rw) <= _w_tol(k) * rw + 2.0 ** -126)
    return rid, rw, roff, rridx, rrow


def test_route_moe_config(h32):
    """1024 tokens, 128 experts, top 8 from U(0,1) logits."""
    cfg = wl.MOE
    _, _, off, ridx, _ = _check_route(h32, wl.moe_logits(cfg), cfg.top_k)
    ridx_ref, off_ref, _ = wl.moe_routing(cfg)
    assert np.array_equal(off, off_ref) and np.array_equal(ridx, ridx_ref)


@pytest.mark.parametrize("T,E,k", [(1, 1, 1), (7, 5, 5), (300, 37, 8), (64, 128, 32),
                                   (33, 1000, 8), (257, 1024, 3), (9, 64, 1)])
def test_route_ragged_and_ties(h32, T, E, k):
    _check_route(h32, _logits(T, E, T * 7 + E), k)


def test_route_wide_logits_and_many_tokens(h32):
    """Logits spread so far apart that weights underflow (exp of differences
    below -87 is subnormal or zero), and a token count whose grouping walks
    many chunks of tokens."""
    r = np.random.default_rng(21)
    wide = (r.standard_normal((300, 40)) * 60.0).astype(np.float32)
    _, rw, _, _, _ = _check_route(h32, wide, 8)
    assert np.any(rw == 0.0) and np.any((rw > 0) & (rw < 2.0 ** -126))
    _check_route(h32, _logits(70000, 16, 22), 2)


def test_route_row_pitch_and_equal_rows(h32):
    l = _logits(40, 48, 5)
    l[3, :] = np.float32(-2.5)     # every logit equal: the k lowest ids, weights fl(1/k)
    rid, rw, _, _, _ = _check_route(h32, l, 6, ldl_pad=16)
    assert rid[3].tolist() == list(range(6))


def test_route_non_finite_logits(h32):
    """Masked experts (-inf), +inf and NaN logits, placed so that a NaN or a
    -inf sits ahead of finite logits in every lane position: ids, offsets and
    row maps exact, weights as the oracle's limits of the softmax."""
    r = np.random.default_rng(23)
    T, E = 96, 70
    l = r.standard_normal((T, E)).astype(np.float32)
    for t in range(T):
        m = r.random(E)
        l[t, m < 0.3] = -np.inf
        l[t, (m >= 0.3) & (m < 0.4)] = np.nan
    l[0, :] = -np.inf                       # every expert masked: equal weights
    l[1, :] = np.nan
    l[2, :5] = np.inf                       # several +inf: they share the weight
    l[3, 0] = np.nan                        # a NaN in the first lane position
    l[4, ::2] = -np.inf
    for k in (1, 4, 8, 32):
        rid, rw, _, _, _ = _check_route(h32, l, k)
    assert np.all(rw[0] == np.float32(1) / np.float32(32))


def test_route_empty_and_bad_args(h32):
    import torch
    l = torch.zeros((0, 16), dtype=torch.float32, device="cuda")
    off = torch.full((17,), 7, dtype=torch.int32, device="cuda")
    h32.h32_moe_route(l, 4, expert_off=off)
    torch.cuda.synchronize()
    assert np.all(np_of(off) == 0)
    lt = torch.zeros((4, 16), dtype=torch.float32, device="cuda")
    with pytest.raises(h32.H32Error):
        h32.h32_moe_route(lt, 17)      # k > E
    with pytest.raises(h32.H32Error):
        h32.h32_moe_route(torch.zeros((4, 1025), dtype=torch.float32, device="cuda"), 2)
    with pytest.raises(h32.H32Error):
        h32.h32_moe_route(torch.zeros((4, 64), dtype=torch.float32, device="cuda"), 33)


def _check_combine(h32, T, k, H, seed, pad=0):
    import torch
    r = np.random.default_rng(seed)
    R = T * k
    y = r.standard_normal((R, H)).astype(np.float32)
    _, rw, _, _, rrow = oracle.moe_route(_logits(T, max(k, 12), seed), k)
    ref = oracle.moe_combine(y, rrow, rw)
    if pad:
        yp = np.zeros((R, H + pad), np.float32)
        yp[:, :H] = y
        yt = torch_of(yp)[:, :H]
        out = torch.zeros((T, H + pad), dtype=torch.float32, device="cuda")[:, :H]
    else:
        yt, out = torch_of(y), None
    got = h32.h32_moe_combine(yt, torch_of(rrow), torch_of(rw), out=out)
    torch.cuda.synchronize()
    assert h32.h32_device_status() == 0
    assert np.array_equal(np_of(got).view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("T,k,H,pad", [(1, 1, 4, 0), (5, 3, 12, 0), (37, 8, 2052, 8),
                                       (16, 32, 640, 0), (3, 8, 8192, 4)])
def test_combine_matches_oracle(h32, T, k, H, pad):
    _check_combine(h32, T, k, H, T + k + H, pad)


def test_combine_moe_config(h32):
    """1024 tokens, top 8, hidden 2048: the size the MoE micro-batch combines."""
    _check_combine(h32, 1024, 8, 2048, 17)


def test_combine_row_guard(h32):
    import torch
    T, k, H = 6, 4, 16
    r = np.random.default_rng(2)
    y = r.standard_normal((T * k, H)).astype(np.float32)
    row_of = r.permutation(T * k).reshape(T, k).astype(np.int32)
    w = r.random((T, k)).astype(np.float32)
    bad = row_of.copy()
    bad[2, 1] = T * k                 # one row past the end
    got = h32.h32_moe_combine(torch_of(y), torch_of(bad), torch_of(w))
    assert h32.h32_device_status() == h32.H32_ERR_DEVICE_GUARD
    w0 = w.copy()
    w0[2, 1] = 0.0                    # the guarded term adds nothing
    ref = oracle.moe_combine(y, row_of, w0)
    assert np.array_equal(np_of(got), ref)
    assert h32.h32_device_status() == 0


def test_moe_layer_sampled(h32):
    """The expert layer on the GPU: route, gather-quantize, expert gate/up GEMM,
    expert down GEMM on its own input (the SwiGLU between them is outside the
    path), combine; sampled tokens against the oracle's pipeline (the combine
    takes the oracle's weights, so the check is exact)."""
    import torch
    cfg = wl.MOE
    logits = wl.moe_logits(cfg)
    x_gu, x_dn = wl.moe_inputs(cfg)
    w_gu, w_dn = wl.moe_weights(cfg)
    ids, w, off, ridx, row_of = h32.h32_moe_route(torch_of(logits), cfg.top_k)
    rid, rw, roff, rridx, rrow = oracle.moe_route(logits, cfg.top_k)
    assert np.array_equal(np_of(off), roff) and np.array_equal(np_of(row_of), rrow)
    R = int(roff[-1])

    def prep(wt):
        E, N, K = wt.shape
        wq, wd = oracle.quantize_weights_q4_0(wt.reshape(E * N, K))
        wp, wsc = h32.h32_prepack_weights_q4_0_tc(torch_of(wq), torch_of(wd.view(np.int16)))
        return wq.reshape(E, N, K // 2), wd.reshape(E, N, K // 32), wp, wsc

    wq_g, wd_g, wp_g, ws_g = prep(w_gu)
    xt = torch.from_numpy(x_gu.view(np.int16)).view(torch.bfloat16).cuda()
    xw, xdt = h32.h32_quantize_act_q4_tc_gather(xt, ridx)
    y_gu = h32.q4_0_x_q4_gemm_tc_experts(wp_g, ws_g, xw, xdt, off, w_gu.shape[1], R=R)
    wq_d, wd_d, wp_d, ws_d = prep(w_dn)
    xn = torch.from_numpy(x_dn.view(np.int16)).view(torch.bfloat16).cuda()
    xw2, xdt2 = h32.h32_quantize_act_q4_tc(xn)
    y_dn = h32.q4_0_x_q4_gemm_tc_experts(wp_d, ws_d, xw2, xdt2, off, w_dn.shape[1], R=R)
    out = h32.h32_moe_combine(y_dn, row_of, torch_of(rw))
    torch.cuda.synchronize()
    assert h32.h32_device_status() == 0
    # oracle: gate/up outputs of a few rows, and the full combine of a few tokens
    xq, xd = oracle.quantize_act_q4(x_gu)
    r = np.random.default_rng(6)
    rows = r.integers(0, R, 200)
    cols = r.integers(0, w_gu.shape[1], 200)
    g32, _, _ = oracle.gemm_experts_sampled(wq_g, wd_g, xq, xd, rridx, roff, w_gu.shape[1],
                                            cfg.hidden, rows, cols)
    assert np.array_equal(np_of(y_gu)[rows, cols].view(np.uint32), g32.view(np.uint32))
    xq2, xd2 = oracle.quantize_act_q4(x_dn)
    H = w_dn.shape[1]
    toks = np.array([0, 1, 511, 1023])
    need = np.unique(rrow[toks].reshape(-1))
    ri = np.repeat(need, H)
    ni = np.tile(np.arange(H), need.size)
    d32, _, _ = oracle.gemm_experts_sampled(wq_d, wd_d, xq2, xd2, None, roff, H, cfg.ffn, ri, ni)
    y_rows = np.zeros((R, H), np.float32)
    y_rows[need] = d32.reshape(need.size, H)
    ref = oracle.moe_combine(y_rows, rrow[toks], rw[toks])
    assert np.array_equal(np_of(out)[toks].view(np.uint32), ref.view(np.uint32))
