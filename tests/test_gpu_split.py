"""GPU parity of the K split of the last wave (the tc GEMMs with a workspace).

Where the tiles of a product do not fill the last wave of the persistent grid,
its tiles are cut into pieces along the tokens, and each piece runs in two
parts along K on two SMs; the second part continues the first part's
accumulators, so every output still takes its 32-blocks in order and the
result must equal the oracle's same-order fp32 result bit for bit ("509 tokens
a second of prompt: the Hadamard route ships", sections "Why prompts are a
matrix-unit problem" and "The rotation")."""
import numpy as np
import pytest

import oracle
from hadamard_rotated_bit_gb300 import workloads as wl
from tests._gpu import np_of, torch_bf16, torch_of

pytestmark = pytest.mark.gpu

# 160 tiles of 128 weight rows x 64 tokens on a 152-SM device: a full wave and
# 8 tiles over, cut into 16-token pieces whose K (two stages) is split in two
SMALL = (64, 20480, 256)


@pytest.fixture(scope="module")
def h32():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import hadamard_rotated_bit_gb300 as m
    from hadamard_rotated_bit_gb300 import _build
    _build.build()
    return m


def _sms():
    import torch
    return torch.cuda.get_device_properties(0).multi_processor_count


def _operands(h32, M, N, K, seed, bits=4):
    x = wl.f32_to_bf16_bits(wl.act_normal_outliers(M, K, 0.01, 20.0, 0, wl.CFG_TEST, seed))
    w = wl.weights_normal(N, K, 0.02, 0, wl.CFG_TEST, seed + 1)
    wq, wd = oracle.quantize_weights_q4_0(w)
    wp, wsc = h32.h32_prepack_weights_q4_0_tc(torch_of(wq), torch_of(wd.view(np.int16)))
    if bits == 4:
        xq, xd = oracle.quantize_act_q4(x)
        xw, xdt = h32.h32_quantize_act_q4_tc(torch_bf16(x))
    else:
        xq, xd = oracle.quantize_act_q8(x)
        xw, xdt = h32.h32_quantize_act_q8_tc(torch_bf16(x))
    return (wq, wd, xq, xd), (wp, wsc, xw, xdt)


def _gemm(h32, bits):
    return h32.q4_0_x_q4_gemm_tc if bits == 4 else h32.q4_0_x_q8_gemm_tc


def _oracle_gemm(bits, wq, wd, xq, xd, K):
    return oracle.gemm(wq, wd, xq, xd, K)[0]   # the route follows from the codes' layout


def test_split_schedules_of_the_chain(h32):
    """On this device the pp512 attention and FFN-down projections and the
    small case take the split (the query and the schedule agree), and a
    workspace-free call does not."""
    sms = _sms()
    for (M, N, K) in (SMALL, (512, 5120, 5120), (512, 5120, 17408)):
        sch = h32.h32_gemm_tc_schedule(M, N, K, sms, True)
        assert h32.h32_gemm_tc_workspace_bytes(M, N, K) == sch["ws_bytes"]
        if sms == 152:
            assert sch["split_p"] > 0, (M, N, K)
        assert h32.h32_gemm_tc_schedule(M, N, K, sms, False)["split_p"] == 0


@pytest.mark.parametrize("bits", [4, 8])
def test_split_all_outputs_bit_exact(h32, bits):
    """Every output of a product whose last wave is split, against the oracle;
    the same product without a workspace (no split) is bit-identical."""
    import torch
    M, N, K = SMALL
    if h32.h32_gemm_tc_workspace_bytes(M, N, K) == 0:
        pytest.skip("this device's schedule does not split the case")
    (wq, wd, xq, xd), (wp, wsc, xw, xdt) = _operands(h32, M, N, K, 900 + bits, bits)
    y = _gemm(h32, bits)(wp, wsc, xw, xdt, M=M)
    y0 = _gemm(h32, bits)(wp, wsc, xw, xdt, M=M, workspace=False)
    torch.cuda.synchronize()
    assert h32.h32_device_status() == 0
    r32 = _oracle_gemm(bits, wq, wd, xq, xd, K)
    assert np.array_equal(np_of(y).view(np.uint32), r32.view(np.uint32))
    assert np.array_equal(np_of(y0).view(np.uint32), r32.view(np.uint32))


@pytest.mark.parametrize("proj,M", [("attn", 512), ("ffn_down", 512), ("ffn_gate_up", 512),
                                    ("attn", 1024), ("ffn_down", 1024)])
def test_split_pieces_pp512_sampled(h32, proj, M):
    """The chain's projections as the chain runs them (split last wave), at
    512 tokens and at the long prompts' 1024-token micro-batch: outputs sampled
    inside the cut tiles (split along K where the schedule splits) and
    elsewhere, against the oracle, bit for bit."""
    import torch
    p = {q.name: q for q in (wl.ATTN, wl.FFN_GATE_UP, wl.FFN_DOWN)}[proj]
    cid = wl.CFG_ATTN if p is wl.ATTN else wl.CFG_FFN
    x = p.activations(M, 1, cid)
    w = p.weights(0, cid)
    wq, wd = oracle.quantize_weights_q4_0(w)
    xq, xd = oracle.quantize_act_q4(x)
    wp, wsc = h32.h32_prepack_weights_q4_0_tc(torch_of(wq), torch_of(wd.view(np.int16)))
    xw, xdt = h32.h32_quantize_act_q4_tc(torch_bf16(x))
    sch = h32.h32_gemm_tc_schedule(M, p.N, p.K, _sms(), True)
    y = np_of(h32.q4_0_x_q4_gemm_tc(wp, wsc, xw, xdt, M=M))
    torch.cuda.synchronize()
    assert h32.h32_device_status() == 0
    r = np.random.default_rng(11)
    # the cut tiles: tile t covers weight rows 128 (t // chunks) and tokens
    # bn (t % chunks) onward
    chunks = (M + sch["bn"] - 1) // sch["bn"]
    cut = np.arange(sch["tail_first"], (sch["total"] - sch["tail_first"]) // max(sch["tail_k"], 1)
                    + sch["tail_first"])
    n_in = 128 * (cut // chunks)
    m_in = sch["bn"] * (cut % chunks)
    pick = r.integers(0, len(cut), 2000) if len(cut) else np.zeros(0, dtype=np.int64)
    mi = np.concatenate([np.minimum(m_in[pick] + r.integers(0, sch["bn"], len(pick)), M - 1),
                         r.integers(0, M, 1000), [M - 1]])
    ni = np.concatenate([np.minimum(n_in[pick] + r.integers(0, 128, len(pick)), p.N - 1),
                         r.integers(0, p.N, 1000), [p.N - 1]])
    r32, _, _ = oracle.gemm_sampled(wq, wd, xq, xd, p.K, mi, ni)
    assert np.array_equal(y[mi, ni].view(np.uint32), r32.view(np.uint32))


def test_split_workspace_reused_across_shapes(h32):
    """One caller-owned workspace (zeroed once) through products of different
    schedules, both routes, back to back on one stream with no host sync:
    every result bit-exact (flags of an earlier call never pass for a later
    one's)."""
    import torch
    cases = [(64, 20480, 256, 4), (48, 20480, 384, 4), (64, 20480, 256, 8), (64, 20480, 256, 4)]
    need = max(h32.h32_gemm_tc_workspace_bytes(M, N, K) for M, N, K, _ in cases)
    if need == 0:
        pytest.skip("this device's schedules do not split the cases")
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    ops, outs = [], []
    for i, (M, N, K, bits) in enumerate(cases):
        o = _operands(h32, M, N, K, 950 + i, bits)
        ops.append(o)
    torch.cuda.synchronize()
    for (M, N, K, bits), (_, (wp, wsc, xw, xdt)) in zip(cases, ops):
        outs.append(_gemm(h32, bits)(wp, wsc, xw, xdt, M=M, workspace=ws))
    torch.cuda.synchronize()
    assert h32.h32_device_status() == 0
    for (M, N, K, bits), ((wq, wd, xq, xd), _), y in zip(cases, ops, outs):
        r32 = _oracle_gemm(bits, wq, wd, xq, xd, K)
        assert np.array_equal(np_of(y).view(np.uint32), r32.view(np.uint32)), (M, N, K, bits)


def test_split_in_a_cuda_graph_replayed(h32):
    """Quantize + split GEMM captured once and replayed on new inputs: the
    kernel advances the workspace's generation itself, so every replay waits
    for its own first parts; bit-exact each time."""
    import torch
    M, N, K = SMALL
    if h32.h32_gemm_tc_workspace_bytes(M, N, K) == 0:
        pytest.skip("this device's schedule does not split the case")
    w = wl.weights_normal(N, K, 0.02, 0, wl.CFG_TEST, 970)
    rwq, rwd = oracle.quantize_weights_q4_0(w)
    wp, wsc = h32.h32_prepack_weights_q4_0_tc(torch_of(rwq), torch_of(rwd.view(np.int16)))
    x = torch.empty((M, K), dtype=torch.float32, device="cuda")
    xw = torch.empty((M, K), dtype=torch.uint8, device="cuda")
    xdt = torch.zeros((K // 32, M), dtype=torch.float32, device="cuda")
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    ws = torch.zeros(h32.h32_gemm_tc_workspace_bytes(M, N, K), dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()

    def step():
        h32.h32_quantize_act_q4_tc(x, xw=xw, xdt=xdt, stream=s)
        h32.q4_0_x_q4_gemm_tc(wp, wsc, xw, xdt, M=M, y=y, stream=s, workspace=ws)

    x.copy_(torch_of(wl.act_normal_outliers(M, K, 0.01, 20.0, 0, wl.CFG_TEST, 971)))
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        step()
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step()
    for tid in (972, 973, 974):
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


def test_split_workspace_checks(h32):
    """A workspace below the query's size is refused, a misaligned one too;
    nothing is launched."""
    import torch
    M, N, K = SMALL
    need = h32.h32_gemm_tc_workspace_bytes(M, N, K)
    if need == 0:
        pytest.skip("this device's schedule does not split the case")
    (_, _, _, _), (wp, wsc, xw, xdt) = _operands(h32, M, N, K, 980)
    small = torch.zeros(need - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(h32.H32Error) as e:
        h32.q4_0_x_q4_gemm_tc(wp, wsc, xw, xdt, M=M, workspace=small)
    assert e.value.status == h32.H32_ERR_INVALID_ARG
    big = torch.zeros(need + 512, dtype=torch.uint8, device="cuda")
    with pytest.raises(h32.H32Error) as e:
        h32.q4_0_x_q4_gemm_tc(wp, wsc, xw, xdt, M=M, workspace=big[16:])
    assert e.value.status == h32.H32_ERR_ALIGNMENT
    torch.cuda.synchronize()
    assert h32.h32_device_status() == 0


@pytest.mark.parametrize("rot", [True, False])
def test_split_fused_producer_bit_exact(h32, rot):
    """The fused producer (output also quantized for the next projection) with
    the K split: y, the next projection's codes and scales all equal the
    oracle's quantizer on the oracle's output, with and without y."""
    import torch
    from tests.test_gpu_tc import e4m3_value
    M, N, K = SMALL
    if h32.h32_gemm_tc_workspace_bytes(M, N, K) == 0:
        pytest.skip("this device's schedule does not split the case")
    (wq, wd, xq, xd), (wp, wsc, xw, xdt) = _operands(h32, M, N, K, 985)
    y, xn, xnd = h32.q4_0_x_q4_gemm_tc_quant_next(wp, wsc, xw, xdt, M=M, rotate_next=rot)
    torch.cuda.synchronize()
    assert h32.h32_device_status() == 0
    r32, _, _ = oracle.gemm(wq, wd, xq, xd, K)
    assert np.array_equal(np_of(y).view(np.uint32), r32.view(np.uint32))
    nq, nd = oracle.quantize_act_q4(r32, rot)
    assert np.array_equal(e4m3_value(np_of(xn)), oracle.decode_act4(nq, N).astype(np.float64))
    assert np.array_equal(np_of(xnd)[:, :M].T.view(np.uint32), nd.view(np.uint32))
    y2, xn2, xnd2 = h32.q4_0_x_q4_gemm_tc_quant_next(wp, wsc, xw, xdt, M=M, want_y=False,
                                                      rotate_next=rot)
    torch.cuda.synchronize()
    assert y2 is None
    assert np.array_equal(np_of(xn2), np_of(xn)) and np.array_equal(np_of(xnd2), np_of(xnd))
