"""Parity of the chain exactly as `bench.py` times it: its resident buffers, its
launch stream, both alternating input sets, the quantizer and GEMM of every
projection launched back to back with overlapping launches.  Sampled outputs
of every projection against the oracle's same-order fp32 value ("509 tokens a
second of prompt: the Hadamard route ships", sections "Why prompts are a
matrix-unit problem" and "The rotation")."""
import functools

import numpy as np
import pytest

import oracle
from hadamard_rotated_bit_gb300 import workloads as wl

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


@functools.lru_cache(maxsize=None)
def _oracle_operands(name):
    import bench
    p = {q.name: q for q in bench.CHAIN}[name]
    cid = wl.CFG_ATTN if p is wl.ATTN else wl.CFG_FFN
    wq, wd = oracle.quantize_weights_q4_0(p.weights(0, cid))
    xq, xd = oracle.quantize_act_q4(p.activations(bench.M_TOKENS, 0, cid))
    return wq, wd, xq, xd, p.K


@pytest.mark.parametrize("form", ["tc", "q4_0", "widen"])
def test_timed_chain_outputs(h32, form):
    import torch
    import bench
    dev = torch.device("cuda", 0)
    chain = bench.Chain(torch, h32, dev, sets=2, form=form)
    stream = torch.cuda.Stream(dev)
    with torch.cuda.stream(stream):
        for i in range(4):
            chain.step(i, stream)
    stream.synchronize()
    assert h32.h32_device_status(stream) == 0
    r = np.random.default_rng(8)
    M = bench.M_TOKENS
    for p, d0, d1 in zip(bench.CHAIN, chain.sets[0], chain.sets[1]):
        y0, y1 = d0["y"].cpu().numpy(), d1["y"].cpu().numpy()
        assert np.array_equal(y0.view(np.uint32), y1.view(np.uint32))   # the cloned set agrees
        wq, wd, xq, xd, K = _oracle_operands(p.name)
        mi = np.concatenate([r.integers(0, M, 2000), [0, M - 1, 0, M - 1]])
        ni = np.concatenate([r.integers(0, p.N, 2000), [0, 0, p.N - 1, p.N - 1]])
        r32, _, _ = oracle.gemm_sampled(wq, wd, xq, xd, K, mi, ni)
        assert np.array_equal(y0[mi, ni].view(np.uint32), r32.view(np.uint32)), p.name
