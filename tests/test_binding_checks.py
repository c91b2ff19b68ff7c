"""The Python binding checks every tensor it passes to the library as a raw
pointer (dtype, shape, layout, device) before any call, so a mismatched tensor
raises instead of letting a kernel read or write past it.  CPU only: the
checks run before the library is reached, and a well-formed CPU tensor is
refused for not being on a CUDA device."""
import pytest
import torch

import hadamard_rotated_bit_gb300 as h32

u8, i8, i32, f32 = torch.uint8, torch.int8, torch.int32, torch.float32


def _tc_operands(N=32, K=128, M=8):
    return (torch.zeros((N, K), dtype=u8), torch.zeros((N, 4), dtype=f32),
            torch.zeros((M, K), dtype=u8), torch.zeros((K // 32, 8), dtype=f32))


def _raises(match, fn, *args, **kwargs):
    with pytest.raises(ValueError, match=match):
        fn(*args, **kwargs)


def test_tc_gemm_operands():
    wp, wsc, xw, xdt = _tc_operands()
    _raises("must be a CUDA tensor", h32.q4_0_x_q4_gemm_tc, wp, wsc, xw, xdt)
    _raises("xw: shape", h32.q4_0_x_q4_gemm_tc, wp, wsc, xw[:, :64].contiguous(), xdt)
    _raises("xw: dtype", h32.q4_0_x_q4_gemm_tc, wp, wsc, xw.to(i8), xdt)
    _raises("xdt: shape", h32.q4_0_x_q4_gemm_tc, wp, wsc, xw, xdt[:2].contiguous())
    _raises("xw: shape", h32.q4_0_x_q4_gemm_tc, wp, wsc, xw, xdt, M=9)     # too few token rows
    _raises("xdt: shape", h32.q4_0_x_q4_gemm_tc, wp, wsc, torch.zeros((9, 128), dtype=u8), xdt,
            M=9)                                                               # too few token columns
    _raises("wsc: shape", h32.q4_0_x_q4_gemm_tc, wp, wsc[:, :3].contiguous(), xw, xdt)
    _raises("xw: shape", h32.q4_0_x_q8_gemm_tc, wp, wsc, xw, xdt)          # 8-bit: 2 bytes a code
    _raises("must be contiguous", h32.q4_0_x_q4_gemm_tc, wp, wsc, xw.t().contiguous().t(), xdt)
    y_t = torch.zeros((32, 8), dtype=f32).t()
    _raises("y must be 2-D with contiguous", h32.q4_0_x_q4_gemm_tc, wp, wsc, xw, xdt, y=y_t)
    _raises("block_sums: shape", h32.q4_0_x_q4_gemm_tc, wp, wsc, xw, xdt,
            block_sums=torch.zeros((8, 32, 3), dtype=i32))
    # the K split's workspace: bytes, one flat array
    _raises("workspace: dtype", h32.q4_0_x_q4_gemm_tc, wp, wsc, xw, xdt,
            workspace=torch.zeros(64, dtype=f32))
    _raises("workspace: shape", h32.q4_0_x_q8_gemm_tc, wp, wsc, torch.zeros((8, 256), dtype=u8),
            xdt, workspace=torch.zeros((8, 8), dtype=u8))
    _raises("workspace: dtype", h32.q4_0_x_q4_gemm_tc_quant_next, *_tc_operands(N=64),
            workspace=torch.zeros(64, dtype=i32))


def test_direct_and_quantizer_outputs():
    x = torch.zeros((4, 64), dtype=torch.bfloat16)
    _raises("xq: shape", h32.h32_quantize_act_q4, x, xq=torch.zeros((4, 31), dtype=u8))
    _raises("xd: dtype", h32.h32_quantize_act_q8, x, xd=torch.zeros((4, 2), dtype=torch.float64))
    _raises("x must be bf16 or fp32", h32.h32_quantize_act_q4, x.to(torch.float16))
    _raises("xdt: shape", h32.h32_quantize_act_q4_tc, x, xdt=torch.zeros((2, 3), dtype=f32))
    wq, wd = torch.zeros((16, 32), dtype=u8), torch.zeros((16, 2), dtype=torch.int16)
    _raises("xq: dtype", h32.q4_0_x_q8_gemm, wq, wd, torch.zeros((4, 64), dtype=torch.int16),
            torch.zeros((4, 2), dtype=f32))
    _raises("must be a CUDA tensor", h32.q4_0_x_q8_gemm, wq, wd, torch.zeros((4, 64), dtype=u8),
            torch.zeros((4, 2), dtype=f32))      # 8-bit codes in a uint8 buffer are accepted
    _raises("wd: shape", h32.q4_0_x_q4_gemm, wq, wd[:, :1].contiguous(),
            torch.zeros((4, 32), dtype=u8), torch.zeros((4, 2), dtype=f32))
    _raises("wp: shape", h32.h32_prepack_weights_q4_0_tc, wq, wd, wp=torch.zeros((16, 63), dtype=u8))
    _raises("wq: shape", h32.h32_rotate_quantize_weights_q4_0, torch.zeros((16, 64), dtype=f32),
            wq=torch.zeros((15, 32), dtype=u8))


def test_experts_and_gather():
    wp, wsc, xw, xdt = _tc_operands(N=64)
    _raises("expert_off: shape", h32.q4_0_x_q4_gemm_tc_experts, wp, wsc, xw, xdt,
            torch.zeros(2, dtype=i32), 32)                       # E = 2 needs 3 offsets
    _raises("wp must be 2-D with E", h32.q4_0_x_q4_gemm_tc_experts, wp, wsc, xw, xdt,
            torch.zeros(3, dtype=i32), 48)
    x = torch.zeros((10, 128), dtype=f32)
    _raises("row_idx: dtype", h32.h32_quantize_act_q4_tc_gather, x, torch.zeros(5, dtype=torch.int64))
    _raises("xw: shape", h32.h32_quantize_act_q4_tc_gather, x, torch.zeros(5, dtype=i32),
            xw=torch.zeros((4, 128), dtype=u8))
    _raises("xw_next: shape", h32.q4_0_x_q4_gemm_tc_quant_next, *_tc_operands(N=64),
            xw_next=torch.zeros((8, 32), dtype=u8))


def test_router_and_combine():
    l = torch.zeros((6, 16), dtype=f32)
    _raises("topk_id: shape", h32.h32_moe_route, l, 4, topk_id=torch.zeros((6, 3), dtype=i32))
    _raises("expert_off: shape", h32.h32_moe_route, l, 4, expert_off=torch.zeros(16, dtype=i32))
    _raises("logits: dtype", h32.h32_moe_route, l.double(), 4)
    _raises("must be a CUDA tensor", h32.h32_moe_route, l, 4)
    y = torch.zeros((24, 8), dtype=f32)
    row_of, w = torch.zeros((6, 4), dtype=i32), torch.zeros((6, 4), dtype=f32)
    _raises("topk_w: shape", h32.h32_moe_combine, y, row_of, w[:, :3].contiguous())
    _raises("out: shape", h32.h32_moe_combine, y, row_of, w, out=torch.zeros((6, 4), dtype=f32))
    _raises("must be a CUDA tensor", h32.h32_moe_combine, y, row_of, w)


def test_need_shapes():
    t = torch.zeros((4, 8), dtype=f32)
    assert h32._need(t, "t", (f32,), (h32._ge(3), 8)) is t
    _raises("t: shape", h32._need, t, "t", (f32,), (5, 8))
    _raises("t: shape", h32._need, t, "t", (f32,), (4, h32._ge(9)))
    _raises("t: shape", h32._need, t, "t", (f32,), (4, 8, 1))


def test_workspace_cache_per_stream(monkeypatch):
    """The binding's K-split workspaces (host logic, faked sizes, CPU tensors):
    one zeroed workspace per (device, stream), kept across calls; a larger need
    replaces it and keeps the old one alive (a captured graph may still use
    it); no workspace when the schedule does not split; inside a graph capture
    a fresh one per call, not cached."""
    need = {"bytes": 1000}
    monkeypatch.setattr(h32, "h32_gemm_tc_workspace_bytes", lambda M, N, K: need["bytes"])
    monkeypatch.setattr(torch.cuda, "is_current_stream_capturing", lambda: False)
    monkeypatch.setattr(h32, "_workspaces", {})
    monkeypatch.setattr(h32, "_retired_workspaces", [])

    class S1:
        cuda_stream = 1234

    class S2:
        cuda_stream = 5678

    dev = torch.device("cpu")
    a = h32._workspace_for(1, 1, 1, dev, S1())
    assert a.dtype == u8 and a.numel() == 1000 and int(a.sum()) == 0
    assert h32._workspace_for(1, 1, 1, dev, S1()) is a
    assert h32._workspace_for(1, 1, 1, dev, S2()) is not a
    need["bytes"] = 4000
    b = h32._workspace_for(1, 1, 1, dev, S1())
    assert b.numel() == 4000 and any(r is a for r in h32._retired_workspaces)
    need["bytes"] = 256
    assert h32._workspace_for(1, 1, 1, dev, S1()) is b     # large enough already
    need["bytes"] = 0
    assert h32._workspace_for(1, 1, 1, dev, S1()) is None
    need["bytes"] = 500
    monkeypatch.setattr(torch.cuda, "is_current_stream_capturing", lambda: True)
    c, d = h32._workspace_for(1, 1, 1, dev, S1()), h32._workspace_for(1, 1, 1, dev, S1())
    assert c is not d and c.numel() == 500 and int(c.sum()) == 0
    assert h32._workspaces[(None, 1234)] is b
