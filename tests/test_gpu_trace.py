"""The call tracer on the device: H32_TRACE=hash gives one line per call with
a positive device time and output hashes that repeat for repeated inputs."""
import numpy as np
import pytest

from hadamard_rotated_bit_gb300 import trace
from hadamard_rotated_bit_gb300 import workloads as wl
from tests._gpu import torch_bf16

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


def test_hash_trace_of_repeated_calls(h32, capsys):
    import torch
    x = torch_bf16(wl.f32_to_bf16_bits(wl.act_normal_outliers(64, 512, 0.01, 20.0, 0,
                                                               wl.CFG_TEST, 280)))
    stream = torch.cuda.Stream()
    trace.set_mode("hash")
    try:
        out1 = h32.h32_quantize_act_q4_tc(x, stream=stream)
        out2 = h32.h32_quantize_act_q4_tc(x, stream=stream)
    finally:
        trace.set_mode("")
    assert h32.h32_device_status() == 0
    lines = [ln for ln in capsys.readouterr().err.splitlines()
             if ln.startswith("h32 trace: h32_quantize_act_q4_tc ")]
    assert len(lines) == 2
    f1, f2 = lines[0].split(), lines[1].split()
    assert float(f1[3]) > 0 and f1[4] == "ms"
    assert f1[5:] == f2[5:] and len(f1[5:]) == 2
    assert f1[5:] == [trace.digest(t) for t in out1]
    assert all(np.array_equal(a.cpu().numpy(), b.cpu().numpy()) for a, b in zip(out1, out2))
