"""The optional call tracer of the binding (H32_TRACE): off by default; with
mode "1" one line per call with its device time, with "hash" also a hash of
each output, equal for equal outputs.  CPU only: the device clock is replaced
by a fake, the traced function is a stand-in that returns CPU tensors."""
import hashlib

import numpy as np
import pytest
import torch

import hadamard_rotated_bit_gb300 as h32
from hadamard_rotated_bit_gb300 import trace


class FakeClock:
    def __init__(self):
        self.streams = []

    def start(self, stream):
        self.streams.append(stream)
        return 0.0

    def stop(self, stream, token):
        self.streams.append(stream)
        return 0.25

    def default_stream(self):
        return "current"


@pytest.fixture
def fake(monkeypatch):
    clock = FakeClock()
    lines = []
    monkeypatch.setattr(trace, "_clock", clock)
    monkeypatch.setattr(trace, "_emit", lines.append)
    yield clock, lines
    trace.set_mode("")


def _op(x, scale=2, stream=None):
    return x + 1, x * scale


def test_off_by_default_and_passthrough(fake):
    clock, lines = fake
    trace.set_mode("")
    f = trace.traced("fake_op")(_op)
    a, b = f(torch.arange(4))
    assert lines == [] and clock.streams == []
    assert a.tolist() == [1, 2, 3, 4] and b.tolist() == [0, 2, 4, 6]


def test_timing_line_uses_the_call_stream(fake):
    clock, lines = fake
    trace.set_mode("1")
    f = trace.traced("fake_op")(_op)
    f(torch.arange(4), stream="s7")
    f(torch.arange(4), 3, "s8")          # stream given positionally
    f(torch.arange(4))
    assert lines == ["h32 trace: fake_op 0.2500 ms"] * 3
    assert clock.streams == ["s7", "s7", "s8", "s8", "current", "current"]


def test_hash_mode_hashes_every_output(fake):
    clock, lines = fake
    trace.set_mode("hash")
    f = trace.traced("fake_op")(_op)
    x = torch.arange(6, dtype=torch.float32).reshape(2, 3)
    f(x)
    f(x.clone())
    f(x + 1)
    want = [hashlib.blake2b(np.ascontiguousarray(t.numpy()).tobytes(), digest_size=8).hexdigest()
            for t in (x + 1, x * 2)]
    assert lines[0] == "h32 trace: fake_op 0.2500 ms " + " ".join(want)
    assert lines[1] == lines[0] and lines[2] != lines[0]
    # a transposed (non-contiguous) output hashes its row-major bytes
    assert trace.digest(x.t()) == trace.digest(x.t().contiguous())


def test_errors_are_traced_and_raised(fake):
    clock, lines = fake
    trace.set_mode("1")

    def bad(stream=None):
        raise ValueError("no")
    with pytest.raises(ValueError):
        trace.traced("bad_op")(bad)()
    assert lines == ["h32 trace: bad_op raised ValueError: no"]
    with pytest.raises(ValueError):
        trace.set_mode("verbose")


def test_every_compute_entry_point_is_wrapped():
    for name in h32._COMPUTE_CALLS:
        fn = getattr(h32, name)
        assert hasattr(fn, "__wrapped__"), name
        assert name in h32.EXPORTED_SYMBOLS
