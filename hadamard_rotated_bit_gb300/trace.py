"""Optional per-call tracing of the library's compute entry points (a debug aid).

Set ``H32_TRACE`` in the environment (or call ``set_mode``):

``1``     every compute call of the Python binding is bracketed by CUDA events on
          the stream it enqueues on; after the call the end event is waited for
          and one line goes to stderr: the entry point and its device time.
``hash``  the same, plus a 64-bit hash of each output tensor's bytes.  Two runs
          of the same inputs then give the same lines, and the first line that
          differs names the first call whose output diverged -- the way the
          pages found a race ("Milestone: the HRX decode race is solved",
          section "How we know": hashing every kernel's output in serial
          execution).

Off by default.  Tracing waits for every call to finish, so a traced run is
serial and slow; timed benchmarks run untraced.
"""
from __future__ import annotations

import functools
import hashlib
import inspect
import os
import sys

_MODE = os.environ.get("H32_TRACE", "").strip().lower()
if _MODE in ("0", "off", "false"):
    _MODE = ""


def mode() -> str:
    """"" (off), "1" (timing) or "hash" (timing and output hashes)."""
    return _MODE


def set_mode(m: str | None) -> None:
    global _MODE
    m = (m or "").strip().lower()
    if m not in ("", "0", "1", "hash"):
        raise ValueError("trace mode is '', '1' or 'hash'")
    _MODE = "" if m == "0" else m


class _CudaClock:
    """Device time between two CUDA events recorded on a stream."""

    def start(self, stream):
        import torch
        e0 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        return e0

    def stop(self, stream, e0) -> float:
        import torch
        e1 = torch.cuda.Event(enable_timing=True)
        e1.record(stream)
        e1.synchronize()
        return e0.elapsed_time(e1)

    def default_stream(self):
        import torch
        return torch.cuda.current_stream()


_clock = _CudaClock()


def _emit(line: str) -> None:
    print(line, file=sys.stderr, flush=True)


def digest(t) -> str:
    """64-bit hash (hex) of a tensor's bytes, in row-major order."""
    import torch
    b = t.detach().contiguous().reshape(-1)
    if b.numel():
        b = b.view(torch.uint8)
    return hashlib.blake2b(b.cpu().numpy().tobytes(), digest_size=8).hexdigest()


def _tensors(obj):
    if obj is None:
        return []
    if isinstance(obj, (tuple, list)):
        return [t for o in obj for t in _tensors(o)]
    return [obj] if hasattr(obj, "data_ptr") else []


def traced(name: str):
    """Decorator for a binding function that enqueues work on its `stream`
    argument (None = the current stream)."""
    def deco(fn):
        sig = inspect.signature(fn)

        @functools.wraps(fn)
        def wrapper(*args, **kwargs):
            if not _MODE:
                return fn(*args, **kwargs)
            bound = sig.bind(*args, **kwargs)
            stream = bound.arguments.get("stream")
            if stream is None:
                stream = _clock.default_stream()
            token = _clock.start(stream)
            try:
                out = fn(*args, **kwargs)
            except Exception as e:
                _emit(f"h32 trace: {name} raised {type(e).__name__}: {e}")
                raise
            ms = _clock.stop(stream, token)
            line = f"h32 trace: {name} {ms:.4f} ms"
            if _MODE == "hash":
                line += " " + " ".join(digest(t) for t in _tensors(out))
            _emit(line)
            return out
        return wrapper
    return deco
