"""A plain C program calls the library through include/h32.h alone (no Python,
no torch: its own cudaMalloc'd buffers and stream) and its result equals the
oracle's same-order fp32 value bit for bit.  The build check runs on the CPU;
the run needs a GPU."""
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle
from hadamard_rotated_bit_gb300 import _build
from hadamard_rotated_bit_gb300 import workloads as wl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c", "h32_c_caller.c")
CUDA = "/usr/local/cuda"


def _compile(tmp_path):
    if shutil.which("gcc") is None or not os.path.exists(os.path.join(CUDA, "include", "cuda_runtime.h")):
        pytest.skip("gcc or the CUDA toolkit headers are missing")
    lib = _build.build()
    libdir = os.path.dirname(lib)
    cudalib = os.path.join(CUDA, "lib64")
    exe = str(tmp_path / "h32_c_caller")
    cmd = ["gcc", "-std=c11", "-O2", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(CUDA, "include"), SRC, "-o", exe, "-L", libdir, "-lh32",
           "-L", cudalib, "-lcudart", f"-Wl,-rpath,{libdir}:{cudalib}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


def test_c_caller_builds(tmp_path):
    assert os.access(_compile(tmp_path), os.X_OK)


@pytest.mark.gpu
@pytest.mark.parametrize("M,N,K", [(70, 144, 384), (70, 144, 512), (64, 20480, 256)])
def test_c_caller_matches_the_oracle(tmp_path, M, N, K):
    """K = 384: the tensor-core route; K = 512: also the widening route; 64 x
    20480 x 256 (a full wave and 8 tiles over on 152 SMs): also the K split with
    the caller's workspace (twice) and the no-alloc form.  Every result
    bit-exact."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    exe = _compile(tmp_path)
    x = wl.act_normal_outliers(M, K, 0.01, 20.0, 0, wl.CFG_TEST, 290)
    w = wl.weights_normal(N, K, 0.02, 0, wl.CFG_TEST, 291)
    inp, out = tmp_path / "in.bin", tmp_path / "out.bin"
    with open(inp, "wb") as f:
        f.write(np.array([M, N, K], np.int64).tobytes())
        f.write(np.ascontiguousarray(x, np.float32).tobytes())
        f.write(np.ascontiguousarray(w, np.float32).tobytes())
    r = subprocess.run([exe, str(inp), str(out)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    raw = np.fromfile(out, np.uint8)
    routes = int(raw[:8].view(np.int64)[0])
    expect = 1 + (K % 256 == 0) + (2 if N == 20480 and torch.cuda.get_device_properties(0)
                                   .multi_processor_count == 152 else 0)
    assert routes == expect
    ys = raw[8:].view(np.float32).reshape(routes, M, N)
    wq, wd = oracle.quantize_weights_q4_0(w)
    xq, xd = oracle.quantize_act_q4(x)
    r32, _, _ = oracle.gemm(wq, wd, xq, xd, K)
    for y in ys:
        assert np.array_equal(y.view(np.uint32), r32.view(np.uint32))
