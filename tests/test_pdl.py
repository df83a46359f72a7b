"""Programmatic dependent launch after a forward call (include/fa.h): every
forward kernel lets a kernel launched next on the stream with programmatic
stream serialization start before it ends; such a kernel that waits for its
prerequisite grids (griddepcontrol.wait) sees the finished O. The successor
is a small helper built here with nvcc."""
import ctypes
import os
import shutil
import subprocess

import numpy as np
import pytest

from exact_attention_91_gb300 import inputs as fin

from .parity_util import to_device

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def successor(tmp_path_factory):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from exact_attention_91_gb300 import build as fa_build
    nvcc = fa_build.nvcc_path()
    if not (os.path.exists(nvcc) or shutil.which(nvcc)):
        pytest.skip("nvcc not available")
    out = str(tmp_path_factory.mktemp("pdl") / "libpdl_successor.so")
    subprocess.run([nvcc, fa_build.ARCH, "-O2", "-std=c++17", "-Xcompiler", "-fPIC", "-shared",
                    os.path.join(HERE, "helpers", "pdl_successor.cu"), "-o", out], check=True)
    lib = ctypes.CDLL(out)
    lib.launch_successor_copy.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
    lib.launch_successor_copy.restype = ctypes.c_int
    return lib


@pytest.mark.parametrize("shape", [(4, 32, 2048, 128, True), (1, 8, 8192, 64, False), (1, 1, 128, 64, False)])
def test_successor_launched_early_sees_the_finished_output(successor, shape):
    import torch
    import exact_attention_91_gb300 as fa
    B, H, N, d, causal = shape
    x = fin.make_inputs(fin.custom(B, H, N, d, causal, seed=4242))
    q, k, v = to_device(x.q), to_device(x.k), to_device(x.v)
    ref, _ = fa.attention_forward(q, k, v, causal=causal)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    for _ in range(3):
        o = torch.full_like(q, float("nan"))
        copy = torch.full_like(q, float("nan"))
        with torch.cuda.stream(s):
            fa.attention_forward(q, k, v, causal=causal, out=o)
            rc = successor.launch_successor_copy(o.data_ptr(), copy.data_ptr(), o.numel(), s.cuda_stream)
            assert rc == 0
        s.synchronize()
        assert torch.equal(copy.view(torch.int16), ref.view(torch.int16))
