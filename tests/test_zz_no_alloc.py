"""The allocation-free entry point, fa_fwd_noalloc, against fa_fwd.

fa_fwd_noalloc exists for callers that cannot let a library call allocate
device memory (allocator or memory-pool callbacks, runtimes that plan every
byte of device memory in advance). It runs the same kernel as fa_fwd with its
scratch in a fixed array inside the library. This file is collected last so a
run that stops at the first failure has already run every other test; it
also passes when run alone in a fresh process, and one case makes
fa_fwd_noalloc the library's very first call in a fresh process (its
first-call setup: the array's device address and the kernels' attributes)
and checks it against the oracle.
"""
import math
import os
import subprocess
import sys

import numpy as np
import pytest

from exact_attention_91_gb300 import inputs as fin

from .parity_util import LSE_MAX_ABS, O_MAX_ABS, O_MEAN_ABS, o_to_numpy, to_device

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("shape", [(2, 3, 777, 128, True), (1, 4, 2048, 64, False)])
def test_noalloc_matches_fa_fwd_twice(shape):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import exact_attention_91_gb300 as fa
    fa.load_library()
    B, H, N, d, causal = shape
    x = fin.make_inputs(fin.custom(B, H, N, d, causal, seed=4242))
    q, k, v = to_device(x.q), to_device(x.k), to_device(x.v)
    scale = 1.0 / math.sqrt(d)
    stream = torch.cuda.current_stream().cuda_stream

    o_ref = torch.empty_like(q)
    lse_ref = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    rc = fa.fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o_ref.data_ptr(), lse_ref.data_ptr(),
                   B, H, N, d, scale, causal, stream)
    assert rc == 0, fa.fa_strerror(rc)
    torch.cuda.synchronize()
    want_o, want_lse = o_to_numpy(o_ref), lse_ref.cpu().numpy()

    for _ in range(2):  # two calls in a row: the shared scratch must be left usable
        o = torch.full_like(q, float("nan"))
        lse = torch.full((B, H, N), float("nan"), dtype=torch.float32, device="cuda")
        rc = fa.fa_fwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                               B, H, N, d, scale, causal, stream)
        assert rc == 0, fa.fa_strerror(rc)
        torch.cuda.synchronize()
        got_o, got_lse = o_to_numpy(o), lse.cpu().numpy()
        assert np.isfinite(got_o).all() and np.isfinite(got_lse).all()
        d_o = np.abs(got_o - want_o)
        assert d_o.max() <= O_MAX_ABS and d_o.mean() <= O_MEAN_ABS
        assert np.abs(got_lse - want_lse).max() <= LSE_MAX_ABS
    rc, bits = fa.fa_device_status(None)
    assert rc == 0, bits


CHILD = r"""
import math
import numpy as np
import torch
import exact_attention_91_gb300 as fa
from exact_attention_91_gb300 import inputs as fin
import oracle
from tests.parity_util import compare, assert_within, o_to_numpy, to_device, visible_keys

lib = fa.load_library()
called = []
class Tripwire:
    def __init__(self, name):
        self.name = name
    def __call__(self, *a):
        called.append(self.name)
        raise AssertionError(self.name + " called")
lib.fa_fwd = Tripwire("fa_fwd")                 # nothing but fa_fwd_noalloc may run here
lib.fa_fwd_varlen = Tripwire("fa_fwd_varlen")
B, H, N, d, causal = 2, 3, 777, 128, True
w = fin.custom(B, H, N, d, causal, seed=4343)
x = fin.make_inputs(w)
q, k, v = to_device(x.q), to_device(x.k), to_device(x.v)
o_ref, lse_ref = oracle.attn_fwd(*x.f64(), w.scale, causal)
keys = np.broadcast_to(visible_keys(N, causal, np.arange(N)), lse_ref.shape)
for rep in range(2):
    o = torch.full_like(q, float("nan"))
    lse = torch.full((B, H, N), float("nan"), dtype=torch.float32, device="cuda")
    rc = fa.fa_fwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                           B, H, N, d, w.scale, causal, torch.cuda.current_stream().cuda_stream)
    assert rc == 0, fa.fa_strerror(rc)
    torch.cuda.synchronize()
    assert_within(compare(o_to_numpy(o), lse.cpu().numpy(), o_ref, lse_ref, f"call {rep}", keys=keys))
assert not called, called
print("noalloc-first OK")
"""


def test_noalloc_as_the_first_call_of_a_fresh_process():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, PYTHONPATH=root + os.pathsep + os.environ.get("PYTHONPATH", ""))
    r = subprocess.run([sys.executable, "-c", CHILD], capture_output=True, text=True, env=env, timeout=600,
                       cwd=root)
    assert r.returncode == 0, (r.stdout[-2000:], r.stderr[-3000:])
    assert "noalloc-first OK" in r.stdout, r.stdout
