"""The allocation-free entry point, fa_fwd_noalloc, against fa_fwd.

fa_fwd_noalloc exists for callers that cannot let a library call allocate
device memory (allocator or memory-pool callbacks, runtimes that plan every
byte of device memory in advance). It runs the same kernel as fa_fwd with its
scratch in a fixed array inside the library. This file is collected last so a
run that stops at the first failure has already run every other test; it
also passes when run alone in a fresh process.
"""
import math

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
