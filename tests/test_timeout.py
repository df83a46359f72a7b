"""Failure detection on the GPU without a fault: a bounded mbarrier wait that
runs out is reported through the device status word, and the context stays
usable afterwards.

fa_selftest_wait_timeout launches one warp that waits, through the forward
kernel's own bounded wait, on a barrier phase that nothing completes. After
the limit it records the timeout and returns; no trap, no fault, no hang.
"""
import numpy as np
import pytest

from exact_attention_91_gb300 import inputs as fin

from .parity_util import assert_within, compare, o_to_numpy, run_gpu

pytestmark = pytest.mark.gpu

STATUS_TIMEOUT_OTHER = 1 << 4


def test_wait_that_runs_out_is_reported(oracle_mod):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import exact_attention_91_gb300 as fa
    torch.cuda.init()
    fa.fa_device_status()  # start from a clear word
    stream = torch.cuda.current_stream().cuda_stream
    assert fa.fa_selftest_wait_timeout(2_000_000, stream) == 0
    rc, bits = fa.fa_device_status(stream)
    assert rc == fa.FA_ERR_DEVICE_TIMEOUT, fa.fa_strerror(rc)
    assert bits == STATUS_TIMEOUT_OTHER
    assert fa.fa_device_status(stream) == (0, 0)  # read and cleared

    # the context still works: a forward pass afterwards matches the oracle
    x = fin.make_inputs(fin.custom(1, 2, 300, 64, True, seed=6060))
    o, lse = run_gpu(x)
    torch.cuda.synchronize()
    q, k, v = x.f64()
    o_ref, lse_ref = oracle_mod.attn_fwd(q, k, v, x.workload.scale, True)
    stats = compare(o_to_numpy(o), lse.cpu().numpy(), o_ref, lse_ref, "after timeout")
    assert_within(stats)
    assert fa.fa_device_status(stream) == (0, 0)


def test_selftest_rejects_limits_out_of_range():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import exact_attention_91_gb300 as fa
    assert fa.fa_selftest_wait_timeout(1_000) == -2
    assert fa.fa_selftest_wait_timeout(5_000_000_000) == -2
