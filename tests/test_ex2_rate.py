"""The exponential unit's throughput probe (fa_selftest_ex2_rate), which
gives the bench's second ceiling (one ex2 per query and visible key) a
measured denominator instead of a nominal one."""
import numpy as np
import pytest


def _lib():
    import exact_attention_91_gb300 as fa
    from exact_attention_91_gb300 import build as fa_build
    import shutil
    if not fa_build.up_to_date():
        if shutil.which(fa_build.nvcc_path()) is None:
            pytest.skip("nvcc not available to build libfa.so")
        fa_build.build()
    fa.load_library()
    return fa


def test_bad_arguments_are_rejected_before_any_device_work():
    fa = _lib()
    fake = 1 << 20  # never dereferenced: the checks come first
    assert fa.fa_selftest_ex2_rate(fake, fake, 0, 16) == -2
    assert fa.fa_selftest_ex2_rate(fake, fake, 4097, 16) == -2
    assert fa.fa_selftest_ex2_rate(fake, fake, 1, 0) == -2
    assert fa.fa_selftest_ex2_rate(fake, fake, 1, (1 << 20) + 1) == -2
    assert fa.fa_selftest_ex2_rate(0, fake, 1, 16) == -1
    assert fa.fa_selftest_ex2_rate(fake, 0, 1, 16) == -1
    assert fa.fa_selftest_ex2_rate(fake + 4, fake, 1, 16) == -4
    assert fa.fa_selftest_ex2_rate(fake, fake + 2, 1, 16) == -4


@pytest.mark.gpu
def test_rate_is_a_plausible_exponential_throughput():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import bench
    fa = _lib()
    dev = torch.device("cuda", torch.cuda.current_device())
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    rate = bench.measure_ex2_rate(fa, torch, dev, sms, iters=1024)
    assert rate is not None
    # one SM's exponential unit: tens of ex2 per clock (32 on GB300), never
    # more than one per lane of its four sub-partitions
    assert 8.0 <= rate <= 128.0, rate
    # the chains' final values are finite and on the map x -> -2^x's orbit
    sink = torch.empty(sms * fa.EX2_RATE_THREADS, dtype=torch.float32, device=dev)
    cycles = torch.zeros(sms, dtype=torch.int64, device=dev)
    assert fa.fa_selftest_ex2_rate(cycles.data_ptr(), sink.data_ptr(), sms, 64,
                                   torch.cuda.current_stream().cuda_stream) == 0
    torch.cuda.synchronize()
    s = sink.cpu().numpy() / fa.EX2_RATE_CHAINS
    assert np.isfinite(s).all() and (s <= -0.5).all() and (s >= -1.0).all()
    assert (cycles.cpu().numpy() > 0).all()
