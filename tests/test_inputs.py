"""The seeded input generator: deterministic, bf16 rounding as torch does it,
and the workload recipes as stated (shapes, distributions, the max-shift spike)."""
import numpy as np
import pytest

from exact_attention_91_gb300 import inputs as fin


def test_bf16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    g = np.random.Generator(np.random.PCG64(5))
    x = np.concatenate([g.standard_normal(20000) * 10.0 ** g.integers(-30, 30, 20000),
                        np.array([0.0, -0.0, 1.0, -1.0, 1.00390625, 1.01171875, 3.0e38,
                                  1e-40, np.inf, -np.inf])])
    ours = fin.bf16_from_f64(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, ref)
    back = fin.bf16_to_f64(ours)
    np.testing.assert_array_equal(back, torch.from_numpy(x).to(torch.bfloat16).double().numpy())


def test_deterministic_per_seed():
    w = fin.custom(1, 2, 50, 64, False, seed=123)
    a, b = fin.make_inputs(w), fin.make_inputs(w)
    for x, y in ((a.q, b.q), (a.k, b.k), (a.v, b.v)):
        np.testing.assert_array_equal(x, y)
    c = fin.make_inputs(fin.custom(1, 2, 50, 64, False, seed=124))
    assert not np.array_equal(a.q, c.q)
    assert not np.array_equal(a.q, a.k)


def test_workload_table():
    W = fin.WORKLOADS
    assert [(w.B, w.H, w.N, w.d, w.causal) for w in W.values()] == [
        (1, 1, 128, 64, False), (2, 4, 1000, 64, True), (4, 32, 4096, 128, True),
        (1, 8, 16384, 64, False), (16, 16, 1024, 128, False)]
    assert [w.seed for w in W.values()] == [20260000 + i for i in range(5)]
    assert W["llm_prefill"].flops == pytest.approx(549.755813888e9)
    assert W["tiny"].hbm_bytes == 66048
    assert W["llm_prefill"].hbm_bytes == 538968064


def test_normal_values():
    x = fin.make_inputs(fin.WORKLOADS["tiny"])
    assert x.q.shape == (1, 1, 128, 64) and x.q.dtype == np.uint16
    q = fin.bf16_to_f64(x.q)
    assert abs(q.mean()) < 0.05 and 0.95 < q.std() < 1.05


def test_max_shift_spike():
    """Each query row's score against its drawn key sits about +20 above what
    it was before the spike (up to Q's bf16 rounding)."""
    w = fin.custom(1, 2, 256, 128, False, seed=fin.SEED_BASE + 4, values="maxshift")
    x = fin.make_inputs(w)
    q, k, v = x.f64()
    assert v.min() >= -1.0 and v.max() <= 1.0
    s = np.einsum("bhic,bhjc->bhij", q, k) * w.scale
    spike = np.take_along_axis(s, x.spike_keys[..., None], axis=3)[..., 0]
    # the un-spiked Q is redrawn from the same stream to measure the rise
    gq = np.random.Generator(np.random.PCG64(np.random.SeedSequence(w.seed).spawn(4)[0]))
    q0 = 3.0 * gq.standard_normal(q.shape)
    s0 = np.einsum("bhic,bhjc->bhij", q0, k) * w.scale
    rise = spike - np.take_along_axis(s0, x.spike_keys[..., None], axis=3)[..., 0]
    assert np.all(np.abs(rise - 20.0) < 0.5)


def test_varlen_inputs():
    """Packed sequences: int32 offsets that start at 0 and add up the counts,
    token-major [total, H, d] bf16 values, the same bits for the same seed,
    and empty sequences allowed."""
    x = fin.make_varlen_inputs([3, 0, 5], [7, 2, 0], 2, 64, seed=9)
    assert x.cu_q.dtype == np.int32 and x.cu_k.dtype == np.int32
    assert x.cu_q.tolist() == [0, 3, 3, 8] and x.cu_k.tolist() == [0, 7, 9, 9]
    assert x.q.shape == (8, 2, 64) and x.k.shape == (9, 2, 64) and x.v.shape == (9, 2, 64)
    assert x.q.dtype == np.uint16
    y = fin.make_varlen_inputs([3, 0, 5], [7, 2, 0], 2, 64, seed=9)
    for a, b in ((x.q, y.q), (x.k, y.k), (x.v, y.v)):
        np.testing.assert_array_equal(a, b)
    assert not np.array_equal(x.k, x.v)
    q, k, v = x.f64()
    np.testing.assert_array_equal(fin.bf16_from_f64(q), x.q)  # values are exact bf16
    big = fin.make_varlen_inputs([4000], [4000], 4, 64, seed=10)
    qb = fin.bf16_to_f64(big.q)
    assert abs(qb.mean()) < 0.02 and 0.98 < qb.std() < 1.02
    with pytest.raises(ValueError):
        fin.make_varlen_inputs([1, 2], [3], 1, 64, seed=1)
