"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on
the same seeded bf16 inputs. Needs a GB300 and the built library."""
import math

import numpy as np
import pytest

from exact_attention_91_gb300 import inputs as fin

from .parity_util import (assert_within, compare, o_to_numpy, oracle_rows, run_gpu, sample_rows,
                          to_device, visible_keys)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa_lib():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import exact_attention_91_gb300 as fa
    fa.load_library()  # raises if the library was not built
    return fa


def _full_check(oracle_mod, x, causal=None, scale=None):
    w = x.workload
    causal = w.causal if causal is None else causal
    scale = w.scale if scale is None else scale
    o, lse = run_gpu(x, causal=causal, scale=scale)
    o_ref, lse_ref = oracle_mod.attn_fwd(*x.f64(), scale, causal)
    keys = np.broadcast_to(visible_keys(w.N, causal, np.arange(w.N)), lse_ref.shape)
    st = compare(o_to_numpy(o), lse.cpu().numpy(), o_ref, lse_ref, w.name, keys=keys)
    assert_within(st)
    return o, lse, o_ref, lse_ref


@pytest.mark.parametrize("name", ["tiny", "ragged_causal"])
def test_small_workloads_full(fa_lib, oracle_mod, name):
    _full_check(oracle_mod, fin.make_inputs(fin.WORKLOADS[name]))


@pytest.mark.parametrize("name", ["llm_prefill", "long_sequence", "max_shift"])
def test_large_workloads(fa_lib, oracle_mod, name):
    """Full-size workloads in the benchmark's launch configuration: every row
    of the first, middle and last head, and a sample of rows of every head
    (tile-boundary rows of four heads, ~3000 random rows), element by element
    against the oracle; every output row checked for finiteness and for the
    convex-combination bound (each O row is a weighted mean of V rows, so it
    lies between the per-column min and max of its head's V, up to bf16
    rounding)."""
    import torch
    w = fin.WORKLOADS[name]
    x = fin.make_inputs(w)
    o, lse = run_gpu(x)
    torch.cuda.synchronize()
    v = to_device(x.v).float().view(w.B * w.H, w.N, w.d)
    of = o.float().view(w.B * w.H, w.N, w.d)
    assert torch.isfinite(of).all() and torch.isfinite(lse).all()
    lo = v.amin(dim=1, keepdim=True)
    hi = v.amax(dim=1, keepdim=True)
    slack = 1e-2 * torch.maximum(lo.abs(), hi.abs()) + 1e-6
    assert bool(((of >= lo - slack) & (of <= hi + slack)).all())
    o_all = o_to_numpy(o).reshape(-1, w.d)
    lse_all = lse.cpu().numpy().reshape(-1)
    BH = w.B * w.H
    whole = np.concatenate([h * w.N + np.arange(w.N) for h in sorted({0, BH // 2, BH - 1})])
    sampled = sample_rows(w.B, w.H, w.N, n_random=3000, seed=w.seed)
    for label, rows in (("whole heads", whole), ("sampled rows", sampled)):
        o_ref, lse_ref = oracle_rows(oracle_mod, x, rows, w.causal, w.scale)
        keys = visible_keys(w.N, w.causal, rows % w.N)
        assert_within(compare(o_all[rows], lse_all[rows], o_ref, lse_ref, f"{name} {label}", keys=keys))


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", [1, 2, 127, 128, 129, 255, 256, 257, 640, 1000])
def test_shapes(fa_lib, oracle_mod, N, d, causal):
    x = fin.make_inputs(fin.custom(1, 2, N, d, causal, seed=7000 + N + d + causal))
    _full_check(oracle_mod, x)


def test_max_shift_full(fa_lib, oracle_mod):
    """The max-shift recipe at a size the oracle does whole: large spiked
    scores move the running max by a lot between key tiles."""
    x = fin.make_inputs(fin.custom(2, 2, 1024, 128, False, seed=fin.SEED_BASE + 4,
                                   values="maxshift"))
    _full_check(oracle_mod, x)
    xc = fin.make_inputs(fin.custom(1, 2, 1000, 64, True, seed=fin.SEED_BASE + 44,
                                    values="maxshift"))
    _full_check(oracle_mod, xc)


@pytest.mark.parametrize("causal", [False, True])
def test_constant_values(fa_lib, causal):
    """V[j] = u for all keys: O = u exactly (u is a bf16 value; the weights sum
    to l, so O = u·l/l up to one fp32 rounding before the bf16 rounding)."""
    w = fin.custom(1, 2, 300, 64, causal, seed=31)
    x = fin.make_inputs(w)
    u = x.v[0, 0, 5].copy()
    x.v[:] = u
    o, _ = run_gpu(x)
    got = o_to_numpy(o)
    want = np.broadcast_to(fin.bf16_to_f64(u), got.shape)
    ulp = np.abs(want) * 2.0 ** -7 + 1e-30
    assert np.all(np.abs(got - want) <= ulp)


@pytest.mark.parametrize("causal", [False, True])
def test_zero_keys(fa_lib, oracle_mod, causal):
    """K = 0: O is the (prefix) mean of V and LSE = ln(visible keys)."""
    w = fin.custom(1, 1, 260, 128, causal, seed=32)
    x = fin.make_inputs(w)
    x.k[:] = 0
    o, lse = run_gpu(x)
    n = np.arange(1, w.N + 1) if causal else np.full(w.N, w.N)
    np.testing.assert_allclose(lse.cpu().numpy()[0, 0], np.log(n), atol=1e-5, rtol=0)
    _full_check(oracle_mod, x)


def test_repeat_and_stream(fa_lib):
    """Same inputs twice (once on a side stream): bit-identical outputs."""
    import torch
    x = fin.make_inputs(fin.custom(2, 3, 777, 128, True, seed=33))
    q, k, v = to_device(x.q), to_device(x.k), to_device(x.v)
    o1, l1 = fa_lib.attention_forward(q, k, v, causal=True)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        o2, l2 = fa_lib.attention_forward(q, k, v, causal=True)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(l1, l2)


@pytest.mark.parametrize("shape", [(1, 2, 4096, 64, False), (1, 3, 200, 64, False), (2, 3, 777, 128, True),
                                   (1, 4, 2048, 128, False)])
def test_repeated_calls_bit_identical(fa_lib, oracle_mod, shape):
    """Eight calls on the same inputs give the same bits, every output
    written (O and LSE start as NaN), and the first matches the oracle. Work
    units land on different CTAs from call to call, so any ordering hazard
    between the kernel's roles shows up as a difference here."""
    import torch
    B, H, N, d, causal = shape
    x = fin.make_inputs(fin.custom(B, H, N, d, causal, seed=36))
    q, k, v = to_device(x.q), to_device(x.k), to_device(x.v)
    first = None
    for _ in range(8):
        o = torch.full_like(q, float("nan"))
        lse = torch.full((B, H, N), float("nan"), dtype=torch.float32, device="cuda")
        fa_lib.attention_forward(q, k, v, causal=causal, out=o, lse=lse)
        torch.cuda.synchronize()
        assert bool(torch.isfinite(o).all()) and bool(torch.isfinite(lse).all())
        if first is None:
            first = (o.clone(), lse.clone())
            rows = sample_rows(B, H, N, n_random=400, seed=37)
            o_ref, lse_ref = oracle_rows(oracle_mod, x, rows, causal, 1.0 / math.sqrt(d))
            st = compare(o_to_numpy(o).reshape(-1, d)[rows], lse.cpu().numpy().reshape(-1)[rows], o_ref,
                         lse_ref, "repeat", keys=visible_keys(N, causal, rows % N))
            assert_within(st)
        else:
            assert torch.equal(o.view(torch.int16), first[0].view(torch.int16))
            assert torch.equal(lse, first[1])


def test_without_lse_and_guard_bands(fa_lib):
    """lse = NULL gives the same O; nothing is written outside O and LSE
    (sentinel bands before and after each buffer stay untouched), also for a
    ragged N whose last tile hangs past the end of every head."""
    import torch
    w = fin.custom(1, 3, 200, 64, False, seed=34)
    x = fin.make_inputs(w)
    q, k, v = to_device(x.q), to_device(x.k), to_device(x.v)
    band = 8192
    n_o = w.B * w.H * w.N * w.d
    o_buf = torch.full((band + n_o + band,), -12345, dtype=torch.int16, device="cuda")
    l_buf = torch.full((band + w.B * w.H * w.N + band,), float("nan"), dtype=torch.float32, device="cuda")
    o = o_buf[band:band + n_o].view(torch.bfloat16).view(w.B, w.H, w.N, w.d)
    lse = l_buf[band:band + w.B * w.H * w.N].view(w.B, w.H, w.N)
    fa_lib.attention_forward(q, k, v, causal=False, out=o, lse=lse)
    o2 = fa_lib.attention_forward(q, k, v, causal=False, return_lse=False)
    torch.cuda.synchronize()
    assert torch.equal(o.view(torch.int16), o2.view(torch.int16))
    assert bool((o_buf[:band] == -12345).all()) and bool((o_buf[band + n_o:] == -12345).all())
    assert bool(torch.isnan(l_buf[:band]).all()) and bool(torch.isnan(l_buf[-band:]).all())
    assert bool(torch.isfinite(lse).all())


def test_status_word_clean(fa_lib):
    rc, bits = fa_lib.fa_device_status(None)
    assert rc == 0 and bits == 0


def test_scale_argument(fa_lib, oracle_mod):
    """A scale other than 1/sqrt(d) reaches the kernel as given."""
    x = fin.make_inputs(fin.custom(1, 2, 300, 64, True, seed=35))
    _full_check(oracle_mod, x, scale=0.05)
    _full_check(oracle_mod, x, scale=1.0 / math.sqrt(64) * 2.0)


@pytest.mark.parametrize("d", [64, 128])
def test_whole_and_half_units_in_one_launch(fa_lib, oracle_mod, d):
    """A non-causal launch with a few more units than SMs runs most units
    whole and its last few as half units (the kernel instantiation that
    carries both kinds of item). Rows of every head are checked, with all
    256 rows of the first query block of the last 8 heads, where the last
    units (heaviest-first order within groups of 16 heads) fall."""
    import torch
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    N = 1024
    nqb = N // 256
    H = (sms + 8 + nqb - 1) // nqb  # units = H * nqb: one wave plus a few
    r = (H * nqb) % sms
    assert 0 < r <= sms // 2
    x = fin.make_inputs(fin.custom(1, H, N, d, False, seed=8100 + d))
    o, lse = run_gpu(x)
    g = np.random.Generator(np.random.PCG64(8200 + d))
    rows = [h * N + g.choice(N, 32, replace=False) for h in range(H)]
    rows += [h * N + np.arange(256) for h in range(max(0, H - 8), H)]
    rows = np.unique(np.concatenate(rows))
    o_ref, lse_ref = oracle_rows(oracle_mod, x, rows, False, x.workload.scale)
    st = compare(o_to_numpy(o).reshape(-1, d)[rows], lse.cpu().numpy().reshape(-1)[rows], o_ref, lse_ref,
                 f"whole+half d={d}", keys=visible_keys(N, False, rows % N))
    assert_within(st)
