"""Pins for the fp64 oracle: each test checks it against something other than
itself (hand-derived worked examples, closed forms, invariants of the
definition, an independent library routine, and the streaming loop that the
pages claim is exact). A plausible slip in the oracle — a dropped scale, a
wrong causal boundary, swapped Q/K roles, a missing max shift, an LSE without
its max, a wrong V stride — fails at least one of them.
"""
import math
import os

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_examples.txt")


def _parse_golden(path):
    cases, cur = [], None
    env = {"ln": math.log, "sqrt": math.sqrt, "__builtins__": {}}
    for raw in open(path, encoding="utf-8"):
        line = raw.split("#", 1)[0].strip()
        if not line:
            continue
        if line.startswith("[case"):
            cur = {"name": line[5:-1].strip()}
            cases.append(cur)
            continue
        key, val = (s.strip() for s in line.split("=", 1))
        if key in ("N", "d", "causal"):
            cur[key] = int(val)
        elif key == "scale":
            cur[key] = float(eval(val, env))
        else:
            rows = [[float(eval(x, env)) for x in r.split(",")] for r in val.split(";")]
            cur[key] = np.array(rows, dtype=np.float64)
    return cases


def _rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


def _rand(seed, B, H, N, d, s=1.0):
    g = _rng(seed)
    return (s * g.standard_normal((B, H, N, d)), s * g.standard_normal((B, H, N, d)),
            s * g.standard_normal((B, H, N, d)))


@pytest.mark.parametrize("case", _parse_golden(GOLDEN), ids=lambda c: c["name"])
def test_worked_examples(oracle_mod, case):
    N, d = case["N"], case["d"]
    q = case["Q"].reshape(1, 1, N, d)
    k = case["K"].reshape(1, 1, N, d)
    v = case["V"].reshape(1, 1, N, d)
    o, lse = oracle_mod.attn_fwd(q, k, v, case["scale"], bool(case["causal"]))
    np.testing.assert_allclose(o[0, 0], case["O"].reshape(N, d), rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse[0, 0], case["LSE"].reshape(N), rtol=0, atol=1e-14)
    # the streaming loop and the row list give the same numbers
    o2, lse2 = oracle_mod.attn_online(q, k, v, case["scale"], bool(case["causal"]), chunk=1)
    np.testing.assert_allclose(o2, o, rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse2, lse, rtol=0, atol=1e-14)
    o3, lse3 = oracle_mod.attn_rows(q, k, v, np.arange(N), case["scale"], bool(case["causal"]))
    np.testing.assert_array_equal(o3, o[0, 0])
    np.testing.assert_array_equal(lse3, lse[0, 0])


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,d", [(1, 4), (5, 3), (64, 16), (200, 64), (256, 128)])
def test_matches_library_sdpa(oracle_mod, causal, N, d):
    """Independent library routine: torch's CPU fp64 scaled_dot_product_attention,
    and scipy's logsumexp of the scores for LSE."""
    torch = pytest.importorskip("torch")
    scipy_special = pytest.importorskip("scipy.special")
    B, H = 2, 3
    q, k, v = _rand(1000 + N * 7 + d + causal, B, H, N, d)
    scale = 1.0 / math.sqrt(d)
    o, lse = oracle_mod.attn_fwd(q, k, v, scale, causal)
    tq, tk, tv = (torch.from_numpy(x) for x in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(
        tq, tk, tv, is_causal=causal, scale=scale).numpy()
    np.testing.assert_allclose(o, ref, rtol=0, atol=1e-12)
    s = np.einsum("bhic,bhjc->bhij", q, k) * scale
    if causal:
        s = np.where(np.tril(np.ones((N, N), bool)), s, -np.inf)
    np.testing.assert_allclose(lse, scipy_special.logsumexp(s, axis=-1), rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_single_key_and_first_row(oracle_mod, causal):
    """N = 1: O = V[0], LSE = S[0,0]. Under the causal mask the same holds for
    row 0 at any N (it sees key 0 only)."""
    q, k, v = _rand(7, 1, 2, 1, 8)
    o, lse = oracle_mod.attn_fwd(q, k, v, 0.3, causal)
    np.testing.assert_allclose(o[:, :, 0], v[:, :, 0], rtol=0, atol=1e-15)
    np.testing.assert_allclose(lse[:, :, 0], 0.3 * np.sum(q[:, :, 0] * k[:, :, 0], -1),
                               rtol=0, atol=1e-14)
    if causal:
        q, k, v = _rand(8, 1, 2, 50, 8)
        o, lse = oracle_mod.attn_fwd(q, k, v, 0.3, True)
        np.testing.assert_allclose(o[:, :, 0], v[:, :, 0], rtol=0, atol=1e-15)
        np.testing.assert_allclose(lse[:, :, 0], 0.3 * np.sum(q[:, :, 0] * k[:, :, 0], -1),
                                   rtol=0, atol=1e-14)


@pytest.mark.parametrize("causal", [False, True])
def test_probability_rows_sum_to_one(oracle_mod, causal):
    g = _rng(11)
    N, d = 97, 32
    q, k = 2.0 * g.standard_normal((N, d)), 2.0 * g.standard_normal((N, d))
    p = oracle_mod.attn_probs(q, k, 1 / math.sqrt(d), causal)
    assert np.all(p >= 0)
    np.testing.assert_allclose(p.sum(axis=1), 1.0, rtol=0, atol=1e-14)
    if causal:
        assert np.all(p[np.triu_indices(N, 1)] == 0.0)
    # O from P matches the forward entry point (P V is the last line of the definition)
    v = g.standard_normal((N, d))
    o, _ = oracle_mod.attn_fwd(q[None, None], k[None, None], v[None, None], 1 / math.sqrt(d), causal)
    np.testing.assert_allclose(o[0, 0], p @ v, rtol=0, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_constant_values(oracle_mod, causal):
    """V[j] = u for every key j gives O[i] = u for every query i."""
    B, H, N, d = 1, 2, 130, 16
    q, k, _ = _rand(12, B, H, N, d, s=2.0)
    u = _rng(13).standard_normal(d)
    v = np.broadcast_to(u, (B, H, N, d)).copy()
    o, _ = oracle_mod.attn_fwd(q, k, v, 0.25, causal)
    np.testing.assert_allclose(o, v, rtol=0, atol=1e-14)


@pytest.mark.parametrize("causal", [False, True])
def test_zero_keys(oracle_mod, causal):
    """K = 0: every score is 0, so O[i] is the mean of the visible V rows and
    LSE_i = ln(number of visible keys): N, or i + 1 under the causal mask."""
    B, H, N, d = 2, 1, 77, 8
    q, _, v = _rand(14, B, H, N, d)
    k = np.zeros_like(q)
    o, lse = oracle_mod.attn_fwd(q, k, v, 0.5, causal)
    if causal:
        counts = np.arange(1, N + 1, dtype=np.float64)
        mean = np.cumsum(v, axis=2) / counts[:, None]
        np.testing.assert_allclose(lse, np.broadcast_to(np.log(counts), lse.shape), rtol=0, atol=1e-14)
    else:
        mean = np.broadcast_to(v.mean(axis=2, keepdims=True), v.shape)
        np.testing.assert_allclose(lse, math.log(N), rtol=0, atol=1e-14)
    np.testing.assert_allclose(o, mean, rtol=0, atol=1e-13)


def test_key_value_permutation(oracle_mod):
    """Without a mask, permuting K and V rows together changes nothing."""
    B, H, N, d = 1, 2, 60, 8
    q, k, v = _rand(15, B, H, N, d)
    perm = _rng(16).permutation(N)
    o, lse = oracle_mod.attn_fwd(q, k, v, 0.4, False)
    o2, lse2 = oracle_mod.attn_fwd(q, k[:, :, perm], v[:, :, perm], 0.4, False)
    np.testing.assert_allclose(o2, o, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse2, lse, rtol=0, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_shift_of_keys(oracle_mod, causal):
    """Adding u to every K row adds scale·<Q[i], u> to every score of row i:
    O is unchanged and LSE_i moves by exactly that amount. u is large, so the
    shifted scores reach several hundred: without the max subtraction the
    exponentials would overflow."""
    B, H, N, d = 1, 2, 40, 8
    q, k, v = _rand(17, B, H, N, d)
    u = 60.0 * _rng(18).standard_normal(d)
    scale = 0.9
    o, lse = oracle_mod.attn_fwd(q, k, v, scale, causal)
    o2, lse2 = oracle_mod.attn_fwd(q, k + u, v, scale, causal)
    shift = scale * (q @ u)
    assert np.max(np.abs(shift)) > 300.0
    np.testing.assert_allclose(o2, o, rtol=0, atol=1e-11)
    np.testing.assert_allclose(lse2, lse + shift, rtol=1e-13, atol=1e-11)


def test_linear_in_values(oracle_mod):
    B, H, N, d = 1, 1, 33, 8
    q, k, v = _rand(19, B, H, N, d)
    o, lse = oracle_mod.attn_fwd(q, k, v, 0.4, True)
    o2, lse2 = oracle_mod.attn_fwd(q, k, 2.0 * v - 1.0, 0.4, True)
    np.testing.assert_allclose(o2, 2.0 * o - 1.0, rtol=0, atol=1e-13)
    np.testing.assert_array_equal(lse2, lse)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("chunk", [1, 7, 64, 128, 1000])
def test_online_equals_definition(oracle_mod, causal, chunk):
    """The chunked running-max/running-sum loop gives the definition's result
    up to fp64 rounding ("Mini FlashAttention", §4; the surrogate-output
    paragraph of "How Did I Write My First FlashAttention Kernel in CUDA?")."""
    B, H, N, d = 1, 3, 300, 32
    q, k, v = _rand(20 + chunk, B, H, N, d, s=1.5)
    o, lse = oracle_mod.attn_fwd(q, k, v, 1 / math.sqrt(d), causal)
    o2, lse2 = oracle_mod.attn_online(q, k, v, 1 / math.sqrt(d), causal, chunk)
    np.testing.assert_allclose(o2, o, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse2, lse, rtol=1e-13, atol=1e-13)


def test_row_subset_and_thread_count(oracle_mod):
    """Selected rows equal the same rows of the full run, bit for bit, whatever
    the thread count."""
    B, H, N, d = 2, 2, 150, 16
    q, k, v = _rand(30, B, H, N, d)
    o, lse = oracle_mod.attn_fwd(q, k, v, 0.25, True, nthreads=1)
    o4, lse4 = oracle_mod.attn_fwd(q, k, v, 0.25, True, nthreads=4)
    np.testing.assert_array_equal(o4, o)
    np.testing.assert_array_equal(lse4, lse)
    rows = np.array([0, 149, 150, 299, 451, 599])
    orow, lrow = oracle_mod.attn_rows(q, k, v, rows, 0.25, True, nthreads=3)
    np.testing.assert_array_equal(orow, o.reshape(-1, d)[rows])
    np.testing.assert_array_equal(lrow, lse.reshape(-1)[rows])


def test_bad_arguments(oracle_mod):
    q = np.zeros((1, 1, 4, 2))
    with pytest.raises(RuntimeError):
        oracle_mod.attn_rows(q, q, q, np.array([4]), 1.0, False)
    with pytest.raises(RuntimeError):
        oracle_mod.attn_online(q, q, q, 1.0, False, chunk=0)
