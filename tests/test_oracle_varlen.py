"""Pins for the oracle's variable-length entry point (sequences of their own
query and key lengths, token-major [total, H, d], causal mask aligned at the
last query and the last key of each sequence). Each test checks it against
something other than itself: the square oracle (pinned in test_oracle.py),
torch's CPU fp64 scaled_dot_product_attention with an explicit mask, scipy's
logsumexp, closed forms, and the independence of sequences."""
import math

import numpy as np
import pytest


def _rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


def _batch(seed, nq, nk, H, d):
    g = _rng(seed)
    cu_q = np.concatenate([[0], np.cumsum(nq)]).astype(np.int64)
    cu_k = np.concatenate([[0], np.cumsum(nk)]).astype(np.int64)
    q = g.standard_normal((cu_q[-1], H, d))
    k = g.standard_normal((cu_k[-1], H, d))
    v = g.standard_normal((cu_k[-1], H, d))
    return q, k, v, cu_q, cu_k


def _visible(nq, nk, causal):
    """[nq, nk] boolean: key j visible to query i (bottom-right causal)."""
    if not causal:
        return np.ones((nq, nk), bool)
    i = np.arange(nq)[:, None]
    j = np.arange(nk)[None, :]
    return j <= i + (nk - nq)


@pytest.mark.parametrize("causal", [False, True])
def test_equal_lengths_match_the_square_oracle(oracle_mod, causal):
    B, H, N, d = 3, 2, 70, 16
    q, k, v, cu_q, cu_k = _batch(11, [N] * B, [N] * B, H, d)
    o, lse = oracle_mod.attn_varlen(q, k, v, cu_q, cu_k, 0.25, causal)
    sq = lambda x: x.reshape(B, N, H, d).transpose(0, 2, 1, 3)  # noqa: E731
    o_sq, lse_sq = oracle_mod.attn_fwd(sq(q), sq(k), sq(v), 0.25, causal)
    np.testing.assert_allclose(sq(o), o_sq, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse.reshape(H, B, N).transpose(1, 0, 2), lse_sq, rtol=0, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_matches_library_sdpa_with_explicit_mask(oracle_mod, causal):
    """Nq < Nk, Nq > Nk (queries that see nothing), an empty sequence and a
    single-query (decode) sequence, against torch's fp64 SDPA with the
    bottom-right mask written out, and scipy's logsumexp for LSE."""
    torch = pytest.importorskip("torch")
    scipy_special = pytest.importorskip("scipy.special")
    nq, nk = [5, 40, 0, 1, 33], [17, 9, 4, 30, 33]
    H, d = 3, 8
    q, k, v, cu_q, cu_k = _batch(12 + causal, nq, nk, H, d)
    scale = 1.0 / math.sqrt(d)
    o, lse = oracle_mod.attn_varlen(q, k, v, cu_q, cu_k, scale, causal)
    for b in range(len(nq)):
        qs, ks, vs = q[cu_q[b]:cu_q[b + 1]], k[cu_k[b]:cu_k[b + 1]], v[cu_k[b]:cu_k[b + 1]]
        if nq[b] == 0:
            continue
        vis = _visible(nq[b], nk[b], causal)
        has = vis.any(axis=1)
        tq, tk, tv = (torch.from_numpy(x.transpose(1, 0, 2).copy()) for x in (qs, ks, vs))
        ref = torch.nn.functional.scaled_dot_product_attention(
            tq, tk, tv, attn_mask=torch.from_numpy(vis), scale=scale).numpy().transpose(1, 0, 2)
        got = o[cu_q[b]:cu_q[b + 1]]
        np.testing.assert_allclose(got[has], ref[has], rtol=0, atol=1e-12)
        np.testing.assert_array_equal(got[~has], 0.0)
        s = np.einsum("ihc,jhc->hij", qs, ks) * scale
        s = np.where(vis[None], s, -np.inf)
        want = scipy_special.logsumexp(s, axis=-1) if has.all() else None
        got_l = lse[:, cu_q[b]:cu_q[b + 1]]
        if want is not None:
            np.testing.assert_allclose(got_l, want, rtol=0, atol=1e-12)
        else:
            np.testing.assert_allclose(got_l[:, has], scipy_special.logsumexp(s[:, has], axis=-1),
                                       rtol=0, atol=1e-12)
            assert np.all(np.isneginf(got_l[:, ~has]))


def test_decode_query_sees_every_key(oracle_mod):
    """One query against Nk keys: the causal mask aligned at the last key
    hides nothing."""
    q, k, v, cu_q, cu_k = _batch(13, [1, 1], [50, 7], 2, 16)
    o1, l1 = oracle_mod.attn_varlen(q, k, v, cu_q, cu_k, 0.2, True)
    o0, l0 = oracle_mod.attn_varlen(q, k, v, cu_q, cu_k, 0.2, False)
    np.testing.assert_array_equal(o1, o0)
    np.testing.assert_array_equal(l1, l0)


def test_zero_keys_give_prefix_means(oracle_mod):
    """K = 0: every visible score is 0, so O is the mean of the visible V rows
    and LSE = ln(number of visible keys)."""
    nq, nk = [6, 3], [4, 8]
    q, k, v, cu_q, cu_k = _batch(14, nq, nk, 2, 4)
    k[:] = 0.0
    o, lse = oracle_mod.attn_varlen(q, k, v, cu_q, cu_k, 0.7, True)
    for b in range(2):
        vis = _visible(nq[b], nk[b], True)
        vs = v[cu_k[b]:cu_k[b + 1]]
        for i in range(nq[b]):
            n = int(vis[i].sum())
            row = o[cu_q[b] + i]
            if n == 0:
                np.testing.assert_array_equal(row, 0.0)
                assert np.all(np.isneginf(lse[:, cu_q[b] + i]))
            else:
                np.testing.assert_allclose(row, vs[:n].mean(axis=0), rtol=0, atol=1e-14)
                np.testing.assert_allclose(lse[:, cu_q[b] + i], math.log(n), rtol=0, atol=1e-14)


def test_sequences_are_independent(oracle_mod):
    """Changing one sequence's keys and values leaves the others unchanged."""
    q, k, v, cu_q, cu_k = _batch(15, [9, 12, 4], [9, 20, 6], 2, 8)
    o, lse = oracle_mod.attn_varlen(q, k, v, cu_q, cu_k, 0.4, True)
    k2, v2 = k.copy(), v.copy()
    k2[cu_k[1]:cu_k[2]] += 3.0
    v2[cu_k[1]:cu_k[2]] *= -2.0
    o2, lse2 = oracle_mod.attn_varlen(q, k2, v2, cu_q, cu_k, 0.4, True)
    for b in (0, 2):
        sl = slice(cu_q[b], cu_q[b + 1])
        np.testing.assert_array_equal(o2[sl], o[sl])
        np.testing.assert_array_equal(lse2[:, sl], lse[:, sl])
    assert not np.allclose(o2[cu_q[1]:cu_q[2]], o[cu_q[1]:cu_q[2]])


def test_bad_offsets_are_rejected(oracle_mod):
    q, k, v, cu_q, cu_k = _batch(16, [3, 3], [3, 3], 1, 4)
    with pytest.raises(ValueError):
        oracle_mod.attn_varlen(q, k, v, cu_q[:-1], cu_k, 1.0, False)
    bad = cu_q.copy()
    bad[1] = 4
    bad[2] = 3
    with pytest.raises((ValueError, RuntimeError)):
        oracle_mod.attn_varlen(q, k, v, bad, cu_k, 1.0, False)
