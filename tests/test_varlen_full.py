"""fa_fwd_varlen on the variable-length bench workloads at full size, in the
launch configuration bench.py times (same batch, seeds, scale and mask), on
sampled query rows that the fp64 oracle computes one by one.

prefill_mix: 16 causal sequences (Nq = Nk) of lengths drawn from U{256..8192};
a row of sequence b, head h is row i of the single-head problem made of that
sequence's tokens. decode_long: 2 sequences of one query against 65536 keys,
each unit's key range split and merged; the query sees every key, so it is
row 0 of a non-causal single-head problem whose other query rows are unused.
"""
import math

import numpy as np
import pytest

import bench
from exact_attention_91_gb300 import inputs as fin

from .parity_util import LSE_MAX_ABS, O_MAX_ABS, O_MEAN_ABS, o_to_numpy, to_device

pytestmark = pytest.mark.gpu


def _run_bench_batch(name):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import exact_attention_91_gb300 as fa
    sq, sk, H, d, causal = bench.varlen_batch(name)
    x = fin.make_varlen_inputs(sq, sk, H, d, seed=fin.SEED_BASE + 71)  # the bench's inputs
    q, k, v = to_device(x.q), to_device(x.k), to_device(x.v)
    cu_q, cu_k = torch.from_numpy(x.cu_q).cuda(), torch.from_numpy(x.cu_k).cuda()
    o, lse = fa.attention_forward_varlen(q, k, v, cu_q, cu_k, max(sq), causal=causal, scale=1.0 / math.sqrt(d))
    torch.cuda.synchronize()
    assert fa.fa_device_status() == (0, 0)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    nsplit = fa.fa_varlen_num_splits(len(sq), H, k.shape[0], max(sq), sms)
    return x, sq, sk, H, d, causal, o_to_numpy(o), lse.cpu().numpy().astype(np.float64), nsplit


def _compare(got_o, got_lse, ref_o, ref_lse):
    d_o = np.abs(got_o - ref_o)
    print("O max", d_o.max(), "mean", d_o.mean(), "LSE max", np.abs(got_lse - ref_lse).max())
    assert np.isfinite(got_o).all() and np.isfinite(got_lse).all()
    assert d_o.max() <= O_MAX_ABS and d_o.mean() <= O_MEAN_ABS
    assert np.abs(got_lse - ref_lse).max() <= LSE_MAX_ABS


def test_prefill_mix_sampled_rows(oracle_mod):
    x, sq, sk, H, d, causal, o, lse, _ = _run_bench_batch("prefill_mix")
    rng = np.random.Generator(np.random.PCG64(71))
    order = np.argsort(sq)
    seqs = sorted({int(order[0]), int(order[-1]), *(int(b) for b in rng.choice(len(sq), 2, replace=False))})
    got_o, got_l, ref_o, ref_l = [], [], [], []
    for b in seqs:
        n = sq[b]
        q0, k0 = int(x.cu_q[b]), int(x.cu_k[b])
        # first and last rows, both sides of the first tile boundaries, and random rows
        rows = np.unique(np.concatenate([[0, 1, 127, 128, 255, 256, n - 129, n - 128, n - 1],
                                         rng.integers(0, n, 40)]).clip(0, n - 1))
        for h in rng.choice(H, 3, replace=False):
            qs = fin.bf16_to_f64(x.q[q0:q0 + n, h])[None, None]
            ks = fin.bf16_to_f64(x.k[k0:k0 + n, h])[None, None]
            vs = fin.bf16_to_f64(x.v[k0:k0 + n, h])[None, None]
            r_o, r_l = oracle_mod.attn_rows(qs, ks, vs, rows, 1.0 / math.sqrt(d), causal)
            ref_o.append(r_o)
            ref_l.append(r_l)
            got_o.append(o[q0 + rows, h])
            got_l.append(lse[h, q0 + rows])
    _compare(np.concatenate(got_o), np.concatenate(got_l), np.concatenate(ref_o), np.concatenate(ref_l))


def test_decode_long_sampled_heads(oracle_mod):
    x, sq, sk, H, d, causal, o, lse, nsplit = _run_bench_batch("decode_long")
    assert nsplit > 1  # this launch configuration splits every unit's key range
    got_o, got_l, ref_o, ref_l = [], [], [], []
    for b in range(len(sq)):
        nk = sk[b]
        q0, k0 = int(x.cu_q[b]), int(x.cu_k[b])
        for h in range(0, H, 4):
            qs = np.zeros((1, 1, nk, d))
            qs[0, 0, 0] = fin.bf16_to_f64(x.q[q0, h])
            ks = fin.bf16_to_f64(x.k[k0:k0 + nk, h])[None, None]
            vs = fin.bf16_to_f64(x.v[k0:k0 + nk, h])[None, None]
            r_o, r_l = oracle_mod.attn_rows(qs, ks, vs, np.array([0]), 1.0 / math.sqrt(d), False)
            ref_o.append(r_o)
            ref_l.append(r_l)
            got_o.append(o[q0:q0 + 1, h])
            got_l.append(lse[h, q0:q0 + 1])
    _compare(np.concatenate(got_o), np.concatenate(got_l), np.concatenate(ref_o), np.concatenate(ref_l))
