"""fa_fwd_varlen (batches of sequences with their own query and key counts,
causal mask aligned at the end of each sequence) against the fp64 oracle."""
import math

import numpy as np
import pytest

from exact_attention_91_gb300 import inputs as fin

from .parity_util import LSE_MAX_ABS, O_MAX_ABS, O_MEAN_ABS, o_to_numpy, to_device

pytestmark = pytest.mark.gpu

CASES = [
    # (seqlens_q, seqlens_k, H, d)
    ([300, 1, 129, 0, 700, 64], [300, 513, 40, 17, 700, 64], 3, 64),
    ([1000, 5, 256, 257], [1000, 900, 128, 300], 2, 128),
    ([1, 1, 1, 1], [4096, 100, 1, 2049], 4, 128),        # decode: one query per sequence
    ([200, 333], [50, 90], 2, 64),                        # more queries than keys
    ([5, 130, 3], [0, 260, 0], 2, 128),                   # sequences without keys
    ([384, 5], [384, 700], 2, 64),                        # last blocks of <= 128 queries
    # few units for the SMs: each unit's key range is split and merged
    ([1, 1], [20000, 9000], 4, 128),                      # decode, long key sets
    ([1, 1, 1], [5000, 16384, 77], 2, 64),                # decode; one key set shorter than a split
    ([3000], [3000], 2, 128),                             # one long sequence (causal: empty splits)
    ([4, 200], [12000, 9000], 2, 64),                     # a few queries against long key sets
    ([1500], [1200], 1, 64),                              # queries that see no key, split
]
SPLIT_CASES = range(6, 11)


def _run(x, H, d, causal):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import exact_attention_91_gb300 as fa
    q, k, v = to_device(x.q), to_device(x.k), to_device(x.v)
    cu_q = torch.from_numpy(x.cu_q).cuda()
    cu_k = torch.from_numpy(x.cu_k).cuda()
    o, lse = fa.attention_forward_varlen(q, k, v, cu_q, cu_k, max(x.seqlens_q), causal=causal,
                                         scale=1.0 / math.sqrt(d))
    torch.cuda.synchronize()
    return o_to_numpy(o), lse.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("case", range(len(CASES)))
def test_varlen_matches_oracle(oracle_mod, case, causal):
    sq, sk, H, d = CASES[case]
    x = fin.make_varlen_inputs(sq, sk, H, d, seed=5150 + case)
    o, lse = _run(x, H, d, causal)
    o_ref, lse_ref = oracle_mod.attn_varlen(*x.f64(), x.cu_q, x.cu_k, 1.0 / math.sqrt(d), causal)
    assert np.isfinite(o).all()
    none = np.isneginf(lse_ref)                      # [H, total_q]: queries that see no key
    np.testing.assert_array_equal(np.isneginf(lse), none)
    assert np.all(o[none.T] == 0.0)
    d_o = np.abs(o - o_ref)
    print(case, causal, "O max", d_o.max(), "mean", d_o.mean())
    assert d_o.max() <= O_MAX_ABS and d_o.mean() <= O_MEAN_ABS
    if (~none).any():
        assert np.abs(lse[~none] - lse_ref[~none]).max() <= LSE_MAX_ABS


def test_split_cases_are_split():
    """The last cases of CASES do run with a split key range on this GPU."""
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import exact_attention_91_gb300 as fa
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for c in SPLIT_CASES:
        sq, sk, H, d = CASES[c]
        assert fa.fa_varlen_num_splits(len(sq), H, sum(sk), max(sq), sms) > 1, c
    assert fa.fa_varlen_num_splits(len(CASES[2][0]), CASES[2][2], sum(CASES[2][1]), 1, sms) > 1


def test_equal_lengths_match_fa_fwd():
    """B sequences of N tokens in the token-major layout give the same rows as
    fa_fwd on the [B, H, N, d] layout (both causal: no key-range split)."""
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import exact_attention_91_gb300 as fa
    B, H, N, d = 3, 2, 777, 128
    x = fin.make_varlen_inputs([N] * B, [N] * B, H, d, seed=77)
    o_v, lse_v = _run(x, H, d, True)
    to_bhnd = lambda a: np.ascontiguousarray(a.reshape(B, N, H, d).transpose(0, 2, 1, 3))  # noqa: E731
    q, k, v = (to_device(to_bhnd(a)) for a in (x.q, x.k, x.v))
    o, lse = fa.attention_forward(q, k, v, causal=True)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(to_bhnd(o_v), o_to_numpy(o))
    np.testing.assert_array_equal(lse_v.reshape(H, B, N).transpose(1, 0, 2), lse.cpu().numpy())


def test_empty_batch_and_validation():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import exact_attention_91_gb300 as fa
    q = torch.zeros((0, 2, 64), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((5, 2, 64), dtype=torch.bfloat16, device="cuda")
    cu = torch.tensor([0, 0], dtype=torch.int32, device="cuda")
    cuk = torch.tensor([0, 5], dtype=torch.int32, device="cuda")
    o, lse = fa.attention_forward_varlen(q, k, k, cu, cuk, 0)
    assert o.shape == (0, 2, 64) and lse.shape == (2, 0)
    rc = fa.fa_fwd_varlen(0, k.data_ptr(), k.data_ptr(), 0, None, cu.data_ptr(), cuk.data_ptr(),
                          1, 2, 0, 5, 3, 64, 0.125, False, None)
    assert rc == -2  # max_seqlen_q > total_q
    rc = fa.fa_fwd_varlen(0, k.data_ptr(), k.data_ptr(), 0, None, cu.data_ptr(), cuk.data_ptr(),
                          1, 2, 4, 5, 3, 64, 0.125, False, None)
    assert rc == -1  # 4 queries but no q / o
