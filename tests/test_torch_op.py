"""The PyTorch custom operators fa91::attention_forward and
fa91::attention_forward_varlen: registered with fake implementations (CPU),
and on the GPU identical to the C-ABI path, also when compiled."""
import pytest

torch = pytest.importorskip("torch")

from exact_attention_91_gb300 import inputs as fin  # noqa: E402
from exact_attention_91_gb300 import torch_op  # noqa: E402,F401  (registers the operator)

from .parity_util import to_device  # noqa: E402


def test_fake_implementation_gives_shapes_without_a_gpu():
    from torch._subclasses.fake_tensor import FakeTensorMode
    with FakeTensorMode():
        q = torch.empty(2, 3, 100, 64, dtype=torch.bfloat16, device="meta")
        o, lse = torch.ops.fa91.attention_forward(q, q, q, True, 0.125)
    assert o.shape == (2, 3, 100, 64) and o.dtype == torch.bfloat16
    assert lse.shape == (2, 3, 100) and lse.dtype == torch.float32


def test_varlen_fake_implementation_gives_shapes_without_a_gpu():
    from torch._subclasses.fake_tensor import FakeTensorMode
    with FakeTensorMode():
        q = torch.empty(300, 4, 128, dtype=torch.bfloat16, device="meta")
        k = torch.empty(900, 4, 128, dtype=torch.bfloat16, device="meta")
        cu = torch.empty(3, dtype=torch.int32, device="meta")
        o, lse = torch.ops.fa91.attention_forward_varlen(q, k, k, cu, cu, 200, True, None)
    assert o.shape == (300, 4, 128) and o.dtype == torch.bfloat16
    assert lse.shape == (4, 300) and lse.dtype == torch.float32


@pytest.mark.gpu
def test_operator_matches_the_c_abi_path():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import exact_attention_91_gb300 as fa
    x = fin.make_inputs(fin.custom(2, 3, 777, 128, True, seed=31))
    q, k, v = to_device(x.q), to_device(x.k), to_device(x.v)
    o1, l1 = torch.ops.fa91.attention_forward(q, k, v, True, None)
    o2, l2 = fa.attention_forward(q, k, v, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(l1, l2)


@pytest.mark.gpu
def test_varlen_operator_matches_the_c_abi_path_and_compiles():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import exact_attention_91_gb300 as fa
    x = fin.make_varlen_inputs([1, 300, 77], [5000, 300, 900], 4, 64, seed=32)
    q, k, v = to_device(x.q), to_device(x.k), to_device(x.v)
    cu_q, cu_k = torch.from_numpy(x.cu_q).cuda(), torch.from_numpy(x.cu_k).cuda()
    o1, l1 = torch.ops.fa91.attention_forward_varlen(q, k, v, cu_q, cu_k, 300, True, None)
    o2, l2 = fa.attention_forward_varlen(q, k, v, cu_q, cu_k, 300, causal=True)

    def f(q, k, v, cu_q, cu_k):
        return torch.ops.fa91.attention_forward_varlen(q, k, v, cu_q, cu_k, 300, True, None)

    o3, l3 = torch.compile(f, fullgraph=True)(q, k, v, cu_q, cu_k)
    torch.cuda.synchronize()
    for o, lse in ((o1, l1), (o3, l3)):
        assert torch.equal(o.view(torch.int16), o2.view(torch.int16))
        assert torch.equal(lse, l2)


@pytest.mark.gpu
@pytest.mark.parametrize("compiled", [False, True])
def test_operator_matches_the_oracle(oracle_mod, compiled):
    """The operator's O and LSE against the fp64 oracle, called eagerly and
    through torch.compile(fullgraph=True), on a ragged causal shape and a
    non-causal one whose last units run as half items."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import numpy as np

    from .parity_util import assert_within, compare, o_to_numpy, visible_keys

    def f(q, k, v, causal, scale):
        return torch.ops.fa91.attention_forward(q, k, v, causal, scale)

    g = torch.compile(f, fullgraph=True) if compiled else f
    for B, H, N, d, causal in ((2, 3, 777, 128, True), (1, 8, 4096, 64, False)):
        w = fin.custom(B, H, N, d, causal, seed=41 + N)
        x = fin.make_inputs(w)
        q, k, v = to_device(x.q), to_device(x.k), to_device(x.v)
        o, lse = g(q, k, v, causal, w.scale)
        torch.cuda.synchronize()
        o_ref, lse_ref = oracle_mod.attn_fwd(*x.f64(), w.scale, causal)
        keys = np.broadcast_to(visible_keys(N, causal, np.arange(N)), lse_ref.shape)
        assert_within(compare(o_to_numpy(o), lse.cpu().numpy(), o_ref, lse_ref,
                              f"op compiled={compiled} {w.name}", keys=keys))


@pytest.mark.gpu
@pytest.mark.parametrize("compiled", [False, True])
def test_varlen_operator_matches_the_oracle(oracle_mod, compiled):
    """fa91::attention_forward_varlen against the oracle, eagerly and
    compiled: a decode query, a ragged pair and a sequence with more queries
    than keys."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import math

    import numpy as np

    from .parity_util import LSE_MAX_ABS, O_MAX_ABS, O_MEAN_ABS, o_to_numpy

    def f(q, k, v, cu_q, cu_k):
        return torch.ops.fa91.attention_forward_varlen(q, k, v, cu_q, cu_k, 400, True, None)

    g = torch.compile(f, fullgraph=True) if compiled else f
    x = fin.make_varlen_inputs([1, 300, 400], [5000, 300, 200], 4, 64, seed=43)
    q, k, v = to_device(x.q), to_device(x.k), to_device(x.v)
    cu_q, cu_k = torch.from_numpy(x.cu_q).cuda(), torch.from_numpy(x.cu_k).cuda()
    o, lse = g(q, k, v, cu_q, cu_k)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle_mod.attn_varlen(*x.f64(), x.cu_q, x.cu_k, 1.0 / math.sqrt(64), True)
    got_o, got_l = o_to_numpy(o), lse.cpu().numpy().astype(np.float64)
    none = np.isneginf(lse_ref)
    np.testing.assert_array_equal(np.isneginf(got_l), none)
    d_o = np.abs(got_o - o_ref)
    assert d_o.max() <= O_MAX_ABS and d_o.mean() <= O_MEAN_ABS, (d_o.max(), d_o.mean())
    assert np.abs(got_l[~none] - lse_ref[~none]).max() <= LSE_MAX_ABS
