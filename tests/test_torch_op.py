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
