"""The forward entry points captured into CUDA graphs (torch.cuda.graph):
a replay gives the same bits as an ordinary call, graphs replayed on two
streams at once do not disturb each other, and a capture made before any
ordinary call on the device is refused without enqueuing anything."""
import math
import os
import subprocess
import sys

import numpy as np
import pytest

from exact_attention_91_gb300 import inputs as fin

from .parity_util import to_device

pytestmark = pytest.mark.gpu

DENSE = [
    # (B, H, N, d, causal): a ragged causal case, a non-causal one with few
    # units (they run as half units), d=128
    (2, 4, 1000, 64, True),
    (1, 8, 4096, 64, False),
    (2, 2, 777, 128, False),
]


def _torch():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch


def _dense_inputs(B, H, N, d, seed):
    w = fin.custom(B, H, N, d, False, seed=seed)
    x = fin.make_inputs(w)
    return to_device(x.q), to_device(x.k), to_device(x.v)


def _capture(torch, fn):
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(g, stream=side):
        fn()
    torch.cuda.synchronize()
    return g


@pytest.mark.parametrize("case", range(len(DENSE)))
def test_captured_dense_call_matches_ordinary_call(case):
    torch = _torch()
    import exact_attention_91_gb300 as fa
    B, H, N, d, causal = DENSE[case]
    q, k, v = _dense_inputs(B, H, N, d, seed=900 + case)
    o_ref, lse_ref = fa.attention_forward(q, k, v, causal=causal)
    o = torch.full_like(q, float("nan"))
    lse = torch.full_like(lse_ref, float("nan"))
    g = _capture(torch, lambda: fa.attention_forward(q, k, v, causal=causal, out=o, lse=lse))
    for _ in range(2):
        o.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)
    assert fa.fa_device_status() == (0, 0)


def test_captured_varlen_and_noalloc_calls_match_ordinary_calls():
    torch = _torch()
    import exact_attention_91_gb300 as fa
    # decode of two sequences against long key sets: a cluster split
    x = fin.make_varlen_inputs([1, 3], [20000, 9000], 4, 128, seed=931)
    q, k, v = to_device(x.q), to_device(x.k), to_device(x.v)
    cu_q, cu_k = torch.from_numpy(x.cu_q).cuda(), torch.from_numpy(x.cu_k).cuda()
    o_ref, lse_ref = fa.attention_forward_varlen(q, k, v, cu_q, cu_k, 3, causal=True)
    o, lse = torch.empty_like(o_ref), torch.empty_like(lse_ref)
    g = _capture(torch, lambda: fa.attention_forward_varlen(q, k, v, cu_q, cu_k, 3, causal=True, out=o, lse=lse))
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)

    qd, kd, vd = _dense_inputs(1, 4, 1500, 128, seed=932)
    od_ref, lsed_ref = fa.attention_forward(qd, kd, vd, causal=True)
    od, lsed = torch.empty_like(od_ref), torch.empty_like(lsed_ref)
    sc = 1.0 / math.sqrt(128)

    def noalloc():
        s = torch.cuda.current_stream()
        rc = fa.fa_fwd_noalloc(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), od.data_ptr(), lsed.data_ptr(),
                               1, 4, 1500, 128, sc, True, s.cuda_stream)
        assert rc == 0, rc

    noalloc()  # an ordinary call first: the entry point's own first-call lookup
    torch.cuda.synchronize()
    g2 = _capture(torch, noalloc)
    od.zero_()
    g2.replay()
    torch.cuda.synchronize()
    assert torch.equal(od, od_ref) and torch.equal(lsed, lsed_ref)
    assert fa.fa_device_status() == (0, 0)


def test_graphs_replayed_on_two_streams_at_once():
    """Each captured launch has a work-queue slot of its own, so replays on
    different streams may overlap on the GPU. Every buffer a graph reads or
    writes is kept alive while it may be replayed (torch.cuda.graph empties
    the allocator cache when a capture begins, so a freed input would be
    unmapped)."""
    torch = _torch()
    import exact_attention_91_gb300 as fa
    shapes = [(1, 8, 2048, 128, True), (2, 4, 1500, 64, False)]
    runs = []
    for i, (B, H, N, d, causal) in enumerate(shapes):
        q, k, v = _dense_inputs(B, H, N, d, seed=940 + i)
        o_ref, lse_ref = fa.attention_forward(q, k, v, causal=causal)
        o, lse = torch.empty_like(o_ref), torch.empty_like(lse_ref)
        g = _capture(torch, lambda q=q, k=k, v=v, o=o, lse=lse, c=causal:
                     [fa.attention_forward(q, k, v, causal=c, out=o, lse=lse) for _ in range(4)])
        runs.append((g, o, lse, o_ref, lse_ref, (q, k, v)))
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    torch.cuda.synchronize()
    for _ in range(5):
        for (g, *_), s in zip(runs, streams):
            with torch.cuda.stream(s):
                g.replay()
    torch.cuda.synchronize()
    for g, o, lse, o_ref, lse_ref, _ in runs:
        assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)
    assert fa.fa_device_status() == (0, 0)


CHILD = r"""
import sys, torch
import exact_attention_91_gb300 as fa
q = torch.zeros((1, 1, 256, 64), dtype=torch.bfloat16, device="cuda")
o = torch.empty_like(q)
lse = torch.empty((1, 1, 256), dtype=torch.float32, device="cuda")
g = torch.cuda.CUDAGraph()
err = None
with torch.cuda.graph(g):
    try:
        fa.attention_forward(q, q, q, out=o, lse=lse)
    except fa.FaError as e:
        err = e.status
print("captured-first", err)
o2, _ = fa.attention_forward(q, q, q)   # an ordinary call still works afterwards
torch.cuda.synchronize()
print("ordinary", bool(torch.isfinite(o2.float()).all()))
"""


def test_capture_before_any_ordinary_call_is_refused():
    _torch()
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, PYTHONPATH=root + os.pathsep + os.environ.get("PYTHONPATH", ""))
    r = subprocess.run([sys.executable, "-c", CHILD], capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    assert "captured-first -7" in r.stdout, r.stdout
    assert "ordinary True" in r.stdout, r.stdout
