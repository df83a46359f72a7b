"""Head-sharded forward (several GPUs, each on a contiguous range of the
flattened B*H heads, no exchange between ranks).

CPU: the partition covers every head once, in order, balanced; two gloo
ranks each compute their range (the fp64 oracle stands in for the per-rank
GPU call) and the gathered shards are the whole problem's result bit for
bit. GPU: calls on the ranges of a partition, made one after the other on one
device, write the same bits as one fa_fwd over all heads."""
import os
import socket

import numpy as np
import pytest

import exact_attention_91_gb300 as fa
from exact_attention_91_gb300 import inputs as fin


@pytest.mark.parametrize("bh,world", [(1, 1), (7, 2), (128, 3), (5, 8), (4096, 7)])
def test_partition_covers_every_head_once_in_order(bh, world):
    shards = fa.head_shards(bh, world)
    assert len(shards) == world
    start = 0
    for s, n in shards:
        assert s == start and n >= 0
        start += n
    assert start == bh
    sizes = [n for _, n in shards]
    assert max(sizes) - min(sizes) <= 1


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch
    import torch.distributed as dist

    import oracle
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = fin.custom(2, 3, 96, 64, True, seed=515)
        x = fin.make_inputs(w)
        BH = w.B * w.H
        start, n = fa.head_shards(BH, world)[rank]
        # this rank's heads only (its own memory), computed without the others
        q, k, v = (a.reshape(BH, w.N, w.d)[start:start + n][None] for a in x.f64())
        o, lse = oracle.attn_fwd(q, k, v, w.scale, w.causal)
        # reassembly: gather every rank's shard (shards differ in size: pad to the largest)
        most = max(c for _, c in fa.head_shards(BH, world))
        pad_o = torch.zeros((most, w.N, w.d), dtype=torch.float64)
        pad_l = torch.zeros((most, w.N), dtype=torch.float64)
        pad_o[:n] = torch.from_numpy(o[0])
        pad_l[:n] = torch.from_numpy(lse[0])
        go = [torch.empty_like(pad_o) for _ in range(world)]
        gl = [torch.empty_like(pad_l) for _ in range(world)]
        dist.all_gather(go, pad_o)
        dist.all_gather(gl, pad_l)
        if rank == 0:
            parts = fa.head_shards(BH, world)
            o_all = np.concatenate([go[r][:c].numpy() for r, (_, c) in enumerate(parts)])
            l_all = np.concatenate([gl[r][:c].numpy() for r, (_, c) in enumerate(parts)])
            o_ref, l_ref = oracle.attn_fwd(*x.f64(), w.scale, w.causal)
            out["same"] = bool(np.array_equal(o_all, o_ref.reshape(BH, w.N, w.d)) and
                               np.array_equal(l_all, l_ref.reshape(BH, w.N)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reassemble_the_whole_result():
    torch = pytest.importorskip("torch")
    world = 2
    ctx = torch.multiprocessing.get_context("spawn")
    out = ctx.Manager().dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(180)
        assert p.exitcode == 0
    assert out.get("same") is True


@pytest.mark.gpu
@pytest.mark.parametrize("shape,world", [((2, 4, 1024, 128, True), 3), ((1, 6, 2048, 64, False), 2),
                                         ((4, 32, 4096, 128, True), 8)])
def test_sharded_calls_equal_one_call(shape, world):
    """Causal launches and launches whose units all run as half units schedule
    every head the same way whatever the head count, so the bits match."""
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from .parity_util import to_device
    B, H, N, d, causal = shape
    x = fin.make_inputs(fin.custom(B, H, N, d, causal, seed=616))
    q, k, v = to_device(x.q), to_device(x.k), to_device(x.v)
    o_ref, l_ref = fa.attention_forward(q, k, v, causal=causal)
    o = torch.full_like(q, float("nan"))
    lse = torch.full_like(l_ref, float("nan"))
    for start, n in fa.head_shards(B * H, world):
        fa.attention_forward_heads(q, k, v, start, n, causal=causal, out=o, lse=lse)
    torch.cuda.synchronize()
    assert torch.equal(o.view(torch.int16), o_ref.view(torch.int16))
    assert torch.equal(lse, l_ref)
