"""No call of the library allocates device memory.

The work-queue counters live in a fixed array inside the library, the tail
of an equal-length launch is balanced inside each CTA (half items), and a
variable-length key-range split is merged through the distributed shared
memory of a thread-block cluster; none of them needs scratch memory. The CPU
test reads the library's source for allocation calls; the GPU test reads the
device's free memory around 100 calls of each forward entry point (after one
call of each has done the device's first-call setup), with every buffer
allocated beforehand.
"""
import os
import re

import numpy as np
import pytest

from exact_attention_91_gb300 import inputs as fin

CSRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "exact_attention_91_gb300", "csrc")
ALLOC_CALL = re.compile(r"\b(cudaMalloc\w*|cudaFree\w*|cudaMemPool\w*|cuMemAlloc\w*|cuMemCreate|cudaHostAlloc|"
                        r"cudaMallocHost|malloc|calloc|realloc|free|new|delete)\s*[(\[]")


def test_library_source_calls_no_allocation_routine():
    found = []
    for name in sorted(os.listdir(CSRC)):
        text = open(os.path.join(CSRC, name), encoding="utf-8").read()
        text = re.sub(r"//[^\n]*", "", text)                    # comments say what is not done
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        found += [f"{name}: {m.group(0)}" for m in ALLOC_CALL.finditer(text)]
    assert not found, found


@pytest.mark.gpu
def test_forward_calls_leave_device_memory_unchanged():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import exact_attention_91_gb300 as fa
    from .parity_util import to_device

    w = fin.WORKLOADS["long_sequence"]          # 512 units on the SMs: its last units run as half items
    x = fin.make_inputs(w)
    q, k, v = to_device(x.q), to_device(x.k), to_device(x.v)
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device="cuda")
    xv = fin.make_varlen_inputs([1, 1], [65536, 65536], 32, 128, seed=77)   # decode: a cluster split
    qv, kv, vv = to_device(xv.q), to_device(xv.k), to_device(xv.v)
    ov = torch.empty_like(qv)
    lv = torch.empty((32, qv.shape[0]), dtype=torch.float32, device="cuda")
    cu_q, cu_k = torch.from_numpy(xv.cu_q).cuda(), torch.from_numpy(xv.cu_k).cuda()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert fa.fa_varlen_num_splits(2, 32, kv.shape[0], 1, sms) > 1
    s = torch.cuda.current_stream().cuda_stream

    def calls():
        for rc in (
            fa.fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                      w.B, w.H, w.N, w.d, w.scale, w.causal, s),
            fa.fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                      w.B, w.H, w.N, w.d, w.scale, True, s),
            fa.fa_fwd_varlen(qv.data_ptr(), kv.data_ptr(), vv.data_ptr(), ov.data_ptr(), lv.data_ptr(),
                             cu_q.data_ptr(), cu_k.data_ptr(), 2, 32, qv.shape[0], kv.shape[0], 1, 128,
                             1.0 / np.sqrt(128), True, s),
            fa.fa_fwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                              w.B, w.H, w.N, w.d, w.scale, w.causal, s),
        ):
            assert rc == 0, fa.fa_strerror(rc)

    calls()
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(100):
        calls()
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, (free0, free1)
    assert fa.fa_device_status() == (0, 0)
