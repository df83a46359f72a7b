"""The C-ABI library without a GPU: it builds, loads, exports every function
that include/fa.h declares, and rejects bad arguments before touching CUDA."""
import ctypes
import os
import re
import shutil

import pytest

import exact_attention_91_gb300 as fa
from exact_attention_91_gb300 import build as fa_build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "fa.h")


def _declared_functions():
    text = open(HEADER, encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[a-z_ ]+\**\s*\**\s*(fa_[a-z_0-9]+)\s*\(", text, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    if not fa_build.up_to_date():
        if shutil.which(fa_build.nvcc_path()) is None and not os.path.exists(fa_build.nvcc_path()):
            pytest.skip("nvcc not available to build libfa.so")
        fa_build.build()
    return fa.load_library()


def test_header_declares_the_entry_points():
    assert _declared_functions() == sorted(fa.EXPORTED_SYMBOLS)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name
    assert fa.fa_abi_version() == 1


def test_strerror_covers_every_code(lib):
    for code in range(0, -11, -1):
        msg = fa.fa_strerror(code)
        assert msg and "unknown" not in msg
    assert "unknown" in fa.fa_strerror(-99)


P = 1 << 20  # a 16-byte-aligned fake address; never dereferenced by these calls


def _call(q=P, k=2 * P, v=3 * P, o=4 * P, lse=5 * P, B=1, H=1, N=128, d=64, scale=0.125,
          causal=0):
    return fa.fa_fwd(q, k, v, o, lse, B, H, N, d, scale, causal, None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=0), -1), (dict(k=0), -1), (dict(v=0), -1), (dict(o=0), -1),
    (dict(B=0), -2), (dict(H=0), -2), (dict(N=0), -2), (dict(N=-5), -2),
    (dict(B=1 << 16, H=1 << 16), -2),
    (dict(d=32), -3), (dict(d=96), -3), (dict(d=256), -3),
    (dict(q=P + 8), -4), (dict(o=4 * P + 2), -4), (dict(lse=5 * P + 2), -4),
    (dict(scale=0.0), -9), (dict(scale=-1.0), -9), (dict(scale=float("inf")), -9),
    (dict(scale=float("nan")), -9),
    (dict(o=P), -10), (dict(o=P + 64 * 128), -10), (dict(lse=4 * P + 16), -10),
])
def test_bad_arguments_are_rejected_before_launch(lib, kw, code):
    assert _call(**kw) == code


def test_valid_call_without_gpu_reports_no_device(lib):
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert _call() == -5
    assert _call(lse=0) == -5
    assert lib.fa_selftest_wait_timeout(None, 1_000_000) == -5


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(FileNotFoundError):
        fa.load_library(str(tmp_path / "libfa.so"))


def test_varlen_bad_arguments_are_rejected_before_launch(lib):
    """fa_fwd_varlen validates on the host before it looks for a device."""
    p = 1 << 20  # aligned stand-in pointers; nothing is dereferenced on these paths
    f = lib.fa_fwd_varlen
    #          q  k  v  o        lse   cu_q  cu_k  B  H  tq tk  mq  d    scale causal stream
    assert f(p, p, p, p + 4096, None, p, p, 0, 2, 8, 8, 8, 64, 0.125, 0, None) == -2   # B < 1
    assert f(p, p, p, p + 4096, None, p, p, 1, 2, 8, 8, 9, 64, 0.125, 0, None) == -2   # max_seqlen_q > total_q
    assert f(p, p, p, p + 4096, None, None, p, 1, 2, 8, 8, 8, 64, 0.125, 0, None) == -1
    assert f(None, p, p, p + 4096, None, p, p, 1, 2, 8, 8, 8, 64, 0.125, 0, None) == -1
    assert f(p, p, p, p + 4096, None, p, p, 1, 2, 8, 8, 8, 96, 0.125, 0, None) == -3
    assert f(p, p, p, p + 4096, None, p, p, 1, 2, 8, 8, 8, 64, 0.0, 0, None) == -9
    assert f(p + 2, p, p, p + 4096, None, p, p, 1, 2, 8, 8, 8, 64, 0.125, 0, None) == -4
    assert f(p, p, p, p + 64, None, p, p, 1, 2, 8, 8, 8, 64, 0.125, 0, None) == -10  # o overlaps q


def test_varlen_split_choice(lib):
    """fa_varlen_num_splits (host only): the key range of a unit is split only
    when the units are too few for the SMs and the key sets are long, and
    every split keeps at least 4 key tiles of 128."""
    f = lib.fa_varlen_num_splits
    #        B   H   total_k        max_seqlen_q  SMs
    assert f(64, 32, 64 * 8192, 1, 152) == 1        # decode, 2048 (sequence, head) pairs: enough units
    assert f(16, 32, 16 * 4096, 4096, 152) == 1     # prefill-sized units
    assert f(1, 8, 32768, 1, 152) > 4               # 8 pairs of one query and 32768 keys
    assert f(2, 4, 2 * 896, 1, 152) == 1            # short key sets: fewer than 8 tiles per sequence
    for B, H, nk in [(1, 8, 32768), (4, 4, 6000), (1, 2, 3000), (2, 1, 1 << 20)]:
        sp = f(B, H, B * nk, 1, 152)
        assert 1 <= sp <= 64 and (sp == 1 or -(-nk // 128) // sp >= 4), (B, H, nk, sp)
    # splits fill more SMs: 8 units never split into fewer than 152 items' worth of tiles
    assert f(1, 8, 32768, 1, 152) * 8 <= 2 * 152
    assert f(0, 8, 100, 1, 152) == -2 and f(1, 8, 100, 1, 0) == -2 and f(1, 8, -1, 1, 152) == -2
