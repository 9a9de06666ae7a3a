"""The C-ABI library loads, exports every function include/pa.h declares,
and rejects bad arguments on the host (no GPU needed for any of this)."""
import ctypes as C
import os
import re

import pytest

from paged_kv_cache_105_gb300 import binding as B
from paged_kv_cache_105_gb300 import build as _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    _build.build()
    return B.lib()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "pa.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w\*]+\s+\**\s*(pa_\w+)\s*\(", text,
                                 flags=re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for fn in ("pa_decode", "pa_reshape_and_cache", "pa_copy_blocks",
               "pa_decode_workspace_bytes", "pa_decode_partition_tokens",
               "pa_status_string", "pa_last_cuda_error"):
        assert fn in names


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), name
    assert set(B.SIGNATURES) == set(declared_functions())


def test_status_strings(L):
    assert L.pa_status_string(0) == b"PA_OK"
    assert L.pa_status_string(1) == b"PA_ERR_INVALID_ARG"
    assert L.pa_status_string(2) == b"PA_ERR_UNSUPPORTED"
    assert L.pa_status_string(3) == b"PA_ERR_CUDA"


def test_partition_choice(L):
    f = L.pa_decode_partition_tokens
    assert f(16, 8, 16, 32768, 512) == 512
    assert f(16, 8, 16, 32768, 100) < 0          # not a multiple of 16
    assert f(16, 8, 32, 32768, 40) < 0           # not a multiple of 16
    assert f(16, 8, 32, 32768, 48) == 48         # may split a 32-token block
    assert f(16, 8, 16, 32768, 128 * 16 + 16) < 0
    assert f(1, 1, 7, 10, 0) < 0                 # unsupported block size
    for args in [(256, 32, 16, 4096), (64, 8, 16, 2048), (5, 8, 16, 1900), (1, 1, 8, 1)]:
        assert f(*args, 0) == 0                  # 0 selects the balanced split


def test_workspace_bytes(L):
    f = L.pa_decode_workspace_bytes
    n = f(16, 64, 8, 128, 16, 32768, 512)
    parts = 32768 // 512
    assert n >= 16 * 64 * parts * (128 * 4 + 8)    # partial O, m and l of every partition
    assert f(16, 64, 8, 96, 16, 32768, 512) == 0      # head_dim 96 unsupported
    assert f(16, 64, 7, 128, 16, 32768, 512) == 0     # heads not divisible
    assert f(16, 64, 2, 128, 16, 32768, 512) == 0     # group of 32 > 16
    assert f(1, 1, 1, 64, 16, 10**6, 64) == 0         # more than 1024 partitions
    # balanced split: two partial slots per CTA (at most 1024 CTAs), whatever
    # the longest sequence
    b = f(16, 64, 8, 128, 16, 32768, 0)
    assert b >= 1024 * 2 * 8 * (128 * 4 + 8)
    assert b == f(16, 64, 8, 128, 16, 512, 0)


# The two tests below pass fake addresses that host validation must reject
# before any launch. They run only where no GPU is present, so that a
# validation bug can never turn into a launch with those addresses.
no_gpu = pytest.mark.skipif(__import__("torch").cuda.is_available(),
                            reason="host-validation tests use fake device addresses")


def _decode(L, **kw):
    args = dict(out=1 << 12, q=1 << 12, k=1 << 12, v=1 << 12, bt=1 << 12, sl=1 << 12, S=2,
                maxb=4, NB=8, Hq=8, Hkv=2, D=128, bs=16, scale=0.1, P=0, maxlen=64,
                ws=1 << 16, wsb=1 << 20, err=None, stream=None)
    args.update(kw)
    a = args
    return L.pa_decode(a["out"], a["q"], a["k"], a["v"], a["bt"], a["sl"], a["S"], a["maxb"],
                       a["NB"], a["Hq"], a["Hkv"], a["D"], a["bs"], a["scale"], a["P"],
                       a["maxlen"], a["ws"], a["wsb"], a["err"], a["stream"])


@no_gpu
def test_decode_host_validation(L):
    INV, UNS = B.PA_ERR_INVALID_ARG, B.PA_ERR_UNSUPPORTED
    assert _decode(L, q=None) == INV
    assert _decode(L, ws=None) == INV
    assert _decode(L, Hq=6, Hkv=4) == INV            # heads not divisible
    assert _decode(L, D=96) == UNS
    assert _decode(L, bs=12) == UNS
    assert _decode(L, Hq=34, Hkv=2) == UNS           # group of 17
    assert _decode(L, P=24) == UNS
    assert _decode(L, maxlen=65) == INV              # beyond 4 blocks of 16
    assert _decode(L, wsb=16) == INV                 # workspace too small
    assert _decode(L, q=(1 << 12) + 2) == INV        # misaligned
    assert _decode(L, ws=(1 << 16) + 16) == INV      # workspace not 256-B aligned
    assert _decode(L, S=-1) == INV
    assert _decode(L, S=0, q=None) == B.PA_OK        # nothing to do, no launch


@no_gpu
def test_cache_calls_host_validation(L):
    INV, UNS = B.PA_ERR_INVALID_ARG, B.PA_ERR_UNSUPPORTED
    p = 1 << 12
    assert L.pa_reshape_and_cache(None, p, p, p, p, 4, 8, 2, 128, 16, None, None) == INV
    assert L.pa_reshape_and_cache(p, p, p, p, p, 4, 8, 2, 80, 16, None, None) == UNS
    assert L.pa_reshape_and_cache(p, p, p, p, p, -1, 8, 2, 128, 16, None, None) == INV
    assert L.pa_reshape_and_cache(p + 8, p, p, p, p, 4, 8, 2, 128, 16, None, None) == INV
    assert L.pa_reshape_and_cache(None, None, None, None, None, 0, 8, 2, 128, 16, None,
                                  None) == B.PA_OK
    assert L.pa_copy_blocks(None, p, p, 3, 2, 128, 16, 8, None, None) == INV
    assert L.pa_copy_blocks(p, p, p, 3, 2, 128, 4, 8, None, None) == UNS
    assert L.pa_copy_blocks(p, p, p, -2, 2, 128, 16, 8, None, None) == INV
    assert L.pa_copy_blocks(None, None, None, 0, 2, 128, 16, 8, None, None) == B.PA_OK


@no_gpu
def test_fp8_calls_host_validation(L):
    INV, UNS = B.PA_ERR_INVALID_ARG, B.PA_ERR_UNSUPPORTED
    p = 1 << 12
    f = L.pa_decode_fp8

    def dec(D=128, ks=0.01, vs=0.01, S=2, q=p):
        return f(p, q, p, p, p, p, S, 4, 8, 8, 2, D, 16, 0.1, ks, vs, 64, 1 << 16, 1 << 20,
                 None, None)

    assert dec(D=64) == UNS                      # fp8 decode: head_dim 128 only
    assert dec(ks=0.0) == INV
    assert dec(vs=float("inf")) == INV
    assert dec(ks=-1.0) == INV
    assert dec(q=None) == INV
    assert dec(S=0) == B.PA_OK
    w = L.pa_reshape_and_cache_fp8
    assert w(p, p, p, p, p, 4, 8, 2, 128, 16, 0.0, 1.0, None, None) == INV
    assert w(p, p, p, p, p, 4, 8, 2, 80, 16, 1.0, 1.0, None, None) == UNS
    assert w(None, None, None, None, None, 0, 8, 2, 128, 16, 1.0, 1.0, None, None) == B.PA_OK
    c = L.pa_copy_blocks_fp8
    assert c(None, p, p, 3, 2, 128, 16, 8, None, None) == INV
    assert c(p, p, p, 3, 2, 128, 4, 8, None, None) == UNS
    assert c(None, None, None, 0, 2, 128, 16, 8, None, None) == B.PA_OK


@no_gpu
def test_prefill_and_swap_host_validation(L):
    INV, UNS = B.PA_ERR_INVALID_ARG, B.PA_ERR_UNSUPPORTED
    p = 1 << 12
    f = L.pa_prefill

    def pre(q=p, cu=p, S=2, TQ=100, Hq=8, Hkv=2, D=128, bs=16, maxq=64, scale=0.1):
        return f(p, q, p, p, p, p, cu, S, TQ, 4, 8, Hq, Hkv, D, bs, scale, maxq, None, None)

    assert pre(D=96) == UNS
    assert pre(bs=12) == UNS
    assert pre(Hq=130, Hkv=2) == UNS             # group of 65 > 64 rows per tile
    assert pre(Hq=6, Hkv=4) == INV
    assert pre(cu=None) == INV
    assert pre(q=p + 2) == INV                   # misaligned
    assert pre(S=0, q=None) == B.PA_OK
    assert pre(maxq=0, q=None) == B.PA_OK
    assert pre(maxq=-1) == INV
    assert pre(TQ=-1) == INV
    assert pre(TQ=0, q=None) == B.PA_OK            # no rows: nothing to do
    assert pre(scale=0.0) == INV                 # the softmax scale must be > 0
    assert pre(scale=-0.1) == INV
    s = L.pa_swap_blocks
    assert s(p, p, p, p, p, 2, 24, 4, 4, None, None) == INV        # block not 16-B multiple
    assert s(p, p, p, p, p, -1, 1024, 4, 4, None, None) == INV
    assert s(None, None, None, None, None, 0, 1024, 4, 4, None, None) == B.PA_OK
    assert s(p, p, p, p, p, 1, 1024, 4, 4, None, None) == INV      # no device to address p
    h = L.pa_copy_host
    assert h(p, p, 0, None) == B.PA_OK                           # nothing to copy
    assert h(None, p, 64, None) == INV
    assert h(p, p, 24, None) == INV                              # not a 16-byte multiple
    assert h(p, p, 64, None) == INV                              # no device to address p
    w = L.pa_check_bounded_wait
    assert w(None, 1000, None) == INV                            # an error word is required
    assert w(p, 0, None) == INV
    assert w(p, 3_000_000_000, None) == INV                      # above the 2 s limit
