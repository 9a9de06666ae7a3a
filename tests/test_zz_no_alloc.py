"""pa_decode_noalloc, called through the C ABI, against the fp64 oracle and
against pa_decode.

pa_decode_noalloc serves callers that cannot allocate device memory where
they decode (an engine that handed all free HBM to its KV pool at start-up, a
plugin whose host framework owns the allocator, code that cannot afford an
allocation that may synchronise the device): it takes no workspace and uses
the library's fixed 64 MiB device scratch instead. Calls in a row on
different batches (a large one, then smaller ones, so that anything a
previous call left in the shared scratch would show) must each match the
oracle within the parity bar and agree with pa_decode; a batch needing more
scratch than the fixed array, or one with a bad argument, is refused before
anything is launched.

Each test sets up everything it uses, so the file passes alone in a fresh
process as well as after the other tests; it is named to be collected last.
"""
import ctypes as C

import numpy as np
import pytest
import torch

from paged_kv_cache_105_gb300 import binding as B
from paged_kv_cache_105_gb300 import workloads as W
from tests.helpers import ATOL, bits, compare, gpu_step, oracle_step, to_dev

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def noalloc_via_cabi(wl, vals, t, err, partition_tokens):
    out = torch.full_like(vals["q"], float("nan"))
    stream = C.c_void_p(torch.cuda.current_stream(DEV).cuda_stream)
    st = B.lib().pa_decode_noalloc(
        C.c_void_p(out.data_ptr()), C.c_void_p(vals["q"].data_ptr()),
        C.c_void_p(vals["k_pool"].data_ptr()), C.c_void_p(vals["v_pool"].data_ptr()),
        C.c_void_p(t["block_tables"].data_ptr()), C.c_void_p(t["seq_lens"].data_ptr()),
        wl.num_seqs, wl.block_tables.shape[1], wl.num_blocks, wl.n_q_heads, wl.n_kv_heads,
        wl.head_dim, wl.block_size, wl.scale, partition_tokens, wl.max_seq_len,
        C.c_void_p(err.data_ptr()), stream)
    assert st == B.PA_OK, B.lib().pa_status_string(st)
    torch.cuda.synchronize()
    return out


BATCHES = [
    # (workload, partition_tokens): large first, then smaller ones
    (lambda: W.config2(), 0),
    (lambda: W.custom([3, 700, 1, 2500, 64], block_size=8, n_q_heads=16, n_kv_heads=2,
                      head_dim=64, seed=31, name="noalloc-small"), 0),
    (lambda: W.custom([40, 1, 900, 0, 17], block_size=32, n_q_heads=8, n_kv_heads=8,
                      head_dim=128, seed=32, name="noalloc-small-fixed"), 64),
]


def test_noalloc_matches_oracle_and_pa_decode_on_calls_in_a_row():
    for make, P in BATCHES:
        wl = make()
        vals_cpu = W.make_values(wl, poison_tails=True)
        ref, kp, vp = oracle_step(wl, vals_cpu)            # the oracle's copy, write, attend
        vals = {k: v.to(DEV) for k, v in vals_cpu.items()}
        err = torch.zeros(1, dtype=torch.int32, device=DEV)
        with_ws, e = gpu_step(wl, vals, partition_tokens=P, err=err)  # writes, then pa_decode
        assert e == 0
        assert np.array_equal(bits(vals["k_pool"]), kp)
        got = noalloc_via_cabi(wl, vals, to_dev(wl, DEV), err, P)
        assert int(err.item()) == 0
        compare(got, ref, wl.name + "-noalloc")
        compare(with_ws, ref, wl.name)
        diff = (got.float() - with_ws.float()).abs().max().item()
        assert diff <= ATOL


def _refused(args):
    st = B.lib().pa_decode_noalloc(*args, C.c_void_p(torch.cuda.current_stream(DEV).cuda_stream))
    torch.cuda.synchronize()
    return st


def test_noalloc_refuses_before_launching():
    wl = W.config5(num_seqs=16, seq_len=32768)
    need = B.pa_decode_workspace_bytes(16, 64, 8, 128, 16, 32768, 64)
    assert need > B.PA_NOALLOC_SCRATCH_BYTES
    # Host-side refusals: nothing is launched, so placeholder buffers suffice;
    # the error word must stay untouched.
    tiny = torch.zeros(16, dtype=torch.int32, device=DEV)
    q = torch.zeros((16, 64, 128), dtype=torch.bfloat16, device=DEV)
    err = torch.full((1,), 12345, dtype=torch.int32, device=DEV)
    p = [C.c_void_p(q.data_ptr())] * 4 + [C.c_void_p(tiny.data_ptr())] * 2
    big = p + [16, 2048, 8, 64, 8, 128, 16, wl.scale, 64, 32768, C.c_void_p(err.data_ptr())]
    assert _refused(big) == B.PA_ERR_INVALID_ARG
    # a length hint beyond the table: refused by the argument checks
    bad = p + [2, 4, 8, 8, 8, 128, 16, wl.scale, 0, 4 * 16 + 1, C.c_void_p(err.data_ptr())]
    assert _refused(bad) == B.PA_ERR_INVALID_ARG
    # a misaligned output pointer
    mis = [C.c_void_p(q.data_ptr() + 2)] + p[1:] + [2, 4, 8, 8, 8, 128, 16, wl.scale, 0, 64,
                                                    C.c_void_p(err.data_ptr())]
    assert _refused(mis) == B.PA_ERR_INVALID_ARG
    assert int(err.item()) == 12345
