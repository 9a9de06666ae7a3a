"""pa_decode_noalloc, called through the C ABI, against pa_decode.

pa_decode_noalloc serves callers that cannot allocate device memory where
they decode (an engine that handed all free HBM to its KV pool at start-up, a
plugin whose host framework owns the allocator, code that cannot afford an
allocation that may synchronise the device): it takes no workspace and uses
the library's fixed 64 MiB device scratch instead. Two calls in a row, on
different batches, must each match pa_decode's output within the parity
tolerance; a batch needing more scratch than the fixed array is refused
before anything is launched.

This file is named to be collected last.
"""
import ctypes as C

import numpy as np
import pytest
import torch

from paged_kv_cache_105_gb300 import binding as B
from paged_kv_cache_105_gb300 import workloads as W
from tests.helpers import ATOL, ROW_RTOL, gpu_step, to_dev

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def noalloc_via_cabi(wl, vals, t, err):
    out = torch.full_like(vals["q"], float("nan"))
    stream = C.c_void_p(torch.cuda.current_stream(DEV).cuda_stream)
    st = B.lib().pa_decode_noalloc(
        C.c_void_p(out.data_ptr()), C.c_void_p(vals["q"].data_ptr()),
        C.c_void_p(vals["k_pool"].data_ptr()), C.c_void_p(vals["v_pool"].data_ptr()),
        C.c_void_p(t["block_tables"].data_ptr()), C.c_void_p(t["seq_lens"].data_ptr()),
        wl.num_seqs, wl.block_tables.shape[1], wl.num_blocks, wl.n_q_heads, wl.n_kv_heads,
        wl.head_dim, wl.block_size, wl.scale, wl.partition_tokens, wl.max_seq_len,
        C.c_void_p(err.data_ptr()), stream)
    assert st == B.PA_OK, B.lib().pa_status_string(st)
    torch.cuda.synchronize()
    return out


def agree(a, b):
    x, y = a.float().cpu().numpy(), b.float().cpu().numpy()
    assert np.all(np.isfinite(x))
    assert np.abs(x - y).max() <= ATOL
    num = np.sqrt(((x - y) ** 2).sum(-1))
    den = np.maximum(np.sqrt((y ** 2).sum(-1)), 1e-30)
    assert (np.where(np.sqrt((y ** 2).sum(-1)) > 0, num / den, num)).max() <= ROW_RTOL


def test_noalloc_matches_pa_decode_on_two_calls_in_a_row():
    batches = [W.config2(), W.custom([3, 700, 1, 2500, 64], block_size=8, n_q_heads=16,
                                     n_kv_heads=2, head_dim=64, seed=31)]
    for wl in batches:
        vals = {k: v.to(DEV) for k, v in W.make_values(wl, poison_tails=True).items()}
        err = torch.zeros(1, dtype=torch.int32, device=DEV)
        ref, e = gpu_step(wl, vals, err=err)      # writes, then pa_decode with a workspace
        assert e == 0
        t = to_dev(wl, DEV)
        got = noalloc_via_cabi(wl, vals, t, err)
        assert int(err.item()) == 0
        agree(got, ref)


def test_noalloc_refuses_a_batch_beyond_its_scratch():
    wl = W.config5(num_seqs=16, seq_len=32768)
    need = B.pa_decode_workspace_bytes(16, 64, 8, 128, 16, 32768, 64)
    assert need > B.PA_NOALLOC_SCRATCH_BYTES
    # Host-side refusal: nothing is launched, so placeholder buffers suffice.
    tiny = torch.zeros(16, dtype=torch.int32, device=DEV)
    q = torch.zeros((16, 64, 128), dtype=torch.bfloat16, device=DEV)
    st = B.lib().pa_decode_noalloc(
        C.c_void_p(q.data_ptr()), C.c_void_p(q.data_ptr()), C.c_void_p(q.data_ptr()),
        C.c_void_p(q.data_ptr()), C.c_void_p(tiny.data_ptr()), C.c_void_p(tiny.data_ptr()),
        16, 2048, 8, 64, 8, 128, 16, wl.scale, 64, 32768, None,
        C.c_void_p(torch.cuda.current_stream(DEV).cuda_stream))
    assert st == B.PA_ERR_INVALID_ARG
