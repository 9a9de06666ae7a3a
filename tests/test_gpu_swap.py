"""GPU parity of block swap (device <-> page-locked host) against the oracle:
byte-exact, for bf16 and fp8 pools."""
import ctypes as C

import numpy as np
import pytest
import torch

from oracle import paref
from paged_kv_cache_105_gb300 import binding as B
from paged_kv_cache_105_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _np(t):
    t = t.detach().cpu().contiguous()
    return t.view(torch.uint8).numpy() if t.dtype != torch.uint8 else t.numpy()


@pytest.mark.parametrize("fp8", [False, True])
def test_swap_out_and_in_byte_exact(fp8):
    wl = W.config2()
    vals = W.make_values_fp8(wl, device=DEV) if fp8 else W.make_values(wl, device=DEV)
    gk, gv = vals["k_pool"], vals["v_pool"]
    # preempt the 8 longest sequences: all their blocks go to host blocks
    order = np.argsort(wl.seq_lens)[::-1][:8]
    ids = np.concatenate([wl.block_tables[s, :-(-int(wl.seq_lens[s]) // wl.block_size)]
                          for s in order]).astype(np.int32)
    n_host = len(ids) + 5
    hk = torch.zeros((n_host,) + tuple(gk.shape[1:]), dtype=gk.dtype).pin_memory()
    hv = torch.zeros_like(hk).pin_memory()
    host_ids = np.random.default_rng(0).permutation(n_host)[:len(ids)].astype(np.int32)
    out_pairs = np.stack([ids, host_ids], 1).astype(np.int32)
    g0k, g0v, h0k, h0v = _np(gk), _np(gv), _np(hk), _np(hv)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    B.pa_swap_blocks(hk, hv, gk, gv, torch.from_numpy(out_pairs).to(DEV), err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    rk, rv = h0k.copy(), h0v.copy()
    assert paref.swap_blocks(rk, rv, g0k, g0v, out_pairs) == 0
    assert np.array_equal(_np(hk), rk) and np.array_equal(_np(hv), rv)
    # swap back in under other device ids: the freed ids, in another order
    back = np.random.default_rng(1).permutation(ids).astype(np.int32)
    assert not np.array_equal(back, ids)
    in_pairs = np.stack([host_ids, back], 1).astype(np.int32)
    B.pa_swap_blocks(gk, gv, hk, hv, torch.from_numpy(in_pairs).to(DEV), err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    wk, wv = g0k.copy(), g0v.copy()
    assert paref.swap_blocks(wk, wv, rk, rv, in_pairs) == 0
    assert np.array_equal(_np(gk), wk) and np.array_equal(_np(gv), wv)
    assert np.array_equal(wk[back], g0k[ids])


def test_swap_bad_pair_flagged_and_skipped():
    g = torch.Generator(device=DEV).manual_seed(1)
    gk = torch.randint(0, 255, (10, 2, 16, 64), generator=g, device=DEV, dtype=torch.uint8)
    gv = torch.randint(0, 255, (10, 2, 16, 64), generator=g, device=DEV, dtype=torch.uint8)
    hk = torch.zeros((4, 2, 16, 64), dtype=torch.uint8).pin_memory()
    hv = torch.zeros_like(hk).pin_memory()
    pairs = np.array([[3, 0], [10, 1], [2, 4], [5, 2]], np.int32)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    B.pa_swap_blocks(hk, hv, gk, gv, torch.from_numpy(pairs).to(DEV), err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == B.PA_DEV_ERR_PAIR
    rk, rv = np.zeros_like(_np(hk)), np.zeros_like(_np(hv))
    assert paref.swap_blocks(rk, rv, _np(gk), _np(gv), pairs) == 2
    assert np.array_equal(_np(hk), rk) and np.array_equal(_np(hv), rv)


def test_swap_refuses_pageable_host_memory():
    # Host-side refusal before any launch: pageable memory is not an address
    # the kernel may use.
    gk = torch.zeros((4, 1, 16, 64), dtype=torch.uint8, device=DEV)
    pageable = np.zeros((4, 1, 16, 64), np.uint8)
    pairs = torch.tensor([[0, 0]], dtype=torch.int32, device=DEV)
    st = B.lib().pa_swap_blocks(
        C.c_void_p(pageable.ctypes.data), C.c_void_p(pageable.ctypes.data),
        C.c_void_p(gk.data_ptr()), C.c_void_p(gk.data_ptr()), C.c_void_p(pairs.data_ptr()), 1,
        1024, 4, 4, None, C.c_void_p(torch.cuda.current_stream(DEV).cuda_stream))
    assert st == B.PA_ERR_INVALID_ARG
    assert np.all(pageable == 0)


@pytest.mark.parametrize("nbytes", [16, 4096, 819712, 3 << 20])
def test_copy_host_both_ways_is_bit_exact(nbytes):
    # pa_copy_host: pinned host -> device and back, checked against the bytes
    g = torch.Generator().manual_seed(nbytes)
    host = torch.randint(0, 256, (nbytes,), generator=g, dtype=torch.uint8).pin_memory()
    dev = torch.full((nbytes,), 7, dtype=torch.uint8, device=DEV)
    back = torch.zeros(nbytes, dtype=torch.uint8).pin_memory()
    B.pa_copy_host(dev, host)
    B.pa_copy_host(back, dev)
    torch.cuda.synchronize()
    assert torch.equal(dev.cpu(), host)
    assert torch.equal(back, host)


def test_copy_host_refuses_pageable_memory():
    src = torch.zeros(64, dtype=torch.uint8)                    # pageable
    dst = torch.zeros(64, dtype=torch.uint8, device=DEV)
    with pytest.raises(ValueError):
        B.pa_copy_host(dst, src)
    st = B.lib().pa_copy_host(dst.data_ptr(), src.data_ptr(), 64, None)
    assert st == B.PA_ERR_INVALID_ARG
