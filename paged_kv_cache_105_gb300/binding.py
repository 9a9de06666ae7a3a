"""Thin ctypes binding of ``libpa.so`` (declared in ``include/pa.h``).

Argument marshalling only: tensors are checked for dtype, device, shape and
contiguity, their sizes and data pointers are passed through, and a
non-zero status becomes an exception. Every step of the computation runs
in the library's CUDA kernels; there is no fallback. If the library has not
been built, ``lib()`` raises.
"""
from __future__ import annotations

import ctypes as C
import os
import threading

import torch

from . import build as _build

PA_OK, PA_ERR_INVALID_ARG, PA_ERR_UNSUPPORTED, PA_ERR_CUDA = 0, 1, 2, 3
PA_DEV_ERR_BLOCK_ID = 0x1
PA_DEV_ERR_SLOT = 0x2
PA_DEV_ERR_PAIR = 0x4
PA_DEV_ERR_SEQ_LEN = 0x8
PA_DEV_ERR_TIMEOUT = 0x10

_lib = None
_lock = threading.Lock()

_vp = C.c_void_p
_i = C.c_int

SIGNATURES = {
    "pa_status_string": (C.c_char_p, [_i]),
    "pa_last_cuda_error": (C.c_char_p, []),
    "pa_decode_partition_tokens": (_i, [_i, _i, _i, _i, _i]),
    "pa_decode_workspace_bytes": (C.c_size_t, [_i, _i, _i, _i, _i, _i, _i]),
    "pa_decode": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, C.c_float,
                       _i, _i, _vp, C.c_size_t, _vp, _vp]),
    "pa_reshape_and_cache": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp, _vp]),
    "pa_copy_blocks": (_i, [_vp, _vp, _vp, _i, _i, _i, _i, _i, _vp, _vp]),
    "pa_decode_noalloc": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i,
                               C.c_float, _i, _i, _vp, _vp]),
    "pa_reshape_and_cache_fp8": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, C.c_float,
                                      C.c_float, _vp, _vp]),
    "pa_copy_blocks_fp8": (_i, [_vp, _vp, _vp, _i, _i, _i, _i, _i, _vp, _vp]),
    "pa_prefill": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _i,
                        C.c_float, _i, _vp, _vp]),
    "pa_swap_blocks": (_i, [_vp, _vp, _vp, _vp, _vp, _i, C.c_size_t, _i, _i, _vp, _vp]),
    "pa_copy_host": (_i, [_vp, _vp, C.c_size_t, _vp]),
    "pa_check_bounded_wait": (_i, [_vp, C.c_int64, _vp]),
    "pa_decode_fp8": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, C.c_float,
                           C.c_float, C.c_float, _i, _vp, C.c_size_t, _vp, _vp]),
}

# Size of the library's fixed scratch used by pa_decode_noalloc (64 MiB).
PA_NOALLOC_SCRATCH_BYTES = 64 << 20


class PAError(RuntimeError):
    def __init__(self, fn, status):
        L = lib()
        name = L.pa_status_string(status).decode()
        detail = L.pa_last_cuda_error().decode() if status == PA_ERR_CUDA else ""
        super().__init__(f"{fn}: {name}" + (f" ({detail})" if detail else ""))
        self.status = status


def lib():
    """The loaded ``libpa.so``; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_build.LIB):
                raise RuntimeError(
                    f"{_build.LIB} is missing: build it first "
                    "(python -c 'import __graft_entry__ as g; g.build()')")
            L = C.CDLL(_build.LIB)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


# The argument types are declared (SIGNATURES), so ctypes takes plain ints
# for the pointer arguments; these helpers stay cheap because every step of
# a serving loop goes through them.
def _ptr(t):
    return None if t is None else t.data_ptr()


# The raw current stream of a device, without building a Stream object.
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream, device):
    if stream is None:
        if _raw_stream is not None:
            return _raw_stream(device.index if device.index is not None else
                               torch.cuda.current_device())
        stream = torch.cuda.current_stream(device)
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check(t, name, dtype, dim=None, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if device is not None and t.get_device() != device.index:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dim is not None and t.dim() != dim:
        raise ValueError(f"{name} must have {dim} dimensions, got {tuple(t.shape)}")


def pa_decode_partition_tokens(num_seqs, n_kv_heads, block_size, max_seq_len,
                               partition_tokens=0) -> int:
    r = lib().pa_decode_partition_tokens(num_seqs, n_kv_heads, block_size, max_seq_len,
                                         partition_tokens)
    if r < 0:
        raise ValueError("unsupported decode arguments")
    return r


def pa_decode_workspace_bytes(num_seqs, n_q_heads, n_kv_heads, head_dim, block_size,
                              max_seq_len, partition_tokens=0) -> int:
    return int(lib().pa_decode_workspace_bytes(num_seqs, n_q_heads, n_kv_heads, head_dim,
                                               block_size, max_seq_len, partition_tokens))


def decode_workspace(num_seqs, n_q_heads, n_kv_heads, head_dim, block_size, max_seq_len,
                     partition_tokens=0, device=None) -> torch.Tensor:
    """A zeroed workspace for pa_decode (it stays zeroed between calls)."""
    n = pa_decode_workspace_bytes(num_seqs, n_q_heads, n_kv_heads, head_dim, block_size,
                                  max_seq_len, partition_tokens)
    if n == 0:
        raise ValueError("unsupported decode arguments")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def pa_decode(out, q, k_pool, v_pool, block_tables, seq_lens, scale, *, max_seq_len,
              workspace, partition_tokens=0, err_word=None, stream=None):
    """out[s, h] = softmax(scale * q[s, h] . K) V over the tokens of sequence s,
    K/V gathered from k_pool/v_pool through block_tables (see include/pa.h)."""
    dev = q.device
    _check(q, "q", torch.bfloat16, 3)
    _check(out, "out", torch.bfloat16, 3, dev)
    _check(k_pool, "k_pool", torch.bfloat16, 4, dev)
    _check(v_pool, "v_pool", torch.bfloat16, 4, dev)
    _check(block_tables, "block_tables", torch.int32, 2, dev)
    _check(seq_lens, "seq_lens", torch.int32, 1, dev)
    _check(workspace, "workspace", torch.uint8, 1, dev)
    if err_word is not None:
        _check(err_word, "err_word", torch.int32, None, dev)
    S, Hq, D = q.shape
    NB, Hkv, bs, D2 = k_pool.shape
    if tuple(out.shape) != (S, Hq, D) or D2 != D or tuple(v_pool.shape) != tuple(k_pool.shape):
        raise ValueError("shape mismatch between q, out and the pools")
    if block_tables.shape[0] != S or seq_lens.shape[0] != S:
        raise ValueError("block_tables / seq_lens must have one row per sequence")
    st = lib().pa_decode(_ptr(out), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(block_tables),
                         _ptr(seq_lens), S, block_tables.shape[1], NB, Hq, Hkv, D, bs,
                         float(scale), int(partition_tokens), int(max_seq_len),
                         _ptr(workspace), workspace.numel(), _ptr(err_word),
                         _stream(stream, dev))
    if st != PA_OK:
        raise PAError("pa_decode", st)
    return out


def pa_reshape_and_cache(k, v, k_pool, v_pool, slot_mapping, *, err_word=None, stream=None):
    """k_pool[slot // bs, :, slot % bs] = k[t] (and v) for every slot >= 0."""
    dev = k.device
    _check(k, "k", torch.bfloat16, 3)
    _check(v, "v", torch.bfloat16, 3, dev)
    _check(k_pool, "k_pool", torch.bfloat16, 4, dev)
    _check(v_pool, "v_pool", torch.bfloat16, 4, dev)
    _check(slot_mapping, "slot_mapping", torch.int32, 1, dev)
    if err_word is not None:
        _check(err_word, "err_word", torch.int32, None, dev)
    T, Hkv, D = k.shape
    NB, Hkv2, bs, D2 = k_pool.shape
    if v.shape != k.shape or Hkv2 != Hkv or D2 != D or v_pool.shape != k_pool.shape:
        raise ValueError("shape mismatch between new K/V and the pools")
    if slot_mapping.shape[0] != T:
        raise ValueError("slot_mapping must have one entry per token")
    st = lib().pa_reshape_and_cache(_ptr(k), _ptr(v), _ptr(k_pool), _ptr(v_pool),
                                    _ptr(slot_mapping), T, NB, Hkv, D, bs, _ptr(err_word),
                                    _stream(stream, dev))
    if st != PA_OK:
        raise PAError("pa_reshape_and_cache", st)


def pa_copy_blocks(k_pool, v_pool, pairs, *, err_word=None, stream=None):
    """Block pairs[p, 1] of both pools becomes a copy of block pairs[p, 0]."""
    dev = k_pool.device
    _check(k_pool, "k_pool", torch.bfloat16, 4)
    _check(v_pool, "v_pool", torch.bfloat16, 4, dev)
    _check(pairs, "pairs", torch.int32, 2, dev)
    if err_word is not None:
        _check(err_word, "err_word", torch.int32, None, dev)
    NB, Hkv, bs, D = k_pool.shape
    if v_pool.shape != k_pool.shape or (pairs.numel() and pairs.shape[1] != 2):
        raise ValueError("pools must match and pairs must be [n, 2]")
    st = lib().pa_copy_blocks(_ptr(k_pool), _ptr(v_pool), _ptr(pairs), pairs.shape[0], Hkv, D,
                              bs, NB, _ptr(err_word), _stream(stream, dev))
    if st != PA_OK:
        raise PAError("pa_copy_blocks", st)


def pa_decode_noalloc(out, q, k_pool, v_pool, block_tables, seq_lens, scale, *, max_seq_len,
                      partition_tokens=0, err_word=None, stream=None):
    """pa_decode without a workspace argument, for callers that cannot
    allocate device memory where they decode (an engine that gave all free
    HBM to its KV pool at start-up, a plugin whose host framework owns the
    allocator, code that cannot afford an allocation that may synchronise the
    device). Its scratch is the library's fixed 64 MiB device array, shared by
    every call in the process: calls must not overlap on the GPU, and the
    first call on a device should come before any stream capture."""
    dev = q.device
    _check(q, "q", torch.bfloat16, 3)
    _check(out, "out", torch.bfloat16, 3, dev)
    _check(k_pool, "k_pool", torch.bfloat16, 4, dev)
    _check(v_pool, "v_pool", torch.bfloat16, 4, dev)
    _check(block_tables, "block_tables", torch.int32, 2, dev)
    _check(seq_lens, "seq_lens", torch.int32, 1, dev)
    if err_word is not None:
        _check(err_word, "err_word", torch.int32, None, dev)
    S, Hq, D = q.shape
    NB, Hkv, bs, D2 = k_pool.shape
    if tuple(out.shape) != (S, Hq, D) or D2 != D or tuple(v_pool.shape) != tuple(k_pool.shape):
        raise ValueError("shape mismatch between q, out and the pools")
    if block_tables.shape[0] != S or seq_lens.shape[0] != S:
        raise ValueError("block_tables / seq_lens must have one row per sequence")
    need = pa_decode_workspace_bytes(S, Hq, Hkv, D, bs, int(max_seq_len), int(partition_tokens))
    if need > PA_NOALLOC_SCRATCH_BYTES:
        raise ValueError(f"pa_decode_noalloc: this batch needs {need} bytes of scratch, the "
                         f"library's fixed scratch holds {PA_NOALLOC_SCRATCH_BYTES}")
    st = lib().pa_decode_noalloc(_ptr(out), _ptr(q), _ptr(k_pool), _ptr(v_pool),
                                 _ptr(block_tables), _ptr(seq_lens), S, block_tables.shape[1],
                                 NB, Hq, Hkv, D, bs, float(scale), int(partition_tokens),
                                 int(max_seq_len), _ptr(err_word), _stream(stream, dev))
    if st != PA_OK:
        raise PAError("pa_decode_noalloc", st)
    return out


# ------------------------------------------------------------ fp8 (E4M3) cache
# Pools are uint8 tensors of E4M3 codes; a code times the tensor's scale is
# the value (include/pa.h, "FP8 KV cache").

def pa_reshape_and_cache_fp8(k, v, k_pool, v_pool, slot_mapping, k_scale, v_scale, *,
                             err_word=None, stream=None):
    """k_pool[slot // bs, :, slot % bs] = E4M3(fp32(k[t]) / k_scale) (and v)."""
    dev = k.device
    _check(k, "k", torch.bfloat16, 3)
    _check(v, "v", torch.bfloat16, 3, dev)
    _check(k_pool, "k_pool", torch.uint8, 4, dev)
    _check(v_pool, "v_pool", torch.uint8, 4, dev)
    _check(slot_mapping, "slot_mapping", torch.int32, 1, dev)
    if err_word is not None:
        _check(err_word, "err_word", torch.int32, None, dev)
    T, Hkv, D = k.shape
    NB, Hkv2, bs, D2 = k_pool.shape
    if v.shape != k.shape or Hkv2 != Hkv or D2 != D or v_pool.shape != k_pool.shape:
        raise ValueError("shape mismatch between new K/V and the pools")
    if slot_mapping.shape[0] != T:
        raise ValueError("slot_mapping must have one entry per token")
    st = lib().pa_reshape_and_cache_fp8(_ptr(k), _ptr(v), _ptr(k_pool), _ptr(v_pool),
                                        _ptr(slot_mapping), T, NB, Hkv, D, bs, float(k_scale),
                                        float(v_scale), _ptr(err_word), _stream(stream, dev))
    if st != PA_OK:
        raise PAError("pa_reshape_and_cache_fp8", st)


def pa_copy_blocks_fp8(k_pool, v_pool, pairs, *, err_word=None, stream=None):
    """Block pairs[p, 1] of both uint8 pools becomes a copy of block pairs[p, 0]."""
    dev = k_pool.device
    _check(k_pool, "k_pool", torch.uint8, 4)
    _check(v_pool, "v_pool", torch.uint8, 4, dev)
    _check(pairs, "pairs", torch.int32, 2, dev)
    if err_word is not None:
        _check(err_word, "err_word", torch.int32, None, dev)
    NB, Hkv, bs, D = k_pool.shape
    if v_pool.shape != k_pool.shape or (pairs.numel() and pairs.shape[1] != 2):
        raise ValueError("pools must match and pairs must be [n, 2]")
    st = lib().pa_copy_blocks_fp8(_ptr(k_pool), _ptr(v_pool), _ptr(pairs), pairs.shape[0], Hkv,
                                  D, bs, NB, _ptr(err_word), _stream(stream, dev))
    if st != PA_OK:
        raise PAError("pa_copy_blocks_fp8", st)


def pa_decode_fp8(out, q, k_pool, v_pool, block_tables, seq_lens, scale, k_scale, v_scale, *,
                  max_seq_len, workspace, err_word=None, stream=None):
    """pa_decode over E4M3 pools: K = code * k_scale, V = code * v_scale.
    The workspace is decode_workspace(..., partition_tokens=0)."""
    dev = q.device
    _check(q, "q", torch.bfloat16, 3)
    _check(out, "out", torch.bfloat16, 3, dev)
    _check(k_pool, "k_pool", torch.uint8, 4, dev)
    _check(v_pool, "v_pool", torch.uint8, 4, dev)
    _check(block_tables, "block_tables", torch.int32, 2, dev)
    _check(seq_lens, "seq_lens", torch.int32, 1, dev)
    _check(workspace, "workspace", torch.uint8, 1, dev)
    if err_word is not None:
        _check(err_word, "err_word", torch.int32, None, dev)
    S, Hq, D = q.shape
    NB, Hkv, bs, D2 = k_pool.shape
    if tuple(out.shape) != (S, Hq, D) or D2 != D or tuple(v_pool.shape) != tuple(k_pool.shape):
        raise ValueError("shape mismatch between q, out and the pools")
    if block_tables.shape[0] != S or seq_lens.shape[0] != S:
        raise ValueError("block_tables / seq_lens must have one row per sequence")
    st = lib().pa_decode_fp8(_ptr(out), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(block_tables),
                             _ptr(seq_lens), S, block_tables.shape[1], NB, Hq, Hkv, D, bs,
                             float(scale), float(k_scale), float(v_scale), int(max_seq_len),
                             _ptr(workspace), workspace.numel(), _ptr(err_word),
                             _stream(stream, dev))
    if st != PA_OK:
        raise PAError("pa_decode_fp8", st)
    return out


# ------------------------------------------------------------------ prefill

def pa_prefill(out, q, k_pool, v_pool, block_tables, seq_lens, cu_q, scale, *, max_q_len,
               err_word=None, stream=None):
    """Causal attention of each sequence's chunk (its last cu_q[s+1]-cu_q[s]
    tokens, rows cu_q[s].. of q) over its whole paged context (include/pa.h)."""
    dev = q.device
    _check(q, "q", torch.bfloat16, 3)
    _check(out, "out", torch.bfloat16, 3, dev)
    _check(k_pool, "k_pool", torch.bfloat16, 4, dev)
    _check(v_pool, "v_pool", torch.bfloat16, 4, dev)
    _check(block_tables, "block_tables", torch.int32, 2, dev)
    _check(seq_lens, "seq_lens", torch.int32, 1, dev)
    _check(cu_q, "cu_q", torch.int32, 1, dev)
    if err_word is not None:
        _check(err_word, "err_word", torch.int32, None, dev)
    TQ, Hq, D = q.shape
    NB, Hkv, bs, D2 = k_pool.shape
    S = seq_lens.shape[0]
    if tuple(out.shape) != (TQ, Hq, D) or D2 != D or tuple(v_pool.shape) != tuple(k_pool.shape):
        raise ValueError("shape mismatch between q, out and the pools")
    if block_tables.shape[0] != S or cu_q.shape[0] != S + 1:
        raise ValueError("block_tables needs one row and cu_q one entry per sequence (+1)")
    st = lib().pa_prefill(_ptr(out), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(block_tables),
                          _ptr(seq_lens), _ptr(cu_q), S, TQ, block_tables.shape[1], NB, Hq,
                          Hkv, D,
                          bs, float(scale), int(max_q_len), _ptr(err_word), _stream(stream, dev))
    if st != PA_OK:
        raise PAError("pa_prefill", st)
    return out


# ------------------------------------------------------------------ swap

def _check_pool_any(t, name, like=None):
    """A contiguous pool tensor on the GPU or in page-locked host memory."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if not t.is_cuda and not t.is_pinned():
        raise ValueError(f"{name} must be a CUDA tensor or page-locked (pinned) host memory")
    if like is not None and (t.dtype != like.dtype or t.shape[1:] != like.shape[1:]):
        raise ValueError(f"{name} blocks must have the dtype and shape of the other pool's")


def pa_swap_blocks(dst_k, dst_v, src_k, src_v, pairs, *, err_word=None, stream=None):
    """Block pairs[p, 1] of (dst_k, dst_v) becomes a copy of block pairs[p, 0]
    of (src_k, src_v); either pool pair may live in pinned host memory (the
    kernel reads or writes it directly). Swap-out: device pools -> host
    pools; swap-in: back."""
    _check_pool_any(src_k, "src_k")
    _check_pool_any(src_v, "src_v", src_k)
    _check_pool_any(dst_k, "dst_k", src_k)
    _check_pool_any(dst_v, "dst_v", src_k)
    if src_v.shape != src_k.shape or dst_v.shape != dst_k.shape:
        raise ValueError("K and V pools of one side must match")
    _check(pairs, "pairs", torch.int32, 2)
    dev = pairs.device
    if err_word is not None:
        _check(err_word, "err_word", torch.int32, None, dev)
    if pairs.numel() and pairs.shape[1] != 2:
        raise ValueError("pairs must be [n, 2]")
    block_bytes = src_k[0].numel() * src_k.element_size()
    st = lib().pa_swap_blocks(_ptr(dst_k), _ptr(dst_v), _ptr(src_k), _ptr(src_v), _ptr(pairs),
                              pairs.shape[0], block_bytes, src_k.shape[0], dst_k.shape[0],
                              _ptr(err_word), _stream(stream, dev))
    if st != PA_OK:
        raise PAError("pa_swap_blocks", st)


def pa_copy_host(dst, src, *, stream=None):
    """Copy src into dst (same byte size, contiguous) with the SMs, where
    either tensor may be a CUDA tensor or page-locked host memory."""
    for t, name in ((dst, "dst"), (src, "src")):
        if not isinstance(t, torch.Tensor):
            raise TypeError(f"{name} must be a torch.Tensor")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        if not t.is_cuda and not t.is_pinned():
            raise ValueError(f"{name} must be a CUDA tensor or page-locked (pinned) host memory")
    n = dst.numel() * dst.element_size()
    if src.numel() * src.element_size() != n:
        raise ValueError("dst and src must hold the same number of bytes")
    dev = dst.device if dst.is_cuda else (src.device if src.is_cuda else
                                          torch.device("cuda", torch.cuda.current_device()))
    st = lib().pa_copy_host(_ptr(dst), _ptr(src), n, _stream(stream, dev))
    if st != PA_OK:
        raise PAError("pa_copy_host", st)


# ------------------------------------------------------------ prepared step

class DecodeStep:
    """One decode step of a fixed batch shape, prepared once: the
    copy-on-write block copies (if `pairs` has rows), the new tokens' cache
    write, and the decode with its merge, in that order on one stream.

    Every check and every pointer extraction happens here, once; enqueue()
    makes only the three library calls, with argument lists built in the
    constructor. The step reads whatever the given tensors hold when it runs,
    so a serving loop refreshes q, the new K/V, the tables, lengths, slots and
    pairs in place between steps (their shapes and storage must not change,
    and they must outlive this object). kv_scales = (k_scale, v_scale) selects
    the E4M3 entry points (uint8 pools). A CUDA graph may capture enqueue().
    """

    def __init__(self, out, q, k_pool, v_pool, block_tables, seq_lens, scale, *, max_seq_len,
                 workspace, k_new, v_new, slot_mapping, pairs=None, partition_tokens=0,
                 err_word=None, kv_scales=None, stream=None):
        fp8 = kv_scales is not None
        dev = q.device
        pool_t = torch.uint8 if fp8 else torch.bfloat16
        _check(q, "q", torch.bfloat16, 3)
        _check(out, "out", torch.bfloat16, 3, dev)
        _check(k_pool, "k_pool", pool_t, 4, dev)
        _check(v_pool, "v_pool", pool_t, 4, dev)
        _check(block_tables, "block_tables", torch.int32, 2, dev)
        _check(seq_lens, "seq_lens", torch.int32, 1, dev)
        _check(workspace, "workspace", torch.uint8, 1, dev)
        _check(k_new, "k_new", torch.bfloat16, 3, dev)
        _check(v_new, "v_new", torch.bfloat16, 3, dev)
        _check(slot_mapping, "slot_mapping", torch.int32, 1, dev)
        if pairs is not None:
            _check(pairs, "pairs", torch.int32, 2, dev)
            if pairs.numel() and pairs.shape[1] != 2:
                raise ValueError("pairs must be [n, 2]")
        if err_word is not None:
            _check(err_word, "err_word", torch.int32, None, dev)
        S, Hq, D = q.shape
        NB, Hkv, bs, D2 = k_pool.shape
        T = k_new.shape[0]
        if tuple(out.shape) != (S, Hq, D) or D2 != D or tuple(v_pool.shape) != tuple(k_pool.shape):
            raise ValueError("shape mismatch between q, out and the pools")
        if block_tables.shape[0] != S or seq_lens.shape[0] != S:
            raise ValueError("block_tables / seq_lens must have one row per sequence")
        if tuple(k_new.shape) != (T, Hkv, D) or v_new.shape != k_new.shape:
            raise ValueError("new K/V must be [tokens, n_kv_heads, head_dim]")
        if slot_mapping.shape[0] != T:
            raise ValueError("slot_mapping must have one entry per new token")
        L = lib()
        self._tensors = (out, q, k_pool, v_pool, block_tables, seq_lens, workspace, k_new,
                         v_new, slot_mapping, pairs, err_word)  # kept alive
        self._dev = dev.index if dev.index is not None else torch.cuda.current_device()
        self._fixed_stream = None if stream is None else _stream(stream, dev)
        err = _ptr(err_word)
        n_pairs = 0 if pairs is None else pairs.shape[0]
        self._copy = None
        if n_pairs:
            fn = L.pa_copy_blocks_fp8 if fp8 else L.pa_copy_blocks
            self._copy = (fn, "pa_copy_blocks_fp8" if fp8 else "pa_copy_blocks",
                          (_ptr(k_pool), _ptr(v_pool), _ptr(pairs), n_pairs, Hkv, D, bs, NB,
                           err))
        if fp8:
            ks, vs = float(kv_scales[0]), float(kv_scales[1])
            self._write = (L.pa_reshape_and_cache_fp8, "pa_reshape_and_cache_fp8",
                           (_ptr(k_new), _ptr(v_new), _ptr(k_pool), _ptr(v_pool),
                            _ptr(slot_mapping), T, NB, Hkv, D, bs, ks, vs, err))
            self._decode = (L.pa_decode_fp8, "pa_decode_fp8",
                            (_ptr(out), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(block_tables),
                             _ptr(seq_lens), S, block_tables.shape[1], NB, Hq, Hkv, D, bs,
                             float(scale), ks, vs, int(max_seq_len), _ptr(workspace),
                             workspace.numel(), err))
        else:
            self._write = (L.pa_reshape_and_cache, "pa_reshape_and_cache",
                           (_ptr(k_new), _ptr(v_new), _ptr(k_pool), _ptr(v_pool),
                            _ptr(slot_mapping), T, NB, Hkv, D, bs, err))
            self._decode = (L.pa_decode, "pa_decode",
                            (_ptr(out), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(block_tables),
                             _ptr(seq_lens), S, block_tables.shape[1], NB, Hq, Hkv, D, bs,
                             float(scale), int(partition_tokens), int(max_seq_len),
                             _ptr(workspace), workspace.numel(), err))

    def enqueue(self):
        """Issue the step on the stream given at construction, else on the
        current stream of the tensors' device."""
        st = self._fixed_stream
        if st is None:
            st = (_raw_stream(self._dev) if _raw_stream is not None else
                  torch.cuda.current_stream(self._dev).cuda_stream)
        for call in (self._copy, self._write, self._decode):
            if call is None:
                continue
            fn, name, args = call
            r = fn(*args, st)
            if r != PA_OK:
                raise PAError(name, r)
