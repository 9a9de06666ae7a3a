"""ctypes front end of the C++ oracle (``libparef.so``), numpy in and out.

Test infrastructure only. bf16 tensors cross as their raw uint16 bit
patterns; the oracle widens them exactly to double.
"""
from __future__ import annotations

import ctypes as C
import threading

import numpy as np

from . import build as _build

_lib = None
_lock = threading.Lock()

i32p = C.POINTER(C.c_int32)
u16p = C.POINTER(C.c_uint16)
u8p = C.POINTER(C.c_uint8)
f64p = C.POINTER(C.c_double)


def lib():
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build()
            L = C.CDLL(path)
            sig = {
                "paref_blocks_for": (C.c_int, [C.c_int, C.c_int]),
                "paref_tail_waste": (C.c_int, [C.c_int, C.c_int]),
                "paref_paged_slots": (C.c_int64, [i32p, C.c_int, C.c_int]),
                "paref_used_tokens": (C.c_int64, [i32p, C.c_int]),
                "paref_naive_slots": (C.c_int64, [C.c_int, C.c_int]),
                "paref_capacity": (C.c_int64, [C.c_int64, C.c_int64, C.c_int]),
                "paref_alloc_new": (C.c_void_p, [C.c_int, C.c_int, i32p]),
                "paref_alloc_delete": (None, [C.c_void_p]),
                "paref_alloc_add_seq": (C.c_int, [C.c_void_p]),
                "paref_alloc_append": (C.c_int, [C.c_void_p, C.c_int, i32p, i32p, i32p]),
                "paref_alloc_fork": (C.c_int, [C.c_void_p, C.c_int]),
                "paref_alloc_free_seq": (C.c_int, [C.c_void_p, C.c_int]),
                "paref_alloc_num_free": (C.c_int, [C.c_void_p]),
                "paref_alloc_usage": (None, [C.c_void_p, C.POINTER(C.c_int64),
                                             C.POINTER(C.c_int64), C.POINTER(C.c_int64)]),
                "paref_alloc_num_blocks": (C.c_int, [C.c_void_p]),
                "paref_alloc_refcount": (C.c_int, [C.c_void_p, C.c_int]),
                "paref_alloc_seq_len": (C.c_int, [C.c_void_p, C.c_int]),
                "paref_alloc_seq_nblocks": (C.c_int, [C.c_void_p, C.c_int]),
                "paref_alloc_seq_alive": (C.c_int, [C.c_void_p, C.c_int]),
                "paref_alloc_table": (C.c_int, [C.c_void_p, C.c_int, i32p, C.c_int]),
                "paref_alloc_free_list": (C.c_int, [C.c_void_p, i32p, C.c_int]),
                "paref_attention_paged": (C.c_int, [f64p, u16p, u16p, u16p, i32p, i32p,
                                                    C.c_int, C.c_int, C.c_int, C.c_int,
                                                    C.c_int, C.c_int, C.c_int, C.c_double,
                                                    i32p, C.c_int]),
                "paref_attention_contiguous": (C.c_int, [f64p, u16p, u16p, u16p, C.c_int,
                                                         C.c_int, C.c_int, C.c_int,
                                                         C.c_double]),
                "paref_reshape_and_cache": (C.c_int, [u16p, u16p, u16p, u16p, i32p, C.c_int,
                                                      C.c_int, C.c_int, C.c_int, C.c_int]),
                "paref_copy_blocks": (C.c_int, [u16p, u16p, i32p, C.c_int, C.c_int, C.c_int,
                                                C.c_int, C.c_int]),
                "paref_prefill_paged": (C.c_int, [f64p, u16p, u16p, u16p, i32p, i32p, i32p,
                                                  C.c_int, C.c_int, C.c_int, C.c_int, C.c_int,
                                                  C.c_int, C.c_int, C.c_double, i32p, C.c_int]),
                "paref_swap_blocks": (C.c_int, [u8p, u8p, u8p, u8p, i32p, C.c_int, C.c_int64,
                                                C.c_int, C.c_int]),
                "paref_e4m3_decode": (C.c_double, [C.c_uint8]),
                "paref_e4m3_encode": (C.c_uint8, [C.c_double]),
                "paref_reshape_and_cache_fp8": (C.c_int, [u16p, u16p, u8p, u8p, i32p, C.c_int,
                                                          C.c_int, C.c_int, C.c_int, C.c_int,
                                                          C.c_float, C.c_float]),
                "paref_attention_paged_fp8": (C.c_int, [f64p, u16p, u8p, u8p, i32p, i32p,
                                                        C.c_int, C.c_int, C.c_int, C.c_int,
                                                        C.c_int, C.c_int, C.c_int, C.c_double,
                                                        C.c_double, C.c_double, i32p, C.c_int]),
            }
            for name, (res, args) in sig.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


def _i32(a):
    a = np.ascontiguousarray(a, dtype=np.int32)
    return a, a.ctypes.data_as(i32p)


def _u16(a):
    a = np.asarray(a)
    if a.dtype != np.uint16 or not a.flags["C_CONTIGUOUS"]:
        raise TypeError("bf16 data must be a C-contiguous uint16 (bit pattern) array")
    return a, a.ctypes.data_as(u16p)


# ----------------------------------------------------------------- accounting

def blocks_for(length: int, block_size: int) -> int:
    return lib().paref_blocks_for(int(length), int(block_size))


def tail_waste(length: int, block_size: int) -> int:
    return lib().paref_tail_waste(int(length), int(block_size))


def paged_slots(lens, block_size: int) -> int:
    a, p = _i32(lens)
    return lib().paref_paged_slots(p, len(a), int(block_size))


def used_tokens(lens) -> int:
    a, p = _i32(lens)
    return lib().paref_used_tokens(p, len(a))


def naive_slots(n: int, max_len: int) -> int:
    return lib().paref_naive_slots(int(n), int(max_len))


def capacity(pool_slots: int, alloc_slots: int, n: int) -> int:
    return lib().paref_capacity(int(pool_slots), int(alloc_slots), int(n))


# ----------------------------------------------------------------- allocator

class OutOfBlocks(RuntimeError):
    pass


class Allocator:
    """Free-list block allocator with refcounts and copy-on-write."""

    def __init__(self, num_blocks: int, block_size: int, free_order=None):
        self.block_size = int(block_size)
        if free_order is not None:
            arr, p = _i32(free_order)
            if len(arr) != num_blocks:
                raise ValueError("free_order must list every block once")
            self._keep = arr
        else:
            p = None
        h = lib().paref_alloc_new(int(num_blocks), int(block_size), p)
        if not h:
            raise ValueError("bad allocator arguments")
        self._h = C.c_void_p(h)

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and _lib is not None:
            _lib.paref_alloc_delete(h)
            self._h = None

    def add_seq(self) -> int:
        return lib().paref_alloc_add_seq(self._h)

    def append(self, seq: int):
        """Append one token; returns (slot, cow_pair_or_None)."""
        slot, src, dst = C.c_int32(), C.c_int32(), C.c_int32()
        rc = lib().paref_alloc_append(self._h, int(seq), C.byref(slot), C.byref(src),
                                      C.byref(dst))
        if rc == -1:
            raise OutOfBlocks(f"no free block for seq {seq}")
        if rc != 0:
            raise ValueError(f"bad sequence id {seq}")
        pair = (src.value, dst.value) if src.value >= 0 else None
        return slot.value, pair

    def fork(self, seq: int) -> int:
        r = lib().paref_alloc_fork(self._h, int(seq))
        if r < 0:
            raise ValueError(f"bad sequence id {seq}")
        return r

    def free(self, seq: int) -> int:
        r = lib().paref_alloc_free_seq(self._h, int(seq))
        if r < 0:
            raise ValueError(f"bad sequence id {seq}")
        return r

    def usage(self):
        """(tokens held, slots of the blocks in use, blocks in use); a shared
        block counts once, holding what its furthest writer put there."""
        t, s, b = C.c_int64(), C.c_int64(), C.c_int64()
        lib().paref_alloc_usage(self._h, C.byref(t), C.byref(s), C.byref(b))
        return t.value, s.value, b.value

    def utilisation(self) -> float:
        """Tokens held / slots allocated ("03 · PagedAttention", Try It: the
        utilisation column); 0.0 for an empty pool."""
        t, s, _ = self.usage()
        return t / s if s else 0.0

    def cache_usage(self) -> float:
        """Blocks in use / pool blocks (the share of the KV pool taken, the
        figure the mlapandio page's closing advice says to watch)."""
        _, _, b = self.usage()
        return b / self.num_blocks if self.num_blocks else 0.0

    @property
    def num_free(self) -> int:
        return lib().paref_alloc_num_free(self._h)

    @property
    def num_blocks(self) -> int:
        return lib().paref_alloc_num_blocks(self._h)

    def refcount(self, block: int) -> int:
        return lib().paref_alloc_refcount(self._h, int(block))

    def refcounts(self) -> np.ndarray:
        return np.array([self.refcount(b) for b in range(self.num_blocks)], dtype=np.int64)

    def seq_len(self, seq: int) -> int:
        return lib().paref_alloc_seq_len(self._h, int(seq))

    def alive(self, seq: int) -> bool:
        return bool(lib().paref_alloc_seq_alive(self._h, int(seq)))

    def table(self, seq: int) -> np.ndarray:
        n = lib().paref_alloc_seq_nblocks(self._h, int(seq))
        out = np.zeros(max(n, 1), dtype=np.int32)
        lib().paref_alloc_table(self._h, int(seq), out.ctypes.data_as(i32p), n)
        return out[:n]

    def free_list(self) -> np.ndarray:
        n = self.num_free
        out = np.zeros(max(n, 1), dtype=np.int32)
        lib().paref_alloc_free_list(self._h, out.ctypes.data_as(i32p), n)
        return out[:n]


# ----------------------------------------------------------------- attention

def attention_paged(q, k_pool, v_pool, block_tables, seq_lens, scale, rows=None):
    """fp64 paged attention. q [S,Hq,d], pools [NB,Hkv,bs,d] as uint16 bits.

    rows: optional int array [n,2] of (seq, q_head); returns [n,d] then,
    else [S,Hq,d].
    """
    q, qp = _u16(q)
    k_pool, kp = _u16(k_pool)
    v_pool, vp = _u16(v_pool)
    bt, btp = _i32(block_tables)
    sl, slp = _i32(seq_lens)
    S, Hq, d = q.shape
    NB, Hkv, bs, d2 = k_pool.shape
    assert d2 == d and v_pool.shape == k_pool.shape
    assert bt.ndim == 2 and bt.shape[0] == S and sl.shape == (S,)
    if rows is None:
        out = np.zeros((S, Hq, d), dtype=np.float64)
        rp, nr = None, 0
    else:
        r, rp = _i32(np.asarray(rows).reshape(-1, 2))
        nr = r.shape[0]
        out = np.zeros((nr, d), dtype=np.float64)
    rc = lib().paref_attention_paged(out.ctypes.data_as(f64p), qp, kp, vp, btp, slp, S,
                                     bt.shape[1], NB, Hq, Hkv, d, bs, float(scale), rp, nr)
    if rc != 0:
        raise ValueError("oracle attention: invalid block table, length or shape")
    return out


def attention_contiguous(q, k, v, scale):
    """fp64 attention for one sequence: q [Hq,d], k/v [len,Hkv,d] (uint16 bits)."""
    q, qp = _u16(q)
    k, kp = _u16(k)
    v, vp = _u16(v)
    Hq, d = q.shape
    n, Hkv, d2 = k.shape
    assert d2 == d and v.shape == k.shape
    out = np.zeros((Hq, d), dtype=np.float64)
    rc = lib().paref_attention_contiguous(out.ctypes.data_as(f64p), qp, kp, vp, n, Hq, Hkv,
                                          d, float(scale))
    if rc != 0:
        raise ValueError("oracle contiguous attention: bad arguments")
    return out


# ----------------------------------------------------------------- writes

def reshape_and_cache(k, v, k_pool, v_pool, slot_mapping) -> int:
    """In place on k_pool / v_pool (uint16 arrays). Returns skipped count."""
    k, kp = _u16(k)
    v, vp = _u16(v)
    k_pool, kpp = _u16(k_pool)
    v_pool, vpp = _u16(v_pool)
    sm, smp = _i32(slot_mapping)
    T, Hkv, d = k.shape
    NB, Hkv2, bs, d2 = k_pool.shape
    assert Hkv2 == Hkv and d2 == d and sm.shape == (T,)
    return lib().paref_reshape_and_cache(kp, vp, kpp, vpp, smp, T, NB, Hkv, d, bs)


def copy_blocks(k_pool, v_pool, pairs) -> int:
    """In place on k_pool / v_pool (uint16 arrays). Returns skipped count."""
    k_pool, kpp = _u16(k_pool)
    v_pool, vpp = _u16(v_pool)
    pr, prp = _i32(np.asarray(pairs).reshape(-1, 2))
    NB, Hkv, bs, d = k_pool.shape
    return lib().paref_copy_blocks(kpp, vpp, prp, pr.shape[0], Hkv, d, bs, NB)


# ----------------------------------------------------------------- prefill

def prefill_paged(q, k_pool, v_pool, block_tables, seq_lens, cu_q, scale, rows=None):
    """Causal attention of each sequence's last c_s tokens (its chunk, rows
    cu_q[s]..cu_q[s+1]-1 of q) over its whole cached context, in fp64."""
    q, qp = _u16(q)
    k_pool, kp = _u16(k_pool)
    v_pool, vp = _u16(v_pool)
    bt, btp = _i32(block_tables)
    sl, slp = _i32(seq_lens)
    cu, cup = _i32(cu_q)
    TQ, Hq, d = q.shape
    NB, Hkv, bs, d2 = k_pool.shape
    S = len(sl)
    assert d2 == d and len(cu) == S + 1 and int(cu[-1]) == TQ
    if rows is None:
        out = np.zeros((TQ, Hq, d), dtype=np.float64)
        rp, nr = None, 0
    else:
        r, rp = _i32(np.asarray(rows).reshape(-1, 2))
        nr = r.shape[0]
        out = np.zeros((nr, d), dtype=np.float64)
    rc = lib().paref_prefill_paged(out.ctypes.data_as(f64p), qp, kp, vp, btp, slp, cup, S,
                                   bt.shape[1], NB, Hq, Hkv, d, bs, float(scale), rp, nr)
    if rc != 0:
        raise ValueError("oracle prefill: invalid table, length or chunk")
    return out


# ----------------------------------------------------------------- swap

def swap_blocks(dst_k, dst_v, src_k, src_v, pairs) -> int:
    """Block pairs[p, 1] of the destination pools becomes a byte copy of block
    pairs[p, 0] of the source pools. Pools are C-contiguous arrays whose
    first axis is the block id (any element type: the copy is of bytes).
    Returns the skipped count."""
    arrs = []
    for a in (dst_k, dst_v, src_k, src_v):
        a = np.asarray(a)
        if not a.flags["C_CONTIGUOUS"]:
            raise TypeError("pools must be C-contiguous")
        arrs.append(a)
    dk, dv, sk, sv = arrs
    if dk.shape[1:] != sk.shape[1:] or dk.dtype != sk.dtype or dv.shape != dk.shape or \
            sv.shape != sk.shape:
        raise ValueError("source and destination blocks must have one shape")
    block_bytes = dk[0].nbytes if len(dk) else sk[0].nbytes
    pr, prp = _i32(np.asarray(pairs).reshape(-1, 2))
    u8 = lambda a: a.ctypes.data_as(u8p)
    return lib().paref_swap_blocks(u8(dk), u8(dv), u8(sk), u8(sv), prp, pr.shape[0],
                                   int(block_bytes), sk.shape[0], dk.shape[0])


# ----------------------------------------------------------------- fp8 (E4M3)

def e4m3_decode(code: int) -> float:
    return lib().paref_e4m3_decode(int(code))


def e4m3_encode(x: float) -> int:
    return lib().paref_e4m3_encode(float(x))


def _u8(a):
    a = np.asarray(a)
    if a.dtype != np.uint8 or not a.flags["C_CONTIGUOUS"]:
        raise TypeError("fp8 pools must be C-contiguous uint8 arrays")
    return a, a.ctypes.data_as(u8p)


def reshape_and_cache_fp8(k, v, k_pool, v_pool, slot_mapping, k_scale, v_scale) -> int:
    """In place on the uint8 pools: E4M3 codes of fp32(k) / k_scale."""
    k, kp = _u16(k)
    v, vp = _u16(v)
    k_pool, kpp = _u8(k_pool)
    v_pool, vpp = _u8(v_pool)
    sm, smp = _i32(slot_mapping)
    T, Hkv, d = k.shape
    NB, Hkv2, bs, d2 = k_pool.shape
    assert Hkv2 == Hkv and d2 == d and sm.shape == (T,)
    return lib().paref_reshape_and_cache_fp8(kp, vp, kpp, vpp, smp, T, NB, Hkv, d, bs,
                                             float(k_scale), float(v_scale))


def attention_paged_fp8(q, k_pool, v_pool, block_tables, seq_lens, scale, k_scale, v_scale,
                        rows=None):
    """fp64 paged attention over E4M3 pools (uint8 codes times the scales)."""
    q, qp = _u16(q)
    k_pool, kp = _u8(k_pool)
    v_pool, vp = _u8(v_pool)
    bt, btp = _i32(block_tables)
    sl, slp = _i32(seq_lens)
    S, Hq, d = q.shape
    NB, Hkv, bs, d2 = k_pool.shape
    assert d2 == d and v_pool.shape == k_pool.shape
    if rows is None:
        out = np.zeros((S, Hq, d), dtype=np.float64)
        rp, nr = None, 0
    else:
        r, rp = _i32(np.asarray(rows).reshape(-1, 2))
        nr = r.shape[0]
        out = np.zeros((nr, d), dtype=np.float64)
    rc = lib().paref_attention_paged_fp8(out.ctypes.data_as(f64p), qp, kp, vp, btp, slp, S,
                                         bt.shape[1], NB, Hq, Hkv, d, bs, float(scale),
                                         float(k_scale), float(v_scale), rp, nr)
    if rc != 0:
        raise ValueError("oracle fp8 attention: invalid block table, length or shape")
    return out
