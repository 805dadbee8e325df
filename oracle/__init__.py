"""CPU oracle for decode attention over a paged or contiguous KV cache.

TEST INFRASTRUCTURE ONLY.  This package is imported by the tests, by the
smoke check and by the benchmark's CPU-baseline leg, and by nothing else.  It
is a plain fp64 restatement of what the decode step computes (see the header
of ``pkv_oracle.c`` for the passages it follows) and shares no code with the
CUDA library.

Arrays are numpy; bf16 tensors are passed as their uint16 bit patterns.
"""
import ctypes

import numpy as np

from .build_oracle import build as _build

_lib = None

_u16p = np.ctypeslib.ndpointer(dtype=np.uint16, flags="C_CONTIGUOUS")
_i32p = np.ctypeslib.ndpointer(dtype=np.int32, flags="C_CONTIGUOUS")
_i64p = np.ctypeslib.ndpointer(dtype=np.int64, flags="C_CONTIGUOUS")
_f64p = np.ctypeslib.ndpointer(dtype=np.float64, flags="C_CONTIGUOUS")


def configure(L):
    """Declare the C signatures on a loaded oracle library handle."""
    i32, i64, dbl = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
    L.pkv_oracle_gather_paged.argtypes = [_u16p, i64, _i32p, i32, i32, i32,
                                          i32, i32, _u16p]
    L.pkv_oracle_gather_contig.argtypes = [_u16p, i32, i32, i64, i32, i32,
                                           i32, i32, _u16p]
    L.pkv_oracle_attend.argtypes = [_u16p, _u16p, _u16p, i32, i32, dbl,
                                    _f64p, _f64p]
    L.pkv_oracle_attend.restype = None
    L.pkv_oracle_paged_decode.argtypes = [_u16p, _u16p, _u16p, i64, _i32p,
                                          i32, _i32p, i32, i32, i32, i32,
                                          i32, dbl, _f64p, ctypes.c_int]
    L.pkv_oracle_contig_decode.argtypes = [_u16p, _u16p, _u16p, _i32p, i32,
                                           _i32p, i32, i32, i32, i32, i64,
                                           dbl, _f64p, ctypes.c_int]
    L.pkv_oracle_paged_prefill.argtypes = [_u16p, _u16p, _u16p, i64, _i32p, i32, _i32p,
                                           _i32p, i32, i32, i32, i32, i32, dbl, _f64p,
                                           ctypes.c_int]
    L.pkv_oracle_kv_append.argtypes = [_i64p, i64, _u16p, _u16p, _u16p,
                                       _u16p, i64, i64, i32, i32]
    L.pkv_oracle_block_copy.argtypes = [_i64p, i64, ctypes.c_void_p,
                                        ctypes.c_void_p, i32, i64, i64]
    for name in ("pkv_oracle_gather_paged", "pkv_oracle_gather_contig",
                 "pkv_oracle_paged_decode", "pkv_oracle_contig_decode",
                 "pkv_oracle_paged_prefill",
                 "pkv_oracle_kv_append", "pkv_oracle_block_copy"):
        getattr(L, name).restype = ctypes.c_int
    return L


def lib():
    """Load (building first if needed) the oracle library."""
    global _lib
    if _lib is None:
        _lib = configure(ctypes.CDLL(_build()))
    return _lib


def _u16(a):
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError("bf16 arrays are passed as uint16 bit patterns")
    return a


def _check(rc, what):
    if rc != 0:
        raise ValueError("%s failed with code %d" % (what, rc))


def gather_paged(cache, block_table_row, ctx, bs, h):
    """Logical rows [ctx, D] of KV head h of one sequence, via its block table."""
    cache = _u16(cache)
    nb, hkv, bs_c, d = cache.shape
    assert bs_c == bs
    out = np.zeros((max(ctx, 0), d), dtype=np.uint16)
    row = np.ascontiguousarray(block_table_row, dtype=np.int32)
    _check(lib().pkv_oracle_gather_paged(cache, nb, row, ctx, hkv, bs, d, h,
                                         out), "gather_paged")
    return out


def gather_contig(buf, req_id, ctx, h):
    """Logical rows [ctx, D] of KV head h of request req_id (offset reqId x S)."""
    buf = _u16(buf)
    max_reqs, hkv, S, d = buf.shape
    out = np.zeros((max(ctx, 0), d), dtype=np.uint16)
    _check(lib().pkv_oracle_gather_contig(buf, max_reqs, req_id, S, ctx, hkv,
                                          d, h, out), "gather_contig")
    return out


def attend(q, K, V, scale):
    """fp64 softmax(scale * q K^T) V for one query [D] over rows K, V [ctx, D]."""
    q, K, V = _u16(q), _u16(K), _u16(V)
    ctx, d = K.shape
    o = np.zeros(d, dtype=np.float64)
    scores = np.zeros(max(ctx, 1), dtype=np.float64)
    lib().pkv_oracle_attend(q, K, V, ctx, d, float(scale), scores, o)
    return o


def paged_decode(q, k_cache, v_cache, block_tables, context_lens, scale,
                 nthreads=0):
    """fp64 decode attention, paged layout.  Returns out [B, Hq, D] float64."""
    q, k_cache, v_cache = _u16(q), _u16(k_cache), _u16(v_cache)
    B, hq, d = q.shape
    nb, hkv, bs, d2 = k_cache.shape
    assert d == d2 and v_cache.shape == k_cache.shape
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    out = np.zeros((B, hq, d), dtype=np.float64)
    _check(lib().pkv_oracle_paged_decode(q, k_cache, v_cache, nb, bt,
                                         bt.shape[1] if bt.ndim == 2 else 0,
                                         cl, B, hq, hkv, d, bs, float(scale),
                                         out, int(nthreads)), "paged_decode")
    return out


def paged_prefill(q, k_cache, v_cache, block_tables, context_lens, cu_q, scale, nthreads=0):
    """fp64 causal prefill, paged layout: q [T, Hq, D] holds every
    sequence's chunk of new tokens (sequence i: rows cu_q[i] .. cu_q[i+1]-1,
    the last positions of its context_lens[i]).  Returns out [T, Hq, D]."""
    q, k_cache, v_cache = _u16(q), _u16(k_cache), _u16(v_cache)
    T, hq, d = q.shape
    nb, hkv, bs, d2 = k_cache.shape
    assert d == d2 and v_cache.shape == k_cache.shape
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    cu = np.ascontiguousarray(cu_q, dtype=np.int32)
    assert cu[-1] == T
    out = np.zeros((T, hq, d), dtype=np.float64)
    _check(lib().pkv_oracle_paged_prefill(q, k_cache, v_cache, nb, bt, bt.shape[1], cl, cu,
                                          len(cl), hq, hkv, d, bs, float(scale), out,
                                          int(nthreads)), "paged_prefill")
    return out


def contig_decode(q, k_buf, v_buf, req_ids, context_lens, scale, nthreads=0):
    """fp64 decode attention, contiguous layout [max_reqs, Hkv, S, D]."""
    q, k_buf, v_buf = _u16(q), _u16(k_buf), _u16(v_buf)
    B, hq, d = q.shape
    max_reqs, hkv, S, d2 = k_buf.shape
    assert d == d2 and v_buf.shape == k_buf.shape
    rid = np.ascontiguousarray(req_ids, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    out = np.zeros((B, hq, d), dtype=np.float64)
    _check(lib().pkv_oracle_contig_decode(q, k_buf, v_buf, rid, max_reqs, cl,
                                          B, hq, hkv, d, S, float(scale), out,
                                          int(nthreads)), "contig_decode")
    return out


def kv_append(slot_mapping, k, v, k_cache, v_cache):
    """Write new K/V rows [T, Hkv, D] into the caches in place at their slots.

    The caches are [num_blocks, Hkv, bs, D] (or [max_reqs, Hkv, S, D] with the
    slot counted in tokens of S)."""
    k, v = _u16(k), _u16(v)
    for c in (k_cache, v_cache):
        if not (isinstance(c, np.ndarray) and c.dtype == np.uint16
                and c.flags["C_CONTIGUOUS"]):
            raise TypeError("caches must be C-contiguous uint16 arrays")
    nb, hkv, bs, d = k_cache.shape
    sm = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    _check(lib().pkv_oracle_kv_append(sm, sm.shape[0], k, v, k_cache, v_cache,
                                      nb * bs, bs, hkv, d), "kv_append")


def block_copy(pairs, k_caches, v_caches):
    """Copy whole blocks src -> dst for every (src, dst) pair in every layer."""
    pairs = np.ascontiguousarray(pairs, dtype=np.int64).reshape(-1, 2)
    L = len(k_caches)
    assert len(v_caches) == L and L > 0
    for c in list(k_caches) + list(v_caches):
        if not (c.dtype == np.uint16 and c.flags["C_CONTIGUOUS"]
                and c.shape == k_caches[0].shape):
            raise TypeError("caches must be C-contiguous uint16 of one shape")
    nb = k_caches[0].shape[0]
    block_elems = int(np.prod(k_caches[0].shape[1:]))
    kp = (ctypes.c_void_p * L)(*[c.ctypes.data for c in k_caches])
    vp = (ctypes.c_void_p * L)(*[c.ctypes.data for c in v_caches])
    _check(lib().pkv_oracle_block_copy(pairs, pairs.shape[0], kp, vp, L, nb,
                                       block_elems), "block_copy")


def block_swap(pairs, src_k, src_v, dst_k, dst_v):
    """Swap of whole blocks between two pools ("Running Out of Cache",
    closing paragraph, and the glossary entry "Pre-emption": an evicted
    request's cache is swapped out and brought back later).  For every
    (src, dst) pair and every layer, block src of the source pool's K and V
    becomes block dst of the destination pool's.  Plain numpy indexing, one
    block at a time, in pair order."""
    pairs = np.asarray(pairs, dtype=np.int64).reshape(-1, 2)
    L = len(src_k)
    assert len(src_v) == len(dst_k) == len(dst_v) == L and L > 0
    for src, dst in pairs:
        for layer in range(L):
            dst_k[layer][dst] = src_k[layer][src]
            dst_v[layer][dst] = src_v[layer][src]
