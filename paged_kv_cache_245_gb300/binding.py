"""Python binding of the C ABI in ``include/pkv.h`` (argument marshalling only).

Every function takes torch CUDA tensors, checks their dtype/shape/contiguity,
and passes raw device pointers and the current CUDA stream to the compiled
library ``libpkv.so``.  All computation happens in the library's kernels;
there is no fallback of any kind: if the library is missing or fails to load,
every call raises.
"""
import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpkv.so")

PKV_OK = 0
PKV_ERR_INVALID_ARG = 1
PKV_ERR_OUT_OF_BLOCKS = 6
STATUS_NAMES = {0: "PKV_OK", 1: "PKV_ERR_INVALID_ARG", 2: "PKV_ERR_UNSUPPORTED",
                3: "PKV_ERR_WORKSPACE", 4: "PKV_ERR_CUDA", 5: "PKV_ERR_DEVICE_BOUNDS",
                6: "PKV_ERR_OUT_OF_BLOCKS"}
DEVERR_NAMES = {0: "none", 1: "block_id", 2: "slot", 3: "req_id", 4: "context",
                5: "copy_pair", 6: "timeout"}

EXPORTED = ("pkv_kv_append", "pkv_decode_num_splits", "pkv_decode_uses_tensor_cores",
            "pkv_decode_workspace_size",
            "pkv_paged_decode_attention", "pkv_contig_decode_attention", "pkv_block_copy",
            "pkv_set_checked", "pkv_get_checked", "pkv_set_split_tiles",
            "pkv_set_decode_variant", "pkv_get_decode_variant", "pkv_debug_stall_next_decode",
            "pkv_debug_drop_next_piece_record",
            "pkv_paged_decode_step", "pkv_contig_decode_step", "pkv_debug_gather_paged",
            "pkv_debug_gather_contig", "pkv_paged_decode_attention_shared",
            "pkv_shared_decode_workspace_size", "pkv_shared_decode_launches",
            "pkv_paged_prefill_attention",
            "pkv_contig_prefill_attention", "pkv_block_swap",
            "pkv_get_device_error", "pkv_status_string", "pkv_last_error")


class PkvError(RuntimeError):
    def __init__(self, status, message):
        super().__init__("%s: %s" % (STATUS_NAMES.get(status, status), message))
        self.status = status


class Heads(ctypes.Structure):
    _fields_ = [("num_q_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32)]


_lib = None


def lib():
    """The loaded C library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError("libpkv.so is not built (%s); run __graft_entry__.build() "
                           "or paged_kv_cache_245_gb300/build.py" % LIB_PATH)
    L = ctypes.CDLL(LIB_PATH)
    vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    L.pkv_kv_append.argtypes = [vp, i64, vp, vp, vp, vp, i64, i64, Heads, vp]
    L.pkv_decode_num_splits.argtypes = [i32, Heads, i32]
    L.pkv_decode_num_splits.restype = i32
    L.pkv_decode_uses_tensor_cores.argtypes = [i32, Heads, i32, i32]
    L.pkv_decode_uses_tensor_cores.restype = i32
    L.pkv_decode_workspace_size.argtypes = [i32, Heads, i32]
    L.pkv_decode_workspace_size.restype = sz
    L.pkv_paged_decode_attention.argtypes = [vp, vp, vp, vp, i32, i32, vp, i32, i32, i32,
                                             ctypes.c_float, Heads, vp, vp, sz, vp]
    L.pkv_contig_decode_attention.argtypes = [vp, vp, vp, vp, i32, vp, i32, i32, i64,
                                              ctypes.c_float, Heads, vp, vp, sz, vp]
    L.pkv_block_copy.argtypes = [vp, i64, vp, vp, i32, i64, i64, vp]
    L.pkv_block_swap.argtypes = [vp, i64, vp, vp, i64, vp, vp, i64, i32, i64, vp]
    L.pkv_paged_decode_step.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i32, vp, i32, i32, i32,
                                        ctypes.c_float, Heads, vp, vp, sz, vp]
    L.pkv_contig_decode_step.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, vp, i32, i32, i64,
                                         ctypes.c_float, Heads, vp, vp, sz, vp]
    L.pkv_paged_prefill_attention.argtypes = [vp, vp, i32, vp, vp, vp, i32, i32, vp, i32, i32,
                                              i32, ctypes.c_float, Heads, vp, vp]
    L.pkv_contig_prefill_attention.argtypes = [vp, vp, i32, vp, vp, vp, i32, vp, i32, i32, i64,
                                               ctypes.c_float, Heads, vp, vp]
    L.pkv_shared_decode_workspace_size.argtypes = [i32, i32, i32, i32, Heads]
    L.pkv_shared_decode_workspace_size.restype = sz
    L.pkv_shared_decode_launches.argtypes = [i32, i32, i32, i32, i32, i32, i32, Heads]
    L.pkv_shared_decode_launches.restype = i32
    L.pkv_paged_decode_attention_shared.argtypes = [vp, vp, vp, vp, i32, i32, vp, i32, i32, i32,
                                                    vp, vp, i32, i32, i32, ctypes.c_float, Heads,
                                                    vp, vp, sz, vp]
    L.pkv_debug_gather_paged.argtypes = [vp, vp, i32, i32, vp, i32, i32, i32, i32, vp, vp]
    L.pkv_debug_gather_contig.argtypes = [vp, vp, i32, vp, i32, i32, i64, i32, vp, vp]
    L.pkv_set_checked.argtypes = [ctypes.c_int]
    L.pkv_set_checked.restype = None
    L.pkv_get_checked.restype = ctypes.c_int
    L.pkv_debug_stall_next_decode.restype = None
    L.pkv_debug_drop_next_piece_record.restype = None
    L.pkv_set_decode_variant.argtypes = [ctypes.c_int]
    L.pkv_set_decode_variant.restype = None
    L.pkv_get_decode_variant.restype = ctypes.c_int
    L.pkv_set_split_tiles.argtypes = [i32]
    L.pkv_set_split_tiles.restype = None
    L.pkv_get_device_error.argtypes = [ctypes.POINTER(ctypes.c_int)]
    L.pkv_status_string.argtypes = [ctypes.c_int]
    L.pkv_status_string.restype = ctypes.c_char_p
    L.pkv_last_error.restype = ctypes.c_char_p
    for name in ("pkv_kv_append", "pkv_paged_decode_attention", "pkv_contig_decode_attention",
                 "pkv_block_copy", "pkv_block_swap", "pkv_get_device_error"):
        getattr(L, name).restype = ctypes.c_int
    _lib = L
    return L


def _check(status):
    if status != PKV_OK:
        raise PkvError(status, lib().pkv_last_error().decode())


def _stream(t):
    return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _need(t, dtype, name, ndim=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError("%s must be a CUDA tensor" % name)
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if ndim is not None and t.dim() != ndim:
        raise ValueError("%s must have %d dims" % (name, ndim))


def heads(num_q_heads, num_kv_heads, head_dim=128):
    return Heads(int(num_q_heads), int(num_kv_heads), int(head_dim))


# ---------------------------------------------------------------- operations

def kv_append(slot_mapping, k, v, k_cache, v_cache):
    """Write new rows k, v [T, Hkv, D] into the caches at slot_mapping [T]
    (int64; slot = block * block_size + offset; negative = skip).  The caches
    are [num_blocks, Hkv, block_size, D] (or [max_reqs, Hkv, S, D])."""
    _need(slot_mapping, torch.int64, "slot_mapping", 1)
    for t, n in ((k, "k"), (v, "v")):
        _need(t, torch.bfloat16, n, 3)
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, torch.bfloat16, n, 4)
    nb, hkv, bs, d = k_cache.shape
    if tuple(v_cache.shape) != tuple(k_cache.shape) or k.shape != v.shape:
        raise ValueError("k/v and cache shapes must match")
    if k.shape[1] != hkv or k.shape[2] != d or k.shape[0] != slot_mapping.shape[0]:
        raise ValueError("k must be [T, Hkv, D] matching the cache and slot_mapping")
    _check(lib().pkv_kv_append(_ptr(slot_mapping), k.shape[0], _ptr(k), _ptr(v),
                               _ptr(k_cache), _ptr(v_cache), nb * bs, bs,
                               heads(hkv, hkv, d), _stream(k_cache)))


def decode_num_splits(num_seqs, num_q_heads, num_kv_heads, max_context, head_dim=128):
    return int(lib().pkv_decode_num_splits(num_seqs, heads(num_q_heads, num_kv_heads, head_dim),
                                           max_context))


def decode_uses_tensor_cores(num_seqs, num_q_heads, num_kv_heads, max_context, block_size,
                             head_dim=128):
    """True when the decode calls run the tensor-core kernel for this batch
    (block_size 0: the contiguous layout)."""
    r = int(lib().pkv_decode_uses_tensor_cores(num_seqs, heads(num_q_heads, num_kv_heads, head_dim),
                                               max_context, block_size))
    if r < 0:
        raise ValueError("bad arguments")
    return r == 1


def decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, max_context, head_dim=128):
    return int(lib().pkv_decode_workspace_size(num_seqs, heads(num_q_heads, num_kv_heads,
                                                               head_dim), max_context))


def shared_decode_launches(num_seqs, num_groups, max_group_size, max_blocks_per_seq, max_context,
                           block_size, max_own_tokens, num_q_heads, num_kv_heads, head_dim=128):
    """Kernel launches of one shared-prefix decode call with these sizes (-1: rejected)."""
    return int(lib().pkv_shared_decode_launches(
        num_seqs, num_groups, max_group_size, max_blocks_per_seq, max_context, block_size,
        max_own_tokens, heads(num_q_heads, num_kv_heads, head_dim)))


def _workspace(workspace, q, nbytes):
    if nbytes == 0:
        return workspace
    if workspace is None:
        # convenience for callers without their own buffer; the C ABI itself never allocates
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    return workspace


def paged_decode_attention(q, k_cache, v_cache, block_tables, context_lens, max_context,
                           scale, out=None, workspace=None):
    """out[i, h] = softmax(scale * q[i, h] . K) V over the context_lens[i]
    positions that block_tables[i] maps into the paged caches."""
    _need(q, torch.bfloat16, "q", 3)
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, torch.bfloat16, n, 4)
    _need(block_tables, torch.int32, "block_tables", 2)
    _need(context_lens, torch.int32, "context_lens", 1)
    B, hq, d = q.shape
    nb, hkv, bs, d2 = k_cache.shape
    if d != d2 or tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("q / cache shapes disagree")
    if block_tables.shape[0] != B or context_lens.shape[0] != B:
        raise ValueError("block_tables / context_lens must have num_seqs rows")
    if out is None:
        out = torch.empty_like(q)
    _need(out, torch.bfloat16, "out", 3)
    h = heads(hq, hkv, d)
    nbytes = lib().pkv_decode_workspace_size(B, h, int(max_context)) if B > 0 else 0
    workspace = _workspace(workspace, q, nbytes)
    ws_ptr = _ptr(workspace) if workspace is not None else ctypes.c_void_p(0)
    ws_len = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib().pkv_paged_decode_attention(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), block_tables.shape[1], nb,
        _ptr(context_lens), B, int(max_context), bs, float(scale), h, _ptr(out), ws_ptr,
        ws_len, _stream(q)))
    return out


def contig_decode_attention(q, k_buf, v_buf, req_ids, context_lens, max_context, scale,
                            out=None, workspace=None):
    """Decode attention over per-request sub-tensors: request i's rows are
    k_buf[req_ids[i], h, :context_lens[i]] (offset reqId x S)."""
    _need(q, torch.bfloat16, "q", 3)
    for t, n in ((k_buf, "k_buf"), (v_buf, "v_buf")):
        _need(t, torch.bfloat16, n, 4)
    _need(req_ids, torch.int32, "req_ids", 1)
    _need(context_lens, torch.int32, "context_lens", 1)
    B, hq, d = q.shape
    max_reqs, hkv, S, d2 = k_buf.shape
    if d != d2 or tuple(v_buf.shape) != tuple(k_buf.shape):
        raise ValueError("q / buffer shapes disagree")
    if req_ids.shape[0] != B or context_lens.shape[0] != B:
        raise ValueError("req_ids / context_lens must have num_seqs rows")
    if out is None:
        out = torch.empty_like(q)
    _need(out, torch.bfloat16, "out", 3)
    h = heads(hq, hkv, d)
    nbytes = lib().pkv_decode_workspace_size(B, h, int(max_context)) if B > 0 else 0
    workspace = _workspace(workspace, q, nbytes)
    ws_ptr = _ptr(workspace) if workspace is not None else ctypes.c_void_p(0)
    ws_len = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib().pkv_contig_decode_attention(
        _ptr(q), _ptr(k_buf), _ptr(v_buf), _ptr(req_ids), max_reqs, _ptr(context_lens), B,
        int(max_context), S, float(scale), h, _ptr(out), ws_ptr, ws_len, _stream(q)))
    return out


def _check_new_rows(slot_mapping, k_new, v_new, B, hkv, d):
    _need(slot_mapping, torch.int64, "slot_mapping", 1)
    for t, n in ((k_new, "k_new"), (v_new, "v_new")):
        _need(t, torch.bfloat16, n, 3)
        if tuple(t.shape) != (B, hkv, d):
            raise ValueError("%s must be [num_seqs, Hkv, D]" % n)
    if slot_mapping.shape[0] != B:
        raise ValueError("slot_mapping must have num_seqs entries")


def paged_decode_step(slot_mapping, k_new, v_new, q, k_cache, v_cache, block_tables,
                      context_lens, max_context, scale, out=None, workspace=None):
    """One decode step of one layer in one call: kv_append(slot_mapping, k_new,
    v_new, k_cache, v_cache) then paged_decode_attention(q, ...); the same
    bytes as the two calls."""
    _need(q, torch.bfloat16, "q", 3)
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, torch.bfloat16, n, 4)
    _need(block_tables, torch.int32, "block_tables", 2)
    _need(context_lens, torch.int32, "context_lens", 1)
    B, hq, d = q.shape
    nb, hkv, bs, d2 = k_cache.shape
    if d != d2 or tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("q / cache shapes disagree")
    if block_tables.shape[0] != B or context_lens.shape[0] != B:
        raise ValueError("block_tables / context_lens must have num_seqs rows")
    _check_new_rows(slot_mapping, k_new, v_new, B, hkv, d)
    if out is None:
        out = torch.empty_like(q)
    _need(out, torch.bfloat16, "out", 3)
    h = heads(hq, hkv, d)
    nbytes = lib().pkv_decode_workspace_size(B, h, int(max_context)) if B > 0 else 0
    workspace = _workspace(workspace, q, nbytes)
    ws_ptr = _ptr(workspace) if workspace is not None else ctypes.c_void_p(0)
    ws_len = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib().pkv_paged_decode_step(
        _ptr(slot_mapping), _ptr(k_new), _ptr(v_new), _ptr(q), _ptr(k_cache), _ptr(v_cache),
        _ptr(block_tables), block_tables.shape[1], nb, _ptr(context_lens), B, int(max_context),
        bs, float(scale), h, _ptr(out), ws_ptr, ws_len, _stream(q)))
    return out


def contig_decode_step(slot_mapping, k_new, v_new, q, k_buf, v_buf, req_ids, context_lens,
                       max_context, scale, out=None, workspace=None):
    """kv_append into the request rows (slot = reqId * S + position) then
    contig_decode_attention, as one call."""
    _need(q, torch.bfloat16, "q", 3)
    for t, n in ((k_buf, "k_buf"), (v_buf, "v_buf")):
        _need(t, torch.bfloat16, n, 4)
    _need(req_ids, torch.int32, "req_ids", 1)
    _need(context_lens, torch.int32, "context_lens", 1)
    B, hq, d = q.shape
    max_reqs, hkv, S, d2 = k_buf.shape
    if d != d2 or tuple(v_buf.shape) != tuple(k_buf.shape):
        raise ValueError("q / buffer shapes disagree")
    if req_ids.shape[0] != B or context_lens.shape[0] != B:
        raise ValueError("req_ids / context_lens must have num_seqs rows")
    _check_new_rows(slot_mapping, k_new, v_new, B, hkv, d)
    if out is None:
        out = torch.empty_like(q)
    _need(out, torch.bfloat16, "out", 3)
    h = heads(hq, hkv, d)
    nbytes = lib().pkv_decode_workspace_size(B, h, int(max_context)) if B > 0 else 0
    workspace = _workspace(workspace, q, nbytes)
    ws_ptr = _ptr(workspace) if workspace is not None else ctypes.c_void_p(0)
    ws_len = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib().pkv_contig_decode_step(
        _ptr(slot_mapping), _ptr(k_new), _ptr(v_new), _ptr(q), _ptr(k_buf), _ptr(v_buf),
        _ptr(req_ids), max_reqs, _ptr(context_lens), B, int(max_context), S, float(scale), h,
        _ptr(out), ws_ptr, ws_len, _stream(q)))
    return out


def paged_decode_attention_shared(q, k_cache, v_cache, block_tables, context_lens, max_context,
                                  scale, group_start, shared_blocks, max_group_size,
                                  max_own_tokens=-1, out=None, workspace=None):
    """Paged decode attention where groups of consecutive sequences share
    their first shared_blocks[g] blocks (group_start [G+1], shared_blocks [G]:
    int32 on the device; max_group_size a host bound): the shared positions
    are read once for several sequences."""
    _need(q, torch.bfloat16, "q", 3)
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, torch.bfloat16, n, 4)
    _need(block_tables, torch.int32, "block_tables", 2)
    _need(context_lens, torch.int32, "context_lens", 1)
    _need(group_start, torch.int32, "group_start", 1)
    _need(shared_blocks, torch.int32, "shared_blocks", 1)
    B, hq, d = q.shape
    nb, hkv, bs, d2 = k_cache.shape
    G = shared_blocks.shape[0]
    if group_start.shape[0] != G + 1:
        raise ValueError("group_start must have num_groups + 1 entries")
    if out is None:
        out = torch.empty_like(q)
    _need(out, torch.bfloat16, "out", 3)
    h = heads(hq, hkv, d)
    nbytes = lib().pkv_shared_decode_workspace_size(B, G, int(max_group_size),
                                                    block_tables.shape[1], h)
    if workspace is None:
        workspace = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=q.device)
    _check(lib().pkv_paged_decode_attention_shared(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), block_tables.shape[1], nb,
        _ptr(context_lens), B, int(max_context), bs, _ptr(group_start), _ptr(shared_blocks), G,
        int(max_group_size), int(max_own_tokens), float(scale), h, _ptr(out), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(q)))
    return out


def paged_prefill_attention(q, cu_seqlens_q, k_cache, v_cache, block_tables, context_lens,
                            max_q_tokens, scale, out=None):
    """Causal prefill: q [T, Hq, D] packs every sequence's chunk of new tokens
    (sequence i: rows cu_seqlens_q[i] .. cu_seqlens_q[i+1]-1, the last
    positions of its context_lens[i]; their K/V already appended)."""
    _need(q, torch.bfloat16, "q", 3)
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, torch.bfloat16, n, 4)
    _need(cu_seqlens_q, torch.int32, "cu_seqlens_q", 1)
    _need(block_tables, torch.int32, "block_tables", 2)
    _need(context_lens, torch.int32, "context_lens", 1)
    T, hq, d = q.shape
    nb, hkv, bs, d2 = k_cache.shape
    B = context_lens.shape[0]
    if cu_seqlens_q.shape[0] != B + 1 or block_tables.shape[0] != B:
        raise ValueError("cu_seqlens_q must have num_seqs + 1 entries, block_tables num_seqs rows")
    if out is None:
        out = torch.empty_like(q)
    _need(out, torch.bfloat16, "out", 3)
    _check(lib().pkv_paged_prefill_attention(
        _ptr(q), _ptr(cu_seqlens_q), T, _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
        block_tables.shape[1], nb, _ptr(context_lens), B, int(max_q_tokens), bs, float(scale),
        heads(hq, hkv, d), _ptr(out), _stream(q)))
    return out


def contig_prefill_attention(q, cu_seqlens_q, k_buf, v_buf, req_ids, context_lens,
                             max_q_tokens, scale, out=None):
    """Causal prefill over per-request sub-tensors: sequence i's rows are
    k_buf[req_ids[i], h, :context_lens[i]] (offset reqId x S); q,
    cu_seqlens_q and out as in paged_prefill_attention."""
    _need(q, torch.bfloat16, "q", 3)
    for t, n in ((k_buf, "k_buf"), (v_buf, "v_buf")):
        _need(t, torch.bfloat16, n, 4)
    _need(cu_seqlens_q, torch.int32, "cu_seqlens_q", 1)
    _need(req_ids, torch.int32, "req_ids", 1)
    _need(context_lens, torch.int32, "context_lens", 1)
    T, hq, d = q.shape
    max_reqs, hkv, S, d2 = k_buf.shape
    B = context_lens.shape[0]
    if d != d2 or tuple(v_buf.shape) != tuple(k_buf.shape):
        raise ValueError("q / buffer shapes disagree")
    if cu_seqlens_q.shape[0] != B + 1 or req_ids.shape[0] != B:
        raise ValueError("cu_seqlens_q must have num_seqs + 1 entries, req_ids num_seqs")
    if out is None:
        out = torch.empty_like(q)
    _need(out, torch.bfloat16, "out", 3)
    _check(lib().pkv_contig_prefill_attention(
        _ptr(q), _ptr(cu_seqlens_q), T, _ptr(k_buf), _ptr(v_buf), _ptr(req_ids), max_reqs,
        _ptr(context_lens), B, int(max_q_tokens), S, float(scale), heads(hq, hkv, d), _ptr(out),
        _stream(q)))
    return out


def debug_gather_paged(cache, block_tables, context_lens, max_context):
    """Test-only: the logical rows [B, Hkv, max_context, D] the decode kernels
    read through block_tables (zeros past each context)."""
    _need(cache, torch.bfloat16, "cache", 4)
    _need(block_tables, torch.int32, "block_tables", 2)
    _need(context_lens, torch.int32, "context_lens", 1)
    nb, hkv, bs, d = cache.shape
    B = context_lens.shape[0]
    out = torch.empty((B, hkv, int(max_context), d), dtype=torch.bfloat16, device=cache.device)
    _check(lib().pkv_debug_gather_paged(_ptr(cache), _ptr(block_tables), block_tables.shape[1],
                                        nb, _ptr(context_lens), B, int(max_context), bs, hkv,
                                        _ptr(out), _stream(cache)))
    return out


def debug_gather_contig(buf, req_ids, context_lens, max_context):
    """Test-only: the logical rows of request rows req_ids (offset reqId x S)."""
    _need(buf, torch.bfloat16, "buf", 4)
    _need(req_ids, torch.int32, "req_ids", 1)
    _need(context_lens, torch.int32, "context_lens", 1)
    max_reqs, hkv, S, d = buf.shape
    B = context_lens.shape[0]
    out = torch.empty((B, hkv, int(max_context), d), dtype=torch.bfloat16, device=buf.device)
    _check(lib().pkv_debug_gather_contig(_ptr(buf), _ptr(req_ids), max_reqs, _ptr(context_lens),
                                         B, int(max_context), S, hkv, _ptr(out), _stream(buf)))
    return out


def block_copy(src_dst_pairs, k_caches, v_caches):
    """Copy whole blocks src -> dst (pairs [n, 2] int64 on the device) in every
    layer's K and V cache (lists of [num_blocks, ...] bf16 tensors)."""
    _need(src_dst_pairs, torch.int64, "src_dst_pairs", 2)
    L = len(k_caches)
    if L != len(v_caches) or L == 0:
        raise ValueError("need one K and one V cache per layer")
    shape = tuple(k_caches[0].shape)
    for t in list(k_caches) + list(v_caches):
        _need(t, torch.bfloat16, "cache")
        if tuple(t.shape) != shape:
            raise ValueError("all caches must have one shape")
    nb = shape[0]
    block_bytes = k_caches[0][0].numel() * 2
    kp = (ctypes.c_void_p * L)(*[t.data_ptr() for t in k_caches])
    vp = (ctypes.c_void_p * L)(*[t.data_ptr() for t in v_caches])
    _check(lib().pkv_block_copy(_ptr(src_dst_pairs), src_dst_pairs.shape[0], kp, vp, L, nb,
                                block_bytes, _stream(k_caches[0])))


def block_swap(pairs, src_k, src_v, dst_k, dst_v):
    """Copy whole blocks from one pool to another, pairs [n, 2] int64 of
    (src block, dst block), in every layer's K and V (lists of [blocks, ...]
    bf16 tensors, one shape per side).  Either side may be page-locked host
    memory (``tensor.pin_memory()``): that is the swap of pre-empted
    sequences out of, and back into, the device cache.  pairs may be a
    device tensor or a pinned host tensor."""
    if pairs.dtype != torch.int64 or pairs.dim() != 2 or pairs.shape[1] != 2 \
            or not pairs.is_contiguous():
        raise ValueError("pairs must be a contiguous [n, 2] int64 tensor")
    L = len(src_k)
    if not (L == len(src_v) == len(dst_k) == len(dst_v)) or L == 0:
        raise ValueError("need one K and one V pool per layer on each side")
    blocks = []
    for side in ((src_k, src_v), (dst_k, dst_v)):
        shape = tuple(side[0][0].shape)
        for t in list(side[0]) + list(side[1]):
            if t.dtype != torch.bfloat16 or not t.is_contiguous() or tuple(t.shape) != shape:
                raise ValueError("pools must be contiguous bf16 tensors of one shape per side")
        blocks.append(shape)
    if blocks[0][1:] != blocks[1][1:]:
        raise ValueError("the two sides must have the same block shape")
    block_bytes = src_k[0][0].numel() * 2
    arr = [(ctypes.c_void_p * L)(*[t.data_ptr() for t in x]) for x in (src_k, src_v, dst_k, dst_v)]
    dev = next((t for t in (src_k[0], dst_k[0], pairs) if t.is_cuda), None)
    if dev is None:
        raise ValueError("one side (or pairs) must be on the GPU")
    _check(lib().pkv_block_swap(_ptr(pairs), pairs.shape[0], arr[0], arr[1], blocks[0][0],
                                arr[2], arr[3], blocks[1][0], L, block_bytes, _stream(dev)))


def set_checked(enable):
    lib().pkv_set_checked(1 if enable else 0)


def get_checked():
    return bool(lib().pkv_get_checked())


# decode kernel selection: automatic, the split (CUDA-core) kernel, or the
# tensor-core kernel in its 8-warp x 3-stage / 12-warp x 2-stage CTA shapes
VARIANT_AUTO, VARIANT_SPLIT, VARIANT_TC_8X3, VARIANT_TC_12X2 = 0, 1, 2, 3


def set_decode_variant(variant):
    lib().pkv_set_decode_variant(int(variant))


def get_decode_variant():
    return int(lib().pkv_get_decode_variant())


def set_split_tiles(tiles):
    lib().pkv_set_split_tiles(int(tiles))


def get_device_error():
    """Read and clear the device error word; returns its code name."""
    code = ctypes.c_int(0)
    st = lib().pkv_get_device_error(ctypes.byref(code))
    if st not in (0, 5):
        _check(st)
    return DEVERR_NAMES.get(code.value, code.value)


# ------------------------------------------------------------ block manager

def _bm_lib():
    L = lib()
    if getattr(L, "_bm_ready", False):
        return L
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    L.pkv_bm_create.argtypes = [i32, i32, vp]
    L.pkv_bm_create.restype = vp
    L.pkv_bm_destroy.argtypes = [vp]
    L.pkv_bm_destroy.restype = None
    L.pkv_bm_add_sequence.argtypes = [vp, i64]
    L.pkv_bm_add_sequence.restype = i32
    L.pkv_bm_fork.argtypes = [vp, i32]
    L.pkv_bm_fork.restype = i32
    L.pkv_bm_append.argtypes = [vp, vp, i32, vp, vp, vp]
    L.pkv_bm_append.restype = ctypes.c_int
    L.pkv_bm_free_sequence.argtypes = [vp, i32]
    L.pkv_bm_free_sequence.restype = ctypes.c_int
    L.pkv_bm_block_table.argtypes = [vp, i32, vp, i32]
    L.pkv_bm_block_table.restype = i32
    L.pkv_bm_export.argtypes = [vp, vp, i32, vp, i32, i32, vp]
    L.pkv_bm_export.restype = ctypes.c_int
    L.pkv_bm_length.argtypes = [vp, i32]
    L.pkv_bm_length.restype = i64
    L.pkv_bm_num_free_blocks.argtypes = [vp]
    L.pkv_bm_num_free_blocks.restype = i32
    L.pkv_bm_set_swap_space.argtypes = [vp, i32]
    L.pkv_bm_set_swap_space.restype = ctypes.c_int
    L.pkv_bm_step_blocks.argtypes = [vp, vp, i32]
    L.pkv_bm_step_blocks.restype = i64
    L.pkv_bm_plan_preemption.argtypes = [vp, vp, i32, vp]
    L.pkv_bm_plan_preemption.restype = ctypes.c_int
    L.pkv_bm_preempt.argtypes = [vp, vp, i32, i32, vp, vp]
    L.pkv_bm_preempt.restype = ctypes.c_int
    L.pkv_bm_resume.argtypes = [vp, vp, i32, vp, vp]
    L.pkv_bm_resume.restype = ctypes.c_int
    L.pkv_bm_state.argtypes = [vp, i32]
    L.pkv_bm_state.restype = i32
    L.pkv_bm_num_free_host_blocks.argtypes = [vp]
    L.pkv_bm_num_free_host_blocks.restype = i32
    L.pkv_bm_host_ref_count.argtypes = [vp, i32]
    L.pkv_bm_host_ref_count.restype = i32
    L.pkv_bm_get_counters.argtypes = [vp, ctypes.POINTER(BmCounters)]
    L.pkv_bm_get_counters.restype = ctypes.c_int
    L.pkv_bm_ref_count.argtypes = [vp, i32]
    L.pkv_bm_ref_count.restype = i32
    L._bm_ready = True
    return L


def _np_ptr(a):
    return ctypes.c_void_p(a.ctypes.data)


class BmCounters(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in (
        "cow_copies", "preempted_recompute", "preempted_swap", "resumed",
        "blocks_swapped_out", "blocks_swapped_in", "tokens_recomputed")]


# sequence states and pre-emption modes of include/pkv_block_manager.h
BM_RETIRED, BM_RUNNING, BM_SWAPPED, BM_RECOMPUTE = 0, 1, 2, 3
PREEMPT_RECOMPUTE, PREEMPT_SWAP = 0, 1


class BlockManager:
    """Host block pool of a paged KV cache (include/pkv_block_manager.h):
    sequences, forks that share blocks, and the decode step's slot mapping
    and copy-on-write pairs.  Arrays are numpy on the host."""

    def __init__(self, num_blocks, block_size, free_order=None):
        import numpy as np
        self._np = np
        L = _bm_lib()
        self.block_size = int(block_size)
        order = None
        if free_order is not None:
            order = np.ascontiguousarray(free_order, dtype=np.int32)
            if order.shape != (num_blocks,):
                raise ValueError("free_order must list every block once")
        h = L.pkv_bm_create(int(num_blocks), int(block_size),
                            _np_ptr(order) if order is not None else None)
        if not h:
            raise PkvError(PKV_ERR_INVALID_ARG, L.pkv_last_error().decode())
        self._h = ctypes.c_void_p(h)

    def close(self):
        if self._h:
            _bm_lib().pkv_bm_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def _id(self, r):
        if r < 0:
            msg = _bm_lib().pkv_last_error().decode()
            raise PkvError(PKV_ERR_OUT_OF_BLOCKS if "free blocks" in msg else PKV_ERR_INVALID_ARG,
                           msg)
        return int(r)

    def add_sequence(self, num_tokens):
        return self._id(_bm_lib().pkv_bm_add_sequence(self._h, int(num_tokens)))

    def fork(self, parent):
        return self._id(_bm_lib().pkv_bm_fork(self._h, int(parent)))

    def append(self, seq_ids):
        """One token for each listed sequence: (slot_mapping [n] int64,
        cow_pairs [k, 2] int64)."""
        np = self._np
        ids = np.ascontiguousarray(seq_ids, dtype=np.int32)
        n = ids.shape[0]
        slots = np.empty(n, dtype=np.int64)
        pairs = np.empty((max(n, 1), 2), dtype=np.int64)
        k = ctypes.c_int32(0)
        _check(_bm_lib().pkv_bm_append(self._h, _np_ptr(ids), n, _np_ptr(slots), _np_ptr(pairs),
                                       ctypes.byref(k)))
        return slots, pairs[:k.value].copy()

    def free_sequence(self, seq):
        _check(_bm_lib().pkv_bm_free_sequence(self._h, int(seq)))

    def block_table(self, seq):
        np = self._np
        n = self.length(seq)
        out = np.empty(max((n + self.block_size - 1) // self.block_size, 1), dtype=np.int32)
        k = _bm_lib().pkv_bm_block_table(self._h, int(seq), _np_ptr(out), out.shape[0])
        if k < 0:
            raise PkvError(PKV_ERR_INVALID_ARG, "bad sequence id")
        return out[:k].copy()

    def export(self, seq_ids, max_blocks, filler=0):
        """(block_tables [n, max_blocks] int32, context_lens [n] int32)."""
        np = self._np
        ids = np.ascontiguousarray(seq_ids, dtype=np.int32)
        tables = np.empty((ids.shape[0], max_blocks), dtype=np.int32)
        ctx = np.empty(ids.shape[0], dtype=np.int32)
        _check(_bm_lib().pkv_bm_export(self._h, _np_ptr(ids), ids.shape[0], _np_ptr(tables),
                                       int(max_blocks), int(filler), _np_ptr(ctx)))
        return tables, ctx

    def length(self, seq):
        n = _bm_lib().pkv_bm_length(self._h, int(seq))
        if n < 0:
            raise PkvError(PKV_ERR_INVALID_ARG, "bad sequence id")
        return int(n)

    def num_free_blocks(self):
        return int(_bm_lib().pkv_bm_num_free_blocks(self._h))

    def ref_count(self, block):
        return int(_bm_lib().pkv_bm_ref_count(self._h, int(block)))

    # ---- pre-emption
    def set_swap_space(self, num_host_blocks):
        _check(_bm_lib().pkv_bm_set_swap_space(self._h, int(num_host_blocks)))

    def _ids(self, seq_ids):
        return self._np.ascontiguousarray(seq_ids, dtype=self._np.int32)

    def step_blocks(self, seq_ids):
        """Free blocks an append of these running sequences needs."""
        ids = self._ids(seq_ids)
        n = _bm_lib().pkv_bm_step_blocks(self._h, _np_ptr(ids), ids.shape[0])
        if n < 0:
            raise PkvError(PKV_ERR_INVALID_ARG, _bm_lib().pkv_last_error().decode())
        return int(n)

    def plan_preemption(self, seq_ids):
        """How many of the listed running sequences, taken from the back,
        must be evicted for the rest to append one token each."""
        ids = self._ids(seq_ids)
        k = ctypes.c_int32(0)
        _check(_bm_lib().pkv_bm_plan_preemption(self._h, _np_ptr(ids), ids.shape[0],
                                                ctypes.byref(k)))
        return int(k.value)

    def _held(self, ids):
        return sum(len(self.block_table(int(s))) for s in ids)

    def preempt(self, seq_ids, mode=PREEMPT_RECOMPUTE):
        """Evict running sequences; returns the (device block, host slot)
        swap-out pairs [k, 2] int64 (empty for recompute)."""
        np = self._np
        ids = self._ids(seq_ids)
        pairs = np.empty((max(self._held(ids), 1), 2), dtype=np.int64)
        k = ctypes.c_int32(0)
        _check(_bm_lib().pkv_bm_preempt(self._h, _np_ptr(ids), ids.shape[0], int(mode),
                                        _np_ptr(pairs), ctypes.byref(k)))
        return pairs[:k.value].copy()

    def resume(self, seq_ids):
        """Bring evicted sequences back; returns the (host slot, device
        block) swap-in pairs [k, 2] int64."""
        np = self._np
        ids = self._ids(seq_ids)
        held = sum(len(self.block_table(int(s))) for s in ids if self.state(int(s)) == BM_SWAPPED)
        pairs = np.empty((max(held, 1), 2), dtype=np.int64)
        k = ctypes.c_int32(0)
        _check(_bm_lib().pkv_bm_resume(self._h, _np_ptr(ids), ids.shape[0], _np_ptr(pairs),
                                       ctypes.byref(k)))
        return pairs[:k.value].copy()

    def state(self, seq):
        return int(_bm_lib().pkv_bm_state(self._h, int(seq)))

    def num_free_host_blocks(self):
        return int(_bm_lib().pkv_bm_num_free_host_blocks(self._h))

    def host_ref_count(self, slot):
        return int(_bm_lib().pkv_bm_host_ref_count(self._h, int(slot)))

    def counters(self):
        c = BmCounters()
        _check(_bm_lib().pkv_bm_get_counters(self._h, ctypes.byref(c)))
        return {n: int(getattr(c, n)) for n, _ in BmCounters._fields_}


# ------------------------------------------------------------ on-demand contiguous buffers

def _vmm_lib():
    L = lib()
    if getattr(L, "_vmm_ready", False):
        return L
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    L.pkv_vmm_create.argtypes = [i32, i32, i64, ctypes.POINTER(vp)]
    L.pkv_vmm_create.restype = ctypes.c_int
    L.pkv_vmm_destroy.argtypes = [vp]
    L.pkv_vmm_destroy.restype = None
    L.pkv_vmm_k.argtypes = [vp]
    L.pkv_vmm_k.restype = vp
    L.pkv_vmm_v.argtypes = [vp]
    L.pkv_vmm_v.restype = vp
    L.pkv_vmm_ensure.argtypes = [vp, i32, i64]
    L.pkv_vmm_ensure.restype = ctypes.c_int
    L.pkv_vmm_release.argtypes = [vp, i32]
    L.pkv_vmm_release.restype = ctypes.c_int
    L.pkv_vmm_backed_tokens.argtypes = [vp, i32]
    L.pkv_vmm_backed_tokens.restype = i64
    L.pkv_vmm_stats.argtypes = [vp, ctypes.POINTER(ctypes.c_size_t), ctypes.POINTER(i64),
                                ctypes.POINTER(i64), ctypes.POINTER(i64),
                                ctypes.POINTER(ctypes.c_double)]
    L.pkv_vmm_stats.restype = ctypes.c_int
    L._vmm_ready = True
    return L


class _DeviceArray:
    """A view of device memory the library owns, for torch.as_tensor."""

    def __init__(self, ptr, shape, owner):
        self._owner = owner
        self.__cuda_array_interface__ = {"version": 3, "shape": tuple(shape), "typestr": "<i2",
                                         "data": (int(ptr), False), "strides": None}


class VmmBuffer:
    """K and V tensors [max_reqs, Hkv, S, 128] bf16 whose physical memory is
    mapped on demand (include/pkv_vmm.h).  .k and .v are torch views of the
    whole virtual range: touch only rows that ensure() has backed."""

    def __init__(self, max_reqs, num_kv_heads, S):
        L = _vmm_lib()
        h = ctypes.c_void_p(0)
        _check(L.pkv_vmm_create(int(max_reqs), int(num_kv_heads), int(S), ctypes.byref(h)))
        self._h = h
        shape = (max_reqs, num_kv_heads, S, 128)
        self.shape = shape
        # torch wraps the pointers without touching the memory (no copy); the
        # explicit device index spares it a pointer query, which a reserved but
        # not yet mapped range cannot answer
        dev = torch.device("cuda", torch.cuda.current_device())
        self.k = torch.as_tensor(_DeviceArray(L.pkv_vmm_k(h), shape, self),
                                 device=dev).view(torch.bfloat16)
        self.v = torch.as_tensor(_DeviceArray(L.pkv_vmm_v(h), shape, self),
                                 device=dev).view(torch.bfloat16)
        assert self.k.data_ptr() == L.pkv_vmm_k(h) and self.v.data_ptr() == L.pkv_vmm_v(h)

    def ensure(self, req, tokens):
        _check(_vmm_lib().pkv_vmm_ensure(self._h, int(req), int(tokens)))

    def release(self, req):
        _check(_vmm_lib().pkv_vmm_release(self._h, int(req)))

    def backed_tokens(self, req):
        return int(_vmm_lib().pkv_vmm_backed_tokens(self._h, int(req)))

    def stats(self):
        pb = ctypes.c_size_t(0)
        mp, cp, mc = ctypes.c_int64(0), ctypes.c_int64(0), ctypes.c_int64(0)
        secs = ctypes.c_double(0.0)
        _check(_vmm_lib().pkv_vmm_stats(self._h, ctypes.byref(pb), ctypes.byref(mp),
                                        ctypes.byref(cp), ctypes.byref(mc), ctypes.byref(secs)))
        return {"page_bytes": pb.value, "mapped_pages": mp.value, "created_pages": cp.value,
                "map_calls": mc.value, "map_seconds": secs.value}

    def close(self):
        if self._h is not None and self._h.value:
            self.k = self.v = None
            _vmm_lib().pkv_vmm_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
