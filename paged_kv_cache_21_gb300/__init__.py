"""Thin Python binding of libpagedkv, the GB300 paged KV-cache decode library.

Argument marshalling only: every step of the decode path (slot mapping,
append, attention, split merge) runs in the native library declared in
``include/paged_kv.h``.  Importing this package without the built library
raises ``ImportError``; there is no fallback.

Typical decode step for one layer::

    alloc = BlockAllocator(num_blocks, kv_heads, head_dim)
    slots, tables, lens, cow = alloc.step(seq_ids, max_blocks)      # host
    kv_copy_blocks(k_cache, v_cache, cow_src, cow_dst)              # if any copy-on-write
    kv_append(k_new, v_new, k_cache, v_cache, slots_dev)            # GPU
    paged_decode_attention(out, q, k_cache, v_cache, tables_dev, lens_dev, scale, ws)  # GPU
"""
import ctypes
import os

import numpy as np

from .build import LIB as _LIB_PATH

KV_OK = 0
KV_ERR_INVALID_ARG = -1
KV_ERR_OUT_OF_BLOCKS = -2
KV_ERR_UNSUPPORTED = -3
KV_ERR_CUDA = -4
KV_ERR_NOT_FOUND = -5
KV_ERR_EXISTS = -6
KV_ERR_TOO_LARGE = -7
NOALLOC_WORKSPACE_BYTES = 16 << 20

BF16 = 0
FP8_E4M3 = 1
F32 = 2
BLOCK_SIZE = 16

DEVERR_SLOT_OUT_OF_RANGE = 1
DEVERR_BLOCK_OUT_OF_RANGE = 2
DEVERR_CONTEXT_TOO_LONG = 4
DEVERR_PIPELINE_TIMEOUT = 8
DEVERR_BAD_PREFIX = 16

# columns of a kv_alloc_trace row (KV_TRACE_*)
TRACE_KEYS = ("seq_id", "slot", "len", "position", "blocks", "shared_blocks", "cache_bytes",
              "reorder_src")
TRACE_FIELDS = len(TRACE_KEYS)

_ERRNAMES = {KV_ERR_INVALID_ARG: "KV_ERR_INVALID_ARG", KV_ERR_OUT_OF_BLOCKS: "KV_ERR_OUT_OF_BLOCKS",
             KV_ERR_UNSUPPORTED: "KV_ERR_UNSUPPORTED", KV_ERR_CUDA: "KV_ERR_CUDA",
             KV_ERR_NOT_FOUND: "KV_ERR_NOT_FOUND", KV_ERR_EXISTS: "KV_ERR_EXISTS",
             KV_ERR_TOO_LARGE: "KV_ERR_TOO_LARGE"}


class KVError(RuntimeError):
    def __init__(self, code, what):
        super().__init__("%s failed: %s (%d)" % (what, _ERRNAMES.get(code, "?"), code))
        self.code = code


if not os.path.exists(_LIB_PATH):
    raise ImportError("libpagedkv.so is not built (expected at %s); run "
                      "`python -c 'import __graft_entry__ as g; g.build()'`" % _LIB_PATH)

_lib = ctypes.CDLL(_LIB_PATH)
_p = ctypes.c_void_p
_i = ctypes.c_int
_i64 = ctypes.c_int64
_f = ctypes.c_float

# exported entry points with their C signatures (include/paged_kv.h)
_SIGS = {
    "kv_bytes": (_i64, [_i, _i, _i, _i64, _i, _i]),
    "kv_cache_alloc": (_i, [ctypes.POINTER(_p), _i, _i, _i, _i, _i]),
    "kv_alloc_destroy": (None, [_p]),
    "kv_seq_add": (_i, [_p, _i64, _i64]),
    "kv_seq_fork": (_i, [_p, _i64, _i64, _i64]),
    "kv_seq_free": (_i, [_p, _i64]),
    "kv_step": (_i, [_p, _p, _i, _p, _p, _i, _p, _p, _p, _i, ctypes.POINTER(_i)]),
    "kv_seq_reorder": (_i, [_p, _p, _p, _i]),
    "kv_seq_info": (_i, [_p, _i64, ctypes.POINTER(_i64), _p, _i, ctypes.POINTER(_i)]),
    "kv_alloc_stats": (_i, [_p, ctypes.POINTER(_i), ctypes.POINTER(_i), ctypes.POINTER(_i), _i,
                            ctypes.POINTER(_i)]),
    "kv_alloc_shape": (_i, [_p, ctypes.POINTER(_i), ctypes.POINTER(_i), ctypes.POINTER(_i),
                            ctypes.POINTER(_i)]),
    "kv_alloc_trace": (_i, [_p, _p, _i, _p, ctypes.POINTER(_i)]),
    "kv_slot_mapping": (_i, [_p, _i, _p, _i, _p]),
    "kv_append": (_i, [_p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _f, _f, _p]),
    "kv_copy_blocks": (_i, [_p, _p, _p, _p, _i, _i, _i, _i, _i, _p]),
    "paged_decode_workspace_bytes": (_i, [_i, _i, _i, _i, _i, ctypes.POINTER(ctypes.c_size_t)]),
    "paged_decode_attention": (_i, [_p, _i, _p, _p, _p, _i, _f, _f, _i, _p, _i, _p, _i, _i, _i,
                                    _i, _f, _p, ctypes.c_size_t, _p]),
    "paged_decode_attention_timed": (_i, [_p, _i, _p, _p, _p, _i, _f, _f, _i, _p, _i, _p, _i,
                                          _i, _i, _i, _f, _p, ctypes.c_size_t, _p, _p, _p, _p]),
    "paged_decode_step": (_i, [_p, _i, _p, _p, _p, _p, _p, _i, _f, _f, _i, _p, _i, _p, _i, _i,
                               _i, _i, _f, _p, ctypes.c_size_t, _p]),
    "paged_decode_attention_noalloc": (_i, [_p, _i, _p, _p, _p, _i, _f, _f, _i, _p, _i, _p, _i,
                                            _i, _i, _i, _f, _p]),
    "kv_prefix_chunks": (_i, [_p, _i, _p, _i, _i, _i, _p, _p, ctypes.POINTER(_i)]),
    "kv_prefix_plan": (_i, [_p, _i, _p, _i, _i, _i, _i, _i, _i, _p, _p, ctypes.POINTER(_i)]),
    "paged_decode_prefix_workspace_bytes": (_i, [_i, _i, _i, _i, _i, _i,
                                                 ctypes.POINTER(ctypes.c_size_t)]),
    "paged_decode": (_i, [_p, _i, _p, _p, _p, _p, _p, _i, _f, _f, _i, _p, _i, _p, _i, _i, _i,
                          _i, _f, _p, _p, _i, ctypes.c_uint, _p, ctypes.c_size_t, _p]),
    "paged_decode_timed": (_i, [_p, _i, _p, _p, _p, _p, _p, _i, _f, _f, _i, _p, _i, _p, _i, _i,
                                _i, _i, _f, _p, _p, _i, ctypes.c_uint, _p, ctypes.c_size_t, _p,
                                _p, _p, _p]),
    "kv_read_ceiling": (_i, [_p, ctypes.c_size_t, _p, _p]),
    "kv_test_pipeline_stall": (_i, [ctypes.c_longlong]),
    "kv_get_device_error": (_i, [ctypes.POINTER(_i), ctypes.POINTER(_i64)]),
    "kv_version": (ctypes.c_char_p, []),
}
for _name, (_res, _args) in _SIGS.items():
    _fn = getattr(_lib, _name)
    _fn.restype = _res
    _fn.argtypes = _args

# The per-step calls go through the CPython-API module _pkvfast when it was
# built (plain integers and floats, no ctypes marshalling); it links the same
# libpagedkv.so, which the dynamic loader shares with the ctypes handle above.
try:
    from . import _pkvfast as _fast
except ImportError:
    _fast = None


def _hot(name):
    return getattr(_fast, name) if _fast is not None else getattr(_lib, name)


_HOT_PAGED_DECODE = _hot("paged_decode")
_HOT_PAGED_DECODE_STEP = _hot("paged_decode_step")
_HOT_PAGED_DECODE_ATTENTION = _hot("paged_decode_attention")
_HOT_KV_APPEND = _hot("kv_append")


def fast_path():
    """True when the per-step calls bypass ctypes (module _pkvfast)."""
    return _fast is not None


def native_library_path():
    return _LIB_PATH


def version():
    return _lib.kv_version().decode()


def _check(rc, what):
    if rc != KV_OK:
        raise KVError(rc, what)


def _np_ptr(a):
    return ctypes.c_void_p(a.ctypes.data)


def _dptr(t):
    """Device (or host) address of a torch tensor."""
    return ctypes.c_void_p(t.data_ptr())


def _stream_ptr(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _stream_int(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _cache_dtype(t):
    import torch
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype in (torch.uint8, getattr(torch, "float8_e4m3fn", torch.uint8)):
        return FP8_E4M3
    raise ValueError("cache tensors must be bfloat16 or uint8 (E4M3 codes)")


# ------------------------------------------------------------------ sizing

def kv_bytes(layers, batch, kv_heads, seq, head_dim, dtype_bytes):
    """2 x layers x batch x kv_heads x seq x head_dim x dtype_bytes (int)."""
    r = _lib.kv_bytes(layers, batch, kv_heads, seq, head_dim, dtype_bytes)
    if r < 0:
        raise ValueError("kv_bytes: negative argument or overflow")
    return r


def slot_mapping(block_tables, positions):
    """Host slot of positions[i] in block-table row i (numpy int32 [n, max_blocks])."""
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    pos = np.ascontiguousarray(positions, dtype=np.int64)
    n = pos.shape[0]
    assert bt.shape[0] == n
    out = np.empty(n, dtype=np.int64)
    _check(_lib.kv_slot_mapping(_np_ptr(bt), bt.shape[1], _np_ptr(pos), n, _np_ptr(out)),
           "kv_slot_mapping")
    return out


# ---------------------------------------------------------------- allocator

class BlockAllocator:
    """Host block pool with free list, reference counts and copy-on-write."""

    def __init__(self, num_blocks, num_kv_heads, head_dim, kv_dtype=BF16):
        h = ctypes.c_void_p()
        _check(_lib.kv_cache_alloc(ctypes.byref(h), num_blocks, num_kv_heads, head_dim,
                                   BLOCK_SIZE, kv_dtype), "kv_cache_alloc")
        self._h = h
        self.num_blocks = num_blocks

    def close(self):
        if self._h:
            _lib.kv_alloc_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def add(self, seq_id, length):
        _check(_lib.kv_seq_add(self._h, seq_id, length), "kv_seq_add")

    def fork(self, parent, child, shared_len):
        _check(_lib.kv_seq_fork(self._h, parent, child, shared_len), "kv_seq_fork")

    def free(self, seq_id):
        _check(_lib.kv_seq_free(self._h, seq_id), "kv_seq_free")

    def step(self, seq_ids, max_blocks, cow_cap=None):
        """Plan one decode step; returns (slot_mapping int64[n], block_tables
        int32[n, max_blocks], context_lens int32[n], (cow_src, cow_dst))."""
        ids = np.ascontiguousarray(seq_ids, dtype=np.int64)
        n = ids.shape[0]
        cap = n if cow_cap is None else cow_cap
        slots = np.empty(n, dtype=np.int64)
        bt = np.empty((n, max_blocks), dtype=np.int32)
        lens = np.empty(n, dtype=np.int32)
        src = np.empty(max(cap, 1), dtype=np.int32)
        dst = np.empty(max(cap, 1), dtype=np.int32)
        ncow = _i(0)
        _check(_lib.kv_step(self._h, _np_ptr(ids), n, _np_ptr(slots), _np_ptr(bt), max_blocks,
                            _np_ptr(lens), _np_ptr(src), _np_ptr(dst), cap, ctypes.byref(ncow)),
               "kv_step")
        return slots, bt, lens, (src[:ncow.value].copy(), dst[:ncow.value].copy())

    def reorder(self, seq_ids, src_index):
        """Row i of seq_ids takes the KV state row src_index[i] had (beam
        reorder / duplication; block tables only, reference counted)."""
        ids = np.ascontiguousarray(seq_ids, dtype=np.int64)
        src = np.ascontiguousarray(src_index, dtype=np.int32)
        assert ids.shape == src.shape
        _check(_lib.kv_seq_reorder(self._h, _np_ptr(ids), _np_ptr(src), ids.shape[0]),
               "kv_seq_reorder")

    def info(self, seq_id, max_blocks=None):
        """(length, block ids) of a sequence."""
        ln = _i64(0)
        nb = _i(0)
        _check(_lib.kv_seq_info(self._h, seq_id, ctypes.byref(ln), None, 0, ctypes.byref(nb)),
               "kv_seq_info")
        row = np.empty(max(nb.value, 1), dtype=np.int32)
        _check(_lib.kv_seq_info(self._h, seq_id, None, _np_ptr(row), row.shape[0], None),
               "kv_seq_info")
        return ln.value, row[:nb.value].copy()

    def stats(self, block=-1):
        """(free blocks, used blocks, live sequences, refcount of `block` or None)."""
        fb, ub, ns, rc = _i(0), _i(0), _i(0), _i(0)
        _check(_lib.kv_alloc_stats(self._h, ctypes.byref(fb), ctypes.byref(ub), ctypes.byref(ns),
                                   block, ctypes.byref(rc)), "kv_alloc_stats")
        return fb.value, ub.value, ns.value, (rc.value if block >= 0 else None)

    def shape(self):
        """Per-layer cache shape [num_blocks, num_kv_heads, 16, head_dim] and dtype."""
        nb, h, d, dt = _i(0), _i(0), _i(0), _i(0)
        _check(_lib.kv_alloc_shape(self._h, ctypes.byref(nb), ctypes.byref(h), ctypes.byref(d),
                                   ctypes.byref(dt)), "kv_alloc_shape")
        return (nb.value, h.value, BLOCK_SIZE, d.value), dt.value

    def trace(self, seq_ids=None):
        """Debug trace of the cache state, one dict per sequence (the given
        ids in order, else every live sequence by ascending id): request id,
        batch slot, length, position offset, blocks, shared blocks, cache
        bytes per layer, the last reorder's source row, and the decode mask
        shape [1, length]."""
        if seq_ids is None:
            n = self.stats()[2]
            ids_ptr = None
        else:
            ids = np.ascontiguousarray(seq_ids, dtype=np.int64)
            n = ids.shape[0]
            ids_ptr = _np_ptr(ids)
        rows = np.empty((max(n, 1), TRACE_FIELDS), dtype=np.int64)
        cnt = _i(0)
        _check(_lib.kv_alloc_trace(self._h, ids_ptr, n, _np_ptr(rows), ctypes.byref(cnt)),
               "kv_alloc_trace")
        out = []
        for r in rows[:cnt.value]:
            rec = dict(zip(TRACE_KEYS, (int(x) for x in r)))
            rec["mask_shape"] = [1, rec["len"]]
            out.append(rec)
        return out

    def dump(self, seq_ids=None):
        """The trace as text: a header line with the pool and cache shape,
        then one JSON line per sequence."""
        import json
        shape, dt = self.shape()
        fb, ub, ns, _ = self.stats()
        head = {"kv_shape": list(shape), "kv_dtype": "fp8_e4m3" if dt == FP8_E4M3 else "bf16",
                "free_blocks": fb, "used_blocks": ub, "num_seqs": ns}
        return "\n".join([json.dumps(head)] + [json.dumps(r) for r in self.trace(seq_ids)])


# -------------------------------------------------------------------- GPU ops

def kv_append(k, v, k_cache, v_cache, slot_mapping, k_scale=1.0, v_scale=1.0, stream=None):
    """Append K/V ([T, Hkv, D] bfloat16, device) at slot_mapping (int64 [T],
    device) into the caches ([NB, Hkv, 16, D], bfloat16 or uint8 E4M3)."""
    T, Hkv, D = k.shape
    NB = k_cache.shape[0]
    _check(_HOT_KV_APPEND(k.data_ptr(), v.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                          slot_mapping.data_ptr(), T, Hkv, D, NB, _cache_dtype(k_cache),
                          float(k_scale), float(v_scale), _stream_int(stream)), "kv_append")


def kv_copy_blocks(k_cache, v_cache, src, dst, stream=None):
    """Copy whole blocks src[i] -> dst[i] (device int32 tensors)."""
    NB, Hkv, _, D = k_cache.shape
    _check(_lib.kv_copy_blocks(_dptr(k_cache), _dptr(v_cache), _dptr(src), _dptr(dst),
                               src.shape[0], Hkv, D, NB, _cache_dtype(k_cache),
                               _stream_ptr(stream)), "kv_copy_blocks")


def workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim, kv_dtype=BF16):
    n = ctypes.c_size_t(0)
    _check(_lib.paged_decode_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                             kv_dtype, ctypes.byref(n)),
           "paged_decode_workspace_bytes")
    return n.value


def alloc_workspace(num_seqs, num_q_heads, num_kv_heads, head_dim, kv_dtype=BF16, device=None):
    import torch
    nbytes = workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim, kv_dtype)
    return torch.empty(max(nbytes, 16), dtype=torch.uint8, device=device or "cuda")


def paged_decode_attention(out, q, k_cache, v_cache, block_tables, context_lens, scale, workspace,
                           k_scale=1.0, v_scale=1.0, stream=None):
    """out[B, Hq, D] (bfloat16 or float32) = decode attention of q [B, Hq, D]
    (bfloat16) over the paged caches; block_tables int32 [B, max_blocks] and
    context_lens int32 [B] on the device; workspace a uint8 device tensor of
    at least workspace_bytes(...) bytes."""
    import torch
    B, Hq, D = q.shape
    NB, Hkv, _, D2 = k_cache.shape
    assert D == D2
    out_dtype = F32 if out.dtype == torch.float32 else BF16
    _check(_HOT_PAGED_DECODE_ATTENTION(
        out.data_ptr(), out_dtype, q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
        _cache_dtype(k_cache), float(k_scale), float(v_scale), NB, block_tables.data_ptr(),
        block_tables.shape[1], context_lens.data_ptr(), B, Hq, Hkv, D, float(scale),
        workspace.data_ptr(), workspace.numel() * workspace.element_size(), _stream_int(stream)),
        "paged_decode_attention")


def paged_decode_attention_timed(out, q, k_cache, v_cache, block_tables, context_lens, scale,
                                 workspace, events, k_scale=1.0, v_scale=1.0, stream=None):
    """paged_decode_attention that also records three torch.cuda.Event objects
    (already recorded once, so that their handles exist, or None) before the
    split kernel, after it and after the merge kernel: events = (begin,
    split_end, end)."""
    import torch
    B, Hq, D = q.shape
    NB, Hkv, _, _ = k_cache.shape
    out_dtype = F32 if out.dtype == torch.float32 else BF16
    ev = [ctypes.c_void_p(e._as_parameter_.value) if e is not None else None for e in events]
    _check(_lib.paged_decode_attention_timed(
        _dptr(out), out_dtype, _dptr(q), _dptr(k_cache), _dptr(v_cache), _cache_dtype(k_cache),
        float(k_scale), float(v_scale), NB, _dptr(block_tables), block_tables.shape[1],
        _dptr(context_lens), B, Hq, Hkv, D, float(scale), _dptr(workspace),
        workspace.numel() * workspace.element_size(), _stream_ptr(stream), ev[0], ev[1], ev[2]),
        "paged_decode_attention_timed")


def paged_decode_step(out, q, k_new, v_new, k_cache, v_cache, block_tables, context_lens, scale,
                      workspace, k_scale=1.0, v_scale=1.0, stream=None):
    """One decode step in one launch: append k_new/v_new ([B, Hkv, D] bfloat16)
    at position context_lens-1 of each sequence, then attend (see
    paged_decode_attention for the other arguments)."""
    import torch
    B, Hq, D = q.shape
    NB, Hkv, _, _ = k_cache.shape
    out_dtype = F32 if out.dtype == torch.float32 else BF16
    _check(_HOT_PAGED_DECODE_STEP(
        out.data_ptr(), out_dtype, q.data_ptr(), k_new.data_ptr(), v_new.data_ptr(),
        k_cache.data_ptr(), v_cache.data_ptr(), _cache_dtype(k_cache), float(k_scale),
        float(v_scale), NB, block_tables.data_ptr(), block_tables.shape[1],
        context_lens.data_ptr(), B, Hq, Hkv, D, float(scale), workspace.data_ptr(),
        workspace.numel() * workspace.element_size(), _stream_int(stream)), "paged_decode_step")


PREFIX_CHUNK_INTS = 18      # KV_PREFIX_CHUNK_INTS
PREFIX_MAX_ROWS = 16        # KV_PREFIX_MAX_ROWS


def prefix_chunks(block_tables, context_lens, group_size, min_blocks=1):
    """Prefix chunks of sequences whose block tables start with the same
    blocks (host numpy int32 arrays in, kv_prefix_chunks): returns
    (chunks int32 [nc, 18], seq_chunk int32 [B])."""
    import numpy as np
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    B, mb = bt.shape
    chunks = np.full((max(B // 2, 1), PREFIX_CHUNK_INTS), -1, dtype=np.int32)
    seq_chunk = np.full(max(B, 1), -1, dtype=np.int32)
    nc = ctypes.c_int(0)
    _check(_lib.kv_prefix_chunks(_np_ptr(bt), mb, _np_ptr(cl), B, int(group_size),
                                 int(min_blocks), _np_ptr(chunks), _np_ptr(seq_chunk),
                                 ctypes.byref(nc)), "kv_prefix_chunks")
    return chunks[:nc.value].copy(), seq_chunk[:B].copy()


def prefix_plan(block_tables, context_lens, num_q_heads, num_kv_heads, head_dim,
                kv_dtype=BF16, resident_warps=0):
    """prefix_chunks with the library's decision whether shared-prefix
    decoding pays for these tables (kv_prefix_plan; resident_warps 0: those
    of the current device): (chunks int32 [nc, 18], seq_chunk int32 [B]),
    nc == 0 for plain decoding."""
    import numpy as np
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    B, mb = bt.shape
    chunks = np.full((max(B // 2, 1), PREFIX_CHUNK_INTS), -1, dtype=np.int32)
    seq_chunk = np.full(max(B, 1), -1, dtype=np.int32)
    nc = ctypes.c_int(0)
    _check(_lib.kv_prefix_plan(_np_ptr(bt), mb, _np_ptr(cl), B, int(num_q_heads),
                               int(num_kv_heads), int(head_dim), int(kv_dtype),
                               int(resident_warps), _np_ptr(chunks),
                               _np_ptr(seq_chunk), ctypes.byref(nc)), "kv_prefix_plan")
    return chunks[:nc.value].copy(), seq_chunk[:B].copy()


def prefix_workspace_bytes(num_seqs, num_chunks, num_q_heads, num_kv_heads, head_dim,
                           kv_dtype=BF16):
    n = ctypes.c_size_t(0)
    _check(_lib.paged_decode_prefix_workspace_bytes(num_seqs, num_chunks, num_q_heads,
                                                    num_kv_heads, head_dim, kv_dtype,
                                                    ctypes.byref(n)),
           "paged_decode_prefix_workspace_bytes")
    return n.value


def alloc_prefix_workspace(num_seqs, num_chunks, num_q_heads, num_kv_heads, head_dim,
                           kv_dtype=BF16, device=None):
    import torch
    nbytes = prefix_workspace_bytes(num_seqs, num_chunks, num_q_heads, num_kv_heads, head_dim,
                                    kv_dtype)
    return torch.empty(max(nbytes, 16), dtype=torch.uint8, device=device or "cuda")


DECODE_EARLY_INPUTS = 1     # KV_DECODE_EARLY_INPUTS


def paged_decode(out, q, k_cache, v_cache, block_tables, context_lens, scale, workspace,
                 k_scale=1.0, v_scale=1.0, k_new=None, v_new=None, chunks=None, seq_chunk=None,
                 early_inputs=False, stream=None):
    """One decode step, general form (paged_decode): with k_new/v_new
    ([B, Hkv, D] bfloat16) the step's token is appended first (as
    paged_decode_step); with chunks (int32 [nc, 18]) and seq_chunk (int32 [B])
    on the device (from prefix_chunks) shared prefix blocks are read once per
    chunk (workspace from alloc_prefix_workspace); early_inputs lets the
    kernel read the block tables, lengths and caches while the previous
    kernel on the stream drains (see KV_DECODE_EARLY_INPUTS in the header for
    the caller's guarantee).  Other arguments as paged_decode_attention."""
    import torch
    B, Hq, D = q.shape
    NB, Hkv, _, _ = k_cache.shape
    out_dtype = F32 if out.dtype == torch.float32 else BF16
    nc = int(chunks.shape[0]) if chunks is not None else 0
    _check(_HOT_PAGED_DECODE(
        out.data_ptr(), out_dtype, q.data_ptr(), k_new.data_ptr() if k_new is not None else 0,
        v_new.data_ptr() if v_new is not None else 0, k_cache.data_ptr(), v_cache.data_ptr(),
        _cache_dtype(k_cache), float(k_scale), float(v_scale), NB, block_tables.data_ptr(),
        block_tables.shape[1], context_lens.data_ptr(), B, Hq, Hkv, D, float(scale),
        chunks.data_ptr() if nc else 0, seq_chunk.data_ptr() if nc else 0, nc,
        DECODE_EARLY_INPUTS if early_inputs else 0, workspace.data_ptr(),
        workspace.numel() * workspace.element_size(), _stream_int(stream)), "paged_decode")


def paged_decode_timed(out, q, k_cache, v_cache, block_tables, context_lens, scale, workspace,
                       events, k_scale=1.0, v_scale=1.0, k_new=None, v_new=None, chunks=None,
                       seq_chunk=None, early_inputs=False, stream=None):
    """paged_decode that also records three torch.cuda.Event objects (already
    recorded once so that their handles exist, or None) before the split
    kernel, after it and after the merge kernel: events = (begin, split_end,
    end).  A measurement hook."""
    import torch
    B, Hq, D = q.shape
    NB, Hkv, _, _ = k_cache.shape
    out_dtype = F32 if out.dtype == torch.float32 else BF16
    nc = int(chunks.shape[0]) if chunks is not None else 0
    ev = [ctypes.c_void_p(e._as_parameter_.value) if e is not None else None for e in events]
    _check(_lib.paged_decode_timed(
        _dptr(out), out_dtype, _dptr(q), _dptr(k_new) if k_new is not None else None,
        _dptr(v_new) if v_new is not None else None, _dptr(k_cache), _dptr(v_cache),
        _cache_dtype(k_cache), float(k_scale), float(v_scale), NB, _dptr(block_tables),
        block_tables.shape[1], _dptr(context_lens), B, Hq, Hkv, D, float(scale),
        _dptr(chunks) if nc else None, _dptr(seq_chunk) if nc else None, nc,
        DECODE_EARLY_INPUTS if early_inputs else 0, _dptr(workspace),
        workspace.numel() * workspace.element_size(), _stream_ptr(stream), ev[0], ev[1], ev[2]),
        "paged_decode_timed")


def read_ceiling(buf, sink, stream=None):
    """Stream the device tensor ``buf`` through shared memory with the decode
    kernel's bulk-copy pattern and no arithmetic (kv_read_ceiling), on
    ``stream``; ``sink`` is a zeroed int32 device tensor of 2 elements.  A
    measurement hook: bytes / elapsed time is a read-only bandwidth ceiling."""
    _check(_lib.kv_read_ceiling(_dptr(buf), buf.numel() * buf.element_size(), _dptr(sink),
                                _stream_ptr(stream)), "kv_read_ceiling")


def set_pipeline_stall(cycles):
    """Test hook (kv_test_pipeline_stall): with cycles > 0 every split-kernel
    warp takes the bounded-wait time-out path on its first wait; 0 turns it
    off."""
    _check(_lib.kv_test_pipeline_stall(int(cycles)), "kv_test_pipeline_stall")


def paged_decode_attention_noalloc(out, q, k_cache, v_cache, block_tables, context_lens, scale,
                                   k_scale=1.0, v_scale=1.0, stream=None):
    """paged_decode_attention without a caller workspace, for callers that
    cannot allocate device memory: the library's own fixed 16 MiB scratch is
    used (shared by every call on the device, so calls must not overlap on
    the GPU).  Shapes needing more raise KVError(KV_ERR_TOO_LARGE)."""
    import torch
    B, Hq, D = q.shape
    NB, Hkv, _, _ = k_cache.shape
    out_dtype = F32 if out.dtype == torch.float32 else BF16
    _check(_lib.paged_decode_attention_noalloc(
        _dptr(out), out_dtype, _dptr(q), _dptr(k_cache), _dptr(v_cache), _cache_dtype(k_cache),
        float(k_scale), float(v_scale), NB, _dptr(block_tables), block_tables.shape[1],
        _dptr(context_lens), B, Hq, Hkv, D, float(scale), _stream_ptr(stream)),
        "paged_decode_attention_noalloc")


def get_device_error():
    """(flags, detail) of the kernels' sticky bounds-check flags; clears them."""
    f = _i(0)
    d = _i64(0)
    _check(_lib.kv_get_device_error(ctypes.byref(f), ctypes.byref(d)), "kv_get_device_error")
    return f.value, d.value


class DecodeStepStaging:
    """Host-to-device plumbing for a stream of decode steps.

    Each of ``slots`` staging slots is one pinned host buffer holding every
    per-step input -- q [B, Hq, D] bf16, k_new / v_new [B, Hkv, D] bf16,
    block_tables [B, max_blocks] int32, context_lens [B] int32 -- at 256-byte
    aligned offsets, mirrored by one device buffer, plus an output buffer on
    each side.  A step costs one host-to-device copy, the fused step kernels
    (paged_decode with the append and KV_DECODE_EARLY_INPUTS) and one
    device-to-host copy of the output.  Uploads
    and downloads run on two copy streams of their own and the slots
    alternate, so step i+1's upload and step i's download overlap the kernels
    of the steps around them.

    The compute stream waits for each upload through an event, which also
    ends the programmatic overlap of consecutive steps.  With
    ``host_ordered=True`` the host instead blocks until the step's upload has
    finished before launching its kernels (the upload was queued a step
    earlier, so the host stays about one step ahead): the compute stream then
    holds only kernel launches and consecutive steps keep their overlap.

    With ``zero_copy=True`` there are no copies and no device slots: the
    kernels read the step's inputs from the pinned host slot and write the
    output into it directly (over NVLink-C2C on a Grace-Blackwell node), and
    the stream of steps stays one chain of kernel launches.

    Use: fill ``host(i)`` views of slot i % slots (``q``, ``k_new``,
    ``v_new``, ``block_tables``, ``context_lens``) once ``ready_for_input(i)``
    holds, call ``step(i, ...)``, and read ``host(i).out`` after
    ``wait_output(i)``."""

    _ALIGN = 256

    class _Slot:
        pass

    def __init__(self, num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks,
                 kv_dtype=BF16, device=None, out_dtype=None, slots=2, zero_copy=False,
                 host_ordered=False):
        import torch
        self.device = torch.device(device or "cuda")
        self.zero_copy = bool(zero_copy)
        self.host_ordered = bool(host_ordered)
        B, Hq, Hkv, D = num_seqs, num_q_heads, num_kv_heads, head_dim
        parts = [("q", (B, Hq, D), torch.bfloat16), ("k_new", (B, Hkv, D), torch.bfloat16),
                 ("v_new", (B, Hkv, D), torch.bfloat16),
                 ("block_tables", (B, max_blocks), torch.int32),
                 ("context_lens", (B,), torch.int32)]
        offs, off = {}, 0
        for name, shape, dt in parts:
            nbytes = int(np.prod(shape)) * torch.empty((), dtype=dt).element_size()
            offs[name] = (off, shape, dt, nbytes)
            off = -(-(off + nbytes) // self._ALIGN) * self._ALIGN
        self.nbytes = off
        od = out_dtype or torch.bfloat16
        self._slots = []
        for _ in range(slots):
            h, d = self._Slot(), self._Slot()
            h.raw = torch.empty(off, dtype=torch.uint8).pin_memory()
            h.out = torch.empty((B, Hq, D), dtype=od).pin_memory()
            if self.zero_copy:
                d = h                   # the kernels address the pinned slot itself
            else:
                d.raw = torch.empty(off, dtype=torch.uint8, device=self.device)
                d.out = torch.empty((B, Hq, D), dtype=od, device=self.device)
            for name, (o, shape, dt, nb) in offs.items():
                setattr(h, name, h.raw[o:o + nb].view(dt).view(shape))
                if d is not h:
                    setattr(d, name, d.raw[o:o + nb].view(dt).view(shape))
            ev = {k: torch.cuda.Event() for k in ("uploaded", "computed", "downloaded")}
            self._slots.append((h, d, ev))
        self.upload_stream = torch.cuda.Stream(self.device)
        self.download_stream = torch.cuda.Stream(self.device)
        self.workspace = alloc_workspace(B, Hq, Hkv, D, kv_dtype, device=self.device)

    def host(self, i):
        return self._slots[i % len(self._slots)][0]

    @property
    def h2d_bytes(self):
        """Bytes of inputs a step moves host to device (copied, or read in
        place with zero_copy)."""
        return self.nbytes

    @property
    def d2h_bytes(self):
        h = self._slots[0][0]
        return h.out.numel() * h.out.element_size()

    def ready_for_input(self, i):
        """Block the host until slot i % slots may be refilled (its previous
        upload has finished; with zero_copy, its previous step)."""
        ev = self._slots[i % len(self._slots)][2]
        (ev["computed"] if self.zero_copy else ev["uploaded"]).synchronize()

    def wait_output(self, i):
        ev = self._slots[i % len(self._slots)][2]
        (ev["computed"] if self.zero_copy else ev["downloaded"]).synchronize()

    def step(self, i, k_cache, v_cache, scale, k_scale=1.0, v_scale=1.0, stream=None):
        """Upload slot i's inputs, run the fused decode step on `stream`,
        download its output (all asynchronous)."""
        import torch
        h, d, ev = self._slots[i % len(self._slots)]
        s = stream or torch.cuda.current_stream(self.device)
        if self.zero_copy:
            # the slot is refilled by the host only after ready_for_input(i),
            # and the kernel before is the previous step's: early reads are safe
            paged_decode(h.out, h.q, k_cache, v_cache, h.block_tables, h.context_lens, scale,
                         self.workspace, k_scale, v_scale, k_new=h.k_new, v_new=h.v_new,
                         early_inputs=True, stream=s)
            ev["computed"].record(s)
            return
        up, down = self.upload_stream, self.download_stream
        # the device slot is free once its previous step has been computed and
        # its output downloaded (the download follows the computation)
        up.wait_event(ev["downloaded"])
        with torch.cuda.stream(up):
            d.raw.copy_(h.raw, non_blocking=True)
            ev["uploaded"].record(up)
        if self.host_ordered:
            ev["uploaded"].synchronize()
        else:
            s.wait_event(ev["uploaded"])
        # the inputs arrive by a copy joined through an event, and the kernel
        # before is the previous step's: the early reads are safe
        paged_decode(d.out, d.q, k_cache, v_cache, d.block_tables, d.context_lens, scale,
                     self.workspace, k_scale, v_scale, k_new=d.k_new, v_new=d.v_new,
                     early_inputs=True, stream=s)
        ev["computed"].record(s)
        down.wait_event(ev["computed"])
        with torch.cuda.stream(down):
            h.out.copy_(d.out, non_blocking=True)
            ev["downloaded"].record(down)

    def join(self, stream=None):
        """Make `stream` wait for every upload and download issued so far."""
        import torch
        s = stream or torch.cuda.current_stream(self.device)
        s.wait_stream(self.upload_stream)
        s.wait_stream(self.download_stream)
