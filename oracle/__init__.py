"""CPU oracle for the paged decode-step hot path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
legs of ``bench.py`` may import this package.  The product library
(``paged_kv_cache_21_gb300``) never imports it, and it never imports the
product library: the two share no code.

Contents
--------
* ``kv_bytes`` -- the KV-cache size formula, 2 (K and V) x layers x batch x
  kv_heads x seq x head_dim x bytes ("KV cache complete guide", section "KV
  cache memory size calculation"; "Transformer attention mask and KV cache
  inference", section "Cache shape and memory calculation").
* ``attention_direct`` -- one-shot softmax(q K^T * scale) V over contiguous
  K/V in float64 ("KV Cache" (heepie), core formula).
* ``tiled_softmax_attention`` -- the same quantity by the running (max, sum)
  tile loop of "KV Cache, Flash Attention and inference optimization",
  sections "Numerical trick" and "Step 2: tiled softmax"; the pages state it
  is exact, so it must equal ``attention_direct`` up to rounding.
* ``causal_attention`` -- full prefill attention with an explicit additive
  causal mask (0 where allowed, -inf where forbidden; "Transformer attention
  mask and KV cache inference", sections "State of scaled dot-product
  attention" and "Causal mask and future positions").  Its last row is what
  one decode step over the same tokens must return.
* ``split_partials`` / ``lse_merge`` -- split-KV: the keys cut into ranges,
  each range's normalised output with its log-sum-exp, then the combine
  out = sum_i e^(lse_i - M) o_i / sum_i e^(lse_i - M), M = max_i lse_i.  Both
  are derived from the running (max, sum) rule of the lesson's "Numerical
  trick" (the pages give no split-KV listing); they must equal
  ``attention_direct`` for any cut.
* ``paged_attention`` / ``append`` / E4M3 and bfloat16 conversions -- thin
  ctypes wrappers over ``oracle.c`` (float64 C, OpenMP over sequence x KV head).
"""
import ctypes
import os

import numpy as np

from .build import build_oracle

BF16 = 0
FP8_E4M3 = 1
BLOCK_SIZE = 16

_lib = None


def lib():
    """Load (building first if needed) the C oracle."""
    global _lib
    if _lib is None:
        path = build_oracle()
        L = ctypes.CDLL(path)
        c_p = ctypes.c_void_p
        L.orc_bf16_to_double.restype = ctypes.c_double
        L.orc_bf16_to_double.argtypes = [ctypes.c_uint16]
        L.orc_double_to_bf16.restype = ctypes.c_uint16
        L.orc_double_to_bf16.argtypes = [ctypes.c_double]
        L.orc_double_to_bf16_array.argtypes = [c_p, c_p, ctypes.c_int64]
        L.orc_bf16_to_double_array.argtypes = [c_p, c_p, ctypes.c_int64]
        L.orc_e4m3_decode.restype = ctypes.c_double
        L.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
        L.orc_e4m3_encode.restype = ctypes.c_uint8
        L.orc_e4m3_encode.argtypes = [ctypes.c_double]
        L.orc_quantize_e4m3.restype = ctypes.c_uint8
        L.orc_quantize_e4m3.argtypes = [ctypes.c_uint16, ctypes.c_float]
        L.orc_quantize_e4m3_array.argtypes = [c_p, c_p, ctypes.c_int64, ctypes.c_float]
        L.orc_append.restype = ctypes.c_int
        L.orc_append.argtypes = [c_p, c_p, c_p, c_p, c_p, ctypes.c_int, ctypes.c_int,
                                 ctypes.c_int, ctypes.c_int64, ctypes.c_int,
                                 ctypes.c_float, ctypes.c_float]
        L.orc_paged_attention.restype = ctypes.c_int
        L.orc_paged_attention.argtypes = [c_p, c_p, c_p, c_p, ctypes.c_int, ctypes.c_double,
                                          ctypes.c_double, c_p, ctypes.c_int, c_p,
                                          ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                          ctypes.c_int, ctypes.c_int64, ctypes.c_double,
                                          c_p, ctypes.c_int]
        L.orc_max_threads.restype = ctypes.c_int
        _lib = L
    return _lib


def _ptr(a):
    return ctypes.c_void_p(a.ctypes.data) if a is not None else None


# ------------------------------------------------------------------ formula

def kv_bytes(layers, batch, kv_heads, seq, head_dim, dtype_bytes):
    """Bytes of K plus V for a whole model: 2 x layers x batch x kv_heads x
    seq x head_dim x dtype_bytes, exact integer arithmetic."""
    return 2 * layers * batch * kv_heads * seq * head_dim * dtype_bytes


# ----------------------------------------------------------- number formats

def bf16_bits_to_f64(bits):
    """uint16 array of bfloat16 patterns -> float64 array."""
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(bits.shape, dtype=np.float64)
    lib().orc_bf16_to_double_array(_ptr(bits), _ptr(out), bits.size)
    return out


def f64_to_bf16_bits(x):
    """float64 array -> nearest bfloat16 (ties to even) as uint16 patterns."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.uint16)
    lib().orc_double_to_bf16_array(_ptr(x), _ptr(out), x.size)
    return out


def round_to_bf16(x):
    """float64 array rounded to the nearest bfloat16 value (still float64)."""
    return bf16_bits_to_f64(f64_to_bf16_bits(x))


def e4m3_decode(code):
    return lib().orc_e4m3_decode(int(code))


def e4m3_encode(x):
    return lib().orc_e4m3_encode(float(x))


def e4m3_decode_array(codes):
    codes = np.asarray(codes, dtype=np.uint8)
    table = np.array([e4m3_decode(c) for c in range(256)], dtype=np.float64)
    return table[codes]


def quantize_e4m3(bits, scale):
    """bfloat16 patterns -> E4M3 codes of x / scale (quotient in binary32)."""
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(bits.shape, dtype=np.uint8)
    lib().orc_quantize_e4m3_array(_ptr(bits), _ptr(out), bits.size, float(scale))
    return out


# ------------------------------------------------------------ paged path

def slot_mapping(block_tables, seq_index, positions):
    """Physical slot of logical position ``pos`` of sequence ``s``: the page
    table entry of the position's 16-token block times 16, plus the offset
    inside the block ("KV Cache, Flash Attention and inference optimization",
    section "PagedAttention").  Vectorised over (seq_index, positions)."""
    bt = np.asarray(block_tables, dtype=np.int64)
    s = np.asarray(seq_index, dtype=np.int64)
    pos = np.asarray(positions, dtype=np.int64)
    return bt[s, pos // BLOCK_SIZE] * BLOCK_SIZE + pos % BLOCK_SIZE


def append(k_cache, v_cache, k_bits, v_bits, slot_mapping, kv_dtype, k_scale=1.0, v_scale=1.0):
    """Write each token's K/V (bfloat16 patterns [T, Hkv, D]) at its slot in the
    host copies ``k_cache``/``v_cache`` (uint8 or uint16 arrays shaped
    [NB, Hkv, 16, D]).  Slots < 0 are skipped.  Returns the C status."""
    assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    k_bits = np.ascontiguousarray(k_bits, dtype=np.uint16)
    v_bits = np.ascontiguousarray(v_bits, dtype=np.uint16)
    slots = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    T, Hkv, D = k_bits.shape
    NB = k_cache.shape[0]
    return lib().orc_append(_ptr(k_cache), _ptr(v_cache), _ptr(k_bits), _ptr(v_bits),
                            _ptr(slots), T, Hkv, D, NB, kv_dtype,
                            float(k_scale), float(v_scale))


def paged_attention(q, k_cache, v_cache, block_tables, context_lens, scale,
                    kv_dtype=BF16, k_scale=1.0, v_scale=1.0, pair_select=None,
                    nthreads=0):
    """Decode attention over a paged cache, float64.

    q: float64 [B, Hq, D]; k_cache/v_cache: uint16 (bf16) or uint8 (e4m3)
    arrays [NB, Hkv, 16, D]; block_tables int32 [B, max_blocks];
    context_lens int32 [B]; pair_select: optional bool [B, Hkv] restricting
    which (sequence, KV head) pairs are computed (others stay NaN).
    Returns float64 [B, Hq, D]."""
    q = np.ascontiguousarray(q, dtype=np.float64)
    B, Hq, D = q.shape
    NB, Hkv, bs, D2 = k_cache.shape
    assert bs == BLOCK_SIZE and D2 == D
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    kc = np.ascontiguousarray(k_cache)
    vc = np.ascontiguousarray(v_cache)
    out = np.full((B, Hq, D), np.nan, dtype=np.float64)
    sel = None
    if pair_select is not None:
        sel = np.ascontiguousarray(pair_select, dtype=np.uint8).reshape(B * Hkv)
    rc = lib().orc_paged_attention(_ptr(out), _ptr(q), _ptr(kc), _ptr(vc), kv_dtype,
                                   float(k_scale), float(v_scale), _ptr(bt), bt.shape[1],
                                   _ptr(cl), B, Hq, Hkv, D, NB, float(scale), _ptr(sel),
                                   int(nthreads))
    if rc != 0:
        raise ValueError("oracle paged_attention failed with status %d" % rc)
    return out


def max_threads():
    return lib().orc_max_threads()


# --------------------------------------------------- contiguous references

def attention_direct(q, K, V, scale):
    """softmax(q K^T * scale) V for one query row q [D] over K, V [L, D]."""
    q = np.asarray(q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    z = scale * (K @ q)
    z = z - z.max()
    w = np.exp(z)
    return (w[:, None] * V).sum(axis=0) / w.sum()


def tiled_softmax_attention(q, K, V, scale, tile=4):
    """Running-maximum softmax over key tiles.

    Keeps, per query, the largest score seen so far ``m``, the running
    denominator ``s`` and an unnormalised output ``o``.  Each new tile raises
    ``m`` to ``m'``; old contributions are multiplied by e^(m - m') (taken as 0
    while no tile has been seen) and the tile adds its own e^(z - m') terms.
    Dividing by ``s`` at the end gives the exact softmax result."""
    q = np.asarray(q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    m = -np.inf
    s = 0.0
    o = np.zeros(V.shape[1], dtype=np.float64)
    for start in range(0, K.shape[0], tile):
        z = scale * (K[start:start + tile] @ q)
        m_new = max(m, float(z.max()))
        carry = 0.0 if m == -np.inf else float(np.exp(m - m_new))
        e = np.exp(z - m_new)
        s = s * carry + float(e.sum())
        o = o * carry + (e[:, None] * V[start:start + tile]).sum(axis=0)
        m = m_new
    return o / s


def split_partials(q, K, V, scale, bounds):
    """Cut the keys at ``bounds`` (increasing indices from 0 to L) and return,
    per range [a, b), the normalised output o = sum_j w_j V_j / sum_j w_j and
    lse = m + log(sum_j e^(z_j - m)) with z = scale * K q, m = max z.  An
    empty range gives (zeros, -inf)."""
    q = np.asarray(q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    parts = []
    for a, b in zip(bounds[:-1], bounds[1:]):
        if b <= a:
            parts.append((np.zeros(V.shape[1]), -np.inf))
            continue
        z = scale * (K[a:b] @ q)
        m = float(z.max())
        w = np.exp(z - m)
        s = float(w.sum())
        parts.append(((w[:, None] * V[a:b]).sum(axis=0) / s, m + float(np.log(s))))
    return parts


def lse_merge(parts):
    """Combine (o_i, lse_i) partials: weights e^(lse_i - M), M = max lse_i;
    partials with lse = -inf (no keys) get weight 0.  No partial with keys
    gives zeros."""
    lse = np.array([p[1] for p in parts], dtype=np.float64)
    if not np.isfinite(lse).any():
        return np.zeros_like(np.asarray(parts[0][0], dtype=np.float64))
    M = lse[np.isfinite(lse)].max()
    w = np.where(np.isfinite(lse), np.exp(lse - M), 0.0)
    o = np.stack([np.asarray(p[0], dtype=np.float64) for p in parts])
    return (w[:, None] * o).sum(axis=0) / w.sum()


def causal_mask(L):
    """Additive causal mask [L, L]: 0 where query t may see key s (s <= t),
    -inf where s > t."""
    allowed = np.tril(np.ones((L, L), dtype=bool))
    return np.where(allowed, 0.0, -np.inf)


def causal_attention(Q, K, V, scale):
    """Full causal self-attention, softmax(Q K^T * scale + mask) V, float64."""
    Q = np.asarray(Q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    scores = scale * (Q @ K.T) + causal_mask(Q.shape[0])
    scores = scores - scores.max(axis=1, keepdims=True)
    w = np.exp(scores)
    w = w / w.sum(axis=1, keepdims=True)
    return w @ V
