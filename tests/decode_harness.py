"""Shared plumbing of the GPU tests: run one decode step through the C ABI and
the same step through the CPU oracle, on the same seeded inputs.

The pool is filled the same way on both sides: every physical slot receives
its vector from ``workloads`` through the append operation (GPU: kv_append
kernel; oracle: its own append), then the step appends each sequence's new
token at position L-1 and attends.  Nothing computed by the GPU feeds the
oracle."""
import numpy as np
import torch

import oracle
import workloads
from workloads import bf16_bits

BS = 16


def tolerance(kv_dtype):
    """Max-abs tolerance on the attention output (before output rounding)."""
    return 3e-2 if kv_dtype == workloads.FP8_E4M3 else 2e-3


def half_ulp_bf16(x):
    """Half a bfloat16 ulp at |x| (the unavoidable rounding of a bf16 output)."""
    ax = np.abs(x)
    e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    e = np.maximum(e, -126)
    return np.where(ax > 0, np.exp2(e - 8), np.exp2(-134))


def gpu_step(case, out_dtype=torch.bfloat16, device="cuda", pool_overrides=None, stream=None,
             fused=False, workspace=None, prefix=None, early_inputs=False):
    """Returns (out, k_cache, v_cache) on the device.  fused=False: kv_append
    then paged_decode_attention (two launches); fused=True: paged_decode_step
    (append and attention in one launch).  prefix=(chunks, seq_chunk) (host
    int32 arrays) runs paged_decode with that chunk table instead.  early_inputs:
    paged_decode with KV_DECODE_EARLY_INPUTS (with fused=True and no prefix,
    the call bench.py times)."""
    import paged_kv_cache_21_gb300 as pk
    NB, Hkv, D = case.num_blocks, case.Hkv, case.D
    cdt = torch.bfloat16 if case.kv_dtype == workloads.BF16 else torch.uint8
    kc = torch.zeros((NB, Hkv, BS, D), dtype=cdt, device=device)
    vc = torch.zeros_like(kc)
    all_slots = torch.arange(NB * BS, dtype=torch.int64, device=device)
    pool_k = case.pool_k.to(device)
    pool_v = case.pool_v.to(device)
    if pool_overrides is not None:
        pool_k, pool_v = pool_overrides(pool_k, pool_v)
    pk.kv_append(pool_k, pool_v, kc, vc, all_slots, case.k_scale, case.v_scale, stream=stream)
    del pool_k, pool_v
    out = torch.empty((case.B, case.Hq, D), dtype=out_dtype, device=device)
    bt = torch.from_numpy(case.block_tables).to(device)
    cl = torch.from_numpy(case.context_lens).to(device)
    if prefix is not None:
        chunks, seq_chunk = prefix
        ws = workspace if workspace is not None else pk.alloc_prefix_workspace(
            case.B, len(chunks), case.Hq, Hkv, D, case.kv_dtype, device=device)
        dch = torch.from_numpy(np.ascontiguousarray(chunks, dtype=np.int32)).to(device)
        dsc = torch.from_numpy(np.ascontiguousarray(seq_chunk, dtype=np.int32)).to(device)
        if fused:
            pk.paged_decode(out, case.q.to(device), kc, vc, bt, cl, case.scale, ws, case.k_scale,
                            case.v_scale, k_new=case.k_new.to(device),
                            v_new=case.v_new.to(device), chunks=dch, seq_chunk=dsc,
                            early_inputs=early_inputs, stream=stream)
        else:
            slots_new = pk.slot_mapping(case.block_tables,
                                        case.context_lens.astype(np.int64) - 1)
            pk.kv_append(case.k_new.to(device), case.v_new.to(device), kc, vc,
                         torch.from_numpy(slots_new).to(device), case.k_scale, case.v_scale,
                         stream=stream)
            pk.paged_decode(out, case.q.to(device), kc, vc, bt, cl, case.scale, ws, case.k_scale,
                            case.v_scale, chunks=dch, seq_chunk=dsc, early_inputs=early_inputs,
                            stream=stream)
        torch.cuda.synchronize()
        return out, kc, vc
    ws = workspace if workspace is not None else pk.alloc_workspace(
        case.B, case.Hq, Hkv, D, case.kv_dtype, device=device)
    if fused and early_inputs:
        # the benchmark's call: fused append, early reads of tables and caches
        pk.paged_decode(out, case.q.to(device), kc, vc, bt, cl, case.scale, ws, case.k_scale,
                        case.v_scale, k_new=case.k_new.to(device), v_new=case.v_new.to(device),
                        early_inputs=True, stream=stream)
    elif fused:
        pk.paged_decode_step(out, case.q.to(device), case.k_new.to(device),
                             case.v_new.to(device), kc, vc, bt, cl, case.scale, ws,
                             case.k_scale, case.v_scale, stream=stream)
    else:
        slots_new = pk.slot_mapping(case.block_tables, case.context_lens.astype(np.int64) - 1)
        pk.kv_append(case.k_new.to(device), case.v_new.to(device), kc, vc,
                     torch.from_numpy(slots_new).to(device), case.k_scale, case.v_scale,
                     stream=stream)
        pk.paged_decode_attention(out, case.q.to(device), kc, vc, bt, cl, case.scale, ws,
                                  case.k_scale, case.v_scale, stream=stream)
    torch.cuda.synchronize()
    return out, kc, vc


def oracle_caches(case, pool_overrides=None):
    """Host caches after the prefill and the step's append (oracle side)."""
    NB, Hkv, D = case.num_blocks, case.Hkv, case.D
    dt = np.uint16 if case.kv_dtype == workloads.BF16 else np.uint8
    kc = np.zeros((NB, Hkv, BS, D), dtype=dt)
    vc = np.zeros_like(kc)
    pk_bits, pv_bits = bf16_bits(case.pool_k), bf16_bits(case.pool_v)
    if pool_overrides is not None:
        pk_bits, pv_bits = pool_overrides(pk_bits, pv_bits)
    rc = oracle.append(kc, vc, pk_bits, pv_bits, np.arange(NB * BS, dtype=np.int64),
                       case.kv_dtype, case.k_scale, case.v_scale)
    assert rc == 0
    L = case.context_lens.astype(np.int64)
    slots = oracle.slot_mapping(case.block_tables, np.arange(case.B), np.maximum(L - 1, 0))
    slots = np.where(L > 0, slots, -1)          # an empty sequence appends nothing
    rc = oracle.append(kc, vc, bf16_bits(case.k_new), bf16_bits(case.v_new), slots,
                       case.kv_dtype, case.k_scale, case.v_scale)
    assert rc == 0
    return kc, vc


def oracle_step(case, kc, vc, pair_select=None):
    q64 = oracle.bf16_bits_to_f64(bf16_bits(case.q))
    return oracle.paged_attention(q64, kc, vc, case.block_tables, case.context_lens, case.scale,
                                  kv_dtype=case.kv_dtype, k_scale=case.k_scale,
                                  v_scale=case.v_scale, pair_select=pair_select)


def head_mask(case, pair_select):
    """bool [B, Hq] of the query heads belonging to selected (seq, KV head) pairs."""
    if pair_select is None:
        return np.ones((case.B, case.Hq), dtype=bool)
    return np.repeat(pair_select, case.G, axis=1)


def compare(case, out_gpu, ref, pair_select=None, what=""):
    """Assert the GPU output matches the fp64 oracle.  float32 outputs: max-abs
    <= tol; bfloat16 outputs: <= tol + half a bf16 ulp of the exact value.
    Returns the max-abs error (before the ulp allowance)."""
    hm = head_mask(case, pair_select)
    g = out_gpu.float().cpu().numpy().astype(np.float64)[hm]
    r = ref[hm]
    assert np.all(np.isfinite(g)), "non-finite GPU output " + what
    err = np.abs(g - r)
    tol = tolerance(case.kv_dtype)
    if out_gpu.dtype == torch.float32:
        bound = tol
    else:
        bound = tol + half_ulp_bf16(r)
    bad = err > bound
    assert not bad.any(), "%s: %d elements beyond tolerance, max err %.3g (tol %.3g)" % (
        what, int(bad.sum()), float(err.max()), tol)
    return float(err.max())
