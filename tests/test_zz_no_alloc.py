"""The allocation-free decode entry point (paged_decode_attention_noalloc).

Some callers cannot allocate device memory -- a plugin inside a host framework
that owns the whole device memory pool, or a latency-critical path that must
not enter the driver's allocator -- so they cannot pass the scratch workspace
that paged_decode_attention needs.  The library then uses its own fixed
16 MiB device array instead.  This file checks, through the C ABI, that the
variant returns bit for bit what the allocating entry point returns (both run
the same deterministic kernels; only the scratch differs), on calls in a row
with different shapes (the shared scratch keeps the previous call's
contents), that its output is within the parity tolerance of the float64
oracle, and that a shape needing more scratch than the array holds is
refused before anything runs.

It is named to be collected last, so that a run stopping at the first failure
has already run every other test."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads
from workloads import bf16_bits

import decode_harness as H

pytestmark = pytest.mark.gpu

BS = 16


@pytest.fixture(scope="module")
def pk():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import paged_kv_cache_21_gb300 as pk
    torch.cuda.set_device(0)
    return pk


def _device_case(pk, case):
    """Caches filled through kv_append, and the device tensors of one step."""
    NB, Hkv, D = case.num_blocks, case.Hkv, case.D
    cdt = torch.bfloat16 if case.kv_dtype == workloads.BF16 else torch.uint8
    kc = torch.zeros((NB, Hkv, BS, D), dtype=cdt, device="cuda")
    vc = torch.zeros_like(kc)
    pk.kv_append(case.pool_k.cuda(), case.pool_v.cuda(), kc, vc,
                 torch.arange(NB * BS, dtype=torch.int64, device="cuda"),
                 case.k_scale, case.v_scale)
    return dict(q=case.q.cuda(), kc=kc, vc=vc,
                bt=torch.from_numpy(case.block_tables).cuda(),
                cl=torch.from_numpy(case.context_lens).cuda())


def _run_both(pk, case, t):
    """Output of the allocating entry point and of the allocation-free one."""
    ref = torch.empty((case.B, case.Hq, case.D), dtype=torch.float32, device="cuda")
    ws = pk.alloc_workspace(case.B, case.Hq, case.Hkv, case.D, case.kv_dtype)
    pk.paged_decode_attention(ref, t["q"], t["kc"], t["vc"], t["bt"], t["cl"], case.scale, ws,
                              case.k_scale, case.v_scale)
    got = torch.full_like(ref, float("nan"))
    pk.paged_decode_attention_noalloc(got, t["q"], t["kc"], t["vc"], t["bt"], t["cl"],
                                      case.scale, case.k_scale, case.v_scale)
    torch.cuda.synchronize()
    return ref.cpu().numpy(), got.cpu().numpy()


def _oracle_out(case):
    """The oracle's attention over the same pool (no step append here)."""
    NB, Hkv, D = case.num_blocks, case.Hkv, case.D
    dt = np.uint16 if case.kv_dtype == workloads.BF16 else np.uint8
    kc = np.zeros((NB, Hkv, BS, D), dtype=dt)
    vc = np.zeros_like(kc)
    assert oracle.append(kc, vc, bf16_bits(case.pool_k), bf16_bits(case.pool_v),
                         np.arange(NB * BS, dtype=np.int64), case.kv_dtype, case.k_scale,
                         case.v_scale) == 0
    return H.oracle_step(case, kc, vc)


def test_noalloc_matches_allocating_entry_point_on_two_calls_in_a_row(pk):
    # call 1: ragged batch, GQA 4, long enough that sequences are split
    # across warps (partials go through the library's scratch)
    a = workloads.make_custom(6, 32, 8, 128, [1, 17, 300, 4097, 9000, 20000], seed=61)
    # call 2: a different shape (MHA, d64, E4M3 cache) reusing the same scratch
    b = workloads.make_custom(5, 16, 16, 64, [5000, 33, 2, 12000, 700],
                              kv_dtype=workloads.FP8_E4M3, seed=62)
    ta, tb = _device_case(pk, a), _device_case(pk, b)
    for n, (case, t) in enumerate(((a, ta), (b, tb), (a, ta))):
        ref, got = _run_both(pk, case, t)
        assert np.all(np.isfinite(got))
        assert np.array_equal(got.view(np.int32), ref.view(np.int32)), "call %d" % n
        if n < 2:
            H.compare(case, torch.from_numpy(got), _oracle_out(case),
                      what="allocation-free call %d" % n)
    flags, detail = pk.get_device_error()
    assert flags == 0, (flags, detail)


def test_noalloc_refuses_shapes_beyond_its_scratch(pk):
    # 20000 sequences x 8 KV heads need far more than 16 MiB of scratch: the
    # call must fail on the host, before any pointer is used or kernel runs
    L = pk._lib
    need = pk.workspace_bytes(20000, 32, 8, 128)
    assert need > pk.NOALLOC_WORKSPACE_BYTES
    rc = L.paged_decode_attention_noalloc(None, 0, None, None, None, 0, 1.0, 1.0, 1, None, 1,
                                          None, 20000, 32, 8, 128, 0.1, None)
    assert rc == pk.KV_ERR_TOO_LARGE
    with pytest.raises(pk.KVError) as e:
        q = torch.zeros((20000, 32, 128), dtype=torch.bfloat16, device="cuda")
        kc = torch.zeros((1, 8, BS, 128), dtype=torch.bfloat16, device="cuda")
        pk.paged_decode_attention_noalloc(torch.empty_like(q), q, kc, kc,
                                          torch.zeros((20000, 1), dtype=torch.int32,
                                                      device="cuda"),
                                          torch.zeros(20000, dtype=torch.int32, device="cuda"),
                                          0.1)
    assert e.value.code == pk.KV_ERR_TOO_LARGE
