"""Shared-prefix decoding on the GPU (paged_decode with a chunk table) against the CPU
oracle.  The result is plain decode attention ("KV Cache" (heepie.pages.dev),
section "Self-Attention") whatever the chunking: the oracle attends each
sequence over its own block-table row; the kernel reads the shared blocks
once per chunk and combines the two partial results."""
import numpy as np
import pytest
import torch

import workloads

import decode_harness as H
from test_gpu_parity import cache_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import paged_kv_cache_21_gb300 as pk  # noqa: F401  (fails loudly without the library)
    torch.cuda.set_device(0)
    pk.get_device_error()
    yield
    flags, detail = pk.get_device_error()
    assert flags == 0, "device error flags %d (detail %d) left set" % (flags, detail)


def chunks_of(case, min_blocks=1):
    import paged_kv_cache_21_gb300 as pk
    return pk.prefix_chunks(case.block_tables, case.context_lens, case.Hq // case.Hkv,
                            min_blocks=min_blocks)


def check_prefix(case, fused, out_dtype=torch.bfloat16, pair_select=None, what="", prefix=None,
                 early_inputs=False):
    prefix = prefix if prefix is not None else chunks_of(case)
    out, kc, vc = H.gpu_step(case, out_dtype=out_dtype, fused=fused, prefix=prefix,
                             early_inputs=early_inputs)
    okc, ovc = H.oracle_caches(case)
    assert np.array_equal(cache_bits(kc), okc), "K cache differs " + what
    assert np.array_equal(cache_bits(vc), ovc), "V cache differs " + what
    ref = H.oracle_step(case, okc, ovc, pair_select)
    return H.compare(case, out, ref, pair_select, what=what), len(prefix[0]), out


def shared_case(Hq, Hkv, D=128, B=24, group=8, kv_dtype=workloads.BF16, n_hi=3000, seed=None):
    """Config-3 structure (groups sharing 38 prefix blocks, log-uniform
    lengths) at a test size."""
    ov = {"B": B, "Hq": Hq, "Hkv": Hkv, "D": D, "group": group, "N_hi": n_hi,
          "kv_dtype": kv_dtype}
    return workloads.make_case("3", override=ov, seed=seed)


@pytest.mark.parametrize("fused,early", [(False, False), (True, False), (True, True)],
                         ids=["append+attend", "fused_step", "fused_step_early_inputs"])
def test_config3_shape_full_compare(fused, early):
    case = workloads.make_case("3", override={"B": 32})
    err, nc, _ = check_prefix(case, fused, what="config 3 B=32 fused=%s" % fused,
                              early_inputs=early)
    assert nc > 0
    print("config 3 B=32 prefix fused=%s: %d chunks, max abs err %.3g" % (fused, nc, err))


@pytest.mark.parametrize("Hq,Hkv,group", [
    (8, 8, 16),      # G=1: 16 members per chunk, 16 query rows
    (16, 8, 8),      # G=2: 8 members, 16 rows
    (32, 8, 8),      # G=4: 4 members
    (64, 8, 8),      # G=8: 2 members
    (24, 8, 8),      # G=3: 5 members, 15 rows
    (40, 8, 8),      # G=5: 3 members, 15 rows
    (56, 8, 8),      # G=7: 2 members, 14 rows
    (8, 8, 4),       # G=1, groups of 4: chunks of 4 rows (one row tile)
])
def test_group_sizes_and_row_tiles(Hq, Hkv, group):
    case = shared_case(Hq, Hkv, B=2 * group, group=group, seed=100 + Hq + group)
    err, nc, _ = check_prefix(case, True, what="Hq %d Hkv %d group %d" % (Hq, Hkv, group))
    assert nc > 0


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("kv_dtype", [workloads.BF16, workloads.FP8_E4M3])
def test_head_dims_and_e4m3(D, kv_dtype):
    case = shared_case(32, 8, D=D, B=16, kv_dtype=kv_dtype, seed=7 + D + kv_dtype)
    for fused in (False, True):
        check_prefix(case, fused, what="D%d dt%d fused=%s" % (D, kv_dtype, fused))


def test_float32_output():
    case = shared_case(32, 8, B=16, seed=31)
    check_prefix(case, True, out_dtype=torch.float32, what="f32 out")


def test_no_chunks_is_plain_decoding_bitwise():
    """num_chunks == 0 runs the plain kernel: bit-identical to paged_decode_step."""
    case = shared_case(32, 8, B=16, seed=5)
    empty = (np.zeros((0, 18), np.int32), np.full(case.B, -1, np.int32))
    _, nc, out_p = check_prefix(case, True, prefix=empty, what="no chunks")
    out, _, _ = H.gpu_step(case, fused=True)
    assert nc == 0 and torch.equal(out.view(torch.int16), out_p.view(torch.int16))


def test_deterministic_and_block_relabelling_invariant():
    """Two runs give the same bits; relabelling the physical blocks (data
    moved with them) gives the same chunks and the same bits."""
    import paged_kv_cache_21_gb300 as pk
    case = shared_case(32, 8, B=24, seed=9)
    pre = chunks_of(case)
    out1, kc, vc = H.gpu_step(case, prefix=pre)
    ws = pk.alloc_prefix_workspace(case.B, len(pre[0]), case.Hq, case.Hkv, case.D)
    dch = torch.from_numpy(pre[0]).cuda()
    dsc = torch.from_numpy(pre[1]).cuda()
    rng = np.random.default_rng(3)
    perm = rng.permutation(case.num_blocks).astype(np.int64)
    kc2, vc2 = torch.empty_like(kc), torch.empty_like(vc)
    pt = torch.from_numpy(perm).cuda()
    kc2[pt] = kc
    vc2[pt] = vc
    bt2 = np.where(case.block_tables >= 0, perm[np.maximum(case.block_tables, 0)], -1)
    bt2 = bt2.astype(np.int32)
    pre2 = pk.prefix_chunks(bt2, case.context_lens, case.Hq // case.Hkv)
    np.testing.assert_array_equal(pre2[0], pre[0])
    np.testing.assert_array_equal(pre2[1], pre[1])
    outs = []
    for _ in range(2):
        o = torch.empty_like(out1)
        pk.paged_decode(o, case.q.cuda(), kc2, vc2, torch.from_numpy(bt2).cuda(),
                        torch.from_numpy(case.context_lens).cuda(), case.scale, ws,
                        chunks=dch, seq_chunk=dsc)
        outs.append(o)
    torch.cuda.synchronize()
    assert torch.equal(out1.view(torch.int16), outs[0].view(torch.int16))
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))


def test_empty_contexts_and_short_members():
    """Empty sequences (no chunk) give zeros next to chunked ones."""
    case = shared_case(32, 8, B=16, seed=13)
    case.context_lens[[3, 11]] = 0
    err, nc, out = check_prefix(case, False, what="empty contexts")
    assert nc > 0
    o = out.float().cpu().numpy()
    assert np.all(o[3] == 0.0) and np.all(o[11] == 0.0)


def test_inconsistent_chunk_entries_are_flagged_and_fall_back():
    """Chunk entries that break the rules are reported through the device
    error word; the sequences concerned are attended alone (correct results),
    every access stays in bounds and the context stays usable."""
    import paged_kv_cache_21_gb300 as pk
    case = shared_case(32, 8, B=24, seed=17)
    chunks, seq_chunk = chunks_of(case)
    assert len(chunks) >= 3
    chunks, seq_chunk = chunks.copy(), seq_chunk.copy()
    bad_seq = int(chunks[0][2])
    seq_chunk[bad_seq] = (len(chunks) + 5) << 4          # names a chunk that does not exist
    chunks[1][1] = 0                                      # a chunk with no members
    chunks[2][0] = 10 ** 6                                # P beyond the block-table width
    pk.get_device_error()
    check_prefix(case, True, prefix=(chunks, seq_chunk), what="bad chunk entries")
    flags, _ = pk.get_device_error()
    assert flags & pk.DEVERR_BAD_PREFIX
    assert flags & ~pk.DEVERR_BAD_PREFIX == 0
    x = torch.ones(4, device="cuda") * 2
    assert float(x.sum()) == 8.0


@pytest.mark.parametrize("kv_dtype", [workloads.BF16, workloads.FP8_E4M3])
def test_config3_full_size_every_pair(kv_dtype):
    """Full-size config 3 through the fused prefix step (early inputs);
    caches and every (sequence, KV head) pair compared with the oracle."""
    case = workloads.make_case("3", override={"kv_dtype": kv_dtype} if kv_dtype else None)
    err, nc, _ = check_prefix(case, True, what="config 3 full size", early_inputs=True)
    assert nc > 0
    print("config 3 full size prefix dt%d: %d chunks, max abs err %.3g over all %d pairs"
          % (kv_dtype, nc, err, case.B * case.Hkv))


@pytest.mark.parametrize("override", [{"B": 32}, None])
def test_long_shared_prompt(override):
    """A 4096-token prompt shared by groups of 8 (the shared blocks are most
    of the bytes): a test-size case, then full size; every pair compared."""
    case = workloads.make_case("3L", override=override)
    err, nc, _ = check_prefix(case, True, what="3L %s" % override, early_inputs=True)
    assert nc > 0
    print("3L %s: %d chunks, max abs err %.3g" % (override, nc, err))


def test_forked_prompt_through_allocator_chunks_and_kernel():
    """A shared system prompt the way a server holds one: a 200-token prompt
    prefilled once, forked to 8 sequences (blocks shared by reference count),
    then 12 decode steps.  Each step: kv_step plans the appends (copy-on-write
    of the shared partial tail block on the first step), kv_prefix_chunks
    finds the shared blocks in the live block tables, and paged_decode
    appends and attends with the chunk table; the oracle replays the same
    tables on its own cache copy."""
    import math
    import paged_kv_cache_21_gb300 as pk
    from workloads import bf16_bits
    import oracle
    Hq, Hkv, D, NB, MB, P0 = 32, 8, 128, 256, 16, 200
    alloc = pk.BlockAllocator(NB, Hkv, D)
    g = torch.Generator().manual_seed(57)
    kc = torch.zeros((NB, Hkv, 16, D), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    okc = np.zeros((NB, Hkv, 16, D), dtype=np.uint16)
    ovc = np.zeros_like(okc)
    alloc.add(100, P0)
    _, row = alloc.info(100)
    pk_ = torch.randn((P0, Hkv, D), generator=g).to(torch.bfloat16)
    pv_ = torch.randn((P0, Hkv, D), generator=g).to(torch.bfloat16)
    slots0 = np.array([row[p // 16] * 16 + p % 16 for p in range(P0)], dtype=np.int64)
    pk.kv_append(pk_.cuda(), pv_.cuda(), kc, vc, torch.from_numpy(slots0).cuda())
    oracle.append(okc, ovc, bf16_bits(pk_), bf16_bits(pv_), slots0, oracle.BF16)
    ids = list(range(8))
    for sid in ids:
        alloc.fork(100, sid, P0)
    alloc.free(100)
    ws = pk.alloc_prefix_workspace(len(ids), len(ids) // 2, Hq, Hkv, D)
    scale = 1 / math.sqrt(D)
    for step in range(12):
        slots, bt, lens, (cs, cd) = alloc.step(ids, MB)
        if len(cs):
            pk.kv_copy_blocks(kc, vc, torch.from_numpy(cs).cuda(), torch.from_numpy(cd).cuda())
            for s_, d_ in zip(cs, cd):
                okc[d_] = okc[s_]
                ovc[d_] = ovc[s_]
        chunks, seq_chunk = pk.prefix_chunks(bt, lens, Hq // Hkv)
        # 200 tokens = 12 full blocks shared by all 8 (the 13th is each one's own copy)
        assert len(chunks) == 2 and all(int(r[0]) >= 12 for r in chunks)
        q = torch.randn((len(ids), Hq, D), generator=g).to(torch.bfloat16)
        k = torch.randn((len(ids), Hkv, D), generator=g).to(torch.bfloat16)
        v = torch.randn((len(ids), Hkv, D), generator=g).to(torch.bfloat16)
        out = torch.empty((len(ids), Hq, D), dtype=torch.float32, device="cuda")
        pk.paged_decode(out, q.cuda(), kc, vc, torch.from_numpy(bt).cuda(),
                        torch.from_numpy(lens).cuda(), scale, ws, k_new=k.cuda(), v_new=v.cuda(),
                        chunks=torch.from_numpy(chunks).cuda(),
                        seq_chunk=torch.from_numpy(seq_chunk).cuda(), early_inputs=True)
        oracle.append(okc, ovc, bf16_bits(k), bf16_bits(v), slots, oracle.BF16)
        ref = oracle.paged_attention(oracle.bf16_bits_to_f64(bf16_bits(q)), okc, ovc, bt, lens,
                                     scale)
        torch.cuda.synchronize()
        assert np.array_equal(kc.cpu().view(torch.int16).numpy().view(np.uint16), okc), step
        assert np.max(np.abs(out.cpu().numpy() - ref)) < H.tolerance(workloads.BF16), step
    for sid in ids:
        alloc.free(sid)
    assert alloc.stats()[0] == NB


def test_general_step_replays_in_a_cuda_graph():
    """paged_decode with a chunk table and early inputs, captured in a CUDA
    graph (programmatic edges inside the graph) and replayed: every replay
    equals the eager call bit for bit (the append rewrites the same token)."""
    import paged_kv_cache_21_gb300 as pk
    case = shared_case(32, 8, B=16, seed=23)
    chunks, seq_chunk = chunks_of(case)
    out_ref, kc, vc = H.gpu_step(case, fused=True, prefix=(chunks, seq_chunk),
                                 early_inputs=True)
    q = case.q.cuda()
    kn, vn = case.k_new.cuda(), case.v_new.cuda()
    bt = torch.from_numpy(case.block_tables).cuda()
    cl = torch.from_numpy(case.context_lens).cuda()
    dch, dsc = torch.from_numpy(chunks).cuda(), torch.from_numpy(seq_chunk).cuda()
    ws = pk.alloc_prefix_workspace(case.B, len(chunks), case.Hq, case.Hkv, case.D)
    out = torch.empty_like(out_ref)

    def call(stream):
        pk.paged_decode(out, q, kc, vc, bt, cl, case.scale, ws, k_new=kn, v_new=vn,
                        chunks=dch, seq_chunk=dsc, early_inputs=True, stream=stream)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        call(s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        call(s)
        call(s)                      # two steps: a programmatic edge inside the graph
    for _ in range(3):
        out.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), out_ref.view(torch.int16))
