"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on the
same seeded inputs.  Append and block indexing must be bit-exact; attention
outputs must be within 2e-3 (bfloat16 KV) or 3e-2 (E4M3 KV) of the float64
oracle, plus half a bfloat16 ulp when the output itself is bfloat16."""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from workloads import bf16_bits

import decode_harness as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import paged_kv_cache_21_gb300 as pk  # noqa: F401  (fails loudly without the library)
    torch.cuda.set_device(0)
    yield
    import paged_kv_cache_21_gb300 as pk
    flags, detail = pk.get_device_error()
    assert flags == 0, "device error flags %d (detail %d) left set" % (flags, detail)


def cache_bits(t):
    t = t.cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def check_case(case, out_dtype=torch.bfloat16, pair_select=None, what="", fused=False,
               early_inputs=False):
    out, kc, vc = H.gpu_step(case, out_dtype=out_dtype, fused=fused, early_inputs=early_inputs)
    okc, ovc = H.oracle_caches(case)
    assert np.array_equal(cache_bits(kc), okc), "K cache differs from oracle " + what
    assert np.array_equal(cache_bits(vc), ovc), "V cache differs from oracle " + what
    ref = H.oracle_step(case, okc, ovc, pair_select)
    return H.compare(case, out, ref, pair_select, what=what)


# ---------------------------------------------------------------- append

@pytest.mark.parametrize("kv_dtype", [workloads.BF16, workloads.FP8_E4M3])
def test_append_bit_exact_with_padding_tokens(kv_dtype):
    import paged_kv_cache_21_gb300 as pk
    rng = np.random.default_rng(5)
    NB, Hkv, D, T = 37, 4, 128, 300
    if kv_dtype == workloads.BF16:
        kc = torch.full((NB, Hkv, 16, D), 3.0, dtype=torch.bfloat16, device="cuda")
    else:
        kc = torch.full((NB, Hkv, 16, D), 0x5A, dtype=torch.uint8, device="cuda")
    vc = kc.clone()
    okc, ovc = cache_bits(kc).copy(), cache_bits(vc).copy()
    g = torch.Generator().manual_seed(9)
    k = (torch.randn((T, Hkv, D), generator=g) * 3).to(torch.bfloat16)
    v = (torch.randn((T, Hkv, D), generator=g) * 0.01).to(torch.bfloat16)
    slots = rng.permutation(NB * 16)[:T].astype(np.int64)
    slots[::7] = -1                                         # padding tokens
    ks, vs = float(np.float32(12.0 / 448)), float(np.float32(0.05 / 448))
    pk.kv_append(k.cuda(), v.cuda(), kc, vc, torch.from_numpy(slots).cuda(), ks, vs)
    assert oracle.append(okc, ovc, bf16_bits(k), bf16_bits(v), slots, kv_dtype, ks, vs) == 0
    assert np.array_equal(cache_bits(kc), okc)
    assert np.array_equal(cache_bits(vc), ovc)


def test_e4m3_encoder_agrees_with_hardware_conversion_on_every_bf16():
    """All 65,536 bfloat16 patterns through kv_append (scale 1): the oracle's
    E4M3 encoder must give the same byte as the GPU conversion (NaN inputs:
    both NaN)."""
    import paged_kv_cache_21_gb300 as pk
    bits = np.arange(65536, dtype=np.uint16)
    k = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).reshape(1, 512, 128)
    kc = torch.zeros((1, 512, 16, 128), dtype=torch.uint8, device="cuda")
    vc = torch.zeros_like(kc)
    pk.kv_append(k.cuda(), k.cuda(), kc, vc, torch.zeros(1, dtype=torch.int64, device="cuda"),
                 1.0, 1.0)
    got = kc[0, :, 0, :].cpu().numpy().reshape(-1)
    want = oracle.quantize_e4m3(bits, 1.0)
    vals = oracle.bf16_bits_to_f64(bits)
    nan_in = np.isnan(vals)
    assert np.array_equal(got[~nan_in], want[~nan_in])
    assert np.all((got[nan_in] & 0x7F) == 0x7F)


def test_copy_blocks_copies_whole_blocks():
    import paged_kv_cache_21_gb300 as pk
    NB, Hkv, D = 9, 2, 64
    g = torch.Generator().manual_seed(3)
    kc = torch.randn((NB, Hkv, 16, D), generator=g).to(torch.bfloat16).cuda()
    vc = torch.randn((NB, Hkv, 16, D), generator=g).to(torch.bfloat16).cuda()
    k0, v0 = kc.clone(), vc.clone()
    src = torch.tensor([1, 4, 7], dtype=torch.int32, device="cuda")
    dst = torch.tensor([2, 0, 8], dtype=torch.int32, device="cuda")
    pk.kv_copy_blocks(kc, vc, src, dst)
    torch.cuda.synchronize()
    for s, d in zip(src.tolist(), dst.tolist()):
        assert torch.equal(kc[d], k0[s]) and torch.equal(vc[d], v0[s])
    for b in (1, 3, 4, 5, 6, 7):
        assert torch.equal(kc[b], k0[b]) and torch.equal(vc[b], v0[b])


# ------------------------------------------------------------- configs

@pytest.mark.parametrize("fused,early", [(False, False), (True, False), (True, True)],
                         ids=["append+attend", "fused_step", "fused_early_inputs"])
@pytest.mark.parametrize("cfg,override", [
    ("1", None),
    ("2", {"B": 3}),                       # 3 x 8193 tokens: many splits + ragged tail
    ("3", {"B": 24}),                      # ragged, 3 groups sharing prefix blocks
    ("4", {"B": 1, "N": 20000}),           # G = 8, long single sequence
    ("5a", {"B": 3}),                      # E4M3 cache
    ("5b", {"B": 2}),                      # MHA, G = 1
])
def test_config_shapes_full_compare(cfg, override, fused, early):
    case = workloads.make_case(cfg, override=override)
    err = check_case(case, what="config %s %s" % (cfg, override), fused=fused,
                     early_inputs=early)
    print("config %s %s fused=%s early=%s: max abs err %.3g" % (cfg, override, fused, early,
                                                                 err))


@pytest.mark.parametrize("cfg", ["2", "3", "4", "5a", "5b"])
def test_config_full_size_every_pair(cfg):
    """Full-size configuration through the call the benchmark times
    (paged_decode: fused append, early inputs); the caches and every
    (sequence, KV head) pair of the output are compared with the oracle."""
    case = workloads.make_case(cfg)
    err = check_case(case, what="config %s full size" % cfg, fused=True, early_inputs=True)
    print("config %s full size: max abs err %.3g over all %d pairs"
          % (cfg, err, case.B * case.Hkv))


@pytest.mark.parametrize("kv_dtype", [workloads.BF16, workloads.FP8_E4M3])
def test_float32_output_within_tolerance(kv_dtype):
    case = workloads.make_custom(5, 32, 8, 128, [1, 17, 300, 4097, 9000], kv_dtype=kv_dtype,
                                 seed=21)
    err = check_case(case, out_dtype=torch.float32, what="f32 out")
    print("f32 output max abs err %.3g" % err)


def query_range_case(kv_dtype, seed=77):
    """Query rows of every bfloat16 magnitude: each (sequence, head) row is
    N(0, 1) times its own power of two 2^E, E from the subnormal range to the
    top of bfloat16, plus one row holding 3e38 and one row whose elements
    each get their own E.  Keys are scaled by 2^-20 so that every score stays
    finite in binary32; values stay N(0, 1), so the output is O(1)."""
    lens = [1, 17, 300, 2000, 33, 4097]
    case = workloads.make_custom(len(lens), 32, 8, 128, lens, kv_dtype=kv_dtype, seed=seed)
    exps = [0, 17, 20, 23, 26, 40, 100, 126, -20, -130]
    rng = np.random.default_rng(seed)
    q = case.q.float()
    E = rng.choice(exps, size=(case.B, case.Hq))
    q = q * torch.from_numpy(np.exp2(E.astype(np.float64))).float()[:, :, None]
    q[0, 1, 5] = 3e38
    q[2, 3] = torch.from_numpy(np.exp2(rng.integers(-130, 127, size=case.D).astype(np.float64))
                               ).float() * torch.sign(q[2, 3] + 0.5)
    case.q = q.to(torch.bfloat16)
    assert torch.isfinite(case.q.float()).all()
    case.pool_k = (case.pool_k.float() * 2.0**-20).to(torch.bfloat16)
    case.k_new = (case.k_new.float() * 2.0**-20).to(torch.bfloat16)
    if kv_dtype == workloads.FP8_E4M3:
        amax_k = max(float(case.pool_k.abs().max()), float(case.k_new.abs().max()))
        case.k_scale = float(np.float32(amax_k) / np.float32(448.0))
    return case


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("kv_dtype", [workloads.BF16, workloads.FP8_E4M3])
def test_query_magnitudes_over_the_whole_bf16_range(kv_dtype, out_dtype):
    """The E4M3 path multiplies q in f16 (exact for bfloat16 values between
    2^-14 and 65504): larger rows are divided by a power of two first and the
    scores multiplied back, so queries up to 3e38 and down to bfloat16
    subnormals give the oracle's result (before, |q| > 65504 gave NaN).  The
    bfloat16 path takes q as it is."""
    case = query_range_case(kv_dtype)
    assert float(case.q.float().abs().max()) > 2.9e38
    err = check_case(case, out_dtype=out_dtype, what="query range dt%d" % kv_dtype)
    check_case(case, out_dtype=out_dtype, what="query range fused dt%d" % kv_dtype, fused=True,
               early_inputs=True)
    print("query magnitudes 2^-130 .. 3e38, dt%d: max abs err %.3g" % (kv_dtype, err))


# ------------------------------------------------------------ edge cases

EDGE_LENS = [1, 2, 15, 16, 17, 31, 32, 33, 255, 256, 257, 4095, 4096, 4097]


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("G", [1, 4, 8])
@pytest.mark.parametrize("kv_dtype", [workloads.BF16, workloads.FP8_E4M3])
def test_edge_lengths(D, G, kv_dtype):
    Hkv = 2
    case = workloads.make_custom(len(EDGE_LENS), G * Hkv, Hkv, D, EDGE_LENS, kv_dtype=kv_dtype,
                                 seed=D + G)
    check_case(case, what="D%d G%d dt%d" % (D, G, kv_dtype))
    check_case(case, what="fused D%d G%d dt%d" % (D, G, kv_dtype), fused=True)


@pytest.mark.parametrize("Hq,Hkv", [(32, 8), (64, 2)])
@pytest.mark.parametrize("kv_dtype", [workloads.BF16, workloads.FP8_E4M3])
@pytest.mark.parametrize("max_len", [40, 300, 600, 2000])
def test_narrow_tables_spread_over_more_warps(max_len, kv_dtype, Hq, Hkv):
    """A block table of w columns sets the minimum range of a warp to
    clamp(ceil(w / 8), 2, 16) blocks: 2, 3, 5 and 16 here (odd and even
    ranges), so short sequences are cut across several warps and merged;
    ragged lengths up to max_len tokens, two-launch and fused paths."""
    rng = np.random.default_rng(max_len)
    lens = rng.integers(1, max_len + 1, size=24)
    lens[0] = max_len
    case = workloads.make_custom(24, Hq, Hkv, 128, lens, kv_dtype=kv_dtype, seed=max_len + 1)
    assert case.block_tables.shape[1] == -(-max_len // 16)
    check_case(case, what="w=%d" % case.block_tables.shape[1])
    check_case(case, what="fused early w=%d" % case.block_tables.shape[1], fused=True,
               early_inputs=True)


@pytest.mark.parametrize("kv_dtype", [workloads.BF16, workloads.FP8_E4M3])
@pytest.mark.parametrize("lens", [[20000, 20000], [100000]])
def test_one_pair_split_over_hundreds_of_warps(lens, kv_dtype):
    """A few long sequences with one KV head: ranges of 16 blocks cut a pair
    into ~80 or ~390 partials, so the merge stages them in several rounds of
    64 (the path beyond one round trip)."""
    case = workloads.make_custom(len(lens), 8, 1, 128, lens, kv_dtype=kv_dtype, seed=len(lens))
    check_case(case, what="%d partials" % (lens[0] // 256))
    check_case(case, what="fused early", fused=True, early_inputs=True)


LARGE_GROUP_LENS = [1, 17, 300, 4097, 2000, 33]


@pytest.mark.parametrize("kv_dtype", [workloads.BF16, workloads.FP8_E4M3])
@pytest.mark.parametrize("Hq,Hkv,D", [(12, 1, 128), (16, 2, 128), (24, 3, 128), (32, 1, 128),
                                      (48, 2, 64), (64, 1, 128), (128, 1, 64), (128, 1, 128),
                                      (256, 2, 128), (80, 1, 128), (96, 1, 128), (72, 1, 128),
                                      (40, 1, 128), (48, 1, 128), (96, 2, 128)])
def test_large_query_groups(Hq, Hkv, D, kv_dtype):
    """G = 12..128, MQA on many-head models ("KV cache complete guide",
    section "(2) GQA": one KV head for all query heads): 9-16 rows run the
    two-row-tile kernel, larger groups run as 2, 4 or 8 sub-groups that read
    the same KV tiles, and above 32 rows (bf16, d128) the tensor-memory
    kernel takes the whole group in one 128-row MMA.  Two-launch and fused
    paths, float32 output, and the append lands once, bit-exact."""
    case = workloads.make_custom(len(LARGE_GROUP_LENS), Hq, Hkv, D, LARGE_GROUP_LENS,
                                 kv_dtype=kv_dtype, seed=Hq + Hkv)
    what = "Hq%d Hkv%d D%d dt%d" % (Hq, Hkv, D, kv_dtype)
    check_case(case, what=what)
    check_case(case, what="fused early " + what, fused=True, early_inputs=True)
    check_case(case, what="f32 " + what, out_dtype=torch.float32)


@pytest.mark.parametrize("Hq", [32, 48, 64, 128])
def test_mqa_full_size_and_deterministic(Hq):
    """One KV head for Hq query heads at the 8B layer's batch and context
    (32 sequences x 8193 tokens, d128): every output against the oracle, and
    two runs bit-identical."""
    import paged_kv_cache_21_gb300 as pk
    case = workloads.make_custom(32, Hq, 1, 128, [8193] * 32, seed=Hq)
    check_case(case, what="MQA %d" % Hq, fused=True, early_inputs=True)
    check_case(case, what="MQA %d f32" % Hq, out_dtype=torch.float32)
    o1, _, _ = H.gpu_step(case, fused=True, early_inputs=True)
    o2, _, _ = H.gpu_step(case, fused=True, early_inputs=True)
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert pk.get_device_error()[0] == 0


@pytest.mark.parametrize("Hq", [48, 64, 128])
@pytest.mark.parametrize("lens", [[100000], [30000, 1, 17, 20000]])
def test_wide_groups_split_over_many_ctas(lens, Hq):
    """48, 64 or 128 query rows on one KV head with pairs cut across tens of CTAs
    of the tensor-memory kernel (partials in sub-groups of 16 rows, then the
    merge), short pairs seen whole by one CTA beside them."""
    case = workloads.make_custom(len(lens), Hq, 1, 128, lens, seed=len(lens) + 77)
    check_case(case, what="wide %s" % lens, fused=True, early_inputs=True)
    check_case(case, what="wide f32 %s" % lens, out_dtype=torch.float32)


@pytest.mark.parametrize("Hq", [48, 64, 128])
def test_wide_groups_flag_bad_block_ids(Hq):
    """A block id outside the pool in the tensor-memory kernel is not
    fetched: its keys are masked, KV_DEVERR_BLOCK_OUT_OF_RANGE is raised with
    the id, nothing faults and the rest of the batch is unaffected."""
    import paged_kv_cache_21_gb300 as pk
    case = workloads.make_custom(3, Hq, 1, 128, [40, 300, 700], seed=91)
    out_ok, kc, vc = H.gpu_step(case, out_dtype=torch.float32)
    pk.get_device_error()
    bt = torch.from_numpy(case.block_tables).cuda()
    bad = bt.clone()
    bad[1, 3] = case.num_blocks + 11
    out = torch.empty_like(out_ok)
    ws = pk.alloc_workspace(case.B, case.Hq, case.Hkv, case.D)
    pk.paged_decode_attention(out, case.q.cuda(), kc, vc, bad,
                              torch.from_numpy(case.context_lens).cuda(), case.scale, ws)
    torch.cuda.synchronize()
    assert pk.get_device_error() == (pk.DEVERR_BLOCK_OUT_OF_RANGE, case.num_blocks + 11)
    assert torch.isfinite(out).all()
    assert torch.equal(out[0], out_ok[0]) and torch.equal(out[2], out_ok[2])


def test_prefix_chunks_refuse_groups_above_eight():
    """A chunk packs at least two members' rows into 16: G > 8 has no chunks,
    and the shared-prefix call refuses a chunk table for it."""
    import paged_kv_cache_21_gb300 as pk
    case = workloads.make_custom(4, 32, 2, 128, [100, 100, 100, 100], seed=3)
    with pytest.raises(pk.KVError):
        pk.prefix_chunks(case.block_tables, case.context_lens, 16)
    with pytest.raises(pk.KVError):
        pk.prefix_workspace_bytes(4, 1, 32, 2, 128)


def test_group_sizes_two_three_five_seven():
    for G in (2, 3, 5, 7):
        case = workloads.make_custom(3, 3 * G, 3, 128, [40, 700, 2000], seed=G)
        check_case(case, what="G=%d" % G)


@pytest.mark.parametrize("Hq,Hkv", [(8, 2), (32, 1)])
def test_many_sequences_beyond_register_scan(Hq, Hkv):
    # more than 256 sequences takes the second scan path of the split kernel
    # (three chunks of 256 here), with some empty contexts mixed in; 32q/1kv
    # runs as two 16-row sub-groups per KV head
    lens = (np.arange(700) * 37) % 500 + 1
    case = workloads.make_custom(700, Hq, Hkv, 64, lens, seed=77)
    case.context_lens[::97] = 0
    check_case(case, what="B=700 G=%d" % (Hq // Hkv))
    check_case(case, what="B=700 fused", fused=True)


@pytest.mark.parametrize("Hq,Hkv", [(8, 2), (16, 1), (64, 2), (128, 1)])
def test_empty_contexts_give_zeros(Hq, Hkv):
    lens = [0, 33, 0, 1, 0]
    case = workloads.make_custom(5, Hq, Hkv, 128, [max(x, 1) for x in lens], seed=4)
    case.context_lens = np.array(lens, dtype=np.int32)
    check_case(case, what="empty contexts")
    # the tolerance without the bf16 output rounding: float32 output
    err = check_case(case, what="empty contexts f32", out_dtype=torch.float32)
    out, _, _ = H.gpu_step(case)
    out_np = out.float().cpu().numpy()
    for s_, L in enumerate(lens):
        if L == 0:
            assert np.all(out_np[s_] == 0.0)
    assert err < 2e-3


@pytest.mark.parametrize("Hq,Hkv", [(16, 4), (48, 1), (64, 1), (128, 1)])
def test_nan_canaries_in_unused_slots_are_never_read(Hq, Hkv):
    case = workloads.make_custom(4, Hq, Hkv, 128, [1, 18, 333, 1000], seed=8, slack=0.5)
    used = np.zeros(case.num_blocks * 16, dtype=bool)
    for s, L in enumerate(case.context_lens):
        for pos in range(int(L)):
            used[case.block_tables[s, pos // 16] * 16 + pos % 16] = True
    nan_bf16 = np.uint16(0x7FC0)

    def poison_np(pk_bits, pv_bits):
        pk_bits, pv_bits = pk_bits.copy(), pv_bits.copy()
        pk_bits[~used] = nan_bf16
        pv_bits[~used] = nan_bf16
        return pk_bits, pv_bits

    def poison_t(pk_t, pv_t):
        m = torch.from_numpy(~used).to(pk_t.device)
        nan = torch.tensor(float("nan"), dtype=torch.bfloat16, device=pk_t.device)
        return torch.where(m[:, None, None], nan, pk_t), torch.where(m[:, None, None], nan, pv_t)

    out, kc, vc = H.gpu_step(case, pool_overrides=poison_t)
    okc, ovc = H.oracle_caches(case, pool_overrides=poison_np)
    assert np.array_equal(cache_bits(kc), okc)
    ref = H.oracle_step(case, okc, ovc)
    H.compare(case, out, ref, what="NaN canaries")


def test_block_permutation_bitwise_invariant_and_deterministic():
    """The same logical cache under two physical block layouts gives
    bit-identical outputs, and repeated runs are bit-identical."""
    import paged_kv_cache_21_gb300 as pk
    case = workloads.make_custom(6, 32, 8, 128, [5, 100, 1000, 3000, 6000, 8193], seed=12)
    out1, kc, vc = H.gpu_step(case)
    # relabel physical blocks with a random permutation, moving the data with them
    rng = np.random.default_rng(99)
    perm = rng.permutation(case.num_blocks).astype(np.int64)
    kc2 = torch.empty_like(kc)
    vc2 = torch.empty_like(vc)
    pt = torch.from_numpy(perm).cuda()
    kc2[pt] = kc
    vc2[pt] = vc
    bt2 = np.where(case.block_tables >= 0, perm[np.maximum(case.block_tables, 0)], -1)
    out2 = torch.empty_like(out1)
    ws = pk.alloc_workspace(case.B, case.Hq, case.Hkv, case.D)
    pk.paged_decode_attention(out2, case.q.cuda(), kc2, vc2,
                              torch.from_numpy(bt2.astype(np.int32)).cuda(),
                              torch.from_numpy(case.context_lens).cuda(), case.scale, ws)
    out3 = torch.empty_like(out1)
    pk.paged_decode_attention(out3, case.q.cuda(), kc2, vc2,
                              torch.from_numpy(bt2.astype(np.int32)).cuda(),
                              torch.from_numpy(case.context_lens).cuda(), case.scale, ws)
    torch.cuda.synchronize()
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))
    assert torch.equal(out2.view(torch.int16), out3.view(torch.int16))


@pytest.mark.parametrize("kv_dtype", [workloads.BF16, workloads.FP8_E4M3])
def test_pool_past_4_gib_with_block_ids_at_its_top(kv_dtype):
    """Largest addresses: the same logical cache placed in a pool of more than
    4 GiB per cache tensor, on block ids at its top end (the last id
    included).  The fused step (append + attention, early inputs) must give
    the same bits as on a compact pool, write the same cache bytes, and agree
    with the oracle; a block copy between two high ids moves the right bytes."""
    import paged_kv_cache_21_gb300 as pk
    case = workloads.make_custom(5, 32, 8, 128, [300, 1000, 17, 2500, 1], kv_dtype=kv_dtype,
                                 seed=61)
    out_ref, kc, vc = H.gpu_step(case, fused=True, early_inputs=True)
    okc, ovc = H.oracle_caches(case)
    assert np.array_equal(cache_bits(kc), okc) and np.array_equal(cache_bits(vc), ovc)
    H.compare(case, out_ref, H.oracle_step(case, okc, ovc), what="compact pool")

    block_bytes = case.Hkv * 16 * case.D * (2 if kv_dtype == workloads.BF16 else 1)
    NB_big = (9 << 29) // block_bytes + 1000            # 4.5 GiB + 1000 blocks per cache
    rng = np.random.default_rng(62)
    off = np.concatenate([[0], 1 + rng.permutation(4 * case.num_blocks)[:case.num_blocks - 1]])
    remap = (NB_big - 1 - off).astype(np.int64)          # distinct, block 0 -> the last id
    assert remap.min() * block_bytes >= 1 << 32
    cdt = torch.bfloat16 if kv_dtype == workloads.BF16 else torch.uint8
    kb = torch.zeros((NB_big, case.Hkv, 16, case.D), dtype=cdt, device="cuda")
    vb = torch.zeros_like(kb)
    c = np.arange(case.num_blocks * 16, dtype=np.int64)
    slots = torch.from_numpy(remap[c // 16] * 16 + c % 16).cuda()
    pk.kv_append(case.pool_k.cuda(), case.pool_v.cuda(), kb, vb, slots, case.k_scale,
                 case.v_scale)
    bt_big = np.where(case.block_tables >= 0, remap[np.maximum(case.block_tables, 0)], -1)
    out_big = torch.empty_like(out_ref)
    ws = pk.alloc_workspace(case.B, case.Hq, case.Hkv, case.D, kv_dtype)
    pk.paged_decode(out_big, case.q.cuda(), kb, vb, torch.from_numpy(bt_big.astype(np.int32)).cuda(),
                    torch.from_numpy(case.context_lens).cuda(), case.scale, ws, case.k_scale,
                    case.v_scale, k_new=case.k_new.cuda(), v_new=case.v_new.cuda(),
                    early_inputs=True)
    torch.cuda.synchronize()
    assert pk.get_device_error()[0] == 0
    assert torch.equal(out_big.view(torch.int16), out_ref.view(torch.int16))
    rt = torch.from_numpy(remap).cuda()
    assert torch.equal(kb[rt].view(torch.uint8), kc.view(torch.uint8))
    assert torch.equal(vb[rt].view(torch.uint8), vc.view(torch.uint8))
    # copy-on-write between two high ids: the top block onto a free one
    free_id = int(np.setdiff1d(np.arange(NB_big - 10, NB_big), remap)[0])
    pk.kv_copy_blocks(kb, vb, torch.tensor([NB_big - 1], dtype=torch.int32, device="cuda"),
                      torch.tensor([free_id], dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert torch.equal(kb[free_id].view(torch.uint8), kc[0].view(torch.uint8))
    assert torch.equal(vb[free_id].view(torch.uint8), vc[0].view(torch.uint8))
    del kb, vb
    torch.cuda.empty_cache()


def test_allocator_driven_steps_with_copy_on_write():
    """Sequences created, forked (shared prefix, copy-on-write) and stepped by
    the host allocator; GPU copies/appends/attends; oracle replays the same
    block tables."""
    import paged_kv_cache_21_gb300 as pk
    Hq, Hkv, D, NB = 8, 2, 128, 64
    alloc = pk.BlockAllocator(NB, Hkv, D)
    g = torch.Generator().manual_seed(31)
    kc = torch.zeros((NB, Hkv, 16, D), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    okc = np.zeros((NB, Hkv, 16, D), dtype=np.uint16)
    ovc = np.zeros_like(okc)
    # prefill sequence 0 with 40 tokens
    alloc.add(0, 40)
    _, row = alloc.info(0)
    pre_k = torch.randn((40, Hkv, D), generator=g).to(torch.bfloat16)
    pre_v = torch.randn((40, Hkv, D), generator=g).to(torch.bfloat16)
    bt0 = np.full((1, 8), -1, dtype=np.int32)
    bt0[0, :len(row)] = row
    pre_slots = np.array([row[p // 16] * 16 + p % 16 for p in range(40)], dtype=np.int64)
    pk.kv_append(pre_k.cuda(), pre_v.cuda(), kc, vc, torch.from_numpy(pre_slots).cuda())
    oracle.append(okc, ovc, bf16_bits(pre_k), bf16_bits(pre_v), pre_slots, oracle.BF16)
    # two forks share the 40-token prefix (tail block 2 is partial and shared)
    alloc.fork(0, 1, 40)
    alloc.fork(0, 2, 40)
    ws = pk.alloc_workspace(3, Hq, Hkv, D)
    for step in range(20):
        ids = [0, 1, 2]
        slots, bt, lens, (cs, cd) = alloc.step(ids, 8)
        if step == 0:
            assert len(cs) == 2        # the first two appenders copy the shared tail
        if len(cs):
            pk.kv_copy_blocks(kc, vc, torch.from_numpy(cs).cuda(), torch.from_numpy(cd).cuda())
            for s_, d_ in zip(cs, cd):
                okc[d_] = okc[s_]
                ovc[d_] = ovc[s_]
        k = torch.randn((3, Hkv, D), generator=g).to(torch.bfloat16)
        v = torch.randn((3, Hkv, D), generator=g).to(torch.bfloat16)
        q = torch.randn((3, Hq, D), generator=g).to(torch.bfloat16)
        pk.kv_append(k.cuda(), v.cuda(), kc, vc, torch.from_numpy(slots).cuda())
        oslots = oracle.slot_mapping(bt, np.arange(3), lens.astype(np.int64) - 1)
        assert np.array_equal(oslots, slots)
        oracle.append(okc, ovc, bf16_bits(k), bf16_bits(v), slots, oracle.BF16)
        out = torch.empty((3, Hq, D), dtype=torch.float32, device="cuda")
        pk.paged_decode_attention(out, q.cuda(), kc, vc, torch.from_numpy(bt).cuda(),
                                  torch.from_numpy(lens).cuda(), 1 / math.sqrt(D), ws)
        ref = oracle.paged_attention(oracle.bf16_bits_to_f64(bf16_bits(q)), okc, ovc, bt, lens,
                                     1 / math.sqrt(D))
        torch.cuda.synchronize()
        assert np.array_equal(cache_bits(kc), okc)
        assert np.max(np.abs(out.cpu().numpy() - ref)) < 2e-3
    alloc.free(1)
    alloc.free(2)
    alloc.free(0)
    assert alloc.stats()[0] == NB


def test_cancelled_request_frees_blocks_for_a_new_one():
    """Request cancellation mid-batch (mask/KV page, implementation and
    verification procedure): a sequence is freed between steps, a new request
    takes its blocks (stale K/V still in them) and the batch goes on through
    the fused step with early inputs.  Every step matches the oracle on the
    same tables; stale slots past a length must get no weight."""
    import paged_kv_cache_21_gb300 as pk
    Hq, Hkv, D, NB, MB = 8, 2, 128, 24, 8
    alloc = pk.BlockAllocator(NB, Hkv, D)
    g = torch.Generator().manual_seed(41)
    kc = torch.zeros((NB, Hkv, 16, D), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    okc = np.zeros((NB, Hkv, 16, D), dtype=np.uint16)
    ovc = np.zeros_like(okc)
    scale = 1 / math.sqrt(D)

    def prefill(sid, n):
        alloc.add(sid, n)
        _, row = alloc.info(sid)
        k = torch.randn((n, Hkv, D), generator=g).to(torch.bfloat16)
        v = torch.randn((n, Hkv, D), generator=g).to(torch.bfloat16)
        sl = np.array([row[p // 16] * 16 + p % 16 for p in range(n)], dtype=np.int64)
        pk.kv_append(k.cuda(), v.cuda(), kc, vc, torch.from_numpy(sl).cuda())
        oracle.append(okc, ovc, bf16_bits(k), bf16_bits(v), sl, oracle.BF16)
        return set(int(b) for b in row)

    def decode(ids, steps):
        ws = pk.alloc_workspace(len(ids), Hq, Hkv, D)
        for _ in range(steps):
            slots, bt, lens, (cs, _) = alloc.step(ids, MB)
            assert len(cs) == 0
            k = torch.randn((len(ids), Hkv, D), generator=g).to(torch.bfloat16)
            v = torch.randn((len(ids), Hkv, D), generator=g).to(torch.bfloat16)
            q = torch.randn((len(ids), Hq, D), generator=g).to(torch.bfloat16)
            out = torch.empty((len(ids), Hq, D), dtype=torch.float32, device="cuda")
            pk.paged_decode(out, q.cuda(), kc, vc, torch.from_numpy(bt).cuda(),
                            torch.from_numpy(lens).cuda(), scale, ws, k_new=k.cuda(),
                            v_new=v.cuda(), early_inputs=True)
            oracle.append(okc, ovc, bf16_bits(k), bf16_bits(v), slots, oracle.BF16)
            ref = oracle.paged_attention(oracle.bf16_bits_to_f64(bf16_bits(q)), okc, ovc, bt,
                                         lens, scale)
            torch.cuda.synchronize()
            assert np.array_equal(cache_bits(kc), okc)
            assert np.max(np.abs(out.cpu().numpy() - ref)) < 2e-3

    prefill(0, 30)
    cancelled = prefill(1, 45)
    prefill(2, 20)
    decode([0, 1, 2], 3)
    alloc.free(1)                                  # cancelled after 48 tokens: 3 blocks
    assert alloc.stats()[2] == 2
    fresh = prefill(3, 40)                         # takes freed blocks, stale data inside
    assert fresh & cancelled
    decode([0, 2, 3], 4)
    decode([3, 0], 2)                              # the batch shrinks and reorders
    assert pk.get_device_error()[0] == 0
    for sid in (0, 2, 3):
        alloc.free(sid)
    assert alloc.stats()[0] == NB


def test_bad_inputs_are_flagged_not_faulted():
    """Out-of-range slots and block ids are skipped and reported through the
    device error word; the context stays usable."""
    import paged_kv_cache_21_gb300 as pk
    pk.get_device_error()
    NB, Hkv, D = 4, 1, 64
    kc = torch.zeros((NB, Hkv, 16, D), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    k = torch.ones((2, Hkv, D), dtype=torch.bfloat16, device="cuda")
    pk.kv_append(k, k, kc, vc, torch.tensor([3, NB * 16 + 5], dtype=torch.int64, device="cuda"))
    torch.cuda.synchronize()
    flags, detail = pk.get_device_error()
    assert flags == pk.DEVERR_SLOT_OUT_OF_RANGE and detail == NB * 16 + 5
    assert float(kc[0, 0, 3, 0]) == 1.0
    out = torch.empty((1, 2, D), dtype=torch.float32, device="cuda")
    ws = pk.alloc_workspace(1, 2, 1, D)
    bt = torch.tensor([[0, 99]], dtype=torch.int32, device="cuda")
    cl = torch.tensor([20], dtype=torch.int32, device="cuda")
    pk.paged_decode_attention(out, torch.ones((1, 2, D), dtype=torch.bfloat16, device="cuda"),
                              kc, vc, bt, cl, 0.125, ws)
    torch.cuda.synchronize()
    flags, detail = pk.get_device_error()
    assert flags == pk.DEVERR_BLOCK_OUT_OF_RANGE and detail == 99
    assert torch.isfinite(out).all()
    # the context is still healthy
    x = torch.ones(4, device="cuda") * 2
    assert float(x.sum()) == 8.0


@pytest.mark.parametrize("prefix", [False, True, "wide", "wide64"],
                         ids=["plain", "prefix_chunks", "wide", "wide64"])
@pytest.mark.parametrize("kv_dtype", [workloads.BF16, workloads.FP8_E4M3])
def test_pipeline_timeout_is_flagged_and_the_context_stays_usable(kv_dtype, prefix):
    """The bounded wait on a bulk copy: with the test hook every warp's first
    wait is on a barrier that nothing arrives on (no copy is lost -- the
    copies it issued are still waited for before it stops).  The time-out
    must raise KV_DEVERR_PIPELINE_TIMEOUT (and nothing else), and the next
    call on the same context must give the oracle's result."""
    import paged_kv_cache_21_gb300 as pk
    case = workloads.make_custom(6, 32, 8, 128, [1, 17, 300, 4097, 2000, 33],
                                 kv_dtype=kv_dtype, seed=93)
    pre = None
    if prefix in ("wide", "wide64"):
        # 128 (or 64) query rows on one KV head: the tensor-memory kernel with
        # the 128-row (64-row) Q buffer (bf16 only; the E4M3 case runs the
        # sub-group kernel)
        case = workloads.make_custom(6, 128 if prefix == "wide" else 64, 1, 128,
                                     [1, 17, 300, 4097, 2000, 33], kv_dtype=kv_dtype, seed=95)
    elif prefix:
        case = workloads.make_case("3", override={"B": 16, "N_hi": 3000, "kv_dtype": kv_dtype},
                                   seed=94)
        pre = pk.prefix_chunks(case.block_tables, case.context_lens, case.G)
        assert len(pre[0]) > 0
    pk.get_device_error()
    pk.set_pipeline_stall(20000)                 # ~10 us of SM clocks
    try:
        H.gpu_step(case, fused=True, early_inputs=True, prefix=pre)
    finally:
        pk.set_pipeline_stall(0)
    flags, detail = pk.get_device_error()
    assert flags == pk.DEVERR_PIPELINE_TIMEOUT, (flags, detail)
    if prefix not in ("wide", "wide64") or kv_dtype != workloads.BF16:
        assert detail == 0, detail               # the split kernel reports the unit
    x = torch.ones(4, device="cuda") * 2
    assert float(x.sum()) == 8.0
    out, kc, vc = H.gpu_step(case, fused=True, early_inputs=True, prefix=pre)
    okc, ovc = H.oracle_caches(case)
    assert np.array_equal(cache_bits(kc), okc) and np.array_equal(cache_bits(vc), ovc)
    H.compare(case, out, H.oracle_step(case, okc, ovc), what="after a time-out")
    assert pk.get_device_error()[0] == 0
    with pytest.raises(pk.KVError):
        pk.set_pipeline_stall(-1)


def test_context_longer_than_its_table_row_is_flagged_and_clamped():
    """A context length past its block-table row (the context-limit overflow
    case) or below zero is reported as KV_DEVERR_CONTEXT_TOO_LONG with the bad
    length, clamped into [0, 16 * max_blocks_per_seq], and nothing faults."""
    import paged_kv_cache_21_gb300 as pk
    # sequence 2 fills its 7-entry row, so the clamped length reads valid blocks
    case = workloads.make_custom(3, 8, 2, 128, [40, 64, 100], seed=21)
    mb = case.block_tables.shape[1]
    assert mb == 7 and (case.block_tables[2] >= 0).all()
    _, kc, vc = H.gpu_step(case)
    pk.get_device_error()
    okc, ovc = H.oracle_caches(case)
    bt = torch.from_numpy(case.block_tables).cuda()
    q64 = oracle.bf16_bits_to_f64(bf16_bits(case.q))
    ws = pk.alloc_workspace(case.B, case.Hq, case.Hkv, case.D)
    for bad, clamped in ((16 * mb + 5, 16 * mb), (-3, 0)):
        lens = case.context_lens.copy()
        lens[2] = bad
        out = torch.empty((case.B, case.Hq, case.D), dtype=torch.float32, device="cuda")
        pk.paged_decode_attention(out, case.q.cuda(), kc, vc, bt, torch.from_numpy(lens).cuda(),
                                  case.scale, ws)
        torch.cuda.synchronize()
        flags, detail = pk.get_device_error()
        assert flags == pk.DEVERR_CONTEXT_TOO_LONG and detail == bad
        ref_lens = lens.copy()
        ref_lens[2] = clamped
        ref = oracle.paged_attention(q64, okc, ovc, case.block_tables, ref_lens, case.scale)
        assert np.max(np.abs(out.cpu().numpy() - ref)) < 2e-3
    assert pk.get_device_error()[0] == 0


def test_workspace_needs_no_initialisation():
    """Garbage-filled workspace, then the same workspace reused: every launch
    writes the pair table and the partial slots it reads, so nothing depends
    on what the workspace held before."""
    import paged_kv_cache_21_gb300 as pk
    case = workloads.make_custom(5, 32, 8, 128, [3000, 9000, 17, 20000, 513], seed=44)
    ws = pk.alloc_workspace(case.B, case.Hq, case.Hkv, case.D)
    g = torch.Generator(device="cuda").manual_seed(5)
    ws.copy_(torch.randint(0, 256, ws.shape, dtype=torch.uint8, device="cuda", generator=g))
    out1, kc, vc = H.gpu_step(case, workspace=ws)
    okc, ovc = H.oracle_caches(case)
    ref = H.oracle_step(case, okc, ovc)
    H.compare(case, out1, ref, what="garbage workspace")
    out2 = torch.empty_like(out1)
    for _ in range(3):
        pk.paged_decode_attention(out2, case.q.cuda(), kc, vc,
                                  torch.from_numpy(case.block_tables).cuda(),
                                  torch.from_numpy(case.context_lens).cuda(), case.scale, ws)
        torch.cuda.synchronize()
        assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))


@pytest.mark.parametrize("Hq,Hkv", [(32, 8), (64, 1), (128, 1)])
def test_fused_step_replays_in_a_cuda_graph(Hq, Hkv):
    """A captured fused step replays with the same arguments: each replay
    appends the same token again and must give the same output (the merge
    reads only what that replay's split kernel wrote).  128 rows on one KV
    head: the tensor-memory kernel in a graph."""
    import paged_kv_cache_21_gb300 as pk
    case = workloads.make_custom(4, Hq, Hkv, 128, [5000, 70, 12000, 4097], seed=45)
    out_ref, kc, vc = H.gpu_step(case, fused=True)          # first call: per-device set-up
    q = case.q.cuda()
    kn, vn = case.k_new.cuda(), case.v_new.cuda()
    bt = torch.from_numpy(case.block_tables).cuda()
    cl = torch.from_numpy(case.context_lens).cuda()
    ws = pk.alloc_workspace(case.B, case.Hq, case.Hkv, case.D)
    out = torch.empty_like(out_ref)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        pk.paged_decode_step(out, q, kn, vn, kc, vc, bt, cl, case.scale, ws, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        pk.paged_decode_step(out, q, kn, vn, kc, vc, bt, cl, case.scale, ws, stream=s)
    for _ in range(3):
        out.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), out_ref.view(torch.int16))


def test_beam_reorder_and_duplication_through_the_kernels():
    """Rows [A0, A1, B0] reordered by [2, 1, 0], then beams duplicated by
    [0, 0, 1] (copy-on-write at the next append), with decode steps in
    between; every step is checked against the oracle on the same tables."""
    import paged_kv_cache_21_gb300 as pk
    Hq, Hkv, D, NB, MB = 8, 2, 128, 64, 8
    alloc = pk.BlockAllocator(NB, Hkv, D)
    g = torch.Generator().manual_seed(77)
    kc = torch.zeros((NB, Hkv, 16, D), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    okc = np.zeros((NB, Hkv, 16, D), dtype=np.uint16)
    ovc = np.zeros_like(okc)
    ids = [10, 11, 12]
    for sid, L in zip(ids, (21, 37, 50)):
        alloc.add(sid, L)
        _, row = alloc.info(sid)
        kk = torch.randn((L, Hkv, D), generator=g).to(torch.bfloat16)
        vv = torch.randn((L, Hkv, D), generator=g).to(torch.bfloat16)
        sl = np.array([row[p // 16] * 16 + p % 16 for p in range(L)], dtype=np.int64)
        pk.kv_append(kk.cuda(), vv.cuda(), kc, vc, torch.from_numpy(sl).cuda())
        oracle.append(okc, ovc, bf16_bits(kk), bf16_bits(vv), sl, oracle.BF16)
    ws = pk.alloc_workspace(3, Hq, Hkv, D)

    def step(expect_lens=None):
        slots, bt, lens, (cs, cd) = alloc.step(ids, MB)
        if expect_lens is not None:
            assert list(lens) == expect_lens
        if len(cs):
            pk.kv_copy_blocks(kc, vc, torch.from_numpy(cs).cuda(), torch.from_numpy(cd).cuda())
            for s_, d_ in zip(cs, cd):
                okc[d_] = okc[s_]
                ovc[d_] = ovc[s_]
        k = torch.randn((3, Hkv, D), generator=g).to(torch.bfloat16)
        v = torch.randn((3, Hkv, D), generator=g).to(torch.bfloat16)
        q = torch.randn((3, Hq, D), generator=g).to(torch.bfloat16)
        out = torch.empty((3, Hq, D), dtype=torch.float32, device="cuda")
        pk.paged_decode_step(out, q.cuda(), k.cuda(), v.cuda(), kc, vc,
                             torch.from_numpy(bt).cuda(), torch.from_numpy(lens).cuda(),
                             1 / math.sqrt(D), ws)
        oracle.append(okc, ovc, bf16_bits(k), bf16_bits(v), slots, oracle.BF16)
        ref = oracle.paged_attention(oracle.bf16_bits_to_f64(bf16_bits(q)), okc, ovc, bt, lens,
                                     1 / math.sqrt(D))
        torch.cuda.synchronize()
        assert np.array_equal(cache_bits(kc), okc)
        assert np.max(np.abs(out.cpu().numpy() - ref)) < 2e-3
        return lens

    step([22, 38, 51])
    alloc.reorder(ids, [2, 1, 0])          # [A0, A1, B0] -> [B0, A1, A0]
    step([52, 39, 23])
    alloc.reorder(ids, [0, 0, 1])          # beam duplication: rows 0 and 1 share B0's history
    for _ in range(20):
        step()
    for sid in ids:
        alloc.free(sid)
    assert alloc.stats()[0] == NB


@pytest.mark.parametrize("host_ordered", [False, True])
def test_staged_host_steps_match_device_step(host_ordered):
    """DecodeStepStaging (per step: one H2D copy of every input on a copy
    stream, fused step, one D2H copy; two alternating slots) gives the same
    bits as the fused step on device inputs, step after step, whether the
    compute stream or the host waits for each upload."""
    import paged_kv_cache_21_gb300 as pk
    case = workloads.make_custom(5, 32, 8, 128, [1, 300, 4097, 9000, 20], seed=81)
    out_ref, kc, vc = H.gpu_step(case, fused=True)
    # the fused step already appended the new tokens; rerunning rewrites them identically
    stg = pk.DecodeStepStaging(case.B, case.Hq, case.Hkv, case.D, case.max_blocks,
                               host_ordered=host_ordered)
    for i in range(5):
        stg.ready_for_input(i)
        hs = stg.host(i)
        hs.q.copy_(case.q)
        hs.k_new.copy_(case.k_new)
        hs.v_new.copy_(case.v_new)
        hs.block_tables.copy_(torch.from_numpy(case.block_tables))
        hs.context_lens.copy_(torch.from_numpy(case.context_lens))
        hs.out.zero_()
        stg.step(i, kc, vc, case.scale)
        if i >= 1:
            stg.wait_output(i - 1)
            assert torch.equal(stg.host(i - 1).out.view(torch.int16),
                               out_ref.cpu().view(torch.int16))
    stg.wait_output(4)
    assert torch.equal(stg.host(4).out.view(torch.int16), out_ref.cpu().view(torch.int16))
    assert stg.h2d_bytes >= (5 * 32 * 128 + 2 * 5 * 8 * 128) * 2


@pytest.mark.parametrize("kv_dtype", [workloads.BF16, workloads.FP8_E4M3])
def test_token_by_token_decode_equals_causal_prefill(kv_dtype):
    """Decode two sequences from empty, one token per step through the fused
    step; step t must equal row t of full causal attention over the same
    tokens (the mask/KV page's check that prefill and token-by-token decode
    agree)."""
    import paged_kv_cache_21_gb300 as pk
    Hq, Hkv, D, T, NB, MB = 8, 2, 64, 70, 16, 8
    g = torch.Generator().manual_seed(91 + kv_dtype)
    Q = torch.randn((2, T, Hq, D), generator=g).to(torch.bfloat16)
    Kt = torch.randn((2, T, Hkv, D), generator=g).to(torch.bfloat16)
    Vt = torch.randn((2, T, Hkv, D), generator=g).to(torch.bfloat16)
    ks = vs = 1.0
    if kv_dtype == workloads.FP8_E4M3:
        ks = float(np.float32(float(Kt.abs().max())) / np.float32(448.0))
        vs = float(np.float32(float(Vt.abs().max())) / np.float32(448.0))
    alloc = pk.BlockAllocator(NB, Hkv, D, kv_dtype)
    alloc.add(0, 0)
    alloc.add(1, 0)
    cdt = torch.bfloat16 if kv_dtype == workloads.BF16 else torch.uint8
    kc = torch.zeros((NB, Hkv, 16, D), dtype=cdt, device="cuda")
    vc = torch.zeros_like(kc)
    ws = pk.alloc_workspace(2, Hq, Hkv, D, kv_dtype)
    # the values the cache holds, as the oracle sees them (dequantised for E4M3)
    if kv_dtype == workloads.FP8_E4M3:
        Kv = oracle.e4m3_decode_array(oracle.quantize_e4m3(bf16_bits(Kt), ks)) * ks
        Vv = oracle.e4m3_decode_array(oracle.quantize_e4m3(bf16_bits(Vt), vs)) * vs
    else:
        Kv, Vv = oracle.bf16_bits_to_f64(bf16_bits(Kt)), oracle.bf16_bits_to_f64(bf16_bits(Vt))
    Qv = oracle.bf16_bits_to_f64(bf16_bits(Q))
    full = np.empty((2, T, Hq, D))
    for s in range(2):
        for h in range(Hq):
            full[s, :, h] = oracle.causal_attention(Qv[s, :, h], Kv[s, :, h // (Hq // Hkv)],
                                                    Vv[s, :, h // (Hq // Hkv)], 1 / math.sqrt(D))
    tol = H.tolerance(kv_dtype)
    for t in range(T):
        _, bt, lens, (cs, cd) = alloc.step([0, 1], MB)
        assert len(cs) == 0 and list(lens) == [t + 1, t + 1]
        out = torch.empty((2, Hq, D), dtype=torch.float32, device="cuda")
        pk.paged_decode_step(out, Q[:, t].contiguous().cuda(), Kt[:, t].contiguous().cuda(),
                             Vt[:, t].contiguous().cuda(), kc, vc, torch.from_numpy(bt).cuda(),
                             torch.from_numpy(lens).cuda(), 1 / math.sqrt(D), ws, ks, vs)
        torch.cuda.synchronize()
        err = np.max(np.abs(out.cpu().numpy() - full[:, t]))
        assert err < tol, (t, err)


@pytest.mark.parametrize("kv_dtype,Hq,Hkv", [(workloads.BF16, 8, 2), (workloads.FP8_E4M3, 8, 2),
                                             (workloads.BF16, 128, 1)])
def test_back_to_back_decode_loop_with_early_inputs(kv_dtype, Hq, Hkv):
    """The token-by-token decode of two sequences as one stream of launches
    with no host synchronisation between steps: every step's tables are
    uploaded before the loop, then paged_decode runs step after step with
    KV_DECODE_EARLY_INPUTS (each step's kernel reads the block tables and the
    cache tiles while the previous step drains, and must still see the
    previous step's append).  Every step equals row t of causal attention,
    and the outputs equal those of the same loop with the default ordering,
    bit for bit."""
    import paged_kv_cache_21_gb300 as pk
    D, T, NB, MB = 128, 90, 16, 8
    g = torch.Generator().manual_seed(191 + kv_dtype)
    Q = torch.randn((2, T, Hq, D), generator=g).to(torch.bfloat16)
    Kt = torch.randn((2, T, Hkv, D), generator=g).to(torch.bfloat16)
    Vt = torch.randn((2, T, Hkv, D), generator=g).to(torch.bfloat16)
    ks = vs = 1.0
    if kv_dtype == workloads.FP8_E4M3:
        ks = float(np.float32(float(Kt.abs().max())) / np.float32(448.0))
        vs = float(np.float32(float(Vt.abs().max())) / np.float32(448.0))
    alloc = pk.BlockAllocator(NB, Hkv, D, kv_dtype)
    alloc.add(0, 0)
    alloc.add(1, 0)
    tables, lens = [], []
    for t in range(T):
        _, bt, ln, (cs, _cd) = alloc.step([0, 1], MB)
        assert len(cs) == 0
        tables.append(bt.copy())
        lens.append(ln.copy())
    d_bt = torch.from_numpy(np.stack(tables)).cuda()          # [T, 2, MB]
    d_len = torch.from_numpy(np.stack(lens)).cuda()           # [T, 2]
    d_q = Q.transpose(0, 1).contiguous().cuda()               # [T, 2, Hq, D]
    d_k = Kt.transpose(0, 1).contiguous().cuda()
    d_v = Vt.transpose(0, 1).contiguous().cuda()
    cdt = torch.bfloat16 if kv_dtype == workloads.BF16 else torch.uint8
    ws = pk.alloc_workspace(2, Hq, Hkv, D, kv_dtype)
    outs = {}
    for early in (False, True):
        kc = torch.zeros((NB, Hkv, 16, D), dtype=cdt, device="cuda")
        vc = torch.zeros_like(kc)
        out = torch.empty((T, 2, Hq, D), dtype=torch.float32, device="cuda")
        torch.cuda.synchronize()
        for t in range(T):
            pk.paged_decode(out[t], d_q[t], kc, vc, d_bt[t], d_len[t], 1 / math.sqrt(D), ws, ks,
                            vs, k_new=d_k[t], v_new=d_v[t], early_inputs=early)
        torch.cuda.synchronize()
        outs[early] = out.cpu()
    assert torch.equal(outs[False], outs[True])
    if kv_dtype == workloads.FP8_E4M3:
        Kv = oracle.e4m3_decode_array(oracle.quantize_e4m3(bf16_bits(Kt), ks)) * ks
        Vv = oracle.e4m3_decode_array(oracle.quantize_e4m3(bf16_bits(Vt), vs)) * vs
    else:
        Kv, Vv = oracle.bf16_bits_to_f64(bf16_bits(Kt)), oracle.bf16_bits_to_f64(bf16_bits(Vt))
    Qv = oracle.bf16_bits_to_f64(bf16_bits(Q))
    tol = H.tolerance(kv_dtype)
    for s in range(2):
        for h in range(Hq):
            ref = oracle.causal_attention(Qv[s, :, h], Kv[s, :, h // (Hq // Hkv)],
                                          Vv[s, :, h // (Hq // Hkv)], 1 / math.sqrt(D))
            err = np.max(np.abs(outs[True][:, s, h].numpy() - ref))
            assert err < tol, (s, h, err)


def test_pinned_host_buffers_read_in_place():
    """The per-step buffers (q, k_new, v_new, block tables, lengths, out) in
    pinned host memory: the kernels read and write them in place, and the
    result equals the device-buffer call bit for bit (caches identical too);
    the zero-copy staging mode runs the same steps."""
    import paged_kv_cache_21_gb300 as pk
    case = workloads.make_custom(6, 32, 8, 128, [1, 40, 700, 3000, 9000, 16], seed=61)
    out_d, kc_d, vc_d = H.gpu_step(case, fused=True, early_inputs=True)
    NB = case.num_blocks
    kc = torch.zeros((NB, case.Hkv, 16, case.D), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    pk.kv_append(case.pool_k.cuda(), case.pool_v.cuda(), kc, vc,
                 torch.arange(NB * 16, dtype=torch.int64, device="cuda"))
    stg = pk.DecodeStepStaging(case.B, case.Hq, case.Hkv, case.D, case.max_blocks,
                               zero_copy=True)
    hs = stg.host(0)
    hs.q.copy_(case.q)
    hs.k_new.copy_(case.k_new)
    hs.v_new.copy_(case.v_new)
    hs.block_tables.copy_(torch.from_numpy(case.block_tables))
    hs.context_lens.copy_(torch.from_numpy(case.context_lens))
    stg.step(0, kc, vc, case.scale)
    stg.wait_output(0)
    assert torch.equal(hs.out.view(torch.int16), out_d.cpu().view(torch.int16))
    assert torch.equal(kc.view(torch.int16), kc_d.view(torch.int16))
    assert torch.equal(vc.view(torch.int16), vc_d.view(torch.int16))


def test_fast_calls_match_ctypes_calls_and_share_the_library():
    """The per-step calls through the CPython-API module and through ctypes
    reach the same library instance: same output bits, and a device flag
    raised by a fast call is what kv_get_device_error (ctypes) reports."""
    import paged_kv_cache_21_gb300 as pk
    if not pk.fast_path():
        pytest.skip("fast-call module not built")
    case = workloads.make_custom(4, 32, 8, 128, [17, 300, 4097, 1000], seed=52)
    out_f, kc, vc = H.gpu_step(case, fused=True, early_inputs=True)
    bt = torch.from_numpy(case.block_tables).cuda()
    cl = torch.from_numpy(case.context_lens).cuda()
    ws = pk.alloc_workspace(case.B, case.Hq, case.Hkv, case.D)
    out_c = torch.empty_like(out_f)
    L = pk._lib
    s = torch.cuda.current_stream().cuda_stream
    kn, vn, q = case.k_new.cuda(), case.v_new.cuda(), case.q.cuda()
    rc = L.paged_decode(out_c.data_ptr(), pk.BF16, q.data_ptr(), kn.data_ptr(), vn.data_ptr(),
                        kc.data_ptr(), vc.data_ptr(), pk.BF16, 1.0, 1.0, case.num_blocks,
                        bt.data_ptr(), bt.shape[1], cl.data_ptr(), case.B, case.Hq, case.Hkv,
                        case.D, case.scale, None, None, 0, pk.DECODE_EARLY_INPUTS,
                        ws.data_ptr(), ws.numel(), s)
    assert rc == pk.KV_OK
    torch.cuda.synchronize()
    assert torch.equal(out_c.view(torch.int16), out_f.view(torch.int16))
    pk.get_device_error()
    bad = bt.clone()
    bad[1, 0] = case.num_blocks + 7
    pk.paged_decode(out_c, q, kc, vc, bad, cl, case.scale, ws)
    torch.cuda.synchronize()
    assert pk.get_device_error() == (pk.DEVERR_BLOCK_OUT_OF_RANGE, case.num_blocks + 7)


def test_read_ceiling_reads_every_piece():
    """The read-only ceiling hook reads every 8 KB piece of its buffer (the
    last one partial here): its XOR sink equals the XOR of the first word of
    every piece, computed on the host, and no copy timed out."""
    import paged_kv_cache_21_gb300 as pk
    nbytes = 8192 * 3001 + 4096 + 16
    g = torch.Generator(device="cuda").manual_seed(11)
    buf = torch.randint(-2**31, 2**31 - 1, (nbytes // 4,), dtype=torch.int32, device="cuda",
                        generator=g)
    sink = torch.zeros(2, dtype=torch.int32, device="cuda")
    pk.read_ceiling(buf, sink)
    torch.cuda.synchronize()
    words = buf.cpu().numpy().view(np.uint32)
    want = np.bitwise_xor.reduce(words[:: 8192 // 4])
    got = sink.cpu().numpy().view(np.uint32)
    assert got[1] == 0
    assert got[0] == want


@pytest.mark.parametrize("kv_dtype", [workloads.BF16, workloads.FP8_E4M3])
def test_timed_call_matches_the_plain_call(kv_dtype):
    """paged_decode_timed runs the same kernels as paged_decode and only adds
    event records: the outputs are bit-identical and the three events are in
    order."""
    import paged_kv_cache_21_gb300 as pk
    case = workloads.make_custom(6, 32, 8, 128, [9000, 17, 4097, 2500, 1, 700], seed=46,
                                 kv_dtype=kv_dtype)
    out_ref, kc, vc = H.gpu_step(case, fused=True)
    q, kn, vn = case.q.cuda(), case.k_new.cuda(), case.v_new.cuda()
    bt = torch.from_numpy(case.block_tables).cuda()
    cl = torch.from_numpy(case.context_lens).cuda()
    ws = pk.alloc_workspace(case.B, case.Hq, case.Hkv, case.D)
    out_a = torch.empty_like(out_ref)
    out_b = torch.empty_like(out_ref)
    # the caches already hold the step's token: both calls rewrite the same bytes
    pk.paged_decode(out_a, q, kc, vc, bt, cl, case.scale, ws, case.k_scale, case.v_scale,
                    k_new=kn, v_new=vn)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    for e in ev:
        e.record()
    pk.paged_decode_timed(out_b, q, kc, vc, bt, cl, case.scale, ws, ev, case.k_scale,
                          case.v_scale, k_new=kn, v_new=vn)
    torch.cuda.synchronize()
    assert torch.equal(out_a.view(torch.int16), out_b.view(torch.int16))
    assert torch.equal(out_a.view(torch.int16), out_ref.view(torch.int16))
    split = ev[0].elapsed_time(ev[1])
    total = ev[0].elapsed_time(ev[2])
    assert 0.0 < split <= total
