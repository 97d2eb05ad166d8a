"""Host logic of shared-prefix decoding: the chunk table kv_prefix_chunks
builds from block tables ("KV cache complete guide", sections "(3) Prefix
Caching" and "(4) PagedAttention": requests with the same system prompt share
its physical blocks).  Checked against the rules the kernels rely on, not
against a second implementation."""
import numpy as np
import pytest

import workloads

MAX_ROWS = 16


@pytest.fixture(scope="module")
def pk():
    import __graft_entry__
    __graft_entry__.build_native()
    import paged_kv_cache_21_gb300 as m
    return m


def check_table(bt, lens, G, chunks, seq_chunk, min_blocks=1):
    """Every rule of the chunk table: sizes, membership, sharing, and the new
    token lying past the shared blocks."""
    B = bt.shape[0]
    assert seq_chunk.shape == (B,)
    seen = set()
    for c, row in enumerate(chunks):
        P, m = int(row[0]), int(row[1])
        members = [int(x) for x in row[2:2 + m]]
        assert 2 <= m <= MAX_ROWS // G and m * G <= MAX_ROWS
        assert all(x == -1 for x in row[2 + m:])
        assert P >= min_blocks
        assert len(set(members)) == m and not (set(members) & seen)
        seen |= set(members)
        for j, s in enumerate(members):
            assert 0 <= s < B
            assert seq_chunk[s] == (c << 4) | j
            assert 16 * P <= int(lens[s]) - 1          # shared blocks end before the new token
            np.testing.assert_array_equal(bt[s, :P], bt[members[0], :P])
    for s in range(B):
        if s not in seen:
            assert seq_chunk[s] == -1


def saved_reads(chunks):
    return sum(int(r[0]) * (int(r[1]) - 1) for r in chunks)


@pytest.mark.parametrize("B", [32, 256])
def test_config3_tables(pk, B):
    case = workloads.make_case("3", override={"B": B})
    G = case.Hq // case.Hkv
    chunks, seq_chunk = pk.prefix_chunks(case.block_tables, case.context_lens, G)
    check_table(case.block_tables, case.context_lens, G, chunks, seq_chunk)
    assert len(chunks) > 0
    # the recipe shares min(38, N // 16) leading blocks within each group of 8:
    # the redundant reads are sum(shared) - (one copy per group)
    groups = B // 8
    shared = case.shared_blocks.astype(np.int64)
    redundant = int(shared.sum()) - sum(int(shared[8 * g:8 * g + 8].max()) for g in range(groups))
    assert 0 < saved_reads(chunks) <= redundant
    assert saved_reads(chunks) >= 0.5 * redundant


def test_no_sharing_gives_no_chunks(pk):
    case = workloads.make_custom(12, 32, 8, 128, [40 + 37 * i for i in range(12)], seed=3)
    chunks, seq_chunk = pk.prefix_chunks(case.block_tables, case.context_lens, 4)
    assert chunks.shape == (0, 18) and (seq_chunk == -1).all()


@pytest.mark.parametrize("G", [1, 2, 3, 4, 5, 7, 8])
def test_chunk_rows_fit_one_tile(pk, G):
    # 20 sequences sharing 6 blocks, lengths 100..290 tokens
    B, mb = 20, 24
    rng = np.random.default_rng(G)
    lens = (100 + 10 * np.arange(B)).astype(np.int32)
    bt = np.full((B, mb), -1, dtype=np.int32)
    ids = rng.permutation(1000).astype(np.int32)
    shared, cur = ids[:6], 6
    for s in range(B):
        nb = -(-int(lens[s]) // 16)
        bt[s, :6] = shared
        bt[s, 6:nb] = ids[cur:cur + nb - 6]
        cur += nb - 6
    chunks, seq_chunk = pk.prefix_chunks(bt, lens, G)
    check_table(bt, lens, G, chunks, seq_chunk)
    per = MAX_ROWS // G
    assert len(chunks) == B // per + (1 if B % per >= 2 else 0)
    assert all(int(r[0]) == 6 for r in chunks)


def test_nested_prefixes_and_short_members(pk):
    # a tree: all 8 share 4 blocks, the first 4 share 10; sequence 7 has only
    # 3 full blocks before its new token (so it shares 3), sequence 6 is empty
    B, mb = 8, 16
    bt = np.full((B, mb), -1, dtype=np.int32)
    base = np.arange(100, 104, dtype=np.int32)
    deep = np.arange(200, 206, dtype=np.int32)
    nxt = 300
    lens = np.array([200, 180, 190, 170, 120, 130, 0, 60], dtype=np.int32)
    for s in range(B):
        nb = -(-int(lens[s]) // 16)
        if nb == 0:
            continue
        row = list(base) + (list(deep) if s < 4 else [])
        row = row[:nb]
        while len(row) < nb:
            row.append(nxt)
            nxt += 1
        bt[s, :nb] = row
    chunks, seq_chunk = pk.prefix_chunks(bt, lens, 4)
    check_table(bt, lens, 4, chunks, seq_chunk)
    assert seq_chunk[6] == -1
    # the four deep members come first (run 10), then the rest (runs 4, 4, 3)
    assert [int(x) for x in chunks[0][:2]] == [10, 4]
    assert sorted(chunks[0][2:6].tolist()) == [0, 1, 2, 3]
    assert [int(x) for x in chunks[1][:2]] == [3, 3]


def test_min_blocks_and_bad_arguments(pk):
    case = workloads.make_case("3", override={"B": 32})
    chunks, _ = pk.prefix_chunks(case.block_tables, case.context_lens, 4, min_blocks=30)
    assert len(chunks) > 0 and all(int(r[0]) >= 30 for r in chunks)
    with pytest.raises(pk.KVError):
        pk.prefix_chunks(case.block_tables, case.context_lens, 9)
    with pytest.raises(pk.KVError):
        pk.prefix_chunks(case.block_tables, case.context_lens, 4, min_blocks=0)
    empty_c, empty_s = pk.prefix_chunks(np.zeros((0, 4), np.int32), np.zeros(0, np.int32), 4)
    assert empty_c.shape[0] == 0 and empty_s.shape[0] == 0


@pytest.mark.parametrize("seed", range(6))
def test_random_prefix_trees_obey_every_rule(pk, seed):
    """Random block tables: groups share random runs of leading blocks
    (prefixes of one another, a tree), some sequences stand alone, some are
    empty; every table kv_prefix_chunks builds obeys the rules, and a chunk
    never spans two groups."""
    rng = np.random.default_rng(1000 + seed)
    G = int(rng.choice([1, 2, 4, 8]))
    B = int(rng.integers(2, 60))
    mb = 40
    bt = np.full((B, mb), -1, dtype=np.int32)
    lens = np.zeros(B, dtype=np.int32)
    next_id = 0
    group_of = rng.integers(0, max(1, B // 4), size=B)
    trunks = {}
    for s in range(B):
        g = int(group_of[s])
        if g not in trunks:
            trunks[g] = list(range(next_id, next_id + mb))
            next_id += mb
        if rng.random() < 0.15:
            continue                                    # empty context
        L = int(rng.integers(1, 16 * mb + 1))
        nb = -(-L // 16)
        run = int(rng.integers(0, nb + 1))              # leading blocks taken from the trunk
        row = trunks[g][:run] + list(range(next_id, next_id + nb - run))
        next_id += nb - run
        bt[s, :nb] = row
        lens[s] = L
    min_blocks = int(rng.integers(1, 4))
    chunks, seq_chunk = pk.prefix_chunks(bt, lens, G, min_blocks=min_blocks)
    check_table(bt, lens, G, chunks, seq_chunk, min_blocks=min_blocks)
    for row in chunks:
        members = [int(x) for x in row[2:2 + int(row[1])]]
        assert len({int(group_of[s]) for s in members}) == 1


def _saved_fraction(chunks, lens):
    saved = sum(int(r[0]) * (int(r[1]) - 1) for r in chunks)
    return saved / float((-(-np.asarray(lens, dtype=np.int64) // 16)).sum())


def _plan_pays(frac, pairs, warps):
    if 5 * pairs >= 2 * warps:
        return frac >= 0.06
    if 5 * pairs >= warps:
        return frac >= 0.30
    return False


@pytest.mark.parametrize("cfg,override,want_chunks", [
    ("3", None, False),                 # 608-token prompt: ~5 % of the blocks saved
    ("3L", None, True),                 # 4096-token prompt: about half saved
    ("3L", {"B": 256, "prefix_blocks": 64}, True),
    ("3L", {"B": 256, "prefix_blocks": 16}, False),                # ~3 % saved
    ("3L", {"B": 128, "prefix_blocks": 32}, True),                 # 1024 pairs, ~6 %
    ("3L", {"B": 64, "prefix_blocks": 32}, True),                  # 512 pairs, ~6 %
    ("3L", {"B": 32}, True),                                       # 256 pairs, ~51 %
    ("3L", {"B": 32, "prefix_blocks": 192}, True),                 # 256 pairs, ~38 %
    ("3L", {"B": 32, "prefix_blocks": 128}, False),                # 256 pairs, ~25 %
    ("3L", {"B": 16}, False),                                      # 128 pairs
])
def test_plan_uses_chunks_only_where_they_pay(pk, cfg, override, want_chunks):
    """kv_prefix_plan keeps kv_prefix_chunks' table when the chunks save a
    fraction f of the blocks read of at least 6 % (5 pairs >= 2 W) or 30 %
    (W <= 5 pairs < 2 W), W = the 1216 resident warps of a GB300 (152 SMs x 2
    CTAs x 4 warps); otherwise it asks for plain decoding (no chunks, seq_chunk
    all -1)."""
    spec, L, bt, NB, _, _ = workloads.make_layout(cfg, override=override)
    G = spec["Hq"] // spec["Hkv"]
    full = pk.prefix_chunks(bt, L, G)
    chunks, seq_chunk = pk.prefix_plan(bt, L, spec["Hq"], spec["Hkv"], spec["D"],
                                       resident_warps=1216)
    frac = _saved_fraction(full[0], L)
    assert _plan_pays(frac, spec["B"] * spec["Hkv"], 1216) == want_chunks, frac
    if want_chunks:
        np.testing.assert_array_equal(chunks, full[0])
        np.testing.assert_array_equal(seq_chunk, full[1])
        check_table(bt, L, G, chunks, seq_chunk)
    else:
        assert len(full[0]) > 0 and len(chunks) == 0 and (seq_chunk == -1).all()


def test_plan_thresholds_follow_the_resident_warps(pk):
    """The same tables planned for a device with other resident warps: the
    tier boundaries move with W (5 pairs against W and 2 W)."""
    spec, L, bt, NB, _, _ = workloads.make_layout("3L", override={"B": 32, "prefix_blocks": 64})
    G = spec["Hq"] // spec["Hkv"]
    frac = _saved_fraction(pk.prefix_chunks(bt, L, G)[0], L)
    assert 0.06 <= frac < 0.30
    pairs = spec["B"] * spec["Hkv"]                       # 256
    for warps, want in ((5 * pairs // 2, True), (5 * pairs // 2 + 1, False),
                        (5 * pairs, False), (5 * pairs + 1, False)):
        chunks, seq_chunk = pk.prefix_plan(bt, L, spec["Hq"], spec["Hkv"], spec["D"],
                                           resident_warps=warps)
        assert (len(chunks) > 0) == want, warps
        assert want or (seq_chunk == -1).all()


def test_plan_refuses_large_groups_and_bad_shapes(pk):
    spec, L, bt, NB, _, _ = workloads.make_layout("3L")
    chunks, seq_chunk = pk.prefix_plan(bt, L, 256, 8, 128, resident_warps=1216)   # G = 32
    assert len(chunks) == 0 and (seq_chunk == -1).all()
    with pytest.raises(pk.KVError):
        pk.prefix_plan(bt, L, 30, 8, 128, resident_warps=1216)                   # Hq % Hkv
