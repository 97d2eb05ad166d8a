"""Host block allocator behind the C ABI: free list, reference counts,
copy-on-write and the per-step slot mapping (no GPU needed)."""
import numpy as np
import pytest

import oracle


@pytest.fixture(scope="module")
def pk():
    import __graft_entry__
    __graft_entry__.build_native()
    import paged_kv_cache_21_gb300 as pk
    return pk


def test_add_and_free_return_blocks(pk):
    a = pk.BlockAllocator(10, 8, 128)
    a.add(1, 33)                         # 3 blocks
    a.add(2, 16)                         # 1 block
    assert a.stats()[:3] == (6, 4, 2)
    ln, row = a.info(1)
    assert ln == 33 and len(row) == 3 and len(set(row)) == 3
    a.free(1)
    assert a.stats()[:3] == (9, 1, 1)
    a.free(2)
    assert a.stats()[:3] == (10, 0, 0)
    with pytest.raises(pk.KVError) as e:
        a.free(2)
    assert e.value.code == pk.KV_ERR_NOT_FOUND


def test_exhaustion_is_reported_and_changes_nothing(pk):
    a = pk.BlockAllocator(4, 1, 64)
    a.add(0, 48)                         # 3 blocks
    with pytest.raises(pk.KVError) as e:
        a.add(1, 17)                     # needs 2
    assert e.value.code == pk.KV_ERR_OUT_OF_BLOCKS
    assert a.stats()[:3] == (1, 3, 1)
    a.add(1, 16)
    # both sequences sit at a block boundary: the step needs 2 fresh blocks
    with pytest.raises(pk.KVError) as e:
        a.step([0, 1], 8)
    assert e.value.code == pk.KV_ERR_OUT_OF_BLOCKS
    assert a.info(0)[0] == 48 and a.info(1)[0] == 16
    with pytest.raises(pk.KVError) as e:
        a.add(0, 1)
    assert e.value.code == pk.KV_ERR_EXISTS


def test_step_slot_mapping_and_block_growth(pk):
    a = pk.BlockAllocator(64, 2, 64)
    a.add(7, 0)
    a.add(9, 15)
    for step in range(40):
        slots, bt, lens, (cs, cd) = a.step([7, 9], 6)
        assert len(cs) == 0
        assert list(lens) == [step + 1, step + 16]
        # the new token goes at position == previous length
        want = oracle.slot_mapping(bt, np.arange(2), lens.astype(np.int64) - 1)
        np.testing.assert_array_equal(slots, want)
        for i in range(2):
            nb = -(-int(lens[i]) // 16)
            assert np.all(bt[i, :nb] >= 0) and np.all(bt[i, nb:] == -1)
    # a row too short for the next append is refused, nothing changes
    with pytest.raises(pk.KVError):
        a.step([9], 3)
    assert a.info(9)[0] == 55


def test_fork_shares_blocks_and_copies_on_write(pk):
    a = pk.BlockAllocator(32, 4, 128)
    a.add(0, 40)                                 # blocks b0 b1 b2, b2 partial (8 tokens)
    _, row0 = a.info(0)
    a.fork(0, 1, 40)
    a.fork(0, 2, 40)
    for b in row0:
        assert a.stats(int(b))[3] == 3
    assert a.stats()[1] == 3                     # no new blocks used by forking
    slots, bt, lens, (cs, cd) = a.step([0, 1, 2], 8)
    # the first two appenders find the shared partial tail and copy it; the
    # third is then its only owner and appends in place
    assert list(cs) == [row0[2], row0[2]]
    assert len(set(cd)) == 2 and row0[2] not in cd
    assert bt[2, 2] == row0[2]
    assert bt[0, 2] == cd[0] and bt[1, 2] == cd[1]
    assert a.stats(int(row0[2]))[3] == 1
    for b in row0[:2]:
        assert a.stats(int(b))[3] == 3           # full prefix blocks stay shared
    np.testing.assert_array_equal(slots, oracle.slot_mapping(bt, np.arange(3), [40, 40, 40]))
    a.free(0)
    a.free(1)
    a.free(2)
    assert a.stats()[:3] == (32, 0, 0)


def test_fork_at_block_boundary_needs_no_copy(pk):
    a = pk.BlockAllocator(16, 1, 64)
    a.add(0, 32)
    a.fork(0, 1, 32)
    slots, bt, lens, (cs, cd) = a.step([0, 1], 4)
    assert len(cs) == 0
    assert bt[0, 2] != bt[1, 2]
    assert bt[0, 0] == bt[1, 0] and bt[0, 1] == bt[1, 1]


def test_fork_of_a_prefix_shorter_than_parent(pk):
    a = pk.BlockAllocator(16, 1, 64)
    a.add(0, 50)
    a.fork(0, 1, 20)                             # shares b0 and the partial b1
    assert a.info(1)[0] == 20 and len(a.info(1)[1]) == 2
    slots, bt, lens, (cs, cd) = a.step([1], 4)
    assert list(cs) == [a.info(0)[1][1]]         # b1 is shared and partial for seq 1
    with pytest.raises(pk.KVError):
        a.fork(0, 2, 51)                         # longer than the parent


def test_step_rejects_bad_requests_atomically(pk):
    a = pk.BlockAllocator(16, 1, 64)
    a.add(0, 5)
    a.add(1, 5)
    before = (a.info(0), a.info(1), a.stats())
    for ids in ([0, 99], [0, 0]):
        with pytest.raises(pk.KVError):
            a.step(ids, 4)
    a.fork(0, 2, 5)
    with pytest.raises(pk.KVError):
        a.step([0, 2], 4, cow_cap=0)             # a copy is needed but not allowed
    assert a.info(0)[0] == before[0][0] and a.info(1)[0] == before[1][0]


def test_random_operations_keep_pool_invariants(pk):
    """Model check: free + used == pool; each block's refcount equals the
    number of live sequences holding it; every block table row matches the
    model's view of the sequence."""
    rng = np.random.default_rng(123)
    NB = 200
    a = pk.BlockAllocator(NB, 2, 64)
    lens = {}
    slot = {}                    # model of the trace: batch row, last reorder source
    rsrc = {}
    next_id = 0
    for _ in range(1500):
        op = rng.integers(0, 5)
        try:
            if op == 0:
                ln = int(rng.integers(0, 80))
                a.add(next_id, ln)
                lens[next_id], slot[next_id], rsrc[next_id] = ln, -1, -1
                next_id += 1
            elif op == 1 and lens:
                sid = int(rng.choice(list(lens)))
                a.free(sid)
                del lens[sid], slot[sid], rsrc[sid]
            elif op == 2 and lens:
                sid = int(rng.choice(list(lens)))
                sl = int(rng.integers(0, lens[sid] + 1))
                a.fork(sid, next_id, sl)
                lens[next_id], slot[next_id], rsrc[next_id] = sl, -1, -1
                next_id += 1
            elif op == 3 and lens:
                ids = rng.choice(list(lens), size=min(len(lens), 5), replace=False)
                slots, bt, ln, _ = a.step(ids, 64)
                for i, sid in enumerate(ids):
                    lens[int(sid)] += 1
                    slot[int(sid)] = i
                    assert ln[i] == lens[int(sid)]
                np.testing.assert_array_equal(
                    slots, oracle.slot_mapping(bt, np.arange(len(ids)), ln.astype(np.int64) - 1))
            elif op == 4 and lens:
                ids = [int(x) for x in rng.choice(list(lens), size=min(len(lens), 4),
                                                  replace=False)]
                src = rng.integers(0, len(ids), size=len(ids))
                a.reorder(ids, src)
                old = [lens[x] for x in ids]
                for i, sid in enumerate(ids):
                    lens[sid], slot[sid], rsrc[sid] = old[src[i]], i, int(src[i])
        except pk.KVError as e:
            assert e.code in (pk.KV_ERR_OUT_OF_BLOCKS, pk.KV_ERR_INVALID_ARG)
        free, used, nseq, _ = a.stats()
        assert free + used == NB and nseq == len(lens)
    holders = {}
    rows = {}
    for sid, ln in lens.items():
        got_len, row = a.info(sid)
        assert got_len == ln and len(row) == -(-ln // 16)
        rows[sid] = row
        for b in row:
            holders[int(b)] = holders.get(int(b), 0) + 1
    for b in range(NB):
        assert a.stats(b)[3] == holders.get(b, 0)
    assert a.stats()[1] == len(holders)
    # the debug trace agrees with the model, field by field
    trace = a.trace()
    assert [r["seq_id"] for r in trace] == sorted(lens)
    for r in trace:
        sid = r["seq_id"]
        nb = len(rows[sid])
        assert (r["slot"], r["reorder_src"]) == (slot[sid], rsrc[sid])
        assert r["len"] == r["position"] == lens[sid] and r["mask_shape"] == [1, lens[sid]]
        assert r["blocks"] == nb and r["cache_bytes"] == nb * 2 * 16 * 2 * 64 * 2
        assert r["shared_blocks"] == sum(holders[int(b)] > 1 for b in rows[sid])


def test_reorder_follows_the_row_permutation(pk):
    # rows [A0, A1, B0] -> [B0, A1, A0]: permutation [2, 1, 0]
    a = pk.BlockAllocator(32, 1, 64)
    a.add(10, 20)      # A0
    a.add(11, 35)      # A1
    a.add(12, 50)      # B0
    before = {sid: a.info(sid) for sid in (10, 11, 12)}
    a.reorder([10, 11, 12], [2, 1, 0])
    assert a.info(10)[0] == before[12][0] and list(a.info(10)[1]) == list(before[12][1])
    assert a.info(11)[0] == before[11][0] and list(a.info(11)[1]) == list(before[11][1])
    assert a.info(12)[0] == before[10][0] and list(a.info(12)[1]) == list(before[10][1])
    assert a.stats()[:3] == (32 - 2 - 3 - 4, 9, 3)


def test_reorder_with_duplicates_shares_and_releases(pk):
    a = pk.BlockAllocator(32, 1, 64)
    a.add(0, 40)                                 # 3 blocks, tail partial
    a.add(1, 17)                                 # 2 blocks
    b0 = a.info(0)[1]
    a.reorder([0, 1], [0, 0])                    # beam 1 becomes a copy of beam 0
    assert list(a.info(1)[1]) == list(b0) and a.info(1)[0] == 40
    assert a.stats()[1] == 3                     # beam 1's old blocks went back to the pool
    for b in b0:
        assert a.stats(int(b))[3] == 2
    slots, bt, lens, (cs, cd) = a.step([0, 1], 8)
    assert list(cs) == [b0[2]] and len(cd) == 1  # the shared tail is copied once
    assert bt[0, 2] != bt[1, 2]
    with pytest.raises(pk.KVError):
        a.reorder([0, 1], [0, 2])                # index out of range
    with pytest.raises(pk.KVError):
        a.reorder([0, 0], [0, 1])                # repeated sequence id


def test_trace_records_the_state_contract_fields(pk):
    # the fields a trace keeps: request id, batch slot, length, position offset,
    # cache shape and bytes, and the reorder permutation; checked against
    # what the operations above imply, and a 2-layer pool's byte count
    a = pk.BlockAllocator(64, 8, 128)
    assert a.shape() == ((64, 8, 16, 128), pk.BF16)
    a.add(10, 20)                          # 2 blocks
    a.add(11, 35)                          # 3 blocks
    a.add(12, 50)                          # 4 blocks
    t = {r["seq_id"]: r for r in a.trace()}
    assert [r["seq_id"] for r in a.trace()] == [10, 11, 12]
    assert t[11] == {"seq_id": 11, "slot": -1, "len": 35, "position": 35, "blocks": 3,
                     "shared_blocks": 0, "cache_bytes": 3 * 2 * 16 * 8 * 128 * 2,
                     "reorder_src": -1, "mask_shape": [1, 35]}
    # one block of K and V for one layer is the pages' per-token formula x 16
    assert t[10]["cache_bytes"] == 2 * pk.kv_bytes(1, 1, 8, 16, 128, 2)
    a.step([12, 10, 11], 8)
    t = {r["seq_id"]: r for r in a.trace()}
    assert [t[s]["slot"] for s in (12, 10, 11)] == [0, 1, 2]
    assert [t[s]["len"] for s in (12, 10, 11)] == [51, 21, 36]
    assert all(t[s]["position"] == t[s]["len"] for s in t)
    # rows [A0, A1, B0] -> [B0, A1, A0] with permutation [2, 1, 0]
    a.reorder([10, 11, 12], [2, 1, 0])
    tr = a.trace([10, 11, 12])
    assert [r["reorder_src"] for r in tr] == [2, 1, 0]
    assert [r["slot"] for r in tr] == [0, 1, 2]
    assert [r["len"] for r in tr] == [51, 36, 21]
    # beam duplication: both rows share every block
    a.reorder([10, 11], [0, 0])
    tr = a.trace([10, 11])
    assert tr[0]["shared_blocks"] == tr[0]["blocks"] == tr[1]["shared_blocks"] == 4
    a.fork(12, 13, 16)
    assert a.trace([13])[0] == {"seq_id": 13, "slot": -1, "len": 16, "position": 16,
                                "blocks": 1, "shared_blocks": 1,
                                "cache_bytes": 2 * 16 * 8 * 128 * 2, "reorder_src": -1,
                                "mask_shape": [1, 16]}
    lines = a.dump().splitlines()
    import json
    head = json.loads(lines[0])
    assert head["kv_shape"] == [64, 8, 16, 128] and head["num_seqs"] == 4
    assert [json.loads(x)["seq_id"] for x in lines[1:]] == [10, 11, 12, 13]
    with pytest.raises(pk.KVError):
        a.trace([99])
    f8 = pk.BlockAllocator(4, 2, 64, kv_dtype=pk.FP8_E4M3)
    f8.add(0, 17)
    assert f8.trace()[0]["cache_bytes"] == 2 * 2 * 16 * 2 * 64 * 1
    assert f8.trace([]) == [] and pk.BlockAllocator(2, 1, 64).trace() == []
