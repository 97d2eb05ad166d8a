"""Model check of the split kernel's work partition and partial-slot scheme
(host arithmetic only, no GPU): the flat (sequence, KV head, block) units are
cut into equal per-warp ranges, q = max(q_min, ceil(T / W)); groups above 16
query rows run as 2^k sub-groups, one team of W / 2^k warps each, every team
with the same ranges and its own run of slots.  A warp's partial of pair x
goes to slot team * (pairs + team warps) + x + w.  The merge reads a pair's
partials as n consecutive slots from the first one.  This checks that no two
partials share a slot, that every slot lies inside the workspace, and that
the n consecutive slots of each pair are exactly its partials."""
import numpy as np
import pytest


def partition(lens, hkv, hshift, warps, q_min):
    nblk = [-(-int(L) // 16) for L in lens]
    teams = 1 << hshift
    wt = warps >> hshift
    total = sum(nb * hkv for nb in nblk)
    pairs_p = len(lens) * hkv                       # pairs per team (physical heads)
    team_slots = pairs_p + wt
    slots = {}                                      # slot -> (virtual pair, team warp)
    first = {}                                      # virtual pair -> (slot, n)
    if total == 0:
        return slots, first, teams * team_slots
    q = max(q_min, -(-total // wt))
    flat = 0
    for s, nb in enumerate(nblk):
        for h in range(hkv):
            if nb == 0:
                continue
            f0, f1 = flat, flat + nb - 1
            w0, w1 = f0 // q, f1 // q
            for team in range(teams):
                pv = (s * hkv + h) * teams + team        # virtual pair
                for wl in range(w0, w1 + 1):
                    slot = team * team_slots + (pv >> hshift) + wl
                    assert slot not in slots, "slot %d taken twice" % slot
                    slots[slot] = (pv, wl)
                first[pv] = (team * team_slots + (pv >> hshift) + w0, w1 - w0 + 1)
            flat += nb
    return slots, first, teams * team_slots


@pytest.mark.parametrize("seed", range(40))
def test_partials_never_share_a_slot(seed):
    rng = np.random.default_rng(seed)
    B = int(rng.integers(1, 40))
    hkv = int(rng.choice([1, 2, 8]))
    hshift = int(rng.choice([0, 0, 1, 2, 3]))
    warps = int(rng.choice([1216, 608, 64, 8])) << 0
    q_min = int(rng.choice([2, 5, 16]))
    lens = rng.integers(0, 3000, size=B)
    lens[rng.random(B) < 0.1] = 0
    slots, first, nslots = partition(lens, hkv, hshift, warps, q_min)
    assert all(0 <= s < nslots for s in slots)
    for pv, (s0, n) in first.items():
        got = [slots[s0 + k] for k in range(n)]
        assert all(p == pv for p, _ in got)
        assert [w for _, w in got] == list(range(got[0][1], got[0][1] + n))
    # every partial is reachable from its pair's entry
    reach = sum(n for _, n in first.values())
    assert reach == len(slots)


def test_without_sub_groups_a_slot_is_pair_plus_warp():
    lens, hkv, warps = [100, 600, 0, 33], 2, 16
    slots, first, nslots = partition(lens, hkv, 0, warps, 2)
    assert nslots == len(lens) * hkv + warps
    assert all(slot == pv + w for slot, (pv, w) in slots.items())


def test_one_run_of_slots_for_all_teams_would_collide():
    """Why each team needs its own run: numbering a sub-group's partials by
    virtual pair + global warp index (pairs of different teams interleave)
    reuses slots."""
    lens, hkv, hshift, warps = [3000] * 4, 1, 1, 64
    nblk = -(-3000 // 16)
    teams, wt = 1 << hshift, warps >> hshift
    q = max(16, -(-(4 * nblk * hkv) // wt))
    seen, clash = set(), False
    for s in range(4):
        f0 = s * nblk
        for team in range(teams):
            pv = s * teams + team
            for wl in range(f0 // q, (f0 + nblk - 1) // q + 1):
                slot = pv + team * wt + wl
                clash |= slot in seen
                seen.add(slot)
    assert clash
