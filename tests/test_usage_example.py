"""The library's basic usage, one decode step of one layer, written the way
a caller writes it: the host allocator plans the step (slot, block table,
length), the caller owns the device tensors, paged_decode appends the new
K/V and attends.  With one key per sequence the result has a closed form:
softmax over a single key is 1, so every query head returns the new V of its
KV head exactly ("KV Cache" (heepie.pages.dev), section "Self-Attention")."""
import pytest
import torch

pytestmark = pytest.mark.gpu


def test_one_step_from_empty_sequences_returns_the_new_values():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import paged_kv_cache_21_gb300 as pk

    NB, Hq, Hkv, D = 4096, 32, 8, 128
    alloc = pk.BlockAllocator(NB, Hkv, D)                      # host: free list, refcounts
    k_cache = torch.zeros((NB, Hkv, 16, D), dtype=torch.bfloat16, device="cuda")
    v_cache = torch.zeros_like(k_cache)
    ws = pk.alloc_workspace(num_seqs=2, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D)

    alloc.add(0, 0)
    alloc.add(1, 0)                                            # two empty sequences
    q = torch.randn((2, Hq, D), device="cuda").bfloat16()
    k_new = torch.randn((2, Hkv, D), device="cuda").bfloat16()
    v_new = torch.randn((2, Hkv, D), device="cuda").bfloat16()
    slots, bt, lens, (cow_src, cow_dst) = alloc.step([0, 1], max_blocks=64)
    out = torch.empty((2, Hq, D), dtype=torch.bfloat16, device="cuda")
    pk.paged_decode(out, q, k_cache, v_cache, torch.from_numpy(bt).cuda(),
                    torch.from_numpy(lens).cuda(), D ** -0.5, ws, k_new=k_new, v_new=v_new)
    torch.cuda.synchronize()
    assert pk.get_device_error()[0] == 0                       # sticky bounds-check flags
    assert list(lens) == [1, 1] and len(cow_src) == 0 and len(cow_dst) == 0
    assert [r["len"] for r in alloc.trace([0, 1])] == [1, 1]   # request id, slot, length ...
    assert torch.equal(out, v_new.repeat_interleave(Hq // Hkv, dim=1))
