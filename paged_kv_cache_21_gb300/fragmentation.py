"""Memory fragmentation of paged vs contiguous KV allocation, by simulation.

"KV Cache, Flash Attention and inference optimization", exercise 3: split
the KV cache into fixed 16-token blocks with a free list, return blocks to
the pool when a sequence ends, simulate 1,000 chat completions of varied
length, and compare the fragmentation with contiguous allocation.  ("KV
cache complete guide", section "(4) PagedAttention": contiguous caches
reserve the maximum sequence length up front and waste what requests never
use; blocks are allocated only as needed.)

The paged side runs entirely on the library's host allocator (kv_seq_add /
kv_step / kv_seq_free through the C ABI); the contiguous side is the plain
model of that guide: each admitted request holds a region of `max_len`
tokens until it ends.  Both serve the same request stream with the same
continuous-batching admission (a fixed number of concurrent requests, each
decode step appends one token to every running request).
"""
from dataclasses import dataclass

import numpy as np

from . import BlockAllocator, BLOCK_SIZE


@dataclass
class FragmentationReport:
    requests: int
    steps: int
    paged_mean_waste: float        # mean over steps of 1 - tokens stored / tokens reserved
    contiguous_mean_waste: float
    paged_peak_blocks: int
    paged_peak_tokens_reserved: int
    contiguous_peak_tokens_reserved: int
    peak_tokens_stored: int

    @property
    def reserved_ratio(self):
        """How many times more memory the contiguous scheme held at peak."""
        return self.contiguous_peak_tokens_reserved / max(self.paged_peak_tokens_reserved, 1)


def chat_lengths(n, seed=0, prompt=(16, 2048), completion=(16, 1024)):
    """Seeded prompt and completion lengths, each log-uniform in its range."""
    rng = np.random.default_rng(seed)
    p = np.exp(rng.uniform(np.log(prompt[0]), np.log(prompt[1]), n)).astype(np.int64)
    c = np.exp(rng.uniform(np.log(completion[0]), np.log(completion[1]), n)).astype(np.int64)
    return p, c


def simulate(num_requests=1000, concurrency=64, max_len=4096, seed=0, num_blocks=None):
    """Serve `num_requests` chats and measure both allocation schemes."""
    prompt, completion = chat_lengths(num_requests, seed)
    prompt = np.minimum(prompt, max_len - 1)
    completion = np.minimum(completion, max_len - prompt)
    max_blocks = -(-max_len // BLOCK_SIZE)
    if num_blocks is None:
        num_blocks = concurrency * max_blocks
    alloc = BlockAllocator(num_blocks, 1, 64)
    next_req = 0
    running = {}                     # request id -> tokens still to generate
    waste_p, waste_c = [], []
    peak_blocks = peak_paged = peak_contig = peak_stored = 0
    steps = 0
    while next_req < num_requests or running:
        while next_req < num_requests and len(running) < concurrency:
            alloc.add(next_req, int(prompt[next_req]))
            running[next_req] = int(completion[next_req])
            next_req += 1
        ids = np.array(sorted(running), dtype=np.int64)
        _, _, lens, _ = alloc.step(ids, max_blocks)
        steps += 1
        stored = int(lens.astype(np.int64).sum())
        free, used, _, _ = alloc.stats()
        paged_reserved = used * BLOCK_SIZE
        contig_reserved = len(ids) * max_len
        waste_p.append(1.0 - stored / paged_reserved)
        waste_c.append(1.0 - stored / contig_reserved)
        peak_blocks = max(peak_blocks, used)
        peak_paged = max(peak_paged, paged_reserved)
        peak_contig = max(peak_contig, contig_reserved)
        peak_stored = max(peak_stored, stored)
        for rid in ids.tolist():
            running[rid] -= 1
            if running[rid] <= 0:
                alloc.free(rid)
                del running[rid]
    assert alloc.stats()[:3] == (num_blocks, 0, 0)
    return FragmentationReport(num_requests, steps, float(np.mean(waste_p)),
                               float(np.mean(waste_c)), peak_blocks, peak_paged, peak_contig,
                               peak_stored)
