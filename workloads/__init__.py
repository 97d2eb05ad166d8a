"""Seeded synthetic inputs for the paged decode step.

Shared by the tests, the benchmark and the smoke check.  This module only
draws numbers and lays out block tables; it holds none of the method's
arithmetic (no slot mapping, no quantisation, no attention), so the oracle and
the CUDA library can both consume what it produces without sharing code.

The shapes follow the pages' Llama-style examples ("KV cache complete guide",
sections "KV cache memory size calculation" and "(2) GQA": 32 query / 8 KV
heads, head_dim 128, batch 32, 8K context; "KV Cache, Flash Attention and
inference optimization", section "KV cache math": a 70B model with 8 KV
heads; the ~600-token shared system prompt of "(3) Prefix Caching"; 16-token
blocks of "(4) PagedAttention").  No public dataset is involved.

Every case is a single decode step for one layer: each sequence holds
``N`` prefilled tokens and appends one more, so its context after the append
is ``L = N + 1``.  The pool content is given as one bfloat16 K and V vector
per physical slot (``pool_k``/``pool_v`` shaped [num_blocks * 16, Hkv, D], in
slot order 0, 1, 2, ...), which both sides write into their caches with the
append operation before the step; unused slots hold random values that the
length mask must exclude.
"""
from dataclasses import dataclass, field
import math

import numpy as np
import torch

BF16 = 0
FP8_E4M3 = 1
BLOCK = 16

# name -> shape recipe.  'N' is the prefilled length (the context after the
# step's append is N + 1).
CONFIGS = {
    "1": dict(desc="tiny decode step: 1 seq, 4q/1kv heads, d64, 128 prefilled + 1 appended, "
                   "16-block pool, random block permutation",
              B=1, Hq=4, Hkv=1, D=64, N=128, kv_dtype=BF16, pool_blocks=16),
    "2": dict(desc="Llama-3.1-8B-shaped layer: 32q/8kv heads, d128, batch 32, 8192 prefilled + 1",
              B=32, Hq=32, Hkv=8, D=128, N=8192, kv_dtype=BF16, slack=0.10),
    "3": dict(desc="ragged continuous batch: 256 seqs, 32q/8kv, d128, prefilled lengths "
                   "log-uniform in [16, 32768], groups of 8 sharing a 608-token prefix",
              B=256, Hq=32, Hkv=8, D=128, N_lo=16, N_hi=32768, group=8, prefix_blocks=38,
              kv_dtype=BF16, slack=0.10),
    "4": dict(desc="Llama-3-70B-shaped long context: 64q/8kv, d128, batch 4, 131072 prefilled + 1",
              B=4, Hq=64, Hkv=8, D=128, N=131072, kv_dtype=BF16, slack=0.10),
    "5a": dict(desc="FP8 E4M3 KV cache, per-tensor scales amax/448, config-2 shapes",
               B=32, Hq=32, Hkv=8, D=128, N=8192, kv_dtype=FP8_E4M3, slack=0.10),
    "5b": dict(desc="MHA 32q/32kv heads, d128, batch 8, 4096 prefilled + 1, bf16",
               B=8, Hq=32, Hkv=32, D=128, N=4096, kv_dtype=BF16, slack=0.10),
    # not among the pages' five workloads: MQA ("KV cache complete guide",
    # section "(2) GQA": one KV head shared by every query head) on a 64- or
    # 128-head model, config 2's batch and context
    "mqa64": dict(desc="MQA: 64 query heads on 1 KV head, d128, batch 32, 8192 prefilled + 1, "
                       "bf16",
                  B=32, Hq=64, Hkv=1, D=128, N=8192, kv_dtype=BF16, slack=0.10),
    "mqa128": dict(desc="MQA: 128 query heads on 1 KV head, d128, batch 32, 8192 prefilled + 1, "
                        "bf16",
                   B=32, Hq=128, Hkv=1, D=128, N=8192, kv_dtype=BF16, slack=0.10),
    # not one of the pages' workloads: config 3's structure with a long shared
    # system prompt, where the shared blocks are most of the bytes
    "3L": dict(desc="shared-prompt batch: 256 seqs, 32q/8kv, d128, groups of 8 sharing a "
                    "4096-token prefix, prefilled lengths log-uniform in [4200, 8192]",
               B=256, Hq=32, Hkv=8, D=128, N_lo=4200, N_hi=8192, group=8, prefix_blocks=256,
               kv_dtype=BF16, slack=0.10),
}

SEED_BASE = 1000
SEED_OFFSET = {"1": 1, "2": 2, "3": 3, "4": 4, "5a": 5, "5b": 6, "3L": 7, "mqa64": 8,
               "mqa128": 9}


@dataclass
class DecodeCase:
    name: str
    B: int
    Hq: int
    Hkv: int
    D: int
    kv_dtype: int
    scale: float
    num_blocks: int
    context_lens: np.ndarray          # int32 [B], after the append
    block_tables: np.ndarray          # int32 [B, max_blocks], -1 beyond each row's blocks
    q: torch.Tensor                   # bf16 [B, Hq, D]
    k_new: torch.Tensor               # bf16 [B, Hkv, D], the appended token's K
    v_new: torch.Tensor               # bf16 [B, Hkv, D]
    pool_k: torch.Tensor              # bf16 [num_blocks*16, Hkv, D], one vector per slot
    pool_v: torch.Tensor
    k_scale: float = 1.0
    v_scale: float = 1.0
    shared_blocks: np.ndarray = field(default=None)  # int32 [B], blocks shared with the group

    @property
    def G(self):
        return self.Hq // self.Hkv

    @property
    def max_blocks(self):
        return self.block_tables.shape[1]

    @property
    def elem_bytes(self):
        return 1 if self.kv_dtype == FP8_E4M3 else 2

    def logical_kv_bytes(self):
        """K plus V bytes one decode step reads: every context position of
        every sequence, for every KV head."""
        return int(2 * int(self.context_lens.astype(np.int64).sum()) * self.Hkv * self.D
                   * self.elem_bytes)

    def unique_kv_bytes(self):
        """Bytes of distinct physical blocks touched (shared prefixes once)."""
        used = set()
        for s in range(self.B):
            nb = -(-int(self.context_lens[s]) // BLOCK)
            used.update(self.block_tables[s, :nb].tolist())
        return int(2 * len(used) * BLOCK * self.Hkv * self.D * self.elem_bytes)


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _randn_bf16(shape, gen, device):
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32).to(torch.bfloat16)


def _layout(rng, nblocks, B, shared=None, slack=0.10, pool_blocks=None, max_blocks=None):
    """Random physical placement.  nblocks[s] logical blocks per sequence;
    shared = (group_of[s], nshared[s], blocks_per_group) places the first
    nshared[s] blocks of a sequence on its group's common blocks."""
    nblocks = np.asarray(nblocks, dtype=np.int64)
    if shared is None:
        n_group_blocks, n_groups = 0, 0
        nshared = np.zeros(B, dtype=np.int64)
    else:
        group_of, nshared, n_group_blocks = shared
        n_groups = int(group_of.max()) + 1
    private = int((nblocks - nshared).sum())
    used = private + n_groups * n_group_blocks
    if pool_blocks is None:
        pool_blocks = int(math.ceil(used * (1.0 + slack)))
    assert pool_blocks >= used
    perm = rng.permutation(pool_blocks).astype(np.int32)
    if max_blocks is None:
        max_blocks = int(nblocks.max()) if B else 1
    bt = np.full((B, max_blocks), -1, dtype=np.int32)
    cursor = 0
    group_ids = []
    for _ in range(n_groups):
        group_ids.append(perm[cursor:cursor + n_group_blocks])
        cursor += n_group_blocks
    for s in range(B):
        ns = int(nshared[s])
        if ns:
            bt[s, :ns] = group_ids[int(group_of[s])][:ns]
        npriv = int(nblocks[s]) - ns
        bt[s, ns:ns + npriv] = perm[cursor:cursor + npriv]
        cursor += npriv
    return bt, pool_blocks, nshared.astype(np.int32)


def make_layout(cfg, seed=None, override=None):
    """The lengths and block placement of configuration ``cfg`` alone (no
    values): (spec, context lengths after the append, block tables, pool
    blocks, shared blocks per sequence, seed) -- the same tables make_case
    builds for the same arguments."""
    spec = dict(CONFIGS[cfg])
    if override:
        spec.update(override)
    if seed is None:
        seed = SEED_BASE + SEED_OFFSET[cfg]
    rng = np.random.default_rng(seed)
    B = spec["B"]
    if "N" in spec:
        N = np.full(B, spec["N"], dtype=np.int64)
    else:
        lo, hi = math.log(spec["N_lo"]), math.log(spec["N_hi"])
        N = np.floor(np.exp(rng.uniform(lo, hi, size=B))).astype(np.int64)
        N = np.clip(N, spec["N_lo"], spec["N_hi"])
    L = N + 1
    nblocks = -(-L // BLOCK)

    shared = None
    if spec.get("group"):
        group_of = np.arange(B) // spec["group"]
        # a sequence shares the full blocks that lie wholly before its new
        # token (the block receiving the append stays private)
        nshared = np.minimum(spec["prefix_blocks"], N // BLOCK)
        shared = (group_of, nshared, spec["prefix_blocks"])
    bt, NB, nshared = _layout(rng, nblocks, B, shared, spec.get("slack", 0.10),
                              spec.get("pool_blocks"), spec.get("max_blocks"))
    return spec, L, bt, NB, nshared, seed


def make_case(cfg, device="cpu", seed=None, override=None):
    """Build the seeded decode-step inputs of configuration ``cfg``.

    ``override`` replaces recipe entries (used by tests to shrink a config
    while keeping its structure, e.g. ``{"B": 4}``)."""
    spec, L, bt, NB, nshared, seed = make_layout(cfg, seed, override)
    gen = _gen(device, seed)
    B, Hq, Hkv, D = spec["B"], spec["Hq"], spec["Hkv"], spec["D"]

    q = _randn_bf16((B, Hq, D), gen, device)
    k_new = _randn_bf16((B, Hkv, D), gen, device)
    v_new = _randn_bf16((B, Hkv, D), gen, device)
    pool_k = _randn_bf16((NB * BLOCK, Hkv, D), gen, device)
    pool_v = _randn_bf16((NB * BLOCK, Hkv, D), gen, device)

    k_scale = v_scale = 1.0
    if spec["kv_dtype"] == FP8_E4M3:
        # per-tensor scale: the largest magnitude maps to the top of E4M3
        amax_k = max(float(pool_k.abs().max()), float(k_new.abs().max()))
        amax_v = max(float(pool_v.abs().max()), float(v_new.abs().max()))
        k_scale = float(np.float32(amax_k) / np.float32(448.0))
        v_scale = float(np.float32(amax_v) / np.float32(448.0))

    return DecodeCase(name=cfg, B=B, Hq=Hq, Hkv=Hkv, D=D, kv_dtype=spec["kv_dtype"],
                      scale=float(spec.get("scale", 1.0 / math.sqrt(D))), num_blocks=NB,
                      context_lens=L.astype(np.int32), block_tables=bt, q=q, k_new=k_new,
                      v_new=v_new, pool_k=pool_k, pool_v=pool_v, k_scale=k_scale,
                      v_scale=v_scale, shared_blocks=nshared)


def make_custom(B, Hq, Hkv, D, lens, kv_dtype=BF16, seed=7, slack=0.25, device="cpu",
                max_blocks=None, scale=None):
    """An arbitrary small case with the given context lengths (after append)."""
    lens = np.asarray(lens, dtype=np.int64)
    rng = np.random.default_rng(seed)
    gen = _gen(device, seed)
    nblocks = -(-lens // BLOCK)
    bt, NB, _ = _layout(rng, nblocks, B, None, slack, None, max_blocks)
    NB = max(NB, 1)
    q = _randn_bf16((B, Hq, D), gen, device)
    k_new = _randn_bf16((B, Hkv, D), gen, device)
    v_new = _randn_bf16((B, Hkv, D), gen, device)
    pool_k = _randn_bf16((NB * BLOCK, Hkv, D), gen, device)
    pool_v = _randn_bf16((NB * BLOCK, Hkv, D), gen, device)
    k_scale = v_scale = 1.0
    if kv_dtype == FP8_E4M3:
        amax_k = max(float(pool_k.abs().max()), float(k_new.abs().max()))
        amax_v = max(float(pool_v.abs().max()), float(v_new.abs().max()))
        k_scale = float(np.float32(amax_k) / np.float32(448.0))
        v_scale = float(np.float32(amax_v) / np.float32(448.0))
    return DecodeCase(name="custom", B=B, Hq=Hq, Hkv=Hkv, D=D, kv_dtype=kv_dtype,
                      scale=float(scale if scale is not None else 1.0 / math.sqrt(D)),
                      num_blocks=NB, context_lens=lens.astype(np.int32), block_tables=bt,
                      q=q, k_new=k_new, v_new=v_new, pool_k=pool_k, pool_v=pool_v,
                      k_scale=k_scale, v_scale=v_scale,
                      shared_blocks=np.zeros(B, dtype=np.int32))


def bf16_bits(t):
    """uint16 numpy view of a bfloat16 torch tensor (CPU copy)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
