#!/usr/bin/env python
"""Benchmark of one decode step of one layer on the GB300:
kv_append (the new token's K/V into the paged cache) + paged decode attention
(split-KV kernel + log-sum-exp merge), on the Llama-3.1-8B-shaped workload:
batch 32, 32 query / 8 KV heads, head_dim 128, bfloat16, every context 8192
prefilled tokens + 1 appended (8193), 16-token blocks scattered at random in a
shared pool.  KV read per step: 1,073,872,896 bytes (larger than the 129 MB
L2, so no flush is needed between steps).

Prints one JSON line (rank 0).  ``value`` is the device-timed loop of the
library's fused call (``paged_decode`` with the append and early inputs);
``e2e`` is the same step through ``DecodeStepStaging`` with the inputs copied
from pinned host memory and the output copied back every step (host-ordered
uploads; ``e2e.stream_ordered`` and ``e2e.zero_copy`` beside it);
``graph_replay`` times CUDA-graph replays; ``roofline`` relates the split
kernel's event-timed duration to the measured copy bandwidth.
``--impl reference`` times the CPU float64 oracle instead, on a bounded sample
of the same workload.

Multi-GPU (torchrun): every rank runs its own replica of the workload (weak
scaling, no data-path collective); the step time is the max over ranks and
``value`` counts the bytes of all ranks.
"""
import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged decode attn: KV-read GB/s (% of HBM peak), µs per layer-step"
FALLBACK_HBM_GBS = 6800.0

# ncu DRAM traffic of the split kernel (dram__bytes_read.sum + dram__bytes_write.sum)
# per launch on this workload, with the hash of the kernel source it was
# measured on; reported as null once the source has changed.
TRAFFIC = {"kernel_sha256": "ceed717c42f2174b1ae20a9d9026475580e9c33fc6a116eeda5e011d810deaf1",
           "bytes_per_launch": 1086476288,
           "source": "ncu dram__bytes_read.sum + dram__bytes_write.sum of the batch-8 launch "
                     "(269,147,648 B + 2,471,424 B), scaled x4 by units processed "
                     "(profiles/smem_bank_conflicts_split_b8.md)"}


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawTextHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="2", help="workload id (see workloads.CONFIGS)")
    ap.add_argument("--soak-s", type=float, default=1.0,
                    help="seconds of untimed steps run just before the timed region "
                         "while clocks are sampled")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="CPU time budget of the oracle baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--batch", type=int, default=None,
                    help="override the workload's batch (profiling a smaller case)")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the per_config block (the other workloads, one after another)")
    ap.add_argument("--ref-seqs", type=int, default=4,
                    help="sequences of the workload per reference-arm step")
    ap.add_argument("--prefix", action="store_true",
                    help="also time the shared-prefix step (paged_decode with the chunks "
                         "kv_prefix_chunks finds) beside the plain one")
    return ap.parse_args(argv)


# ---------------------------------------------------------------- plumbing

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world, backend):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend, init_method="env://")
    return dist


def reduce_max(value, world, device):
    """Max of a float over ranks (identity for one rank)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def reduce_sum(value, world, device):
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_sha():
    """Hash of the split kernel's source with comments and blank lines removed
    (an edit to comments leaves the recorded counters valid)."""
    import re
    h = hashlib.sha256()
    for name in ("paged_decode.cu", "device_common.cuh"):
        with open(os.path.join(ROOT, "paged_kv_cache_21_gb300", "csrc", name)) as f:
            src = f.read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        src = re.sub(r"//[^\n]*", "", src)
        src = "\n".join(line.rstrip() for line in src.splitlines() if line.strip())
        h.update(src.encode())
    return h.hexdigest()


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while running."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------- CPU oracle

def oracle_sample_case(cfg, seqs):
    import workloads
    spec = workloads.CONFIGS[cfg]
    override = {"B": min(seqs, spec["B"])}
    return workloads.make_case(cfg, device="cpu", override=override, seed=4242)


def oracle_prepare(case):
    import numpy as np
    import oracle
    from workloads import bf16_bits
    NB, Hkv, D = case.num_blocks, case.Hkv, case.D
    dt = np.uint16 if case.kv_dtype == 0 else np.uint8
    kc = np.zeros((NB, Hkv, 16, D), dtype=dt)
    vc = np.zeros_like(kc)
    oracle.append(kc, vc, bf16_bits(case.pool_k), bf16_bits(case.pool_v),
                  np.arange(NB * 16, dtype=np.int64), case.kv_dtype, case.k_scale, case.v_scale)
    q64 = oracle.bf16_bits_to_f64(bf16_bits(case.q))
    kb, vb = bf16_bits(case.k_new), bf16_bits(case.v_new)
    return kc, vc, q64, kb, vb


def oracle_step(case, prep, nthreads=0):
    """One oracle decode step on the sample: append + attention (float64).
    nthreads 0 = all host cores."""
    import numpy as np
    import oracle
    kc, vc, q64, kb, vb = prep
    slots = oracle.slot_mapping(case.block_tables, np.arange(case.B),
                                case.context_lens.astype(np.int64) - 1)
    oracle.append(kc, vc, kb, vb, slots, case.kv_dtype, case.k_scale, case.v_scale)
    return oracle.paged_attention(q64, kc, vc, case.block_tables, case.context_lens, case.scale,
                                  kv_dtype=case.kv_dtype, k_scale=case.k_scale,
                                  v_scale=case.v_scale, nthreads=nthreads)


def cpu_baseline(cfg, budget_s, seqs=4):
    import oracle
    case = oracle_sample_case(cfg, seqs)
    prep = oracle_prepare(case)
    oracle_step(case, prep)                       # warm
    n, t0 = 0, time.perf_counter()
    while True:
        oracle_step(case, prep)
        n += 1
        el = time.perf_counter() - t0
        if el >= budget_s or n >= 10000:
            break
    gbs = case.logical_kv_bytes() * n / el / 1e9
    # the same sample on one thread (up to 3 steps)
    n1, t1 = 0, time.perf_counter()
    while n1 < 3 and time.perf_counter() - t1 < budget_s / 2:
        oracle_step(case, prep, nthreads=1)
        n1 += 1
    gbs1 = case.logical_kv_bytes() * n1 / (time.perf_counter() - t1) / 1e9
    return {"value": gbs, "unit": "GB/s", "cores": oracle.max_threads(), "kind": "oracle",
            "value_1_thread": gbs1,
            "sample": "%d of %d sequences of this workload (%d (seq, KV head) pairs, "
                      "%d bytes of KV per step), float64 C oracle with OpenMP, %d steps in %.1f s"
                      % (case.B, 32 if cfg in ("2", "5a") else case.B, case.B * case.Hkv,
                         case.logical_kv_bytes(), n, el),
            "us_per_sample_step": el / n * 1e6}


# ---------------------------------------------------------- reference arm

def run_reference(args):
    world, rank, local = dist_env()
    if world > 1 and rank != 0:
        return 0
    import oracle
    import workloads
    spec = workloads.CONFIGS[args.config]
    case = oracle_sample_case(args.config, max(2, args.ref_seqs))
    prep = oracle_prepare(case)
    for _ in range(max(args.warmup, 0)):
        oracle_step(case, prep)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(case, prep)
    el = time.perf_counter() - t0
    ms = el / args.steps * 1e3
    gbs = case.logical_kv_bytes() / (ms * 1e-3) / 1e9
    sample = ("%d of %d sequences of the workload per step (%d (sequence, KV head) pairs, %d "
              "bytes of KV), float64 C oracle with OpenMP over the pairs"
              % (case.B, spec["B"], case.B * case.Hkv, case.logical_kv_bytes()))
    # n_gpus is the launch's N, as in our arm's line; the oracle itself uses
    # the host cores of rank 0 and no GPU
    line = {"impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s",
            "n_gpus": max(world, args.gpus), "gpu_used": False,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": line_config(args.config, args.batch,
                                                       max(world, args.gpus)),
            "cpu_baseline": {"value": gbs, "unit": "GB/s", "kind": "oracle",
                             "cores": oracle.max_threads(), "sample": sample},
            "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


def line_config(cfg, batch, world):
    """The `config` of the JSON line: the workload plus how it is run (the
    same dict for both arms)."""
    return dict(workload_config(cfg, batch),
                parallelism="replicas x%d" % world if world > 1 else "single GPU")


def workload_config(cfg, batch=None):
    """The workload description shared by both arms (from the recipe only)."""
    import workloads
    spec = dict(workloads.CONFIGS[cfg])
    if batch:
        spec["B"] = batch
    es = 1 if spec["kv_dtype"] == workloads.FP8_E4M3 else 2
    c = {"workload": spec["desc"], "config_id": cfg, "batch": spec["B"],
         "q_heads": spec["Hq"], "kv_heads": spec["Hkv"], "head_dim": spec["D"],
         "kv_dtype": "e4m3" if es == 1 else "bf16", "block_size": 16,
         "l2": "inputs larger than L2: the KV read per step exceeds the 129 MB L2, no flush"}
    if "N" in spec:
        c["context_after_append"] = spec["N"] + 1
        c["kv_bytes_per_step"] = 2 * spec["B"] * (spec["N"] + 1) * spec["Hkv"] * spec["D"] * es
        if c["kv_bytes_per_step"] < 129e6:
            c["l2"] = ("L2-resident: the %d B of KV a step reads fit in the 129 MB L2 and stay "
                       "there across steps, no flush (a latency case)" % c["kv_bytes_per_step"])
    return c


# -------------------------------------------------------------- our arm

def timed_loop(K, body, nev, stream, world, tail=None):
    """Run exactly K steps between a barrier + sync on both sides; events
    ev[i][0..nev-1] (created and recorded once beforehand, so their handles
    exist) are handed to the body of step i; `tail` runs before the end event
    is recorded (to join work on other streams).  Returns (ms per step, ev)."""
    import torch
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(nev)] for _ in range(K)]
    for e in ev:
        for x in e:
            x.record(stream)
    t_beg = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    t_beg.record(stream)
    for i in range(K):
        body(ev[i])
    if tail is not None:
        tail()
    t_end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    return t_beg.elapsed_time(t_end) / K, ev


def device_case(pk, case, device):
    """Device tensors of one decode step of `case`: caches filled through
    kv_append with the pool, tables, lengths, q, new K/V, output, workspace."""
    import torch
    import workloads
    cdt = torch.bfloat16 if case.kv_dtype == workloads.BF16 else torch.uint8
    kc = torch.empty((case.num_blocks, case.Hkv, 16, case.D), dtype=cdt, device=device)
    vc = torch.empty_like(kc)
    pk.kv_append(case.pool_k.to(device), case.pool_v.to(device), kc, vc,
                 torch.arange(case.num_blocks * 16, dtype=torch.int64, device=device),
                 case.k_scale, case.v_scale)
    case.pool_k = case.pool_v = None
    torch.cuda.synchronize()
    return dict(kc=kc, vc=vc, bt=torch.from_numpy(case.block_tables).to(device),
                cl=torch.from_numpy(case.context_lens).to(device), q=case.q.to(device),
                k_new=case.k_new.to(device), v_new=case.v_new.to(device),
                out=torch.empty((case.B, case.Hq, case.D), dtype=torch.bfloat16, device=device),
                ws=pk.alloc_workspace(case.B, case.Hq, case.Hkv, case.D, case.kv_dtype,
                                      device=device))


def measure_fused(pk, case, t, stream, K, W, world):
    """The benchmark's step (paged_decode: fused append, early inputs) timed
    as K back-to-back steps, then the same loop through paged_decode_timed
    with events before the split kernel, after it and after the merge, for
    the split kernel's own duration in the same mode."""
    def step():
        pk.paged_decode(t["out"], t["q"], t["kc"], t["vc"], t["bt"], t["cl"], case.scale, t["ws"],
                        case.k_scale, case.v_scale, k_new=t["k_new"], v_new=t["v_new"],
                        early_inputs=True, stream=stream)

    def step_ev(e):
        pk.paged_decode_timed(t["out"], t["q"], t["kc"], t["vc"], t["bt"], t["cl"], case.scale,
                              t["ws"], e, case.k_scale, case.v_scale, k_new=t["k_new"],
                              v_new=t["v_new"], early_inputs=True, stream=stream)

    for _ in range(W):
        step()
    ms_local, _ = timed_loop(K, lambda e: step(), 0, stream, world)
    for _ in range(W):
        step_ev([None, None, None])
    ev_ms, ev = timed_loop(K, step_ev, 3, stream, world)
    split_ms = statistics.mean(ev[i][0].elapsed_time(ev[i][1]) for i in range(K))
    merge_ms = statistics.mean(ev[i][1].elapsed_time(ev[i][2]) for i in range(K))
    return {"ms_local": ms_local, "split_ms": split_ms, "merge_ms": merge_ms,
            "evented_ms_per_step": ev_ms}


def read_ceiling(pk, device, stream, nbytes=1 << 30, reps=10):
    """Same-run read-only ceiling: kv_read_ceiling streams a 1 GiB buffer
    through shared memory in the decode kernel's bulk-copy pattern."""
    import torch
    buf = torch.ones(nbytes // 2, dtype=torch.int16, device=device)
    sink = torch.zeros(2, dtype=torch.int32, device=device)
    for _ in range(3):
        pk.read_ceiling(buf, sink, stream=stream)
    r0, r1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    r0.record(stream)
    for _ in range(reps):
        pk.read_ceiling(buf, sink, stream=stream)
    r1.record(stream)
    torch.cuda.synchronize()
    assert int(sink[1]) == 0, "read ceiling: a bulk copy timed out"
    gbs = reps * nbytes / (r0.elapsed_time(r1) * 1e-3) / 1e9
    del buf, sink
    return {"gbs": gbs, "how": "kv_read_ceiling: 1 GiB streamed into shared memory by bulk "
                               "copies in the decode kernel's pattern (persistent grid, 4 warps "
                               "x 3 x 8 KB stages per CTA, evict-first), no arithmetic; bytes "
                               "read only; mean of %d launches" % reps}


def split_kernel_name(case):
    """The kernel the plain step (no prefix chunks) runs for the attention part:
    the tcgen05 group kernel for bf16, head dim 128 and more than 32 query heads
    per KV head, else the mma.sync split kernel."""
    import workloads
    wide = case.D == 128 and case.kv_dtype == workloads.BF16 and case.Hq // case.Hkv > 32
    if wide:
        return "paged_decode_wide_kernel<%d> (tcgen05)" % (64 if case.Hq // case.Hkv <= 64 else 128)
    return "paged_decode_split_kernel<%d,%s> (mma.sync)" % (
        case.D, "bf16" if case.kv_dtype == workloads.BF16 else "e4m3")


def per_config(pk, cfgs, device, stream, K, W, world, peak, read_gbs):
    """Each of the other workloads on its own: fused step time, split and
    merge durations in the same loop mode, KV GB/s and the fractions of the
    measured copy peak and of the same-run read ceiling."""
    import torch
    import workloads
    res = {}
    for cfg in cfgs:
        case = workloads.make_case(cfg, device=device)
        t = device_case(pk, case, device)
        m = measure_fused(pk, case, t, stream, K, W, world)
        flags, detail = pk.get_device_error()
        assert flags == 0, "config %s: device error flags %d (detail %d)" % (cfg, flags, detail)
        ms = reduce_max(m["ms_local"], world, device)
        kvb = case.logical_kv_bytes()
        gbs = kvb / (ms * 1e-3) / 1e9
        split_gbs = kvb / (m["split_ms"] * 1e-3) / 1e9
        r = {"config": workload_config(cfg), "us_per_step": ms * 1e3,
             "kernel": split_kernel_name(case),
             "kv_bytes_per_step": kvb, "kv_gbs": gbs,
             "frac_of_copy_peak": gbs / peak, "frac_of_read_ceiling": gbs / read_gbs,
             "split_us": m["split_ms"] * 1e3, "merge_us": m["merge_ms"] * 1e3,
             "split_gbs": split_gbs, "split_frac_of_copy_peak": split_gbs / peak}
        if cfg == "3":
            r["kv_bytes_unique"] = case.unique_kv_bytes()
        if kvb < 129e6:
            r["note"] = "L2-resident latency case: GB/s is nominal"
        res[cfg] = r
        del t
        torch.cuda.empty_cache()
    return res


def run_ours(args):
    import numpy as np
    import torch

    world, rank, local = dist_env()
    assert torch.cuda.is_available(), "bench.py needs a CUDA device"
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    init_dist(world, "nccl")

    import paged_kv_cache_21_gb300 as pk
    import workloads

    cfg = args.config
    case = workloads.make_case(cfg, device=device,
                               override={"B": args.batch} if args.batch else None)
    B, Hq, Hkv, D = case.B, case.Hq, case.Hkv, case.D
    t = device_case(pk, case, device)
    kc, vc, bt, cl = t["kc"], t["vc"], t["bt"], t["cl"]
    q, k_new, v_new, out, ws = t["q"], t["k_new"], t["v_new"], t["out"], t["ws"]
    slots_np = pk.slot_mapping(case.block_tables, case.context_lens.astype(np.int64) - 1)
    slots = torch.from_numpy(slots_np).to(device)
    stream = torch.cuda.current_stream(device)
    kv_bytes = case.logical_kv_bytes()
    W = max(args.warmup, 3)

    def step():
        # one decode step of the layer in a decode loop: append the new token
        # and attend (split + merge launches); consecutive steps overlap the
        # next step's block-table scan and first tile copies with the previous
        # step's merge (KV_DECODE_EARLY_INPUTS: the kernel before is the
        # previous step's, and nothing else writes the tables or the caches)
        pk.paged_decode(out, q, kc, vc, bt, cl, case.scale, ws, case.k_scale, case.v_scale,
                        k_new=k_new, v_new=v_new, early_inputs=True, stream=stream)

    def step_default():
        # the same step with every read after the previous kernel completes
        pk.paged_decode_step(out, q, k_new, v_new, kc, vc, bt, cl, case.scale, ws,
                             case.k_scale, case.v_scale, stream=stream)

    def step_unfused(evs):
        pk.kv_append(k_new, v_new, kc, vc, slots, case.k_scale, case.v_scale, stream=stream)
        pk.paged_decode_attention_timed(out, q, kc, vc, bt, cl, case.scale, ws, evs,
                                        case.k_scale, case.v_scale, stream=stream)

    def timed(K, body, nev, tail=None):
        return timed_loop(K, body, nev, stream, world, tail=tail)

    def unfused_body(e):
        e[0].record(stream)
        step_unfused(e[1:])

    # warm-up (W >= 3), then a short untimed soak while the clock sampler runs
    for _ in range(W):
        step()
    torch.cuda.synchronize()
    sampler = ClockSampler(local)
    sampler.start()
    t_soak = time.perf_counter()
    while time.perf_counter() - t_soak < args.soak_s:
        for _ in range(20):
            step()
        torch.cuda.synchronize()

    # timed region: exactly K back-to-back steps (no events between them)
    K = args.steps
    ms_local, _ = timed(K, lambda e: step(), 0)
    clocks = sampler.stop()
    ms = reduce_max(ms_local, world, device)
    total_bytes = reduce_sum(float(kv_bytes), world, device)
    value = total_bytes / (ms * 1e-3) / 1e9
    flags, detail = pk.get_device_error()
    assert flags == 0, "device error flags %d (detail %d)" % (flags, detail)

    # the split kernel's own duration in the same loop (fused append, early
    # inputs), from events recorded before and after it in every step
    fm = measure_fused(pk, case, t, stream, K, W, world)
    split_ms, merge_ms = fm["split_ms"], fm["merge_ms"]

    # the same loop with the default ordering (every read after the previous
    # kernel completes: paged_decode_step)
    for _ in range(W):
        step_default()
    dms_local, _ = timed(K, lambda e: step_default(), 0)
    default_step_us = reduce_max(dms_local, world, device) * 1e3

    # shared-prefix step: the chunk table is built once on the host from the
    # block tables (kv_prefix_chunks), the step reads each shared tile once
    # per chunk of sequences
    prefix = None
    if args.prefix:
        def time_chunks(chunks_np, seq_chunk_np):
            nc = len(chunks_np)
            dch = torch.from_numpy(chunks_np).to(device) if nc else None
            dsc = torch.from_numpy(seq_chunk_np).to(device) if nc else None
            wsp = pk.alloc_prefix_workspace(B, nc, Hq, Hkv, D, case.kv_dtype, device=device)

            def step_prefix():
                pk.paged_decode(out, q, kc, vc, bt, cl, case.scale, wsp, case.k_scale,
                                case.v_scale, k_new=k_new, v_new=v_new, chunks=dch,
                                seq_chunk=dsc, early_inputs=True, stream=stream)

            for _ in range(W):
                step_prefix()
            pms = reduce_max(timed(K, lambda e: step_prefix(), 0)[0], world, device)
            flags, detail = pk.get_device_error()
            assert flags == 0, "device error flags %d (detail %d)" % (flags, detail)
            read_bytes = kv_bytes - sum(int(r[0]) * (int(r[1]) - 1) for r in chunks_np) * \
                Hkv * 2 * 16 * D * case.elem_bytes
            return {"us_per_step": pms * 1e3, "chunks": nc,
                    "kv_gbs_logical": kv_bytes / (pms * 1e-3) / 1e9,
                    "kv_bytes_read": read_bytes,
                    "kv_gbs_read": read_bytes / (pms * 1e-3) / 1e9,
                    "plain_us_per_step": ms * 1e3, "speedup_vs_plain": ms / pms}

        # the library's decision (kv_prefix_plan: chunks only where they pay),
        # and every chunk kv_prefix_chunks finds, used regardless
        prefix = time_chunks(*pk.prefix_plan(case.block_tables, case.context_lens, Hq, Hkv, D,
                                             case.kv_dtype))
        prefix["how"] = "kv_prefix_plan"
        prefix["all_chunks"] = time_chunks(*pk.prefix_chunks(case.block_tables,
                                                             case.context_lens, Hq // Hkv))

    # one fused step captured in a CUDA graph and replayed, each replay
    # bracketed by events: the median is the per-layer-step latency
    gs = torch.cuda.Stream(device)
    gs.wait_stream(stream)
    with torch.cuda.stream(gs):
        pk.paged_decode_step(out, q, k_new, v_new, kc, vc, bt, cl, case.scale, ws,
                             case.k_scale, case.v_scale, stream=gs)
    stream.wait_stream(gs)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=gs):
        pk.paged_decode_step(out, q, k_new, v_new, kc, vc, bt, cl, case.scale, ws,
                             case.k_scale, case.v_scale, stream=gs)
    n_rep = max(K, 100)
    g_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in range(n_rep)]
    with torch.cuda.stream(gs):
        for _ in range(W):
            graph.replay()
        for a, b in g_ev:
            a.record(gs)
            graph.replay()
            b.record(gs)
    torch.cuda.synchronize()
    g_us = sorted(a.elapsed_time(b) * 1e3 for a, b in g_ev)
    graph_replay = {"median_us": statistics.median(g_us), "min_us": g_us[0],
                    "p90_us": g_us[int(0.9 * (len(g_us) - 1))], "replays": n_rep,
                    "kv_gbs_at_median": kv_bytes / (statistics.median(g_us) * 1e-6) / 1e9}
    del graph

    # many steps of the benchmark's call captured in one graph: the device
    # time per step without the host's launch cost (which bounds the eager
    # loop of a tiny workload)
    S_graph = 32
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=gs):
        for _ in range(S_graph):
            pk.paged_decode(out, q, kc, vc, bt, cl, case.scale, ws, case.k_scale, case.v_scale,
                            k_new=k_new, v_new=v_new, early_inputs=True, stream=gs)
    n_rep = 100
    gb_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
             for _ in range(n_rep)]
    with torch.cuda.stream(gs):
        for _ in range(3):
            graph.replay()
        for a, b in gb_ev:
            a.record(gs)
            graph.replay()
            b.record(gs)
    torch.cuda.synchronize()
    gb_us = sorted(a.elapsed_time(b) * 1e3 / S_graph for a, b in gb_ev)
    gb_med = statistics.median(gb_us)
    graph_replay["batched"] = {"steps_per_graph": S_graph, "replays": n_rep,
                               "median_us_per_step": gb_med, "min_us_per_step": gb_us[0],
                               "kv_gbs_at_median": kv_bytes / (gb_med * 1e-6) / 1e9,
                               "call": "paged_decode (fused append, KV_DECODE_EARLY_INPUTS)"}
    del graph

    # the same step as separate launches (kv_append, then paged_decode_attention)
    for _ in range(W):
        step_unfused([None, None, None])
    un_ms_local, un_ev = timed(K, unfused_body, 4)
    unfused = {"us_per_step": reduce_max(un_ms_local, world, device) * 1e3,
               "append_us": statistics.mean(un_ev[i][0].elapsed_time(un_ev[i][1])
                                            for i in range(K)) * 1e3,
               "split_us": statistics.mean(un_ev[i][1].elapsed_time(un_ev[i][2])
                                           for i in range(K)) * 1e3,
               "merge_us": statistics.mean(un_ev[i][2].elapsed_time(un_ev[i][3])
                                           for i in range(K)) * 1e3}

    # end to end through the public API with host buffers: every step copies
    # its inputs (staged in one pinned buffer) to the device, runs the fused
    # step and copies its output back; the copies run on copy streams with
    # two alternating staging slots, overlapping the neighbouring steps.  The
    # headline mode has the host wait for each upload (host_ordered), so the
    # compute stream holds only kernels; the stream-ordered mode (an event
    # wait on the compute stream per step) is reported beside it.
    e2e = None
    if not args.no_e2e:
        def staged_run(**kw):
            stg = pk.DecodeStepStaging(B, Hq, Hkv, D, case.max_blocks, case.kv_dtype,
                                       device=device, **kw)
            for j in range(2):
                hs = stg.host(j)
                hs.q.copy_(q.cpu())
                hs.k_new.copy_(k_new.cpu())
                hs.v_new.copy_(v_new.cpu())
                hs.block_tables.copy_(torch.from_numpy(case.block_tables))
                hs.context_lens.copy_(torch.from_numpy(case.context_lens))
            counter = [0]

            def e2e_step(_e=None):
                stg.step(counter[0], kc, vc, case.scale, case.k_scale, case.v_scale,
                         stream=stream)
                counter[0] += 1

            for _ in range(W):
                e2e_step()
            torch.cuda.synchronize()
            # the end event waits for the last download on its copy stream
            ms_local, _ = timed(K, e2e_step, 0, tail=lambda: stg.join(stream))
            ms_ = reduce_max(ms_local, world, device)
            torch.cuda.synchronize()
            assert torch.equal(stg.host(counter[0] - 1).out.view(torch.int16),
                               out.cpu().view(torch.int16))
            rec = {"value": total_bytes / (ms_ * 1e-3) / 1e9, "unit": "GB/s",
                   "ms_per_step": ms_, "h2d_bytes_per_step": stg.h2d_bytes,
                   "d2h_bytes_per_step": stg.d2h_bytes}
            del stg
            return rec

        e2e = staged_run(host_ordered=True)
        e2e["how"] = ("DecodeStepStaging(host_ordered=True): one pinned H2D copy of every "
                      "input and one D2H copy of the output per step, the host waits for "
                      "each upload before launching the step")
        e2e["stream_ordered"] = staged_run(host_ordered=False)
        e2e["stream_ordered"]["how"] = "same copies, an event wait on the compute stream per step"

        # the same with the kernels reading the pinned host slots in place
        # (no copies: NVLink-C2C on a Grace-Blackwell node)
        zc = pk.DecodeStepStaging(B, Hq, Hkv, D, case.max_blocks, case.kv_dtype, device=device,
                                  zero_copy=True)
        for j in range(2):
            hs = zc.host(j)
            hs.q.copy_(q.cpu())
            hs.k_new.copy_(k_new.cpu())
            hs.v_new.copy_(v_new.cpu())
            hs.block_tables.copy_(torch.from_numpy(case.block_tables))
            hs.context_lens.copy_(torch.from_numpy(case.context_lens))
        zcount = [0]

        def zc_step(_e=None):
            zc.step(zcount[0], kc, vc, case.scale, case.k_scale, case.v_scale, stream=stream)
            zcount[0] += 1

        for _ in range(W):
            zc_step()
        torch.cuda.synchronize()
        zc_ms = reduce_max(timed(K, zc_step, 0)[0], world, device)
        torch.cuda.synchronize()
        assert torch.equal(zc.host(zcount[0] - 1).out.view(torch.int16),
                           out.cpu().view(torch.int16))
        e2e["zero_copy"] = {"value": total_bytes / (zc_ms * 1e-3) / 1e9, "unit": "GB/s",
                            "ms_per_step": zc_ms, "h2d_bytes_per_step": zc.h2d_bytes,
                            "d2h_bytes_per_step": zc.d2h_bytes,
                            "how": "inputs read and output written in pinned host memory "
                                   "by the kernels (NVLink-C2C), no copies"}
        del zc

    # same-run copy ceiling: a plain device-to-device copy of 1 GiB (read + write bytes)
    src = torch.ones(1 << 29, dtype=torch.int16, device=device)
    dst = torch.empty_like(src)
    with torch.cuda.stream(stream):
        for _ in range(3):
            dst.copy_(src)
        r0, r1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        r0.record(stream)
        for _ in range(10):
            dst.copy_(src)
        r1.record(stream)
    torch.cuda.synchronize()
    copy_ceiling = {"gbs": 10 * 2 * src.numel() * 2 / (r0.elapsed_time(r1) * 1e-3) / 1e9,
                    "how": "torch copy_ of a 1 GiB buffer, read + write bytes, same run"}
    del src, dst

    rc = read_ceiling(pk, device, stream)

    peak, peak_kind = measured_peaks()
    achieved = kv_bytes / (split_ms * 1e-3) / 1e9
    # the recorded counters belong to the default workload (config 2, batch 32)
    traffic = (TRAFFIC["bytes_per_launch"]
               if TRAFFIC["kernel_sha256"] == kernel_sha() and cfg == "2" and not args.batch
               else None)
    roofline = {"bound": "hbm",
                "kernel": split_kernel_name(case),
                "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "peak_source": "%s (MEASURED_PEAKS.json hbm_gbs)" % peak_kind
                if peak_kind == "measured" else "fallback 6.8 TB/s",
                "traffic": traffic, "algorithmic_bytes_per_launch": kv_bytes,
                "split_us": split_ms * 1e3, "merge_us": merge_ms * 1e3,
                "split_timing": "events before and after the split kernel in every step of "
                                "the benchmark's loop (paged_decode_timed: fused append, "
                                "early inputs); %.1f us per step with the events"
                                % (fm["evented_ms_per_step"] * 1e3),
                "copy_ceiling": copy_ceiling, "read_ceiling": rc,
                "frac_vs_read_ceiling": achieved / rc["gbs"],
                "step_frac_vs_read_ceiling": (kv_bytes / (ms * 1e-3) / 1e9) / rc["gbs"]}

    line = {"metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": K,
            "warmup": W, "ms_per_step": ms,
            "us_per_layer_step": ms * 1e3, "pct_of_hbm_peak": 100.0 * (kv_bytes / (ms * 1e-3)
                                                                      / 1e9) / peak,
            "pct_of_8tbs_nameplate": 100.0 * (kv_bytes / (ms * 1e-3) / 1e9) / 8000.0,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" if case.kv_dtype == workloads.BF16 else "e4m3",
            "data": "synthetic (seeded N(0,1) bf16 q/K/V, random block placement)",
            "config": line_config(cfg, args.batch, world),
            "roofline": roofline, "e2e": e2e, "gpu_launches": 2 * K, "clocks": clocks,
            "decode_call": "paged_decode (fused append, KV_DECODE_EARLY_INPUTS)",
            "default_step_us": default_step_us,
            "unfused": unfused, "graph_replay": graph_replay}
    if not args.no_per_config and not args.batch:
        others = [c for c in ("1", "2", "3", "4", "5a", "5b", "mqa64", "mqa128") if c != cfg]
        line["per_config"] = per_config(pk, others, device, stream, K, W, world, peak,
                                        rc["gbs"])
    if prefix is not None:
        line["prefix"] = prefix
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(cfg, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
