"""Host side of the multi-rank benchmark path, on CPU with the gloo backend
and two ranks: the step time reported is the max over ranks and the bytes
are summed over ranks (weak scaling, replicas only, no data-path
collective)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    bench.init_dist(world, "gloo")
    bench.barrier(world)
    ms = bench.reduce_max(1.5 + rank, world, "cpu")        # rank 1 is slower
    total = bench.reduce_sum(1000.0 * (rank + 1), world, "cpu")
    q.put((rank, ms, total, bench.dist_env()))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_rank_gloo_aggregation():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, total, env in res:
        assert ms == 2.5 and total == 3000.0
        assert env == (world, rank, rank)


def test_bench_cli_defaults_single_gpu():
    import bench
    a = bench.parse_args([])
    assert a.gpus == 1 and a.warmup >= 3 and a.impl == "ours" and a.config == "2"


def test_kernel_named_for_each_workload():
    """The roofline names the kernel the step runs: the tcgen05 group kernel for
    bf16, d128 and more than 32 query heads per KV head, else the mma.sync split
    kernel."""
    import bench
    import workloads
    names = {}
    for cfg in ("1", "2", "4", "5a", "5b", "mqa64", "mqa128"):
        case = workloads.make_case(cfg, device="cpu", override={"B": 1})
        names[cfg] = bench.split_kernel_name(case)
    assert names["2"] == "paged_decode_split_kernel<128,bf16> (mma.sync)"
    assert names["5a"] == "paged_decode_split_kernel<128,e4m3> (mma.sync)"
    assert names["mqa64"] == "paged_decode_wide_kernel<64> (tcgen05)"
    assert names["mqa128"] == "paged_decode_wide_kernel<128> (tcgen05)"
    assert all("split_kernel" in names[c] for c in ("1", "4", "5b"))
