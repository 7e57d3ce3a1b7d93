"""The benchmark's roofline arithmetic reproduces the figures the pages print when fed the
pages' own hardware parameters (A100: 1.935 TB/s, 312 TFLOP/s fp16), and the
multi-rank aggregation takes the slowest rank's time (world size 2 over gloo)."""
import os

import pytest

import bench

HERE = os.path.dirname(os.path.abspath(__file__))


def golden():
    out = {}
    with open(os.path.join(HERE, "golden", "page_numbers.txt"), encoding="utf-8") as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                name, value, tol = line.split()
                out[name] = (float(value), float(tol))
    return out


def computed():
    n = 8192
    raw = bench.gemm_tiled_traffic(n, n, n, 128, 2)
    floor = bench.gemm_min_bytes(n, n, n, 2, 2)
    compute_s = bench.gemm_flops(n, n, n) / 312e12
    # multicast: A and B contribute equally; the shared operand is cut by the cluster size
    cut = lambda c: 0.5 * (1 - 1 / c)
    import math
    stages = math.ceil(500 / 200 + 1)
    return {
        "naive_intensity_fp32": bench.gemm_flops(1, 1, 1) / (2 * 4),
        "tiled_intensity_t32_fp32": 32 / 4,
        "tiled_intensity_t32_16bit": bench.tile_intensity(32, 32, 2),
        "tile_128x128_16bit": bench.tile_intensity(128, 128, 2),
        "tile_256x256_16bit": bench.tile_intensity(256, 256, 2),
        "gemm8192_raw_traffic_gb": raw / 1e9,
        "gemm8192_raw_time_ms": raw / 1.935e12 * 1e3,
        "gemm8192_compute_ms": compute_s * 1e3,
        "gemm8192_floor_mb": floor / 1e6,
        "gemm8192_floor_ms": floor / 1.935e12 * 1e3,
        "gemm8192_threshold_gb": compute_s * 1.935e12 / 1e9,
        "multicast_cluster2_cut": cut(2),
        "multicast_cluster4_cut": cut(4),
        "stages_500cy_200cy": stages,
        "stages_smem_bytes": stages * 2 * 32 * 32 * 4,
    }


@pytest.mark.parametrize("name", sorted(golden()))
def test_page_figure(name):
    want, tol = golden()[name]
    got = computed()[name]
    assert abs(got - want) <= tol * abs(want) + 1e-12, (name, got, want)


def test_copy_bytes_of_the_workload():
    # 4100 x 8200 bf16 read once (67,240,000 B) + image of 33 x 129 boxes of 16 KiB
    assert bench.copy_bytes(4100, 8200, 2, 64, 128) == 67_240_000 + 69_746_688


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import torch

    def amax(x):
        t = torch.tensor([x], dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())

    def asum(x):
        t = torch.tensor([x], dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.SUM)
        return float(t.item())

    local_time = 1.0 + rank          # rank 1 is the slow one
    value, t = bench.aggregate(local_time, 100.0, world, amax, asum)
    q.put((rank, value, t))
    dist.destroy_process_group()


def test_aggregate_two_ranks_gloo():
    import multiprocessing as mp
    import socket
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # 2 ranks x 100 units over the slowest rank's 2 s
    assert res == [(0, 100.0, 2.0), (1, 100.0, 2.0)]


def test_aggregate_single_rank():
    assert bench.aggregate(2.0, 10.0, 1) == (5.0, 2.0)


def test_nameplate_from_the_probe_cycle_count():
    # 152 SMs; one pair did 2 * 8192 flop per cycle over 1,000,000 cycles in 512 us: the
    # per-SM rate is 8192 flop per cycle whatever clock was sampled, and the nameplate is
    # 152 x 8192 x the maximum clock
    timed = {"flop_per_pair": 2 * 8192 * 1_000_000, "cycles": 1_000_000, "ns": 512_000}
    clk = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": []}
    line = bench.nameplate_line(2.4e15, 152, clk, 1900.0, timed)
    assert line["per_sm_flop_per_clk"] == 8192
    assert abs(line["probe_mhz_measured"] - 1953.125) < 1e-9
    assert abs(line["peak"] - 152 * 8192 * 2070e6 / 1e12) < 1e-6
    assert abs(line["frac"] - 1900.0 / line["peak"]) < 1e-12
    # without the timed launch: the event rate over the sampled clock
    line = bench.nameplate_line(2.4e15, 152, clk, 1900.0)
    assert abs(line["per_sm_flop_per_clk"] - 2.4e15 / 152 / 2070e6) < 1e-6
    assert bench.nameplate_line(2.4e15, 152, {}, 1900.0)["peak"] is None
