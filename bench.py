#!/usr/bin/env python3
"""Benchmark of the TMA-fed bf16 GEMM and the TMA tile copy on one GB300.

One step = one pass of the whole hot path over one batch of synthetic input:
  * gemm_bf16: C = A*B with M = N = K = 8192, A and B uniform in [-1, 1] rounded to bf16
    (seed 3), fp32 accumulation, bf16 output, alpha = 1, beta = 0;
  * tma_tile_copy: the 4100 x 8200 bf16 tensor bf16((row*8200 + col) mod 65521), boxes
    of 128 rows x 64 columns, 128-byte swizzle, zero out-of-bounds fill.
`value` is the GEMM's throughput (2*M*N*K flops per launch over the device time of the
launches, CUDA events on the launching stream); the copy's GB/s is reported beside it.
`workloads` adds every other GEMM configuration of the set (256^3, 4096^3, the FFN
up/down and weight-gradient shapes of a BERT-large-like training step, and the ragged
3000 x 5000 x 2056 case with beta = 0.5), each in its default launch with its own
roofline fraction, launch plan, sampled parity against the oracle and oracle timing.
Before every timed kernel L2 is flushed (256 MiB written, then 256 MiB read, so no
dirty lines are left for the timed kernel to evict), outside its events.

--impl reference times the CPU oracle (the only reference this method has) on a bounded
sample of the same workload on the host cores.  Under torchrun every rank runs its own
full problem (independent replicas, weak scaling, no collective on the data path); the
reported time is the maximum over ranks.
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "bf16 GEMM TFLOP/s and % of GB300 dense peak at 8192³; TMA copy GB/s vs HBM"
GEMM_WORKLOAD = "gemm_8192"
F8_WORKLOAD = "gemm_8192_e4m3"
MX_WORKLOAD = "gemm_8192_mxe4m3"
COPY_H, COPY_W, COPY_BOX_W, COPY_BOX_H = 4100, 8200, 64, 128
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
FLUSH_BYTES = 256 << 20
FP8_PER_BF16 = 4.5 / 2.25   # nominal dense fp8 / bf16 tensor rates of the part
TF32_PER_BF16 = 1.1 / 2.25  # nominal dense tf32 / bf16 tensor rates of the part
KERNEL_SOURCES = ["tma_pipelined_tensor_gb300/csrc/gemm.cu",
                  "tma_pipelined_tensor_gb300/csrc/gemm_pair.cu",
                  "tma_pipelined_tensor_gb300/csrc/gemm_common.cuh",
                  "tma_pipelined_tensor_gb300/csrc/tile_copy.cu",
                  "tma_pipelined_tensor_gb300/csrc/ptx.cuh",
                  "tma_pipelined_tensor_gb300/csrc/tg_internal.h"]


# ------------------------------------------------------------------------------------
# Roofline arithmetic ("GEMM: la moltiplicazione di matrici sull'hardware": 2MNK flops;
# tile intensity I = 2*BM*BN / ((BM + BN) * s); naive intensity 1/4 flop/byte in fp32).
# ------------------------------------------------------------------------------------
def gemm_flops(M, N, K):
    return 2.0 * M * N * K


def tile_intensity(bm, bn, elem_bytes):
    return 2.0 * bm * bn / ((bm + bn) * elem_bytes)


def gemm_min_bytes(M, N, K, in_bytes=2, out_bytes=2, read_c=False):
    """Each operand read once and C written once (the page's 'floor')."""
    b = (M * K + N * K) * in_bytes + M * N * out_bytes
    return b + (M * N * out_bytes if read_c else 0)


def gemm_tiled_traffic(M, N, K, tile, elem_bytes):
    """Traffic when every tile's operand strips come from DRAM: 2*M*N*K/T elements."""
    return 2.0 * M * N * K / tile * elem_bytes


def copy_bytes(H, W, es, box_w, box_h):
    """Algorithmic bytes of one tile-copy pass: in-bounds read + image write."""
    nbi, nbj = -(-H // box_h), -(-W // box_w)
    return H * W * es + nbi * nbj * box_w * box_h * es


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        d = dict(FALLBACK_PEAKS)
        d["source"] = "fallback"
        return d


def kernel_source_hash():
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def committed_traffic(kernel):
    """DRAM bytes per launch from the committed ncu summary, if the kernel is unchanged."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            t = json.load(f)
        e = t[kernel]
        if e.get("source_hash") != kernel_source_hash():
            return None
        return float(e["dram_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        return None


def nameplate_line(probe_rate, sms, clk, achieved_tflops, timed=None):
    """Nameplate bf16 peak from the rate probe: SMs x measured FLOP per SM per clock x the
    maximum SM clock.  The per-SM rate comes from a probe launch timed in SM cycles on the
    GPU (clock64), so it does not depend on the clock the SMs ran at; the event-timed rate
    over the sampled clock is kept beside it."""
    if not clk.get("sm_max_mhz"):
        return {"peak": None, "why": "no clock samples"}
    line = {"sms": sms, "max_mhz": clk["sm_max_mhz"], "probe_mhz_sampled": clk.get("sm_mhz"),
            "probe_reasons": clk.get("reasons", []), "unit": "TFLOP/s"}
    if clk.get("sm_mhz"):
        line["per_sm_flop_per_clk_sampled"] = probe_rate / sms / (clk["sm_mhz"] * 1e6)
    if timed and timed["cycles"] > 0 and timed["ns"] > 0:
        per_clk = timed["flop_per_pair"] / 2 / timed["cycles"]
        line["per_sm_flop_per_clk"] = per_clk
        line["probe_mhz_measured"] = 1e3 * timed["cycles"] / timed["ns"]
        how = ("tg_tensor_rate_probe_timed: 256x256x16 pair MMAs back to back on operands in "
               "shared memory, every SM; FLOP per SM per cycle from the first pair's clock64 "
               "count of its MMA loop")
    elif clk.get("sm_mhz"):
        per_clk = line["per_sm_flop_per_clk_sampled"]
        line["per_sm_flop_per_clk"] = per_clk
        how = "tg_tensor_rate_probe timed with CUDA events for 0.6 s, over the sampled clock"
    else:
        return {"peak": None, "why": "no clock samples"}
    peak = sms * per_clk * clk["sm_max_mhz"] * 1e6 / 1e12
    line.update({"peak": peak, "frac": achieved_tflops / peak, "how": how})
    return line


def aggregate(local_seconds, local_units, world_size, allreduce_max=None, allreduce_sum=None):
    """Whole-job throughput: units of all ranks over the slowest rank's time."""
    t = allreduce_max(local_seconds) if allreduce_max else local_seconds
    u = allreduce_sum(local_units) if allreduce_sum else local_units * world_size
    return u / t, t


# ------------------------------------------------------------------------------------
# Clock sampling during the timed region
# ------------------------------------------------------------------------------------
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = os.path.join("/tmp", "tg_clocks_%d_%d.csv" % (os.getpid(), index))

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.QUERY,
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.2)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for name, val in zip(names, parts[5:9]):
                    if val.lower() == "active":
                        reasons.add(name)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        busy = sorted(sm)[len(sm) // 2:]  # the upper half: samples taken under load
        return {"sm_mhz": statistics.median(busy), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------------------------
# Our arm
# ------------------------------------------------------------------------------------
def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def physical_gpu_index(local):
    """nvidia-smi index of this process's GPU (CUDA_VISIBLE_DEVICES maps it)."""
    vis = [v.strip() for v in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if v.strip()]
    if local < len(vis) and vis[local].isdigit():
        return int(vis[local])
    return local


def cpu_baseline_gemm(A, B, M, N, K, budget_s=10.0):
    """The oracle as it stands on the host cores, over leading rows of the workload."""
    import oracle
    threads = oracle.threads()
    t0 = time.perf_counter()
    oracle.gemm(A, B, M, N, K, rows=(0, threads))   # calibration: one row per thread
    per_batch = max(time.perf_counter() - t0, 1e-6)
    rows = threads * max(1, int(budget_s / per_batch))
    rows = min(rows, M - threads)
    t0 = time.perf_counter()
    oracle.gemm(A, B, M, N, K, rows=(threads, threads + rows))
    elapsed = time.perf_counter() - t0
    flops = 2.0 * rows * N * K
    return {"value": flops / elapsed / 1e12, "unit": "TFLOP/s", "cores": threads,
            "kind": "oracle",
            "sample": "rows %d..%d of the 8192^3 GEMM (%d of 8192 rows, fp64 triple loop, "
                      "OpenMP over rows), %.1f s" % (threads, threads + rows - 1, rows, elapsed)}


def run_ours(args):
    import numpy as np
    import torch

    from tma_pipelined_tensor_gb300 import inputs as gen
    from tma_pipelined_tensor_gb300 import tg

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist

    M, N, K, _, _, _, _, seed, out, alpha, beta = gen.GEMM_WORKLOADS[GEMM_WORKLOAD]
    A, B, _ = gen.gemm_inputs(GEMM_WORKLOAD)
    T = gen.copy_tensor(COPY_H, COPY_W)
    to_bf16 = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    A_host = to_bf16(A).pin_memory()
    B_host = to_bf16(B).pin_memory()
    Ad, Bd = A_host.to(dev), B_host.to(dev)
    Cd = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    C_host = torch.empty((M, N), dtype=torch.bfloat16).pin_memory()
    Td = to_bf16(T).to(dev)
    img_bytes = tg.image_bytes(COPY_H, COPY_W, 2, COPY_BOX_W, COPY_BOX_H)
    img = torch.empty(img_bytes, dtype=torch.uint8, device=dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_src = torch.ones(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def flush_l2():
        # write 256 MiB, then read another 256 MiB: the timed kernel starts with an L2
        # holding neither its own data nor dirty lines it would have to write back
        flush.zero_()
        return flush_src.sum()
    stream = torch.cuda.current_stream(dev)
    cfg = tg.make_config(**args.gemm_config) if args.gemm_config else None

    def gemm():
        tg.gemm(Ad, Bd, Cd, alpha=alpha, beta=beta, config=cfg)

    def copy():
        tg.tile_copy(Td, COPY_BOX_W, COPY_BOX_H, tg.TG_SWZ_128B, img, stages=args.copy_stages,
                     blocks_per_sm=args.copy_blocks)

    for _ in range(args.warmup):
        gemm()
        copy()
    st = tg.tg_status_sync(None)
    if st != tg.TG_OK:
        raise SystemExit("warm-up failed: %s" % tg.tg_status_string(st))

    n = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(n)]
    clocks = ClockSampler(physical_gpu_index(local))
    clocks.start()
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    for i in range(n):
        flush_l2()
        ev[i][0].record(stream)
        gemm()
        ev[i][1].record(stream)
        flush_l2()
        ev[i][2].record(stream)
        copy()
        ev[i][3].record(stream)
    torch.cuda.synchronize()
    if pg:
        pg.barrier()
    wall = time.perf_counter() - wall0
    clk = clocks.stop()
    st = tg.tg_status_sync(None)
    if st != tg.TG_OK:
        raise SystemExit("timed region failed: %s" % tg.tg_status_string(st))
    gemm_ms = [ev[i][0].elapsed_time(ev[i][1]) for i in range(n)]
    copy_ms = [ev[i][2].elapsed_time(ev[i][3]) for i in range(n)]
    gemm_s, copy_s = sum(gemm_ms) / 1e3, sum(copy_ms) / 1e3

    # Steady-state copy: back-to-back copies of distinct tensors (about 1.1 GB of traffic,
    # far beyond L2), so that write-backs of earlier images are paid inside the region.
    ss_copies = 8
    ss_in = [Td.clone() for _ in range(ss_copies)]
    ss_out = [torch.empty_like(img) for _ in range(ss_copies)]
    ss_times = []
    for _ in range(3):
        flush_l2()
        ss_ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        ss_ev[0].record(stream)
        for j in range(ss_copies):
            tg.tile_copy(ss_in[j], COPY_BOX_W, COPY_BOX_H, tg.TG_SWZ_128B, ss_out[j],
                         stages=args.copy_stages, blocks_per_sm=args.copy_blocks)
        ss_ev[1].record(stream)
        torch.cuda.synchronize()
        ss_times.append(ss_ev[0].elapsed_time(ss_ev[1]) / 1e3)
    ss_s = statistics.median(ss_times)
    del ss_in, ss_out

    # The same product with E4M3 operands (8192^3, bf16 out; not part of the step): each
    # launch timed by CUDA events after an L2 flush.
    A8, B8, _ = gen.gemm_inputs(F8_WORKLOAD)
    A8d = torch.from_numpy(A8).to(dev).view(torch.float8_e4m3fn)
    B8d = torch.from_numpy(B8).to(dev).view(torch.float8_e4m3fn)
    del A8, B8
    f8_ms = []
    for i in range(args.warmup + n):
        flush_l2()
        f8_ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        f8_ev[0].record(stream)
        tg.gemm(A8d, B8d, Cd, config=cfg)
        f8_ev[1].record(stream)
        torch.cuda.synchronize()
        if i >= args.warmup:
            f8_ms.append(f8_ev[0].elapsed_time(f8_ev[1]))
    # The same E4M3 elements with one E8M0 scale per 32 elements of K (MX), each launch
    # timed the same way; sampled outputs checked against the oracle afterwards.
    SA8, SA8p, SB8, SB8p = gen.gemm_mx_scale_inputs(MX_WORKLOAD)
    SA8d, SB8d = torch.from_numpy(SA8p).to(dev), torch.from_numpy(SB8p).to(dev)
    mx_ms = []
    for i in range(args.warmup + n):
        flush_l2()
        mx_ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        mx_ev[0].record(stream)
        tg.gemm_mx(A8d, SA8d, B8d, SB8d, Cd, kind="e4m3", stream=stream)
        mx_ev[1].record(stream)
        torch.cuda.synchronize()
        if i >= args.warmup:
            mx_ms.append(mx_ev[0].elapsed_time(mx_ev[1]))
    _, mx_plan = tg.tg_gemm_last_plan()
    mx_got = gen.bf16_bits_to_f32(Cd.view(torch.int16).cpu().numpy().view(np.uint16))
    del A8d, B8d, SA8d, SB8d
    st = tg.tg_status_sync(None)
    if st != tg.TG_OK:
        raise SystemExit("E4M3 / MX region failed: %s" % tg.tg_status_string(st))
    mx_parity = None
    if not args.no_cpu_baseline:
        mx_parity = mx_sampled_parity(mx_got, SA8p, SB8p, M, N, K)
    del SA8, SB8, SA8p, SB8p, mx_got

    # End to end through the public API: every step copies its inputs in from pinned host
    # memory, multiplies, and reads C back to pinned host memory.  Two streams with their
    # own device buffers let step i+1's copies overlap step i's GEMM (wall-clock timed).
    e2e_steps = max(4, min(n, 20))
    # two streams of their own: the legacy default stream would serialise with them
    streams = [torch.cuda.Stream(dev), torch.cuda.Stream(dev)]
    bufs = [(Ad, Bd, Cd), (torch.empty_like(Ad), torch.empty_like(Bd), torch.empty_like(Cd))]
    C_hosts = [C_host, torch.empty_like(C_host).pin_memory()]

    def e2e_step(i):
        s_i = streams[i % 2]
        a_d, b_d, c_d = bufs[i % 2]
        with torch.cuda.stream(s_i):
            a_d.copy_(A_host, non_blocking=True)
            b_d.copy_(B_host, non_blocking=True)
            tg.gemm(a_d, b_d, c_d, alpha=alpha, beta=beta, config=cfg, stream=s_i)
            C_hosts[i % 2].copy_(c_d, non_blocking=True)
    for i in range(2):          # one untimed step on each stream
        e2e_step(i)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(e2e_steps):
        e2e_step(i)
    torch.cuda.synchronize()
    e2e_s = time.perf_counter() - t0
    st = tg.tg_status_sync(None)
    if st != tg.TG_OK:
        raise SystemExit("end-to-end region failed: %s" % tg.tg_status_string(st))

    # CUDA-graph batch of copies: the same 8 distinct copies as the steady-state region,
    # captured once and replayed, so that no launch gap separates them.
    graph_s, graph_err = None, None
    try:
        g_in = [Td.clone() for _ in range(ss_copies)]
        g_out = [torch.empty_like(img) for _ in range(ss_copies)]
        for j in range(ss_copies):      # outside the capture: first use of each tensor
            tg.tile_copy(g_in[j], COPY_BOX_W, COPY_BOX_H, tg.TG_SWZ_128B, g_out[j])
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for j in range(ss_copies):
                tg.tile_copy(g_in[j], COPY_BOX_W, COPY_BOX_H, tg.TG_SWZ_128B, g_out[j],
                             stages=args.copy_stages, blocks_per_sm=args.copy_blocks)
        g_times = []
        for _ in range(3):
            flush_l2()
            gev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
            gev[0].record(stream)
            graph.replay()
            gev[1].record(stream)
            torch.cuda.synchronize()
            g_times.append(gev[0].elapsed_time(gev[1]) / 1e3)
        graph_s = statistics.median(g_times)
        del graph, g_in, g_out
    except RuntimeError as exc:      # capture not available: report why
        graph_err = str(exc).splitlines()[0][:120]
    st = tg.tg_status_sync(None)
    if st != tg.TG_OK:
        raise SystemExit("graph copy region failed: %s" % tg.tg_status_string(st))

    # Nameplate peak: SMs x the tensor cores' own per-SM FLOP per clock (the rate probe:
    # back-to-back pair MMAs on operands already in shared memory) x the maximum clock.
    probe_iters = 1 << 14
    tg.tensor_rate_probe(tg.TG_IN_BF16, 256)
    torch.cuda.synchronize()
    probe_clk = ClockSampler(physical_gpu_index(local))
    probe_clk.start()
    pev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    pev[0].record(stream)
    probe_flops, probe_n, t_probe0 = 0, 0, time.perf_counter()
    while time.perf_counter() - t_probe0 < 0.6:
        pst, pairs, f = tg.tensor_rate_probe(tg.TG_IN_BF16, probe_iters)
        if pst != tg.TG_OK:
            raise SystemExit("rate probe failed: %s" % tg.tg_status_string(pst))
        probe_flops += f
        probe_n += 1
        if probe_n % 8 == 0:
            torch.cuda.synchronize()
    pev[1].record(stream)
    torch.cuda.synchronize()
    pclk = probe_clk.stop()
    if tg.tg_status_sync(None) != tg.TG_OK:
        raise SystemExit("rate probe failed on the device")
    probe_rate = probe_flops / (pev[0].elapsed_time(pev[1]) * 1e-3)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    # ... and one more launch timed by the GPU itself (SM cycles and ns of the first
    # pair's MMA loop): the per-SM FLOP per clock at the clock the SMs really ran at
    ptim = torch.zeros(2, dtype=torch.int64, device=dev)
    pst, pairs, f = tg.tensor_rate_probe_timed(ptim.data_ptr(), tg.TG_IN_BF16, probe_iters)
    torch.cuda.synchronize()
    if pst != tg.TG_OK or tg.tg_status_sync(None) != tg.TG_OK:
        raise SystemExit("timed rate probe failed")
    probe_cycles, probe_ns = (int(x) for x in ptim.cpu().tolist())
    probe_timed = {"flop_per_pair": f / pairs, "cycles": probe_cycles, "ns": probe_ns}

    workloads = None
    if not args.no_workloads:
        workloads = time_workloads(dev, max(5, min(n, 20)), flush_l2, peaks(), args.workload_cpu)

    allmax = allsum = None
    if pg:
        def allmax(x):
            t = torch.tensor([x], dtype=torch.float64, device=dev)
            pg.all_reduce(t, op=pg.ReduceOp.MAX)
            return float(t.item())

        def allsum(x):
            t = torch.tensor([x], dtype=torch.float64, device=dev)
            pg.all_reduce(t, op=pg.ReduceOp.SUM)
            return float(t.item())
    flops = gemm_flops(M, N, K)
    value, gemm_s_max = aggregate(gemm_s, flops * n, world, allmax, allsum)
    cvalue, copy_s_max = aggregate(copy_s, copy_bytes(COPY_H, COPY_W, 2, COPY_BOX_W, COPY_BOX_H) * n,
                                   world, allmax, allsum)
    e2e_value, _ = aggregate(e2e_s, flops * e2e_steps, world, allmax, allsum)

    if rank != 0:
        if pg:
            pg.destroy_process_group()
        return
    pk = peaks()
    plan_st, plan = tg.tg_gemm_plan_for(M, N, K, tg.TG_C_BF16, cfg, 0)
    gemm_avg = gemm_s / n
    achieved = flops / gemm_avg / 1e12
    copy_avg = copy_s / n
    cb = copy_bytes(COPY_H, COPY_W, 2, COPY_BOX_W, COPY_BOX_H)
    line = {
        "metric": METRIC,
        "value": value / 1e12,
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": n,
        "warmup": args.warmup,
        "ms_per_step": (gemm_s_max + copy_s_max) / n * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {
            "workload": "gemm_8192 (M=N=K=8192, A,B U[-1,1] bf16 seed 3, fp32 accumulate, "
                        "bf16 out, alpha=1 beta=0) + tma_tile_copy (4100x8200 bf16, box 128x64, "
                        "128B swizzle, zero fill)",
            "gemm_launch": {"tile": [plan.tile_m, plan.tile_n, plan.tile_k], "stages": plan.stages,
                            "cluster": plan.cluster, "mma": "cta pair" if plan.mma == 2 else
                            "per cta", "grid": plan.grid,
                            "smem_bytes": plan.smem_bytes} if plan_st == 0 else None,
            "l2": "flushed before every timed kernel (256 MiB written, then 256 MiB read; "
                  "outside the events)",
            "parallelism": "replicas" if world > 1 else "single GPU",
        },
        "roofline": {
            "bound": "tensor", "achieved": achieved, "peak": pk["bf16_tflops"],
            "unit": "TFLOP/s", "frac": achieved / pk["bf16_tflops"],
            "traffic": committed_traffic("gemm_bf16_pair_kernel<256, 0, 0>" if plan.mma == 2
                                         else "gemm_bf16_kernel<256, 0>"),
            "peak_source": "%s bf16 burst" % pk["source"],
            "nameplate": nameplate_line(probe_rate, sms, pclk, value / 1e12, probe_timed),
        },
        "tma_copy": {
            "value": cvalue / 1e9, "unit": "GB/s", "ms_per_launch": copy_avg * 1e3,
            "roofline": {"bound": "hbm", "achieved": cb / copy_avg / 1e9, "peak": pk["hbm_gbs"],
                         "unit": "GB/s", "frac": cb / copy_avg / 1e9 / pk["hbm_gbs"],
                         "traffic": committed_traffic("tma_tile_copy_kernel"),
                         "peak_source": "%s HBM copy" % pk["source"]},
            "steady_state": {"value": cb * ss_copies / ss_s / 1e9, "unit": "GB/s",
                             "frac": cb * ss_copies / ss_s / 1e9 / pk["hbm_gbs"],
                             "how": "%d back-to-back copies of distinct 4100x8200 tensors into "
                                    "distinct images after one L2 flush (CUDA events, median "
                                    "of 3)" % ss_copies},
            "graph": ({"value": cb * ss_copies / graph_s / 1e9, "unit": "GB/s",
                       "frac": cb * ss_copies / graph_s / 1e9 / pk["hbm_gbs"],
                       "how": "the same %d copies captured in one CUDA graph and replayed after "
                              "an L2 flush (CUDA events, median of 3)" % ss_copies}
                      if graph_s else {"value": None, "why": graph_err}),
            "note": "at 137 MB per launch part of the image is still in L2 when a launch "
                    "ends (see traffic); steady_state pays those write-backs",
        },
        "gemm_e4m3": {
            "workload": "gemm_8192_e4m3 (the same shape and U[-1,1] draws rounded to E4M3, "
                        "fp32 accumulate, bf16 out)",
            "value": flops / (statistics.mean(f8_ms) * 1e-3) / 1e12, "unit": "TFLOP/s",
            "ms_per_launch": statistics.mean(f8_ms), "launches": len(f8_ms),
            "roofline": {"bound": "tensor",
                         "achieved": flops / (statistics.mean(f8_ms) * 1e-3) / 1e12,
                         "peak": pk["bf16_tflops"] * FP8_PER_BF16, "unit": "TFLOP/s",
                         "frac": flops / (statistics.mean(f8_ms) * 1e-3) / 1e12
                                 / (pk["bf16_tflops"] * FP8_PER_BF16),
                         "traffic": committed_traffic("gemm_bf16_pair_kernel<256, 1, 0>"
                                                      if plan.mma == 2 else
                                                      "gemm_bf16_kernel<256, 1>"),
                         "peak_source": "%s bf16 burst x %g (nominal fp8 / bf16 dense rates)"
                                        % (pk["source"], FP8_PER_BF16)},
        },
        "gemm_mxe4m3": {
            "workload": "gemm_8192_mxe4m3 (E4M3 elements as above; one E8M0 scale per 32 "
                        "elements of K, exponents drawn from [120, 134]; fp32 accumulate, "
                        "bf16 out)",
            "value": flops / (statistics.mean(mx_ms) * 1e-3) / 1e12, "unit": "TFLOP/s",
            "ms_per_launch": statistics.mean(mx_ms), "launches": len(mx_ms),
            "launch": {"tile": [mx_plan.tile_m, mx_plan.tile_n, mx_plan.tile_k],
                       "stages": mx_plan.stages, "grid": mx_plan.grid, "mma": mx_plan.mma},
            "roofline": {"bound": "tensor",
                         "achieved": flops / (statistics.mean(mx_ms) * 1e-3) / 1e12,
                         "peak": pk["bf16_tflops"] * FP8_PER_BF16, "unit": "TFLOP/s",
                         "frac": flops / (statistics.mean(mx_ms) * 1e-3) / 1e12
                                 / (pk["bf16_tflops"] * FP8_PER_BF16),
                         "traffic": committed_traffic("gemm_bf16_pair_kernel<256, 3, 0>"
                                                      if mx_plan.mma == 2 else
                                                      "gemm_bf16_kernel<128, 3>"),
                         "peak_source": "%s bf16 burst x %g (nominal fp8 / bf16 dense rates)"
                                        % (pk["source"], FP8_PER_BF16)},
            "parity": mx_parity,
        },
        "e2e": {"value": e2e_value / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": (A_host.numel() + B_host.numel()) * 2,
                "d2h_bytes_per_step": C_host.numel() * 2, "steps": e2e_steps,
                "how": "wall clock; pinned host A, B copied in and C copied out every step; "
                       "two streams overlap step i+1's copies with step i's GEMM"},
        "workloads": workloads,
        "gpu_launches": 2 * n,
        "clocks": clk,
        "wall_s": wall,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_gemm(A, B, M, N, K, budget_s=args.cpu_budget)
    print(json.dumps(line), flush=True)
    if pg:
        pg.destroy_process_group()


# ------------------------------------------------------------------------------------
# Every GEMM configuration of the workload set in the bench line itself
# ------------------------------------------------------------------------------------
LINE_WORKLOADS = ["gemm_256", "gemm_4096", "ffn_up", "ffn_down", "dw", "ragged"]


def mx_sampled_parity(got, sa_packed, sb_packed, M, N, K):
    """The MX product's outputs at 1002 sampled positions (the corners among them) against
    the oracle, at the fp32-accumulation bound plus bf16 rounding of C."""
    import numpy as np

    import oracle
    from tma_pipelined_tensor_gb300 import inputs as gen

    A8, B8, _ = gen.gemm_inputs(MX_WORKLOAD)
    rng = np.random.default_rng(7)
    ii = np.concatenate([rng.integers(0, M, 1000), [0, M - 1]])
    jj = np.concatenate([rng.integers(0, N, 1000), [0, N - 1]])
    ref, mag = oracle.gemm_mx_entries(A8, sa_packed, B8, sb_packed, M, N, K, ii, jj)
    bound = 2.0 * K * 2.0 ** -24 * mag + 2.0 ** -8 * np.abs(ref)
    err = np.abs(got[ii, jj].astype(np.float64) - ref)
    return {"samples": int(len(ii)), "within_bound": bool((err <= bound).all()),
            "max_err_over_bound": float((err / np.maximum(bound, 1e-300)).max())}


def time_workloads(dev, reps, flush_l2, pk, cpu_budget):
    """Each configuration in the default launch: device time per launch (CUDA events on
    the launching stream, L2 flushed before every launch), the launch plan, a check of
    sampled outputs against the oracle at the error bound, and the oracle itself timed on
    a row sample on the host cores."""
    import concurrent.futures as cf

    import numpy as np
    import torch

    import oracle
    from tma_pipelined_tensor_gb300 import inputs as gen
    from tma_pipelined_tensor_gb300 import tg

    to_bf16 = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    with cf.ThreadPoolExecutor(4) as ex:      # numpy releases the GIL while drawing
        inputs = dict(zip(LINE_WORKLOADS, ex.map(gen.gemm_inputs, LINE_WORKLOADS)))
    stream = torch.cuda.current_stream(dev)
    rows = []
    for name in LINE_WORKLOADS:
        M, N, K, _, _, _, _, seed, out, alpha, beta = gen.GEMM_WORKLOADS[name]
        A, B, C0 = inputs.pop(name)
        out_bf16 = out == "bf16"
        Ad, Bd = to_bf16(A).to(dev), to_bf16(B).to(dev)
        if C0 is not None:
            Cinit = to_bf16(C0).to(dev) if out_bf16 else torch.from_numpy(C0).to(dev)
        else:
            Cinit = torch.zeros((M, N), device=dev,
                                dtype=torch.bfloat16 if out_bf16 else torch.float32)
        Cd = Cinit.clone()
        for _ in range(3):
            Cd.copy_(Cinit)
            tg.gemm(Ad, Bd, Cd, alpha=alpha, beta=beta)
        ms = []
        for _ in range(reps):
            Cd.copy_(Cinit)
            flush_l2()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            tg.gemm(Ad, Bd, Cd, alpha=alpha, beta=beta)
            e1.record(stream)
            torch.cuda.synchronize()
            ms.append(e0.elapsed_time(e1))
        st = tg.tg_status_sync(None)
        if st != tg.TG_OK:
            raise SystemExit("workload %s failed: %s" % (name, tg.tg_status_string(st)))
        _, last = tg.tg_gemm_last_plan()
        if out_bf16:
            got = gen.bf16_bits_to_f32(Cd.view(torch.int16).cpu().numpy().view(np.uint16))
        else:
            got = Cd.cpu().numpy()
        got = got.astype(np.float64)
        del Ad, Bd, Cd, Cinit
        torch.cuda.empty_cache()
        # parity on sampled outputs (and the first and last rows' first columns)
        rng = np.random.default_rng(seed)
        ii = np.concatenate([rng.integers(0, M, 2000), [0, M - 1, M - 1]])
        jj = np.concatenate([rng.integers(0, N, 2000), [0, 0, N - 1]])
        ref, mag = oracle.gemm_entries(A, B, K, ii, jj, C0=C0, ldc=N, alpha=alpha, beta=beta)
        bound = 2.0 * K * 2.0 ** -24 * abs(alpha) * mag
        if out_bf16:
            bound = bound + 2.0 ** -8 * np.abs(ref)
        if beta != 0.0:
            c0v = gen.bf16_bits_to_f32(C0[ii, jj]).astype(np.float64) if out_bf16 else C0[ii, jj]
            bound = bound + 2.0 ** -23 * np.abs(beta * c0v)
        err = np.abs(got[ii, jj] - ref)
        # the oracle as it stands, on a row sample sized to about cpu_budget seconds
        threads = oracle.threads()
        t0 = time.perf_counter()
        oracle.gemm(A, B, M, N, K, C0=C0, ldc=N, alpha=alpha, beta=beta, rows=(0, min(M, threads)))
        per = max(time.perf_counter() - t0, 1e-6)
        r2 = min(M, threads * max(1, int(cpu_budget / per)))
        t0 = time.perf_counter()
        oracle.gemm(A, B, M, N, K, C0=C0, ldc=N, alpha=alpha, beta=beta, rows=(0, r2))
        cpu_s = time.perf_counter() - t0
        mean_ms = statistics.mean(ms)
        achieved = gemm_flops(M, N, K) / (mean_ms * 1e-3) / 1e12
        entry = {
            "workload": name, "M": M, "N": N, "K": K, "out": out, "alpha": alpha, "beta": beta,
            "ms_per_launch": mean_ms, "ms_median": statistics.median(ms), "launches": reps,
            "value": achieved, "unit": "TFLOP/s",
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": pk["bf16_tflops"],
                         "unit": "TFLOP/s", "frac": achieved / pk["bf16_tflops"],
                         "peak_source": "%s bf16 burst" % pk["source"]},
            "launch": {"tile": [last.tile_m, last.tile_n, last.tile_k], "stages": last.stages,
                       "grid": last.grid, "units": int(last.tiles_n * -(-last.tiles_m // last.cluster)),
                       "dp_units": last.dp_units, "sk_iters": int(last.sk_iters),
                       "split_units": last.split_units},
            "parity": {"samples": int(len(ii)), "within_bound": bool((err <= bound).all()),
                       "max_err_over_bound": float((err / np.maximum(bound, 1e-300)).max())},
            "oracle": {"value": gemm_flops(r2, N, K) / cpu_s / 1e12, "unit": "TFLOP/s",
                       "rows": int(r2), "seconds": cpu_s, "cores": threads},
        }
        if name == "gemm_256":
            entry["us_per_launch"] = mean_ms * 1e3
            entry["roofline"]["note"] = "launch-latency bound: 3.4e7 flop per launch"
        rows.append(entry)
    return rows


# ------------------------------------------------------------------------------------
# Per-workload report (every GEMM configuration, default launch) written as JSON
# ------------------------------------------------------------------------------------
def run_report(args):
    import numpy as np
    import torch

    import oracle
    from tma_pipelined_tensor_gb300 import inputs as gen
    from tma_pipelined_tensor_gb300 import tg

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    pk = peaks()
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_src = torch.ones(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    to_bf16 = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    f8_dtypes = {"e4m3": torch.float8_e4m3fn, "e5m2": torch.float8_e5m2}
    cfg = tg.make_config(**args.gemm_config) if args.gemm_config else None
    rows = []
    only = [w for w in args.report_workloads.split(",") if w]
    items = [(name, w) for name, w in gen.GEMM_WORKLOADS.items() if not only or name in only]
    if args.report_shape:
        # an ad-hoc problem: A, B uniform in [-1, 1] as bf16 (seed 0), bf16 C, alpha 1
        dims = [int(x) for x in args.report_shape.split(",")[:3]]
        sb = float(args.report_shape.split(",")[3]) if args.report_shape.count(",") >= 3 else 0.0
        items.append(("shape_%dx%dx%d" % tuple(dims),
                      (dims[0], dims[1], dims[2], "uniform", None, "uniform", None, 0, "bf16", 1.0, sb)))
    for name, (M, N, K, _, _, _, _, seed, out, alpha, beta) in items:
        if name.startswith("shape_"):
            A = gen.bf16_matrix(M, K, 0, gen.STREAM_A, "uniform") if K else np.zeros((M, 0), np.uint16)
            B = gen.bf16_matrix(N, K, 0, gen.STREAM_B, "uniform") if K else np.zeros((N, 0), np.uint16)
            C0 = gen.bf16_matrix(M, N, 0, gen.STREAM_C, "uniform") if beta != 0.0 else None
        else:
            A, B, C0 = gen.gemm_inputs(name)
        in_type = gen.WORKLOAD_IN_TYPE.get(name, "bf16")
        if in_type == "bf16":
            Ad, Bd = to_bf16(A).to(dev), to_bf16(B).to(dev)
            if args.report_pad:
                # rows of A and B padded by report_pad elements (row strides K + pad)
                Ap = torch.zeros((M, K + args.report_pad), dtype=torch.bfloat16, device=dev)
                Bp = torch.zeros((N, K + args.report_pad), dtype=torch.bfloat16, device=dev)
                Ap[:, :K] = Ad
                Bp[:, :K] = Bd
                Ad, Bd = Ap[:, :K], Bp[:, :K]
            peak, peak_how = pk["bf16_tflops"], "%s bf16 burst" % pk["source"]
        elif in_type == "tf32":
            Ad, Bd = torch.from_numpy(A).to(dev), torch.from_numpy(B).to(dev)
            peak = pk["bf16_tflops"] * TF32_PER_BF16
            peak_how = "%s bf16 burst x %.3f (nominal tf32 / bf16 dense rates)" % (pk["source"],
                                                                                 TF32_PER_BF16)
        else:
            Ad = torch.from_numpy(A).to(dev).view(f8_dtypes[in_type.replace("mx", "")])
            Bd = torch.from_numpy(B).to(dev).view(f8_dtypes[in_type.replace("mx", "")])
            if in_type.startswith("mx"):
                _, SAp, _, SBp = gen.gemm_mx_scale_inputs(name)
                SAd, SBd = torch.from_numpy(SAp).to(dev), torch.from_numpy(SBp).to(dev)
            peak = pk["bf16_tflops"] * FP8_PER_BF16
            peak_how = "%s bf16 burst x %g (nominal fp8 / bf16 dense rates)" % (pk["source"],
                                                                               FP8_PER_BF16)
        if C0 is not None:
            Cinit = to_bf16(C0).to(dev) if out == "bf16" else torch.from_numpy(C0).to(dev)
        else:
            Cinit = torch.zeros((M, N), device=dev,
                                dtype=torch.bfloat16 if out == "bf16" else torch.float32)
        Cd = Cinit.clone()

        def ours():
            if K == 0:   # C <- beta * C: the epilogue alone, no operand is read
                st0 = tg.gemm_bf16_ex(M, N, 0, None, 0, None, 0, Cd.data_ptr(), N, alpha, beta,
                                      tg.TG_C_BF16 if out == "bf16" else tg.TG_C_F32, cfg,
                                      torch.cuda.current_stream().cuda_stream)
                if st0 != tg.TG_OK:
                    raise tg.TgError(st0, "gemm_bf16_ex")
            elif in_type.startswith("mx"):
                tg.gemm_mx(Ad, SAd, Bd, SBd, Cd, alpha=alpha, beta=beta,
                           kind=in_type[2:], config=cfg)
            else:
                tg.gemm(Ad, Bd, Cd, alpha=alpha, beta=beta, config=cfg)
        for _ in range(3):
            Cd.copy_(Cinit)
            ours()
        ms = []
        for _ in range(args.report_reps):
            Cd.copy_(Cinit)
            flush.zero_()
            flush_src.sum()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            ours()
            e1.record()
            torch.cuda.synchronize()
            ms.append(e0.elapsed_time(e1))
        chain_tflops = None
        if args.report_chain > 0 and K > 0:
            # back-to-back launches with no flush in between (inputs stay in L2 where they
            # fit): each launch's start overlaps the previous one's tail.  Context for a
            # sequence of GEMMs, not a flushed per-launch figure.
            chain_ms = []
            for _ in range(3):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                for _ in range(args.report_chain):
                    ours()
                e1.record()
                torch.cuda.synchronize()
                chain_ms.append(e0.elapsed_time(e1) / args.report_chain)
            chain_tflops = gemm_flops(M, N, K) / (statistics.median(chain_ms) * 1e-3) / 1e12
        st = tg.tg_status_sync(None)
        lib_tflops = None
        if args.report_cublas and K > 0 and (in_type == "tf32" or (in_type == "bf16" and out == "bf16")):
            # the same product through torch.matmul (cuBLAS), timed the same way: a
            # comparison column only, never part of the path
            prev_tf32 = torch.backends.cuda.matmul.allow_tf32
            torch.backends.cuda.matmul.allow_tf32 = in_type == "tf32"
            Cl = Cinit.clone() if in_type == "bf16" else torch.empty((M, N), device=dev)
            lib = lambda: torch.addmm(Cl, Ad, Bd.t(), beta=beta, alpha=alpha, out=Cl)
            for _ in range(3):
                lib()
            lms = []
            for _ in range(args.report_reps):
                flush.zero_()
                flush_src.sum()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                lib()
                e1.record()
                torch.cuda.synchronize()
                lms.append(e0.elapsed_time(e1))
            lib_tflops = gemm_flops(M, N, K) / (statistics.median(lms) * 1e-3) / 1e12
            torch.backends.cuda.matmul.allow_tf32 = prev_tf32
            del Cl
        layout = tg.TG_C_BF16 if out == "bf16" else tg.TG_C_F32
        layout |= {"bf16": tg.TG_IN_BF16, "e4m3": tg.TG_IN_E4M3, "e5m2": tg.TG_IN_E5M2,
                   "tf32": tg.TG_IN_TF32, "mxe4m3": tg.TG_IN_MXE4M3,
                   "mxe5m2": tg.TG_IN_MXE5M2}[in_type]
        _, plan = tg.tg_gemm_last_plan()     # the launch just timed
        med = statistics.median(ms)
        tflops = gemm_flops(M, N, K) / (med * 1e-3) / 1e12
        # oracle on a bounded sample of rows (about args.report_cpu seconds)
        r2, cpu_s = 0, float("nan")
        if K > 0:
            def oracle_rows(nr):
                if in_type.startswith("mx"):
                    ii, jj = np.meshgrid(np.arange(nr), np.arange(N), indexing="ij")
                    oracle.gemm_mx_entries(A, SAp, B, SBp, M, N, K, ii.ravel(), jj.ravel(),
                                           in_type[2:], C0=C0, ldc=N, alpha=alpha, beta=beta)
                else:
                    oracle.gemm(A, B, M, N, K, C0=C0, ldc=N, alpha=alpha, beta=beta,
                                rows=(0, nr), in_kind=in_type)
            t0 = time.perf_counter()
            r = max(1, oracle.threads())
            oracle_rows(r)
            per = time.perf_counter() - t0
            r2 = min(M, r * max(1, int(args.report_cpu / max(per, 1e-6))))
            t0 = time.perf_counter()
            oracle_rows(r2)
            cpu_s = time.perf_counter() - t0
        units = plan.tiles_n * -(-plan.tiles_m // plan.cluster)
        slots = torch.cuda.get_device_properties(dev).multi_processor_count // plan.cluster
        rows.append({
            "workload": name, "M": M, "N": N, "K": K, "in": in_type, "out": out, "beta": beta,
            "lda": int(Ad.stride(0)), "ldb": int(Bd.stride(0)),
            "status": tg.tg_status_string(st), "ms_median": med, "ms_min": min(ms),
            "tflops": tflops, "frac_of_measured_peak": tflops / peak, "peak": peak,
            "peak_source": peak_how,
            "tiles": [plan.tiles_m, plan.tiles_n], "units": units, "grid": plan.grid,
            "mma": plan.mma, "tile_n": plan.tile_n, "cluster": plan.cluster,
            "dp_units": plan.dp_units, "sk_iters": plan.sk_iters,
            "waves": units / slots, "wave_efficiency": units / (slots * -(-units // slots)),
            "oracle_tflops": gemm_flops(r2, N, K) / cpu_s / 1e12 if r2 else None,
            "oracle_sample_rows": r2, "oracle_s": cpu_s, "oracle_cores": oracle.threads(),
            "cublas_tflops": lib_tflops,
            "chain_tflops": chain_tflops, "chain_launches": args.report_chain,
        })
        del Ad, Bd, Cd, Cinit
        torch.cuda.empty_cache()
    with open(args.report, "w") as f:
        json.dump({"peak_bf16_tflops": pk["bf16_tflops"], "peak_source": pk["source"],
                   "config": args.gemm_config or "default", "workloads": rows}, f, indent=1)
    for r in rows:
        lib = "  cuBLAS %6.1f" % r["cublas_tflops"] if r["cublas_tflops"] else ""
        if r["chain_tflops"]:
            lib += "  chained %6.1f" % r["chain_tflops"]
        print("%-10s %6.1f TFLOP/s  %5.1f%% of peak  waves %.2f (eff %.2f)  sk %d  oracle %.4f%s"
              % (r["workload"], r["tflops"], 100 * r["frac_of_measured_peak"], r["waves"],
                 r["wave_efficiency"], r["sk_iters"], r["oracle_tflops"] or 0.0, lib), file=sys.stderr)


# ------------------------------------------------------------------------------------
# Reference arm: the CPU oracle, bounded samples of the same workload
# ------------------------------------------------------------------------------------
def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle
    from tma_pipelined_tensor_gb300 import inputs as gen

    M, N, K = gen.GEMM_WORKLOADS[GEMM_WORKLOAD][:3]
    A, B, _ = gen.gemm_inputs(GEMM_WORKLOAD)
    rows_per_step = max(1, args.reference_rows)
    for w in range(args.warmup):
        oracle.gemm(A, B, M, N, K, rows=(w, w + 1))
    times = []
    for s in range(args.steps):
        r0 = (s * rows_per_step) % M
        t0 = time.perf_counter()
        oracle.gemm(A, B, M, N, K, rows=(r0, r0 + rows_per_step))
        times.append(time.perf_counter() - t0)
    total = sum(times)
    value = gemm_flops(rows_per_step, N, K) * args.steps / total / 1e12
    sample = "%d rows of the 8192^3 GEMM per step (fp64 triple loop)" % rows_per_step
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": total / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "gemm_8192 (M=N=K=8192, A,B U[-1,1] bf16 seed 3), bounded row "
                               "sample on the host cores", "parallelism": "host threads"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle.threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=100)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-budget", type=float, default=10.0)
    p.add_argument("--reference-rows", type=int, default=4)
    p.add_argument("--no-workloads", action="store_true",
                   help="leave the other GEMM configurations out of the bench line")
    p.add_argument("--workload-cpu", type=float, default=2.0,
                   help="seconds of oracle time per configuration for its row sample")
    p.add_argument("--stages", type=int, default=0)
    p.add_argument("--cluster", type=int, default=0)
    p.add_argument("--tile-n", type=int, default=0)
    p.add_argument("--group-m", type=int, default=0)
    p.add_argument("--mma", type=int, default=0)
    p.add_argument("--schedule", type=int, default=0)
    p.add_argument("--copy-stages", type=int, default=0)
    p.add_argument("--copy-blocks", type=int, default=0)
    p.add_argument("--report", default="", help="write a per-workload JSON report here")
    p.add_argument("--report-reps", type=int, default=10)
    p.add_argument("--report-chain", type=int, default=0,
                   help="also time this many back-to-back launches per workload (no flush)")
    p.add_argument("--report-cpu", type=float, default=3.0)
    p.add_argument("--report-cublas", action="store_true",
                   help="also time torch.matmul (cuBLAS) on each bf16/tf32 workload, for comparison")
    p.add_argument("--report-shape", default="",
                   help="--report: also an ad-hoc problem M,N,K[,beta] (uniform bf16 inputs, "
                        "bf16 C); K = 0 runs the epilogue alone (C <- beta*C)")
    p.add_argument("--report-pad", type=int, default=0,
                   help="--report: pad the rows of bf16 A and B by this many elements")
    p.add_argument("--report-workloads", default="",
                   help="comma-separated workload names for --report (default: all)")
    a = p.parse_args(argv)
    a.gemm_config = {k: v for k, v in (("stages", a.stages), ("cluster", a.cluster),
                                       ("tile_n", a.tile_n), ("group_m", a.group_m),
                                       ("mma", a.mma), ("schedule", a.schedule)) if v}
    return a


def check_launch(args, world):
    """Refuses, before anything touches a GPU, the launches this bench does not make:
    a world size other than --gpus (N > 1 runs one rank per GPU under torchrun), and the
    per-CTA kernel's cluster-multicast load (--cluster 2 --mma 1) on more than one rank,
    since that load is a single-GPU option.  Returns an error message or None."""
    if args.gpus < 1:
        return "--gpus must be at least 1"
    if world != args.gpus:
        return ("--gpus %d but WORLD_SIZE is %d: for N > 1 launch one rank per GPU with "
                "torchrun --nproc-per-node %d" % (args.gpus, world, args.gpus))
    if world > 1 and args.gemm_config.get("cluster") == 2 and args.gemm_config.get("mma") == 1:
        return ("--cluster 2 --mma 1 selects the TMA multicast kernel, a single-GPU option: "
                "refused with more than one rank")
    return None


def main(argv=None):
    args = parse_args(argv)
    err = check_launch(args, dist_env()[1])
    if err:
        raise SystemExit("bench.py: " + err)
    if args.report:
        run_report(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
