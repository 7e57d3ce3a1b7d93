"""The stream-K workspace: one per stream (told apart by stream ID, so each host thread's
per-thread default stream has its own), a caller-owned one when the caller passes it, and
a reported fall-back to whole tiles when no workspace can be had.

Stream-K splits the k-blocks of the last wave's tiles over all clusters ("GEMM: la
moltiplicazione di matrici sull'hardware", "In pratica": wave quantisation); partial sums
go through the workspace in fp32.  Every result is compared with the fp64 oracle at the
bound |C - C_ref| <= 2*K*2^-24*(|A||B|) (fp32 C)."""
import ctypes
import threading

import numpy as np
import pytest

import oracle
from tma_pipelined_tensor_gb300 import inputs as gen
from tma_pipelined_tensor_gb300 import tg

from gpu_util import assert_within, gemm_bound, to_device_bf16

pytestmark = pytest.mark.gpu

M, N, K = 1100, 1300, 2000
PER_THREAD = ctypes.c_void_p(2)   # cudaStreamPerThread


def _problem(seed):
    A = gen.bf16_matrix(M, K, seed, 0, "normal")
    B = gen.bf16_matrix(N, K, seed, 1, "normal")
    ref, mag = oracle.gemm(A, B, M, N, K)
    return A, B, ref, gemm_bound(ref, mag, K, 1.0, 0.0, None, False)


def _gemm(Ad, Bd, Cd, cfg, stream):
    return tg.gemm_bf16_ex(M, N, K, Ad.data_ptr(), K, Bd.data_ptr(), K, Cd.data_ptr(), N, 1.0,
                           0.0, tg.TG_C_F32, cfg, stream)


def test_two_host_threads_on_the_per_thread_default_stream():
    """Two host threads, each on its own per-thread default stream (the same handle),
    run stream-K GEMMs at the same time: each gets a workspace of its own."""
    import torch
    cfg = tg.make_config(schedule=2)
    probs = [_problem(seed) for seed in (61, 62)]
    dev = [(to_device_bf16(A), to_device_bf16(B),
            torch.full((M, N), np.nan, dtype=torch.float32, device="cuda")) for A, B, _, _ in probs]
    torch.cuda.synchronize()
    results = [None, None]

    def worker(i):
        Ad, Bd, Cd = dev[i]
        sts = [_gemm(Ad, Bd, Cd, cfg, PER_THREAD) for _ in range(6)]
        sync = tg.tg_status_sync(PER_THREAD)
        st, plan = tg.tg_gemm_last_plan()
        results[i] = (sts, sync, st, plan.sk_iters, plan.workspace, plan.sk_fallback)

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    torch.cuda.synchronize()
    for i, (sts, sync, st, sk, ws, fb) in enumerate(results):
        assert all(s == tg.TG_OK for s in sts) and sync == tg.TG_OK and st == tg.TG_OK, (
            i, [tg.tg_status_string(s) for s in sts], tg.tg_status_string(sync), st)
        # stream-K ran on the library's workspace (the per-thread streams of a fresh
        # process are among the first 16 streams to ask for one)
        assert sk > 0 and fb == 0 and ws == 1, (i, sk, fb, ws)
        _, _, ref, bound = probs[i]
        assert_within(dev[i][2].cpu().numpy().astype(np.float64), ref, bound, "thread %d" % i)


def test_caller_owned_workspace():
    import torch
    A, B, ref, bound = _problem(63)
    Ad, Bd = to_device_bf16(A), to_device_bf16(B)
    cfg = tg.make_config(schedule=2)
    st, plan = tg.tg_gemm_plan_for(M, N, K, tg.TG_C_F32, cfg, 0)
    assert st == tg.TG_OK and plan.sk_iters > 0 and plan.workspace_bytes > 0
    need = plan.workspace_bytes
    ws = torch.zeros(need + 256, dtype=torch.uint8, device="cuda")    # zero-filled once
    Cd = torch.full((M, N), np.nan, dtype=torch.float32, device="cuda")
    # too small: refused before launch
    small = tg.make_config(schedule=2, workspace=ws.data_ptr(), workspace_bytes=need - 16)
    assert _gemm(Ad, Bd, Cd, small, None) == tg.TG_ERR_BUFFER_TOO_SMALL
    # host memory as the workspace: refused
    host = torch.zeros(need, dtype=torch.uint8, pin_memory=True)
    hcfg = tg.make_config(schedule=2, workspace=host.data_ptr(), workspace_bytes=need)
    assert _gemm(Ad, Bd, Cd, hcfg, None) == tg.TG_ERR_INVALID_VALUE
    torch.cuda.synchronize()
    assert bool(torch.isnan(Cd).all())
    # the right size, three launches in a row on the same workspace
    good = tg.make_config(schedule=2, workspace=ws.data_ptr(), workspace_bytes=need)
    for _ in range(3):
        Cd.fill_(np.nan)
        assert _gemm(Ad, Bd, Cd, good, None) == tg.TG_OK
        st, last = tg.tg_gemm_last_plan()
        assert st == tg.TG_OK and last.workspace == 2 and last.sk_iters == plan.sk_iters
        assert tg.tg_status_sync(None) == tg.TG_OK
        assert_within(Cd.cpu().numpy().astype(np.float64), ref, bound, "caller workspace")
    assert bool((ws[need:] == 0).all())      # nothing written past the stated size


_CHILD = r"""
import ctypes, json, sys
sys.path[:0] = sys.argv[1:3]
import numpy as np, torch
import oracle
from tma_pipelined_tensor_gb300 import inputs as gen, tg
M, N, K = %d, %d, %d
A = gen.bf16_matrix(M, K, 64, 0, "normal")
B = gen.bf16_matrix(N, K, 64, 1, "normal")
ref, mag = oracle.gemm(A, B, M, N, K)
bound = 2.0 * K * 2.0 ** -24 * mag
to_dev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
Ad, Bd = to_dev(A), to_dev(B)
cfg = tg.make_config(schedule=2)
# torch hands out streams from a pool of 32 per priority: 40 requests cover it
streams = [torch.cuda.Stream() for _ in range(40)]
outs = [torch.full((M, N), np.nan, dtype=torch.float32, device="cuda") for _ in streams]
torch.cuda.synchronize()
seen, bad = {}, []
for s, Cd in zip(streams, outs):
    st = tg.gemm_bf16_ex(M, N, K, Ad.data_ptr(), K, Bd.data_ptr(), K, Cd.data_ptr(), N, 1.0, 0.0,
                         tg.TG_C_F32, cfg, ctypes.c_void_p(s.cuda_stream))
    lst, last = tg.tg_gemm_last_plan()
    if st != 0 or lst != 0:
        bad.append("status %%d %%d" %% (st, lst))
    if last.sk_fallback:
        if not (last.sk_fallback == 1 and last.sk_iters == 0 and last.workspace == 0):
            bad.append("fallback plan %%d %%d %%d" %% (last.sk_fallback, last.sk_iters, last.workspace))
    elif not (last.sk_iters > 0 and last.workspace == 1):
        bad.append("stream-K plan %%d %%d" %% (last.sk_iters, last.workspace))
    seen[s.cuda_stream] = last.sk_fallback
torch.cuda.synchronize()
sync = tg.tg_status_sync(None)
within = [bool((np.abs(Cd.cpu().numpy().astype(np.float64) - ref) <= bound).all()) for Cd in outs]
print(json.dumps({"streams": len(seen), "with_ws": sum(1 for f in seen.values() if f == 0),
                  "fallbacks": sum(1 for f in seen.values() if f == 1), "bad": bad,
                  "sync": sync, "within": all(within)}))
""" % (M, N, K)


def test_seventeenth_stream_falls_back_and_says_so():
    """At most 16 streams of a device hold a library workspace; a stream-K GEMM on any
    further stream runs with whole tiles, correctly, and tg_gemm_last_plan reports it.
    Run in a child process: the workspaces it creates last until that process exits and
    would otherwise take the stream-K schedule away from later tests' streams."""
    import json
    import os
    import subprocess
    import sys
    here = os.path.dirname(os.path.abspath(__file__))
    root = os.path.dirname(here)
    r = subprocess.run([sys.executable, "-c", _CHILD, root, here], capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    res = json.loads(r.stdout.strip().splitlines()[-1])
    assert res["bad"] == [] and res["sync"] == tg.TG_OK and res["within"], res
    assert res["streams"] > 16
    assert 0 < res["with_ws"] <= 16 and res["fallbacks"] >= res["streams"] - 16, res


@pytest.mark.parametrize("own_workspace", [False, True])
def test_capture_runs_stream_k_only_with_a_caller_workspace(own_workspace):
    """Inside a stream capture the library neither allocates nor looks up a stream's
    workspace (asking a capturing stream for its ID would invalidate the capture): a
    stream-K GEMM is captured with whole tiles (reported as sk_fallback 2), or with
    stream-K when the caller passes a workspace; either graph replays a correct product."""
    import torch
    A, B, ref, bound = _problem(65)
    Ad, Bd = to_device_bf16(A), to_device_bf16(B)
    Cd = torch.full((M, N), np.nan, dtype=torch.float32, device="cuda")
    cfg = tg.make_config(schedule=2)
    ws = None
    if own_workspace:
        _, plan = tg.tg_gemm_plan_for(M, N, K, tg.TG_C_F32, cfg, 0)
        ws = torch.zeros(plan.workspace_bytes, dtype=torch.uint8, device="cuda")
        cfg = tg.make_config(schedule=2, workspace=ws.data_ptr(), workspace_bytes=ws.numel())
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        st = _gemm(Ad, Bd, Cd, cfg, ctypes.c_void_p(s.cuda_stream))
        last_st, last = tg.tg_gemm_last_plan()
    assert st == tg.TG_OK and last_st == tg.TG_OK
    if own_workspace:
        assert last.workspace == 2 and last.sk_iters > 0 and last.sk_fallback == 0
    else:
        assert last.sk_fallback == 2 and last.sk_iters == 0 and last.workspace == 0
    for _ in range(2):
        Cd.fill_(np.nan)
        g.replay()
        torch.cuda.synchronize()
        assert tg.tg_status_sync(None) == tg.TG_OK
        assert_within(Cd.cpu().numpy().astype(np.float64), ref, bound, "graph replay")
