"""bench.py refuses, before anything touches a GPU, the launches it does not make: a
world size other than --gpus, and the per-CTA kernel's cluster-multicast load on more
than one rank (that load is a single-GPU option; "2 . Le Tensor Memory Accelerator" 2.5
describes multicast within one GPU's cluster)."""
import subprocess
import sys
import os

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_world_size_must_match_gpus():
    assert bench.check_launch(bench.parse_args([]), 1) is None
    assert bench.check_launch(bench.parse_args(["--gpus", "8"]), 8) is None
    assert "WORLD_SIZE" in bench.check_launch(bench.parse_args(["--gpus", "2"]), 1)
    assert "WORLD_SIZE" in bench.check_launch(bench.parse_args(["--gpus", "1"]), 4)
    assert bench.check_launch(bench.parse_args(["--gpus", "0"]), 1) is not None


def test_multicast_is_refused_on_more_than_one_rank():
    mc = ["--cluster", "2", "--mma", "1"]
    assert bench.check_launch(bench.parse_args(mc), 1) is None            # one GPU: allowed
    err = bench.check_launch(bench.parse_args(["--gpus", "2"] + mc), 2)
    assert err is not None and "multicast" in err
    # a cluster of two without per-CTA MMAs is the CTA-pair kernel: no multicast load
    assert bench.check_launch(bench.parse_args(["--gpus", "2", "--cluster", "2"]), 2) is None
    assert bench.check_launch(bench.parse_args(["--gpus", "2", "--mma", "1"]), 2) is None


def test_refusal_exits_non_zero_before_any_gpu_work():
    # two "ranks" as seen through the environment, multicast requested: the process must
    # stop with an error before it imports torch or touches a device
    env = dict(os.environ, WORLD_SIZE="2", RANK="0", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2",
                        "--cluster", "2", "--mma", "1"], env=env, capture_output=True,
                       text=True, timeout=120)
    assert r.returncode != 0
    assert "multicast" in r.stderr
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "3"],
                       env=dict(os.environ, WORLD_SIZE="1"), capture_output=True, text=True,
                       timeout=120)
    assert r.returncode != 0 and "WORLD_SIZE" in r.stderr
