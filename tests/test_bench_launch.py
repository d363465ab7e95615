"""bench.py's launch contract on the CPU: it drives one GPU from one process.

The expert GEMMs use cluster multicast, which belongs to one-GPU calls only,
so a multi-process launch (WORLD_SIZE > 1) or --gpus other than 1 must fail
loudly for our arm instead of running replicas; the reference arm (the float64
oracle on the host cores) runs on rank 0 of such a launch and the other ranks
exit 0 without work.  Also the host-side helpers that turn the run's clocks
and the kernels' stamps into the bench line's numbers."""
from __future__ import annotations

import os
import subprocess
import sys

import numpy as np
import torch

import bench
import sparse_mixture_experts_55_b300 as moe

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench(args, **env):
    e = dict(os.environ, **{k: str(v) for k, v in env.items()})
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], capture_output=True, text=True,
                          env=e, timeout=300, cwd=ROOT)


def test_multi_process_launch_is_refused():
    r = _bench(["--steps", "1", "--warmup", "1"], WORLD_SIZE=2, RANK=0, LOCAL_RANK=0)
    assert r.returncode != 0
    assert "refusing" in r.stderr and r.stdout == ""


def test_more_than_one_gpu_is_refused():
    r = _bench(["--gpus", "2", "--steps", "1", "--warmup", "1"])
    assert r.returncode != 0
    assert "refusing" in r.stderr and r.stdout == ""


def test_reference_arm_off_rank_zero_exits_without_work():
    r = _bench(["--impl", "reference", "--steps", "1", "--warmup", "1"], WORLD_SIZE=2, RANK=1, LOCAL_RANK=1)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


def test_peak_follows_the_run_clocks():
    peaks = {"bf16_tflops": 1755.4, "bf16_tflops_sustained": 1377.5, "hbm_gbs": 6484.9}
    p, kind, _ = bench.tensor_peak(peaks, {"sm_mhz": 2032, "sm_max_mhz": 2032, "reasons": []})
    assert (p, kind) == (1755.4, "burst")
    p, kind, _ = bench.tensor_peak(peaks, {"sm_mhz": 2032, "sm_max_mhz": 2032, "reasons": ["sw_power_cap"]})
    assert (p, kind) == (1377.5, "sustained")
    p, kind, _ = bench.tensor_peak(peaks, {"sm_mhz": 1500, "sm_max_mhz": 2032, "reasons": []})
    assert kind == "sustained"
    p, kind, _ = bench.tensor_peak(peaks, {"sm_mhz": 2000, "sm_max_mhz": 2032, "reasons": []}, ratio=2.0)
    assert (p, kind) == (2 * 1755.4, "burst")


def test_stage_stats_from_stamps():
    n = moe._lib.MOE_NUM_STAGES
    never = np.iinfo(np.uint64).max
    rows = []
    for base in (10_000_000, 20_000_000):
        b = np.full(n, never, dtype=np.uint64)
        e = np.zeros(n, dtype=np.uint64)
        # route 10 us, group 5 us, gather 5 us, gate/up 1 ms, down 0.5 ms; 2 us gaps
        spans = {0: (0, 10_000), 1: (12_000, 17_000), 2: (19_000, 24_000), 3: (26_000, 1_026_000),
                 5: (1_028_000, 1_528_000)}
        for s, (lo, hi) in spans.items():
            b[s], e[s] = base + lo, base + hi
        rows.append(np.concatenate([b, e]).view(np.int64))
    stamps = torch.from_numpy(np.stack(rows))
    stages, span, gaps = bench.stage_stats(moe, stamps, 2)
    assert set(stages) == {"route", "group", "gather", "gate_up_gemm", "down_gemm"}
    assert abs(stages["gate_up_gemm"] - 1.0) < 1e-12 and abs(stages["down_gemm"] - 0.5) < 1e-12
    assert abs(span - 1.528) < 1e-12
    assert abs(gaps - 0.008) < 1e-12


def test_exclusive_spans_clip_overlap():
    n = moe._lib.MOE_NUM_STAGES
    never = np.iinfo(np.uint64).max
    b = np.full(n, never, dtype=np.uint64)
    e = np.zeros(n, dtype=np.uint64)
    # gather 0-5 us; gate/up starts at 3 us (overlap 2 us) and ends at 100 us;
    # down starts at 90 us (overlap 10 us) and ends at 150 us
    for s_, (lo, hi) in {2: (0, 5_000), 3: (3_000, 100_000), 5: (90_000, 150_000)}.items():
        b[s_], e[s_] = 1_000_000 + lo, 1_000_000 + hi
    stamps = torch.from_numpy(np.concatenate([b, e]).view(np.int64)[None])
    stages, span, gaps = bench.stage_stats(moe, stamps, 1)
    excl = bench.exclusive_stage_ms(moe, stamps)
    assert abs(stages["down_gemm"] - 0.060) < 1e-12 and abs(excl["down_gemm"] - 0.050) < 1e-12
    assert abs(excl["gate_up_gemm"] - 0.095) < 1e-12 and abs(excl["gather"] - 0.005) < 1e-12
    assert abs(sum(excl.values()) - span) < 1e-12 and gaps < 0
