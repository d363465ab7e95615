"""Benchmark of the MoE layer forward on one B300: one JSON line.

    python bench.py [--gpus 1] [--steps K] [--warmup W] [--config prefill] [--impl ours|reference]

A step is one full forward pass of the layer (router, grouping, gather,
gate/up GEMM + SwiGLU, down GEMM x gate, combine) over one batch of seeded
synthetic tokens, with random-init Mixtral-shaped weights resident in HBM.
The run uses one GPU from one process; multi-process launches are refused.

  value        tokens/s, device-timed with CUDA events around K back-to-back
               forwards
  stages_ms    each kernel's span inside that same region, from the
               global-timer stamps every kernel writes (moe_forward_stamped)
  stages_exclusive_ms  the part of each span after the previous kernels
               ended (spans overlap under programmatic dependent launch)
  roofline     the gate/up expert GEMM (the dominant kernel): algorithmic
               FLOPs (or bytes at decode sizes) per launch over its in-run
               span, against MEASURED_PEAKS.json (burst or sustained peak as
               the run's own clocks say)
  decode       (prefill line) the decode batch sizes 1, 8, 32, 128 through the
               same weights: ms per step and achieved HBM bandwidth of the
               layer and of each expert GEMM
  e2e          the same metric through the C ABI with host buffers: pinned x
               copied in, the layer, y copied out, every step
  cpu_baseline the float64 oracle on a token sample, timed on the host cores
  --impl reference   the oracle alone, timed on the host cores
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import math
import os
import pathlib
import re
import statistics
import sys
import threading
import time

ROOT = pathlib.Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

import torch  # noqa: E402

import workloads as W  # noqa: E402

METRIC = "MoE layer tokens/s and TFLOP/s (% bf16 peak; % HBM BW at decode) on 1 B300"
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}

CONFIGS = {
    "prefill": dict(T=4096, d=4096, f=14336, E=8, K=2),
    "decode1": dict(T=1, d=4096, f=14336, E=8, K=2),
    "decode8": dict(T=8, d=4096, f=14336, E=8, K=2),
    "decode32": dict(T=32, d=4096, f=14336, E=8, K=2),
    "decode128": dict(T=128, d=4096, f=14336, E=8, K=2),
    "skew": dict(T=16384, d=4096, f=14336, E=8, K=2),
    "stack32": dict(T=8192, d=4096, f=14336, E=8, K=2, layers=32),
    # profiling stand-in: two experts of Mixtral size with ~1024 rows each, the
    # per-expert GEMM shape of the prefill layer at a quarter of its memory
    "prefill_e2": dict(T=1024, d=4096, f=14336, E=2, K=2),
    # training step of the prefill layer: forward keeping activations + backward
    "train": dict(T=4096, d=4096, f=14336, E=8, K=2, train=True),
    # decode with the expert banks in pinned host memory and C device slots
    # (LRU), over a trace with the pages' temporal locality, or without it
    "decode1_cache": dict(T=1, d=4096, f=14336, E=8, K=2, cache_slots=4, keep=0.35),
    "decode1_cache_nolocality": dict(T=1, d=4096, f=14336, E=8, K=2, cache_slots=4, keep=0.0),
    # profiling stand-in of the training step: two Mixtral-sized experts with ~1024 rows each
    "train_e2": dict(T=1024, d=4096, f=14336, E=2, K=2, train=True),
}
# the same workloads with e4m3 expert weights (quantised once, untimed)
for _n in ("prefill", "decode1", "decode8", "decode32", "decode128", "skew"):
    CONFIGS[_n + "_fp8"] = dict(CONFIGS[_n], fp8=True)
WORKLOAD_TEXT = {
    "prefill": "Mixtral-shaped MoE layer prefill: T=4096 tokens, d=4096, f=14336, E=8 experts, top-2, bf16, "
               "fp32 accumulate",
    "skew": "skewed-routing MoE layer: T=16384, d=4096, f=14336, E=8, top-2, Zipf(1.2) expert loads, bf16",
}
WORKLOAD_TEXT["stack32"] = ("32-layer attention-free MoE stack h <- h + MoE_l(RMSNorm(h)): T=8192 tokens, "
                            "d=4096, f=14336, E=8, top-2, bf16, own seeded weights per layer (90.2 GB resident)")
WORKLOAD_TEXT["train"] = ("Mixtral-shaped MoE layer training step (forward keeping activations, then backward to "
                          "dx, dWg, dW1, dW3, dW2 in fp32): T=4096 tokens, d=4096, f=14336, E=8, top-2, bf16")
WORKLOAD_TEXT["train_e2"] = ("profiling stand-in of the training step: T=1024 tokens, d=4096, f=14336, E=2 experts, "
                             "top-2, bf16")
for _n, _k in (("decode1_cache", "65% of consecutive tokens sharing an expert, as the pages' Table 5"),
               ("decode1_cache_nolocality", "independent routing, ~46% sharing by chance")):
    WORKLOAD_TEXT[_n] = ("Mixtral-shaped MoE layer decode, one token per step, expert banks in pinned host memory "
                         f"with 4 of 8 experts cached on the GPU (LRU); routing trace: {_k}; bf16")
CACHE_METRIC = "MoE layer decode tokens/s with experts offloaded to host memory (4 of 8 cached) on 1 B300"
TRAIN_METRIC = "MoE layer training tokens/s (forward + backward) and TFLOP/s on 1 B300"
WORKLOAD_TEXT["prefill_e2"] = "profiling stand-in: T=1024 tokens, d=4096, f=14336, E=2 experts, top-2, bf16"
for _t in (1, 8, 32, 128):
    WORKLOAD_TEXT[f"decode{_t}"] = f"Mixtral-shaped MoE layer decode batch: T={_t} tokens, d=4096, f=14336, " \
                                   f"E=8, top-2, bf16 (weight-streaming)"
for _n in ("prefill", "decode1", "decode8", "decode32", "decode128", "skew"):
    WORKLOAD_TEXT[_n + "_fp8"] = WORKLOAD_TEXT[_n].replace("bf16", "e4m3 expert weights (per-column scales), " \
                                                           "bf16 tokens")


# ---------------------------------------------------------------------------
def load_peaks():
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        try:
            d = json.loads(p.read_text())
            return {k: float(d[k]) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained")}, "measured"
        except Exception:
            pass
    return dict(FALLBACK_PEAKS), "fallback"


def code_sha256(path: pathlib.Path) -> str:
    """sha256 of a C++/CUDA source with its // comments, trailing blanks and
    empty lines removed: it changes when the code does, not when a comment
    does (the kernel sources hold no // inside string literals)."""
    lines = []
    for line in path.read_text().splitlines():
        code = line.split("//", 1)[0].rstrip()
        if code:
            lines.append(code)
    return hashlib.sha256("\n".join(lines).encode()).hexdigest()


def traffic_from_profiles(kernel_file: pathlib.Path, key: str, summary: str = "gate_up_gemm_traffic.md"):
    """dram bytes per launch recorded by an ncu capture (profiles/<summary>), if
    the kernel's code is unchanged since (code_sha256)."""
    prof = ROOT / "profiles" / summary
    if not prof.exists():
        return None
    text = prof.read_text()
    m_sha = re.search(r"code_sha256:\s*([0-9a-f]{64})", text)
    m_val = re.search(rf"{key}:\s*([0-9.eE+]+)", text)
    if not m_sha or not m_val:
        return None
    return float(m_val.group(1)) if code_sha256(kernel_file) == m_sha.group(1) else None


class _CtypesNVML:
    """Minimal NVML binding over libnvidia-ml.so.1 (for hosts without pynvml)."""
    SOURCE = "nvml-ctypes"
    NVML_CLOCK_SM = 1

    def __init__(self):
        import ctypes
        self.ct = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")

    def _ok(self, rc, what):
        if rc != 0:
            raise RuntimeError(f"{what} returned {rc}")

    def nvmlInit(self):
        self._ok(self.lib.nvmlInit_v2(), "nvmlInit_v2")

    def nvmlDeviceGetHandleByUUID(self, uuid):
        h = self.ct.c_void_p()
        self._ok(self.lib.nvmlDeviceGetHandleByUUID(uuid.encode(), self.ct.byref(h)), "GetHandleByUUID")
        return h

    def nvmlDeviceGetHandleByIndex(self, i):
        h = self.ct.c_void_p()
        self._ok(self.lib.nvmlDeviceGetHandleByIndex_v2(self.ct.c_uint(i), self.ct.byref(h)), "GetHandleByIndex")
        return h

    def _uint(self, fn, h, *args):
        v = self.ct.c_uint()
        self._ok(getattr(self.lib, fn)(h, *args, self.ct.byref(v)), fn)
        return v.value

    def nvmlDeviceGetClockInfo(self, h, kind):
        return self._uint("nvmlDeviceGetClockInfo", h, self.ct.c_int(kind))

    def nvmlDeviceGetMaxClockInfo(self, h, kind):
        return self._uint("nvmlDeviceGetMaxClockInfo", h, self.ct.c_int(kind))

    def nvmlDeviceGetPowerUsage(self, h):
        return self._uint("nvmlDeviceGetPowerUsage", h)

    def nvmlDeviceGetCurrentClocksEventReasons(self, h):
        v = self.ct.c_ulonglong()
        fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(self.lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
        self._ok(fn(h, self.ct.byref(v)), "GetCurrentClocksEventReasons")
        return v.value


def _nvml_module():
    try:
        import pynvml
        return pynvml
    except ImportError:
        return _CtypesNVML()


class ClockSampler:
    """Samples SM clock, power and clock-event reasons while the timed region runs.

    Uses NVML (pynvml) when it imports, else a background
    ``nvidia-smi --query-gpu=... -lms 20`` process whose CSV lines are parsed
    as they arrive.  The sampler is started before the timed region and waits
    for its first sample, so the samples cover that region."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown", 0x2: "applications_clocks_setting",
               0x10: "sync_boost"}
    SMI_FIELDS = ("clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active")

    def __init__(self, device_index: int, period_s: float = 0.005):
        self.samples = []
        self.reasons = set()
        self.ok = False
        self.max_mhz = None
        self.source = None
        self._stop = threading.Event()
        self.period = period_s
        self._proc = None
        self.err = None
        try:
            self.uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            if not self.uuid.startswith("GPU-"):
                self.uuid = "GPU-" + self.uuid
        except Exception:
            self.uuid = None
        self._first = threading.Event()
        try:
            self.nv = _nvml_module()
            self.nv.nvmlInit()
            h = None
            try:
                h = self.nv.nvmlDeviceGetHandleByUUID(self.uuid)
            except Exception:
                h = None
            if h is None:
                vis = os.environ.get("CUDA_VISIBLE_DEVICES")
                idx = int(vis.split(",")[device_index]) if vis and vis.split(",")[0].isdigit() else device_index
                h = self.nv.nvmlDeviceGetHandleByIndex(idx)
            self.h = h
            self.max_mhz = self.nv.nvmlDeviceGetMaxClockInfo(h, self.nv.NVML_CLOCK_SM)
            self._reasons_fn = getattr(self.nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                getattr(self.nv, "nvmlDeviceGetCurrentClocksThrottleReasons")
            self.ok = True
            self.source = getattr(self.nv, "SOURCE", "pynvml")
            self._t = threading.Thread(target=self._run_nvml, daemon=True)
        except Exception as e:
            self.err = f"nvml: {e!r}"
            import shutil
            if shutil.which("nvidia-smi"):
                self.ok = True
                self.source = "nvidia-smi"
                self._t = threading.Thread(target=self._run_smi, daemon=True)

    def _add(self, sm, pw, reasons_mask):
        self.samples.append((sm, pw))
        for bit, name in self.REASONS.items():
            if reasons_mask & bit:
                self.reasons.add(name)
        self._first.set()

    def _run_nvml(self):
        while not self._stop.is_set():
            try:
                sm = self.nv.nvmlDeviceGetClockInfo(self.h, self.nv.NVML_CLOCK_SM)
                r = self._reasons_fn(self.h)
                pw = self.nv.nvmlDeviceGetPowerUsage(self.h) / 1000.0
                self._add(sm, pw, r)
            except Exception:
                pass
            time.sleep(self.period)

    def _run_smi(self):
        import subprocess
        cmd = ["nvidia-smi", "--query-gpu=" + ",".join(self.SMI_FIELDS), "--format=csv,noheader,nounits",
               "-lms", "20"]
        if self.uuid:
            cmd += ["-i", self.uuid]
        try:
            self._proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception as e:
            self.err = f"nvidia-smi: {e!r}"
            self._first.set()
            return
        for line in self._proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 4:
                continue
            try:
                sm, mx = float(parts[0]), float(parts[1])
                pw = float(parts[2]) if parts[2] not in ("[N/A]", "N/A") else float("nan")
                mask = int(parts[3], 16) if parts[3].startswith("0x") else 0
            except ValueError:
                continue
            self.max_mhz = mx
            self._add(sm, pw, mask)
            if self._stop.is_set():
                break

    def __enter__(self):
        if self.ok:
            self._t.start()
            self._first.wait(timeout=10.0)   # the first sample precedes the timed region
        return self

    def __exit__(self, *a):
        self._stop.set()
        if self._proc is not None:
            self._proc.terminate()
        if self.ok:
            self._t.join(timeout=10.0)

    def summary(self):
        if not self.ok or not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [], "samples": 0,
                    "note": self.err or "no samples"}
        sms = [s for s, _ in self.samples]
        pws = [p for _, p in self.samples if p == p]
        out = {"sm_mhz": statistics.median(sms), "sm_max_mhz": self.max_mhz, "reasons": sorted(self.reasons),
               "samples": len(sms), "source": self.source}
        if pws:
            out["power_w_max"] = round(max(pws), 1)
        return out


# ---------------------------------------------------------------------------
def launch_rank(args) -> int:
    """This benchmark drives one GPU from one process.  The layer shards by
    tokens with no exchange, so N GPUs would be N independent replicas; this
    build runs none: the expert GEMMs use cluster multicast, which is for
    one-GPU calls only.  A multi-process launch (WORLD_SIZE > 1) or --gpus
    other than 1 is refused for our arm.  The reference arm (the oracle on the
    host cores, no GPU kernel of this library) runs on rank 0 of such a launch
    and the other ranks exit without work.  Returns this process's rank."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        return rank
    if world != 1 or args.gpus != 1:
        sys.stderr.write(f"bench.py: refusing --gpus {args.gpus} with WORLD_SIZE={world}: this build runs one GPU "
                         "per process and no multi-GPU path\n")
        sys.exit(2)
    return rank


def tensor_peak(peaks, clocks, ratio: float = 1.0):
    """The tensor roofline that matches the run's own clocks: the burst peak
    when the median SM clock under load stayed within 3% of its maximum with no
    power-cap event, else the sustained (power-capped) peak.  ratio scales the
    measured bf16 figures (2 for e4m3, the nominal dense-rate ratio).  Returns
    (peak, kind, reason)."""
    sm, mx = clocks.get("sm_mhz"), clocks.get("sm_max_mhz")
    capped = "sw_power_cap" in (clocks.get("reasons") or [])
    if sm and mx and sm >= 0.97 * mx and not capped:
        return (peaks["bf16_tflops"] * ratio, "burst",
                f"median SM clock {sm:.0f} MHz of {mx:.0f} MHz with no power cap during the timed region")
    why = "sw_power_cap active" if capped else f"median SM clock {sm} MHz below its maximum {mx}"
    return peaks["bf16_tflops_sustained"] * ratio, "sustained", f"{why} during the timed region"


def stage_stats(moe, stamps, steps: int):
    """Per-stage mean kernel span (ms) over the stamped steps, the mean span
    from the first kernel's start to the last kernel's end of a step, and the
    launch gaps (step span minus the sum of the stage spans)."""
    spans = moe.stage_spans(stamps)
    names = [n for n in moe._lib.STAGES if any(n in s for s in spans)]
    out = {n: statistics.mean((s[n][1] - s[n][0]) / 1e6 for s in spans if n in s) for n in names}
    step = statistics.mean((max(e for _, e in s.values()) - min(b for b, _ in s.values())) / 1e6 for s in spans)
    return out, step, step - sum(out.values())


def exclusive_stage_ms(moe, stamps) -> dict:
    """Per-stage mean exclusive span (ms): a kernel's end minus the later of
    its own start and the latest end among the kernels that started before
    it.  With programmatic dependent launch a kernel starts (and issues its
    weight copies) while the previous one drains, so the raw spans overlap;
    the exclusive spans are what each kernel adds to the step and sum to the
    step span less the launch gaps."""
    acc: dict = {}
    for s in moe.stage_spans(stamps):
        done = None
        for name, (b, e) in sorted(s.items(), key=lambda kv: kv[1][0]):
            lo = b if done is None else max(b, done)
            acc.setdefault(name, []).append(max(0, e - lo) / 1e6)
            done = e if done is None else max(done, e)
    return {n: statistics.mean(v) for n, v in acc.items()}


def make_inputs(cfg_name: str, dev, weights=None):
    c = CONFIGS[cfg_name]
    cfg_name = cfg_name.replace("_fp8", "")
    if weights is None:
        weights = W.mixtral_weights(c["d"], c["f"], c["E"], seed=W.BASE_SEED, device=dev)
    if cfg_name in ("prefill", "prefill_e2", "train", "train_e2"):
        return W.prefill(T=c["T"], seed=W.BASE_SEED, device=dev, weights=weights), weights
    if cfg_name.startswith("decode"):
        return W.decode(c["T"], seed=W.BASE_SEED, device=dev, weights=weights), weights
    if cfg_name == "skew":
        return W.skew(T=c["T"], seed=W.BASE_SEED, device=dev, weights=weights), weights
    raise ValueError(cfg_name)


def algorithmic(c, n_touched):
    """Per layer: FLOPs of the whole layer and of the gate/up GEMM; bytes of the
    whole layer and of the gate/up GEMM (touched experts' weights once, one
    byte per weight with e4m3 weights, plus their scales)."""
    T, d, f, E, K = c["T"], c["d"], c["f"], c["E"], c["K"]
    wb = 1 if c.get("fp8") else 2
    scales = (3 * f * 4 + d * 4) if c.get("fp8") else 0            # fp32 column scales per expert
    flops = T * K * 6 * d * f + 2 * T * d * E
    gate_up_flops = T * K * 4 * d * f
    bytes_step = n_touched * (3 * d * f * wb + scales) + 2 * d * E + 2 * T * d * 2
    gate_up_bytes = n_touched * (2 * d * f * wb + 2 * f * 4)
    return flops, gate_up_flops, bytes_step, gate_up_bytes


def down_bytes(c, n_touched):
    """Algorithmic bytes of the down GEMM: each touched expert's W2 once (e4m3:
    one byte per weight plus the fp32 column scales)."""
    d, f = c["d"], c["f"]
    return n_touched * (f * d * (1 if c.get("fp8") else 2) + (d * 4 if c.get("fp8") else 0))


# ---------------------------------------------------------------------------
def f64_banks(inp):
    """Host float64 copies of the router and expert banks, filled one expert at a time."""
    import numpy as np
    E, d, f = inp.W1.shape
    Wg = inp.Wg.float().cpu().numpy().astype(np.float64)
    W1 = np.empty((E, d, f)); W3 = np.empty((E, d, f)); W2 = np.empty((E, f, d))
    for e in range(E):
        W1[e] = inp.W1[e].float().cpu().numpy()
        W3[e] = inp.W3[e].float().cpu().numpy()
        W2[e] = inp.W2[e].float().cpu().numpy()
    return Wg, W1, W3, W2


def blas_threads() -> int:
    """Threads the oracle's BLAS runs with (threadpoolctl if present, else the CPU affinity set)."""
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 1) for i in threadpool_info() if i.get("internal_api") == "openblas"]
        if n:
            return max(n)
    except Exception:
        pass
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        if os.environ.get(var, "").isdigit():
            return int(os.environ[var])
    return len(os.sched_getaffinity(0))


def cpu_oracle_rate(inp, n_tokens: int):
    """Time the unchanged float64 oracle on the first n_tokens tokens of the batch.
    Weights are copied to the host and upcast once, before timing.  Returns
    the rate, the time, the threads and the oracle's output on those tokens."""
    import numpy as np
    import oracle
    x = inp.x[:n_tokens].float().cpu().numpy().astype(np.float64)
    Wg, W1, W3, W2 = f64_banks(inp)
    t0 = time.perf_counter()
    ref = oracle.moe_layer(x, Wg, W1, W3, W2, inp.K)
    dt = time.perf_counter() - t0
    return n_tokens / dt, dt, blas_threads(), ref.y


def oracle_check(inp, idx_gpu, y_gpu, y_ref):
    """The bench line's parity record: the GPU output on the oracle's sampled
    tokens, and the routing of every token against the oracle's (tokens whose
    K-th/(K+1)-th logit gap is below 1e-3 are counted as near ties, not
    compared)."""
    import numpy as np
    import oracle
    x = inp.x.float().cpu().numpy().astype(np.float64)
    Wg = inp.Wg.float().cpu().numpy().astype(np.float64)
    g = oracle.gating(x, Wg, inp.K)
    gap_io, _ = oracle.logit_gaps(oracle.router_logits(x, Wg), inp.K)
    near = (gap_io > 0) & (gap_io < 1e-3)
    gpu = np.sort(np.asarray(idx_gpu), axis=1)
    ref = np.sort(g.idx, axis=1)
    mism = int(np.sum(np.any(gpu != ref, axis=1) & ~near))
    y = np.asarray(y_gpu, dtype=np.float64)
    err = float(np.abs(y - y_ref).max() / (np.abs(y_ref).max() + 1e-6))
    return {"tokens_checked": int(y_ref.shape[0]), "max_rel_err": err, "tolerance": 2e-2,
            "routing_tokens": int(x.shape[0]), "near_ties": int(near.sum()), "index_mismatches": mism}


def reference_line(args, c, value, ms, steps, warmup, sample, metric):
    return {"impl": "reference", "metric": metric, "value": value, "unit": "tokens/s", "n_gpus": 1,
            "steps": steps, "warmup": warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD_TEXT[args.config], **c},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": blas_threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def run_reference_stack(args, c, dev, steps, warmup):
    """stack32 reference arm: the float64 oracle's pre-norm block on a few
    tokens through layer 0 per step, scaled to the stack's layer count."""
    import numpy as np
    import oracle
    L, K = c["layers"], c["K"]
    Wg, W1, W3, W2 = W.stack_layer_weights(0, c["d"], c["f"], c["E"], device=dev)
    E = W1.shape[0]
    Wg64 = Wg.float().cpu().numpy().astype(np.float64)
    b1 = np.stack([W1[e].float().cpu().numpy() for e in range(E)]).astype(np.float64)
    b3 = np.stack([W3[e].float().cpu().numpy() for e in range(E)]).astype(np.float64)
    b2 = np.stack([W2[e].float().cpu().numpy() for e in range(E)]).astype(np.float64)
    del W1, W3, W2
    h0 = W.stack_h0(c["T"], c["d"], device=dev).float().cpu().numpy().astype(np.float64)
    per_step_budget_s = min(2.0, 150.0 / (steps + warmup))
    n_tok = max(1, min(c["T"], int(per_step_budget_s / 0.02)))
    times = []
    for i in range(warmup + steps):
        lo = (i * n_tok) % max(1, c["T"] - n_tok + 1)
        t0 = time.perf_counter()
        oracle.moe_block(h0[lo:lo + n_tok], Wg64, b1, b3, b2, K)
        dt = time.perf_counter() - t0
        if i >= warmup:
            times.append(dt)
    ms = 1e3 * L * sum(times) / len(times)        # one step = all layers of the stack
    value = n_tok / (ms / 1e3)
    sample = (f"{n_tok} tokens per step through layer 0's pre-norm block, time scaled by {L} layers "
              f"(weights upcast to float64 once, untimed)")
    print(json.dumps(reference_line(args, c, value, ms, steps, warmup, sample, METRIC)), flush=True)


def run_reference(args, rank):
    """The oracle as the reference arm: host cores only, bounded sample per step."""
    if rank != 0:
        return
    import numpy as np
    import oracle
    c = CONFIGS[args.config]
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    steps, warmup = args.steps, max(args.warmup, 3)
    if args.config == "stack32":
        return run_reference_stack(args, c, dev, steps, warmup)
    inp, _ = make_inputs(args.config, dev)
    # sample per step: bounded so the whole run stays within a few minutes
    per_step_budget_s = min(2.0, 150.0 / (steps + warmup))
    n_tok = max(1, min(c["T"], int(per_step_budget_s / 0.02)))
    x = inp.x.float().cpu().numpy().astype(np.float64)
    Wg, W1, W3, W2 = f64_banks(inp)
    del inp
    train = bool(c.get("train"))
    if train:
        n_tok = max(1, n_tok // 3)  # the backward costs about twice the forward
        dy = W.randn((c["T"], c["d"]), 1.0, W.BASE_SEED + 77, "cpu").numpy().astype(np.float64)
    times = []
    for i in range(warmup + steps):
        lo = (i * n_tok) % max(1, c["T"] - n_tok + 1)
        t0 = time.perf_counter()
        oracle.moe_layer(x[lo:lo + n_tok], Wg, W1, W3, W2, c["K"])
        if train:
            oracle.moe_layer_backward(x[lo:lo + n_tok], Wg, W1, W3, W2, c["K"], dy[lo:lo + n_tok])
        dt = time.perf_counter() - t0
        if i >= warmup:
            times.append(dt)
    ms = 1e3 * sum(times) / len(times)
    value = n_tok / (ms / 1e3)
    sample = f"{n_tok} tokens of the {args.config} batch per step (weights upcast to float64 once, untimed)"
    metric = TRAIN_METRIC if train else (CACHE_METRIC if "cache_slots" in c else METRIC)
    print(json.dumps(reference_line(args, c, value, ms, steps, warmup, sample, metric)), flush=True)


# ---------------------------------------------------------------------------
def oracle_block_rate(h_rows, layer_weights, K: int):
    """Time the unchanged float64 oracle on one pre-norm block (RMSNorm, MoE,
    residual) for the given rows; the layer's banks are upcast once, untimed."""
    import numpy as np
    import oracle
    Wg, W1, W3, W2 = layer_weights
    E = W1.shape[0]
    Wg64 = Wg.float().cpu().numpy().astype(np.float64)
    W164 = np.stack([W1[e].float().cpu().numpy() for e in range(E)]).astype(np.float64)
    W364 = np.stack([W3[e].float().cpu().numpy() for e in range(E)]).astype(np.float64)
    W264 = np.stack([W2[e].float().cpu().numpy() for e in range(E)]).astype(np.float64)
    h = h_rows.float().cpu().numpy().astype(np.float64)
    t0 = time.perf_counter()
    oracle.moe_block(h, Wg64, W164, W364, W264, K)
    return time.perf_counter() - t0


def run_ours_stack(args):
    """stack32: a step is one pass of h0 through all layers of the stack, each
    layer a stamped pre-norm block (per-layer stage spans from the same run)."""
    import sparse_mixture_experts_55_b300 as moe
    from sparse_mixture_experts_55_b300 import build as _build
    _build.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    c = CONFIGS[args.config]
    T, d, f, E, K, L = c["T"], c["d"], c["f"], c["E"], c["K"], c["layers"]
    layers = [W.stack_layer_weights(l, d, f, E, device=dev) for l in range(L)]
    h0 = W.stack_h0(T, d, device=dev)
    ws = moe.Workspace(T, d, f, E, K, torch.bfloat16, dev)
    h = torch.empty_like(h0)
    stream = torch.cuda.current_stream(dev)
    steps, warmup = args.steps, max(args.warmup, 3)
    stamps = moe.new_stamps(steps * L, dev)

    def step(hbuf, i=None):
        hbuf.copy_(h0)
        for l in range(L):
            if i is None:
                moe.moe_block_forward(hbuf, *layers[l], K, workspace=ws, stream=stream)
            else:
                moe.moe_block_forward_stamped(hbuf, *layers[l], K, stamps[i * L + l], workspace=ws, stream=stream)

    for _ in range(warmup):
        step(h)
    torch.cuda.synchronize(dev)
    if moe.moe_read_status(ws) != 0:
        raise RuntimeError(f"device status {moe.moe_read_status(ws)}")
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    with ClockSampler(0) as clk:
        start.record(stream)
        for i in range(steps):
            step(h, i)
        end.record(stream)
        torch.cuda.synchronize(dev)
    ms = start.elapsed_time(end) / steps
    clocks = clk.summary()
    stage_ms, layer_span_ms, _ = stage_stats(moe, stamps, steps * L)

    # end to end with host buffers: h0 in, the whole stack, h out
    e2e_steps = max(2, min(steps, 5))
    h0_host = h0.cpu().pin_memory()
    h_host = torch.empty_like(h0_host).pin_memory()

    def step_host():
        with torch.cuda.stream(stream):
            h.copy_(h0_host, non_blocking=True)
            for l in range(L):
                moe.moe_block_forward(h, *layers[l], K, workspace=ws, stream=stream)
            h_host.copy_(h, non_blocking=True)

    step_host()
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        step_host()
    torch.cuda.synchronize(dev)
    e2e_ms = 1e3 * (time.perf_counter() - t0) / e2e_steps

    peaks, peak_src = load_peaks()
    flops_layer, gu_flops, _, _ = algorithmic(c, E)
    flops = L * (flops_layer + 4 * T * d)          # + RMSNorm (square, sum, scale, round) per layer
    peak, kind, why = tensor_peak(peaks, clocks)
    gu_ms = stage_ms["gate_up_gemm"]
    achieved = gu_flops / (gu_ms / 1e3) / 1e12
    roof = {"kernel": "gate_up_gemm", "bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
            "frac": achieved / peak, "frac_of_burst": achieved / peaks["bf16_tflops"],
            "frac_of_sustained": achieved / peaks["bf16_tflops_sustained"],
            "traffic": None, "algorithmic_flops_per_launch": gu_flops, "launches_averaged": steps * L,
            "kernel_ms": gu_ms, "share_of_step": gu_ms * L / ms,
            "peak_kind": kind, "peak_source": f"MEASURED_PEAKS.json bf16_tflops{'' if kind == 'burst' else '_sustained'} "
                                              f"({peak_src}): {why}"}
    line = {
        "metric": METRIC, "value": T / (ms / 1e3), "unit": "tokens/s", "n_gpus": 1, "steps": steps,
        "warmup": warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic: seeded random-init Mixtral-shaped weights per layer, h0 ~ N(0,1)",
        "config": {"workload": WORKLOAD_TEXT[args.config], **c, "parallelism": "one GPU",
                   "l2": "inputs larger than L2: %.1f GB of expert weights streamed per step" % (
                       L * E * 3 * d * f * 2 / 1e9)},
        "tflops": flops / (ms / 1e3) / 1e12,
        "tflops_frac_of_peak": flops / (ms / 1e3) / 1e12 / peak,
        "tflops_frac_of_burst_peak": flops / (ms / 1e3) / 1e12 / peaks["bf16_tflops"],
        "stages_ms_per_layer": {k: round(v, 4) for k, v in stage_ms.items()},
        "layer_span_ms": layer_span_ms,
        "roofline": roof,
        "e2e": {"value": T / (e2e_ms / 1e3), "unit": "tokens/s", "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": h0_host.numel() * h0_host.element_size(),
                "d2h_bytes_per_step": h_host.numel() * h_host.element_size()},
        # per layer: RMSNorm, then the layer's kernels
        "gpu_launches": (1 + moe._lib.load().moe_forward_launches(T, d, f, E, K, moe.MOE_BF16)) * L * steps,
        "stage_timing": "global-timer stamps written by every kernel inside the timed region "
                        "(moe_block_forward_stamped), averaged over the steps and layers",
        "clocks": clocks,
    }
    if not args.no_cpu_baseline:
        n_tok = min(T, max(1, args.cpu_tokens // 4))
        dt = oracle_block_rate(h0[:n_tok], layers[0], K)
        line["cpu_baseline"] = {"value": n_tok / (L * dt), "unit": "tokens/s", "cores": blas_threads(),
                                "kind": "oracle",
                                "sample": f"{n_tok} tokens through layer 0 of the stack, float64 oracle block "
                                          f"({dt:.1f} s), scaled to {L} layers; banks upcast once, untimed"}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
def run_ours_cache(args):
    """Decode steps through moe_forward_cached over a seeded locality trace."""
    import sparse_mixture_experts_55_b300 as moe
    from sparse_mixture_experts_55_b300 import build as _build
    _build.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    c = CONFIGS[args.config]
    T, d, f, E, K, C = c["T"], c["d"], c["f"], c["E"], c["K"], c["cache_slots"]
    Wg, W1, W3, W2 = W.mixtral_weights(d, f, E, seed=W.BASE_SEED, device=dev)
    steps, warmup = args.steps, max(args.warmup, 3)
    xs, _ = W.decode_trace(warmup + steps, Wg, T=T, keep=c["keep"], seed=W.BASE_SEED, device=dev)
    cache = moe.ExpertCache(W1, W3, W2, C, dev)
    ws = moe.Workspace(T, d, f, E, K, torch.bfloat16, dev)
    y = torch.empty(T, d, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream(dev)

    # host-to-device link: pinned copies of one expert matrix, event-timed
    mat = cache.host[0][0]
    dst = torch.empty_like(mat, device=dev)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    dst.copy_(mat, non_blocking=True)
    torch.cuda.synchronize(dev)
    ev0.record(stream)
    for _ in range(5):
        dst.copy_(mat, non_blocking=True)
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    link_gbs = 5 * mat.numel() * 2 / (ev0.elapsed_time(ev1) / 1e3) / 1e9
    del dst

    for i in range(warmup):
        cache.forward(xs[i], Wg, K, y=y, workspace=ws, stream=stream)
    torch.cuda.synchronize(dev)
    st = cache.state
    h0, m0, b0 = st.hits, st.misses, st.bytes_loaded
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(0) as clk:
        t0 = time.perf_counter()
        start.record(stream)
        for i in range(warmup, warmup + steps):
            cache.forward(xs[i], Wg, K, y=y, workspace=ws, stream=stream)
        end.record(stream)
        torch.cuda.synchronize(dev)
        wall_ms = 1e3 * (time.perf_counter() - t0) / steps
    ms = start.elapsed_time(end) / steps
    if moe.moe_read_status(ws) != 0:
        raise RuntimeError("device status set during timed run")
    hits, misses, loaded = st.hits - h0, st.misses - m0, st.bytes_loaded - b0

    # the same steps with every expert resident (moe_forward on the full banks)
    for i in range(warmup):
        moe.moe_forward(xs[i], Wg, W1, W3, W2, K, y=y, workspace=ws, stream=stream)
    start.record(stream)
    for i in range(warmup, warmup + steps):
        moe.moe_forward(xs[i], Wg, W1, W3, W2, K, y=y, workspace=ws, stream=stream)
    end.record(stream)
    torch.cuda.synchronize(dev)
    resident_ms = start.elapsed_time(end) / steps

    # end to end: each step's token copied in from pinned memory and its output back
    x_h = xs[warmup:warmup + steps].cpu().pin_memory()
    y_h = torch.empty(steps, T, d, dtype=torch.bfloat16).pin_memory()
    xd = torch.empty(T, d, dtype=torch.bfloat16, device=dev)
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for i in range(steps):
        xd.copy_(x_h[i], non_blocking=True)
        cache.forward(xd, Wg, K, y=y, workspace=ws, stream=stream)
        y_h[i].copy_(y, non_blocking=True)
    torch.cuda.synchronize(dev)
    e2e_ms = 1e3 * (time.perf_counter() - t0) / steps

    achieved = loaded / (ms * steps / 1e3) / 1e9
    line = {
        "metric": CACHE_METRIC, "value": T / (ms / 1e3), "unit": "tokens/s", "n_gpus": 1,
        "steps": steps, "warmup": warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic: seeded random-init Mixtral-shaped weights, Markov-chain locality trace of steered tokens",
        "config": {"workload": WORKLOAD_TEXT[args.config], **c, "parallelism": "one GPU",
                   "l2": "expert matrices of 117 MB each, larger than L2"},
        "cache": {"slots": C, "experts": E, "hits": hits, "misses": misses,
                  "hit_rate": hits / max(1, hits + misses), "bytes_loaded_per_step": loaded / steps,
                  "wall_ms_per_step": wall_ms, "all_resident_ms_per_step": resident_ms,
                  "device_weight_bytes": 3 * C * d * f * 2, "full_bank_bytes": 3 * E * d * f * 2},
        "roofline": {"kernel": "host-to-device expert copies", "bound": "h2d", "achieved": achieved,
                     "peak": link_gbs, "unit": "GB/s", "frac": achieved / link_gbs, "traffic": None,
                     "peak_source": "pinned host-to-device copy of one 117 MB expert matrix, timed in this run"},
        "e2e": {"value": T / (e2e_ms / 1e3), "unit": "tokens/s", "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": T * d * 2, "d2h_bytes_per_step": T * d * 2},
        "gpu_launches": moe._lib.load().moe_forward_launches(T, d, f, E, K, moe.MOE_BF16) * steps,
        "clocks": clk.summary(),
    }
    if not args.no_cpu_baseline:
        import numpy as np
        import oracle
        n_tok = 8
        x64 = xs[:n_tok, 0].float().cpu().numpy().astype(np.float64)
        banks = [t.float().cpu().numpy().astype(np.float64) for t in (Wg, W1, W3, W2)]
        t0 = time.perf_counter()
        for j in range(n_tok):
            oracle.moe_layer(x64[j:j + 1], *banks, K)
        dt = time.perf_counter() - t0
        line["cpu_baseline"] = {"value": n_tok / dt, "unit": "tokens/s", "cores": blas_threads(), "kind": "oracle",
                                "sample": f"first {n_tok} trace tokens one at a time, float64 oracle with every "
                                          f"expert in host memory ({dt:.1f} s; weights upcast once, untimed)"}
    print(json.dumps(line), flush=True)


BWD_STAGES = ("prep", "dgrad_h", "wgrad_w2", "dgrad_x", "wgrad_w13", "dx", "dwg")


def run_ours_train(args):
    """Training step: moe_forward_train then moe_backward (fp32 gradients) on
    the prefill batch with a fixed seeded output gradient."""
    import sparse_mixture_experts_55_b300 as moe
    from sparse_mixture_experts_55_b300 import build as _build
    _build.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    c = CONFIGS[args.config]
    T, d, f, E, K = c["T"], c["d"], c["f"], c["E"], c["K"]
    inp, _ = make_inputs(args.config, dev)
    dy = W.randn((T, d), 1.0, W.BASE_SEED + 77, dev, torch.bfloat16)
    stream = torch.cuda.current_stream(dev)
    steps, warmup = args.steps, max(args.warmup, 3)
    ws = moe.TrainWorkspace(T, d, f, E, K, torch.bfloat16, dev)
    y = torch.empty_like(inp.x)
    z = dict(dtype=torch.float32, device=dev)
    grads = moe.LayerGrads(torch.empty(T, d, **z), torch.empty(d, E, **z), torch.empty(E, d, f, **z),
                           torch.empty(E, d, f, **z), torch.empty(E, f, d, **z))
    lib = moe._lib.load()

    def step(x, g_out, dyv):
        moe.moe_forward_train(x, inp.Wg, inp.W1, inp.W3, inp.W2, K, ws, y=y, stream=stream)
        moe.moe_backward(x, inp.Wg, inp.W1, inp.W3, inp.W2, dyv, K, ws, grads=g_out, stream=stream)

    for _ in range(warmup):
        step(inp.x, grads, dy)
    torch.cuda.synchronize(dev)
    if moe.moe_read_status(ws) != 0:
        raise RuntimeError(f"device status {moe.moe_read_status(ws)}")
    start, mid, end = (torch.cuda.Event(enable_timing=True) for _ in range(3))
    torch.cuda.synchronize(dev)
    with ClockSampler(0) as clk:
        start.record(stream)
        for _ in range(steps):
            step(inp.x, grads, dy)
        end.record(stream)
        torch.cuda.synchronize(dev)
    ms = start.elapsed_time(end) / steps
    clocks = clk.summary()
    if moe.moe_read_status(ws) != 0:
        raise RuntimeError("device status set during timed run")

    # per-stage durations: forward as one region, backward stages from the
    # library's stage events (separate pass of the same steps, scaled below to
    # the headline step so that they add up to it)
    nst = len(BWD_STAGES) + 1
    fwd_ms, st_ms, pass_ms = [], {k: [] for k in BWD_STAGES}, []
    for _ in range(steps):
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(nst)]
        mid.record(stream)
        moe.moe_forward_train(inp.x, inp.Wg, inp.W1, inp.W3, inp.W2, K, ws, y=y, stream=stream)
        for ev in evs:
            ev.record(stream)  # create the handles; the library re-records them
        arr = (ctypes.c_void_p * nst)(*[ev.cuda_event for ev in evs])
        rc = lib.moe_backward_timed(*(ctypes.c_void_p(t.data_ptr()) for t in (inp.x, inp.Wg, inp.W1, inp.W3, inp.W2,
                                                                              dy, *grads)),
                                    T, d, f, E, K, moe.MOE_BF16, ctypes.c_void_p(ws.buf.data_ptr()), ws.nbytes, 0,
                                    ctypes.c_void_p(stream.cuda_stream), arr)
        moe._lib.check("moe_backward_timed", rc)
        torch.cuda.synchronize(dev)
        fwd_ms.append(mid.elapsed_time(evs[0]))
        pass_ms.append(mid.elapsed_time(evs[-1]))
        for j, k in enumerate(BWD_STAGES):
            st_ms[k].append(evs[j].elapsed_time(evs[j + 1]))
    stage_pass = {"forward_train": statistics.mean(fwd_ms), **{k: statistics.mean(v) for k, v in st_ms.items()}}
    scale = ms / statistics.mean(pass_ms)
    stage_ms = {k: v * scale for k, v in stage_pass.items()}

    # end to end with host buffers: x and dy copied in from pinned memory,
    # dx copied out, every step (the weight gradients stay on the device for
    # the optimiser).  As moe.HostPipeline does for the forward: two device
    # buffer sets, the next step's copies in and the previous step's dx out on
    # their own streams, ordered by events against the steps, which run in
    # order on the compute stream (the workspace holds one step's activations).
    x_h, dy_h = inp.x.cpu().pin_memory(), dy.cpu().pin_memory()
    dx_h = [torch.empty(T, d, dtype=torch.float32).pin_memory() for _ in range(2)]
    xs = [torch.empty_like(inp.x) for _ in range(2)]
    dys = [torch.empty_like(dy) for _ in range(2)]
    gbuf = [grads, moe.LayerGrads(torch.empty(T, d, **z), grads.dWg, grads.dW1, grads.dW3, grads.dW2)]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    in_done, run_done, out_done = ([torch.cuda.Event() for _ in range(2)] for _ in range(3))

    def submit(n):
        b = n & 1
        if n >= 2:
            s_in.wait_event(run_done[b])      # xs[b], dys[b] were read by the step two batches ago
        with torch.cuda.stream(s_in):
            xs[b].copy_(x_h, non_blocking=True)
            dys[b].copy_(dy_h, non_blocking=True)
            in_done[b].record(s_in)
        stream.wait_event(in_done[b])
        if n >= 2:
            stream.wait_event(out_done[b])    # dx[b] was copied out two batches ago
        step(xs[b], gbuf[b], dys[b])
        run_done[b].record(stream)
        s_out.wait_event(run_done[b])
        with torch.cuda.stream(s_out):
            dx_h[b].copy_(gbuf[b].dx, non_blocking=True)
            out_done[b].record(s_out)

    e2e_steps = max(3, min(steps, 20))
    for n in range(2):
        submit(n)
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for n in range(2, 2 + e2e_steps):
        submit(n)
    for sx in (s_in, stream, s_out):
        sx.synchronize()
    e2e_ms = 1e3 * (time.perf_counter() - t0) / e2e_steps

    peaks, peak_src = load_peaks()
    unit = 2.0 * T * K * d * f  # one expert-GEMM pass over the routed rows
    flops = 9 * unit + 3 * 2.0 * T * d * E  # 3 forward + 6 backward products; router fwd, dx, dWg
    prods = {"dgrad_h": unit, "wgrad_w2": unit, "dgrad_x": 2 * unit, "wgrad_w13": 2 * unit}
    top = max(prods, key=lambda k: stage_ms[k])  # the longest product
    achieved = prods[top] / (stage_ms[top] / 1e3) / 1e12
    peak, kind, why = tensor_peak(peaks, clocks)
    roof = {"kernel": f"bwd_gemm_kernel ({top})", "bound": "tensor", "achieved": achieved, "peak": peak,
            "unit": "TFLOP/s", "frac": achieved / peak, "frac_of_burst": achieved / peaks["bf16_tflops"],
            "frac_of_sustained": achieved / peaks["bf16_tflops_sustained"],
            "traffic": traffic_from_profiles(ROOT / "sparse_mixture_experts_55_b300" / "csrc" / "gemm_bwd.cu",
                                             f"{args.config}_{top}_traffic_bytes_per_launch", "bwd_gemm_traffic.md"),
            "algorithmic_flops_per_launch": prods[top], "kernel_ms": stage_ms[top],
            "peak_kind": kind, "peak_source": f"MEASURED_PEAKS.json bf16_tflops{'' if kind == 'burst' else '_sustained'} "
                                              f"({peak_src}): {why}"}
    line = {
        "metric": TRAIN_METRIC, "value": T / (ms / 1e3), "unit": "tokens/s", "n_gpus": 1,
        "steps": steps, "warmup": warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16 (fp32 accumulate, fp32 gradients)",
        "data": "synthetic: seeded random-init Mixtral-shaped weights, RMS-normalised N(0,1) tokens, N(0,1) dy",
        "config": {"workload": WORKLOAD_TEXT[args.config], **c, "parallelism": "one GPU",
                   "l2": "inputs larger than L2: %.2f GB of expert weights and %.2f GB of fp32 weight gradients "
                         "per step" % (3 * E * d * f * 2 / 1e9, 3 * E * d * f * 4 / 1e9)},
        "tflops": flops / (ms / 1e3) / 1e12,
        "tflops_frac_of_peak": flops / (ms / 1e3) / 1e12 / peak,
        "stages_ms": {k: round(v, 4) for k, v in stage_ms.items()},
        "stages_ms_separate_pass": {k: round(v, 4) for k, v in stage_pass.items()},
        "roofline": roof,
        "e2e": {"value": T / (e2e_ms / 1e3), "unit": "tokens/s", "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": x_h.numel() * x_h.element_size() + dy_h.numel() * dy_h.element_size(),
                "d2h_bytes_per_step": dx_h[0].numel() * dx_h[0].element_size()},
        "gpu_launches": (moe._lib.load().moe_forward_launches(T, d, f, E, K, moe.MOE_BF16) + 8) * steps,
        "stage_timing": "shares from a separate pass of the same steps with library-recorded backward stage "
                        "events, scaled to the headline step",
        "clocks": clocks,
    }
    if not args.no_cpu_baseline:
        import numpy as np
        import oracle
        n_tok = max(1, min(T, args.cpu_tokens // 4))
        x64 = inp.x[:n_tok].float().cpu().numpy().astype(np.float64)
        dy64 = dy[:n_tok].float().cpu().numpy().astype(np.float64)
        Wg64, W164, W364, W264 = f64_banks(inp)
        t0 = time.perf_counter()
        oracle.moe_layer(x64, Wg64, W164, W364, W264, K)
        oracle.moe_layer_backward(x64, Wg64, W164, W364, W264, K, dy64)
        dt = time.perf_counter() - t0
        line["cpu_baseline"] = {"value": n_tok / dt, "unit": "tokens/s", "cores": blas_threads(), "kind": "oracle",
                                "sample": f"first {n_tok} tokens, float64 oracle forward + backward ({dt:.1f} s; "
                                          f"weights upcast once, untimed)"}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
class LayerRunner:
    """The forward of one configuration (bf16 or e4m3 weights) through the C
    ABI, plain or stamped, with its own workspace."""

    def __init__(self, moe, c, x, weights, q8, dev, stream, flags=0):
        T, d, f, E, K = c["T"], c["d"], c["f"], c["E"], c["K"]
        self.moe, self.x, self.w, self.q8, self.K, self.stream = moe, x, weights, q8, K, stream
        self.flags = flags
        self.ws = moe.Workspace(T, d, f, E, K, torch.float8_e4m3fn if q8 else torch.bfloat16, dev)
        self.y = torch.empty_like(x)

    def __call__(self, stamps=None):
        m, Wg = self.moe, self.w[0]
        kw = dict(y=self.y, workspace=self.ws, flags=self.flags, stream=self.stream)
        if self.q8 is not None:
            if stamps is None:
                m.moe_forward_fp8(self.x, Wg, *self.q8, self.K, **kw)
            else:
                m.moe_forward_fp8_stamped(self.x, Wg, *self.q8, self.K, stamps, **kw)
        elif stamps is None:
            m.moe_forward(self.x, *self.w, self.K, **kw)
        else:
            m.moe_forward_stamped(self.x, *self.w, self.K, stamps, **kw)


def timed_region(moe, run, steps: int, dev, stream, stamped: bool):
    """K back-to-back forwards between two events (kernels chained by
    programmatic dependent launch), NVML clocks sampled meanwhile; with
    stamped, every forward writes its stage stamps into its own row."""
    stamps = moe.new_stamps(steps, dev) if stamped else None
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    with ClockSampler(dev.index or 0) as clk:
        start.record(stream)
        for i in range(steps):
            run(stamps[i] if stamped else None)
        end.record(stream)
        torch.cuda.synchronize(dev)
    if moe.moe_read_status(run.ws) != 0:
        raise RuntimeError("device status set during timed run")
    return start.elapsed_time(end) / steps, clk.summary(), stamps


def decode_record(moe, weights, q8, dev, stream, steps: int, warmup: int, peaks, fp8: bool):
    """The decode half of the metric: for each decode batch size of the sweep,
    the stamped layer over `steps` forwards of that batch through the prefill
    weights: ms per step, algorithmic bytes (touched experts' weights once)
    per second against the measured HBM copy bandwidth, and the same for each
    expert GEMM from its in-run kernel span (which starts when the kernel
    issues its first weight copies, possibly before the previous kernel has
    finished; negative launch gaps are that overlap)."""
    out = {}
    for T in (1, 8, 32, 128):
        c = dict(CONFIGS[f"decode{T}"], fp8=fp8)
        inp = W.decode(T, seed=W.BASE_SEED, device=dev, weights=weights)
        counts = moe.moe_route(inp.x, inp.Wg, c["K"])[3]
        n_touched = int(((counts[1:] - counts[:-1]) > 0).sum())
        run = LayerRunner(moe, c, inp.x, weights, q8, dev, stream)
        for _ in range(warmup):
            run()
        ms, clocks, stamps = timed_region(moe, run, steps, dev, stream, stamped=True)
        stages, span, gaps = stage_stats(moe, stamps, steps)
        excl = exclusive_stage_ms(moe, stamps)
        _, _, bytes_step, gu_bytes = algorithmic(c, n_touched)
        dn_bytes = down_bytes(c, n_touched)
        gbs = bytes_step / (ms / 1e3) / 1e9
        gu_gbs = gu_bytes / (stages["gate_up_gemm"] / 1e3) / 1e9
        dn_gbs = dn_bytes / (stages["down_gemm"] / 1e3) / 1e9
        out[f"T={T}"] = {
            "ms_per_step": ms, "tokens_per_s": T / (ms / 1e3), "touched_experts": n_touched,
            "algorithmic_bytes_per_step": bytes_step, "gbs": gbs, "frac_of_hbm": gbs / peaks["hbm_gbs"],
            "gate_up_gemm": {"ms": stages["gate_up_gemm"], "bytes": gu_bytes, "gbs": gu_gbs,
                             "frac_of_hbm": gu_gbs / peaks["hbm_gbs"],
                             "exclusive_ms": excl["gate_up_gemm"],
                             "frac_of_hbm_exclusive": gu_bytes / (excl["gate_up_gemm"] / 1e3) / 1e9
                             / peaks["hbm_gbs"]},
            "down_gemm": {"ms": stages["down_gemm"], "bytes": dn_bytes, "gbs": dn_gbs,
                          "frac_of_hbm": dn_gbs / peaks["hbm_gbs"],
                          "exclusive_ms": excl["down_gemm"],
                          "frac_of_hbm_exclusive": dn_bytes / (excl["down_gemm"] / 1e3) / 1e9
                          / peaks["hbm_gbs"]},
            "stages_ms": {k: round(v, 4) for k, v in stages.items()},
            "stages_exclusive_ms": {k: round(v, 4) for k, v in excl.items()},
            "launch_gaps_ms": gaps, "clocks": clocks}
        del run
    return out


def run_ours(args):
    import sparse_mixture_experts_55_b300 as moe
    from sparse_mixture_experts_55_b300 import build as _build
    _build.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    c = CONFIGS[args.config]
    T, d, f, E, K = c["T"], c["d"], c["f"], c["E"], c["K"]
    inp, weights = make_inputs(args.config, dev)
    fp8 = bool(c.get("fp8"))
    stream = torch.cuda.current_stream(dev)
    steps, warmup = args.steps, max(args.warmup, 3)
    # e4m3 expert weights: quantised once before timing (weight preparation)
    q8 = [t for W_ in (inp.W1, inp.W3, inp.W2) for t in moe.quantize_weights_fp8(W_)] if fp8 else None
    form_flags = {"auto": 0, "pair": moe.MOE_GEMM_PAIR_MMA, "mc2": moe.MOE_GEMM_MULTICAST_PAIRS,
                  "quad": moe.MOE_GEMM_QUAD}[args.gemm_form]
    run = LayerRunner(moe, c, inp.x, weights, q8, dev, stream, form_flags)

    # touched experts of this routing (algorithmic bytes at decode sizes)
    route_idx, _, _, offs, _ = moe.moe_route(inp.x, inp.Wg, K)
    n_touched = int(((offs[1:] - offs[:-1]) > 0).sum())

    # the decode half of the metric first (light on power), then a pause, so
    # that neither set of numbers is taken in the other's power-management tail
    decode = None
    if args.config in ("prefill", "prefill_fp8") and not args.no_decode:
        decode = decode_record(moe, weights, q8, dev, stream, max(steps, 100), warmup, load_peaks()[0], fp8)
        time.sleep(1.0)

    for _ in range(warmup):
        run()
    torch.cuda.synchronize(dev)
    if moe.moe_read_status(run.ws) != 0:
        raise RuntimeError(f"device status {moe.moe_read_status(run.ws)}")

    # headline: K back-to-back stamped forwards; every kernel writes its
    # begin/end global-timer stamps, so the per-kernel spans come from this
    # very region and add up to its step time (less launch gaps)
    ms, clocks, stamps = timed_region(moe, run, steps, dev, stream, stamped=True)
    stage_ms, step_span_ms, gaps_ms = stage_stats(moe, stamps, steps)
    excl_ms = exclusive_stage_ms(moe, stamps)
    y_out = run.y.clone()
    # the same steps through plain moe_forward (no stamps), for comparison
    ms_plain, clocks_plain, _ = timed_region(moe, run, steps, dev, stream, stamped=False)

    # end to end through the C ABI with host buffers: every step copies its
    # batch in from pinned host memory and its result out; the copies of
    # neighbouring steps overlap the layer (moe.HostPipeline)
    e2e_steps = max(3, min(steps, 50))
    x_hosts = [inp.x.cpu().pin_memory() for _ in range(2)]
    y_hosts = [torch.empty_like(x_hosts[0]).pin_memory() for _ in range(2)]
    pipe = moe.HostPipeline(inp.Wg, inp.W1, inp.W3, inp.W2, K, T, dev, workspace=run.ws, fp8_weights=q8)
    for i in range(3):
        pipe.submit(x_hosts[i & 1], y_hosts[i & 1])
    pipe.synchronize()
    t0 = time.perf_counter()
    for i in range(e2e_steps):
        pipe.submit(x_hosts[i & 1], y_hosts[i & 1])
    pipe.synchronize()
    e2e_ms = 1e3 * (time.perf_counter() - t0) / e2e_steps
    x_host, y_host = x_hosts[0], y_hosts[0]

    peaks, peak_src = load_peaks()
    flops, gu_flops, bytes_step, gu_bytes = algorithmic(c, n_touched)
    tokens_per_s = T / (ms / 1e3)
    gu_ms = stage_ms["gate_up_gemm"]
    hbm_bound = args.config.startswith("decode")
    # e4m3 contractions take the bf16 measured peaks times the nominal fp8/bf16 ratio (4.5 / 2.25)
    ratio = 2.0 if fp8 else 1.0
    peak_note = " x 2 (nominal e4m3/bf16 dense ratio)" if fp8 else ""
    kernel_file = ROOT / "sparse_mixture_experts_55_b300" / "csrc" / "gemm_tc.cu"
    traffic = traffic_from_profiles(kernel_file, f"{args.config}_traffic_bytes_per_launch")
    if hbm_bound:
        achieved = gu_bytes / (gu_ms / 1e3) / 1e9
        roof = {"kernel": "gate_up_gemm", "bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"], "traffic": traffic,
                "algorithmic_bytes_per_launch": gu_bytes, "kernel_ms": gu_ms, "share_of_step": gu_ms / ms,
                "peak_source": f"MEASURED_PEAKS.json hbm_gbs ({peak_src})"}
    else:
        peak, kind, why = tensor_peak(peaks, clocks, ratio)
        achieved = gu_flops / (gu_ms / 1e3) / 1e12
        roof = {"kernel": "gate_up_gemm", "bound": "tensor", "achieved": achieved, "peak": peak,
                "unit": "TFLOP/s", "frac": achieved / peak,
                "frac_of_burst": achieved / (peaks["bf16_tflops"] * ratio),
                "frac_of_sustained": achieved / (peaks["bf16_tflops_sustained"] * ratio),
                "traffic": traffic, "algorithmic_flops_per_launch": gu_flops,
                "kernel_ms": gu_ms, "share_of_step": gu_ms / ms, "peak_kind": kind,
                "peak_source": f"MEASURED_PEAKS.json bf16_tflops{'' if kind == 'burst' else '_sustained'}"
                               f"{peak_note} ({peak_src}): {why}"}
        dn_ms = stage_ms["down_gemm"]
        dn_flops = T * K * 2 * d * f
        dn_x = excl_ms["down_gemm"]
        roof["down_gemm"] = {"kernel_ms": dn_ms, "achieved": dn_flops / (dn_ms / 1e3) / 1e12,
                             "frac": dn_flops / (dn_ms / 1e3) / 1e12 / peak, "algorithmic_flops_per_launch": dn_flops,
                             "exclusive_ms": dn_x, "frac_exclusive": dn_flops / (dn_x / 1e3) / 1e12 / peak,
                             "frac_of_burst_exclusive": dn_flops / (dn_x / 1e3) / 1e12
                             / (peaks["bf16_tflops"] * ratio)}
    line = {
        "metric": METRIC, "value": tokens_per_s, "unit": "tokens/s", "n_gpus": 1, "steps": steps,
        "warmup": warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "e4m3 experts, bf16 tokens" if fp8 else "bf16",
        "data": "synthetic: seeded random-init Mixtral-shaped weights, RMS-normalised N(0,1) tokens",
        "config": {"workload": WORKLOAD_TEXT[args.config], **c, "parallelism": "one GPU",
                   "l2": "inputs larger than L2: %.2f GB of expert weights streamed per step" % (
                       n_touched * 3 * d * f * (1 if fp8 else 2) / 1e9), "touched_experts": n_touched},
        "tflops": flops / (ms / 1e3) / 1e12,
        "hbm_gbs_algorithmic": bytes_step / (ms / 1e3) / 1e9,
        "stages_ms": {k: round(v, 4) for k, v in stage_ms.items()},
        "stages_exclusive_ms": {k: round(v, 4) for k, v in excl_ms.items()},
        "step_span_ms": step_span_ms, "launch_gaps_ms": gaps_ms,
        "roofline": roof,
        "e2e": {"value": T / (e2e_ms / 1e3), "unit": "tokens/s", "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": x_host.numel() * x_host.element_size(),
                "d2h_bytes_per_step": y_host.numel() * y_host.element_size()},
        "gpu_launches": moe._lib.load().moe_forward_launches(T, d, f, E, K, moe.MOE_FP8_E4M3 if fp8 else moe.MOE_BF16)
        * steps,
        "timed_call": ("moe_forward_fp8_stamped" if fp8 else "moe_forward_stamped") +
                      ": the plain call's kernels, each CTA also writing two global-timer stamps",
        "stage_timing": "global-timer stamps written by every kernel inside the timed region, averaged over the steps",
        "plain": {"ms_per_step": ms_plain, "tokens_per_s": T / (ms_plain / 1e3), "clocks": clocks_plain,
                  "call": "moe_forward_fp8" if fp8 else "moe_forward", "region": "the next K steps, unstamped"},
        "clocks": clocks,
    }
    if args.gemm_form != "auto":
        line["config"]["gemm_form"] = args.gemm_form
    if not hbm_bound:
        line["tflops_frac_of_peak"] = line["tflops"] / roof["peak"]
    if decode is not None:
        line["decode"] = decode
    if not args.no_cpu_baseline and not fp8:
        n_tok = min(T, args.cpu_tokens)
        rate, dt, threads, y_ref = cpu_oracle_rate(inp, n_tok)
        line["cpu_baseline"] = {"value": rate, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                                "sample": f"first {n_tok} tokens of the batch, float64 oracle ({dt:.1f} s; "
                                          f"weights upcast once, untimed)"}
        line["parity"] = oracle_check(inp, route_idx.cpu().numpy(), y_out[:n_tok].float().cpu().numpy(), y_ref)
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1, help="1 (the only supported value)")
    ap.add_argument("--steps", type=int, default=None, help="default: 100 (10 for stack32)")
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--config", default="prefill", choices=sorted(CONFIGS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-tokens", type=int, default=256)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-decode", action="store_true", help="omit the decode sweep of the prefill line")
    ap.add_argument("--gemm-form", default="auto", choices=["auto", "pair", "mc2", "quad"],
                    help="expert-GEMM form (the library's MOE_GEMM_* flags; results are identical)")
    args = ap.parse_args()
    if args.steps is None:
        args.steps = 10 if args.config == "stack32" else 100
    rank = launch_rank(args)
    if args.impl == "reference":
        run_reference(args, rank)
    elif args.config == "stack32":
        run_ours_stack(args)
    elif CONFIGS[args.config].get("train"):
        run_ours_train(args)
    elif "cache_slots" in CONFIGS[args.config]:
        run_ours_cache(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
