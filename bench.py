#!/usr/bin/env python
"""Benchmark of the MoE finalize (+ RMSNorm) path on GB300.

Default workload: finalize + RMSNorm over 32768 tokens, hidden 4096, top-k 8,
gemm2_permuted BF16 [288358, 4096] ~N(0, 2) (262144 indexed rows plus 10%
never-indexed padding rows), a random permutation index map with 1% invalid
slots, FP32 softmax weights, norm_weight ~N(0, 0.1), gain_center 1.0,
eps 1e-6.  One step = one call over the whole batch; weight_before_norm
alternates between steps so both orderings are timed.  The inputs (2.42 GB
per call) are larger than L2, so every call reads its rows from HBM.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload roofline|padded|beam|beam_residual|small|decode|custom|beam_custom]
                    [--tokens T]
                    [--hidden H --top-k K --weights fp32|bf16|packed]

Prints one JSON line (rank 0).  ``--impl reference`` times the CPU oracle (the
reference arm of this path) on the host cores instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time
from concurrent.futures import ThreadPoolExecutor

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth_inputs as si  # noqa: E402

METRIC = "finalize tokens/s and achieved HBM GB/s vs GB300 peak (1 GPU)"
FALLBACK_HBM_GBS = 6800.0
CSRC = os.path.join(ROOT, "moe_finalize_rmsnorm_gb300", "csrc")
PROFILES = os.path.join(ROOT, "profiles")


# ---------------------------------------------------------------------------
# host-side helpers (also exercised by the CPU tests)

# More than twice the GB300's 129 MB L2: the scratch write of --cold.
L2_FLUSH_BYTES = 288 * 1024 * 1024
# GB300's L2; a launch's inputs count as cold when the launches since their
# last use have moved at least four times this much.
L2_BYTES = 129 * 10 ** 6


def rank_seed(base_seed: int, rank: int) -> int:
    """Each rank finalizes its own independent batch (weak scaling)."""
    return base_seed + 1000003 * rank


def reduce_max(value: float, group=None) -> float:
    """Max of a per-rank float over the default process group (identity at N=1)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return value
    dev = "cuda" if dist.get_backend(group) == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    return float(t.item())


def code_only(text: str) -> str:
    """C++ source without its comments, whitespace runs collapsed (the sources
    hold no string literal with a comment marker)."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def source_digest(kernel: str) -> str:
    """Digest of the code a kernel is built from (its family's .cu file and the
    shared device headers, comments left out); a recorded traffic figure
    applies only to the code it was measured on."""
    family = "beam_finalize.cu" if kernel.startswith("beam_") else "tp_finalize.cu"
    h = hashlib.sha256()
    for name in ("common.cuh", "kernels.h", family):
        with open(os.path.join(CSRC, name), encoding="utf-8") as f:
            h.update(name.encode() + b"\0" + code_only(f.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str) -> float | None:
    """DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum)
    recorded from an ncu capture in profiles/*.md, if it matches the current
    sources.  Lines look like:
    ``traffic: kernel=<name> workload=<name> bytes_per_launch=<n> sources=<digest>``"""
    if not os.path.isdir(PROFILES):
        return None
    digest = source_digest(kernel)
    pat = re.compile(r"traffic: kernel=(\S+) workload=(\S+) bytes_per_launch=(\d+) sources=(\S+)")
    for name in sorted(os.listdir(PROFILES)):
        if not name.endswith((".md", ".txt")):
            continue
        with open(os.path.join(PROFILES, name)) as f:
            for line in f:
                m = pat.search(line)
                if m and m.group(1) == kernel and m.group(2) == workload and m.group(4) == digest:
                    return float(m.group(3))
    return None


def measured_peaks() -> tuple[float, str]:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples every 50 ms in the background."""

    FIELDS = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, uuid: str | None):
        self.uuid = (uuid or "").lower().replace("gpu-", "")
        self.samples: list[tuple[float, list[str]]] = []
        self.proc = None
        self.error = None

    def start(self) -> None:
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError as e:
            self.error = f"nvidia-smi unavailable: {e}"
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        t0 = time.time()
        while not self.samples and time.time() - t0 < 10 and self.proc.poll() is None:
            time.sleep(0.02)

    def _read(self) -> None:
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.samples.append((time.time(), parts))

    def stop(self) -> None:
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float) -> dict:
        if self.error:
            return {"unavailable": self.error}
        mine = [p for _, p in self.samples if not self.uuid or p[0].lower().replace("gpu-", "") == self.uuid]
        if not mine:
            mine = [p for _, p in self.samples]
        inwin = [p for (t, p) in self.samples if t0 <= t <= t1 and p in mine]
        use = inwin or mine
        if not use:
            return {"unavailable": "no nvidia-smi samples"}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [v for v in (num(p[1]) for p in use) if v is not None]
        mx = [v for v in (num(p[2]) for p in use) if v is not None]
        pw = [v for v in (num(p[3]) for p in use) if v is not None]
        reasons = sorted({name for p in use for name, v in zip(self.REASONS, p[5:9])
                          if v.strip().lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(pw) if pw else None,
                "reasons": reasons, "samples": len(use), "samples_in_timed_region": len(inwin)}


class NvmlClock:
    """Read-only NVML queries of one GPU (SM clock, power draw, clock-event
    reasons), polled from the host thread while the timed launches run, so a
    timed region of a few milliseconds still holds samples.  Nothing is set."""

    # nvmlClocksEventReason* bits (nvml.h) of the reasons the record reports
    REASON_BITS = (("sw_power_cap", 0x4), ("hw_slowdown", 0x8),
                   ("sw_thermal_slowdown", 0x20), ("hw_thermal_slowdown", 0x40))
    NVML_CLOCK_SM = 1

    def __init__(self, uuid: str | None):
        import ctypes
        self.ct = ctypes
        self.error = None
        self.max_mhz = None
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                raise OSError("nvmlInit_v2 failed")
            if not uuid:
                raise OSError("no device UUID")
            u = "GPU-" + uuid.lower().replace("gpu-", "")
            h = ctypes.c_void_p()
            if lib.nvmlDeviceGetHandleByUUID(u.encode(), ctypes.byref(h)) != 0:
                raise OSError(f"no NVML device {u}")
            self.reasons_fn = (getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None)
                               or lib.nvmlDeviceGetCurrentClocksThrottleReasons)
            mx = ctypes.c_uint()
            if lib.nvmlDeviceGetMaxClockInfo(h, self.NVML_CLOCK_SM, ctypes.byref(mx)) == 0:
                self.max_mhz = float(mx.value)
            self.lib, self.h = lib, h
        except (OSError, AttributeError) as e:
            self.error = f"NVML unavailable: {e}"

    def sample(self):
        """(wall time, SM MHz, watts, reason bits) or None."""
        if self.error:
            return None
        c = self.ct
        clk, mw, rs = c.c_uint(), c.c_uint(), c.c_ulonglong()
        if self.lib.nvmlDeviceGetClockInfo(self.h, self.NVML_CLOCK_SM, c.byref(clk)) != 0:
            return None
        self.lib.nvmlDeviceGetPowerUsage(self.h, c.byref(mw))
        self.reasons_fn(self.h, c.byref(rs))
        return (time.time(), float(clk.value), mw.value / 1000.0, int(rs.value))

    def poll(self, end_event, into: list, interval_s: float = 0.0005) -> None:
        """Sample until end_event (recorded after the timed launches) completes."""
        while not end_event.query():
            smp = self.sample()
            if smp is None:
                return
            into.append(smp)
            time.sleep(interval_s)

    def summary(self, samples: list) -> dict:
        if not samples:
            return {"samples": 0}
        reasons = sorted({name for _, _, _, bits in samples for name, b in self.REASON_BITS
                          if bits & b})
        return {"sm_mhz": statistics.median(s[1] for s in samples), "sm_max_mhz": self.max_mhz,
                "power_w_max": max(s[2] for s in samples), "reasons": reasons,
                "samples": len(samples)}


def clock_record(smi: dict, nvml: NvmlClock, inwin: list) -> dict:
    """The line's clock record: NVML samples taken inside the timed region
    (the host polls while the launches run), with the nvidia-smi background
    samples as the fallback and for context."""
    if nvml.error or not inwin:
        rec = dict(smi)
        rec["source"] = "nvidia-smi every 50 ms" + (f" ({nvml.error})" if nvml.error else "")
        return rec
    rec = nvml.summary(inwin)
    rec["reasons"] = sorted(set(rec["reasons"]) | set(smi.get("reasons", [])))
    rec["samples_in_timed_region"] = len(inwin) + smi.get("samples_in_timed_region", 0)
    rec["samples"] = len(inwin) + smi.get("samples", 0)
    rec["source"] = ("NVML (read-only) polled by the host while the timed launches ran, "
                     "plus nvidia-smi every 50 ms")
    return rec


def gpu_uuid(device_index: int) -> str | None:
    import torch
    try:
        return str(torch.cuda.get_device_properties(device_index).uuid)
    except Exception:
        return None


# ---------------------------------------------------------------------------
# workloads

class Job:
    """Device-resident inputs of one workload and how to launch one step."""

    def __init__(self, name, units_per_step, bytes_per_launch, kernel, launch, host, describe):
        self.name = name
        self.units_per_step = units_per_step
        self.bytes_per_launch = bytes_per_launch
        self.kernel = kernel
        self.launch = launch
        self.host = host
        self.describe = describe


def _dev_bf16(torch, bits, device):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(
        device)


def make_tp_job(torch, mf, case: si.TpCase, device, variant: str, alternate: bool) -> Job:
    g = _dev_bf16(torch, case.gemm2, device)[:, :case.hidden]
    w = (_dev_bf16(torch, case.weights, device) if case.weights.dtype == np.uint16
         else torch.from_numpy(case.weights).to(device))
    idx = torch.from_numpy(case.idx).to(device)
    nw = _dev_bf16(torch, case.norm_weight, device)
    out = torch.empty((case.num_tokens, case.hidden), dtype=torch.bfloat16, device=device)
    T = case.num_tokens
    wbytes = case.weights.dtype.itemsize

    def launch(step: int, tensors=(g, w, idx, nw, out)):
        before = (step % 2 == 1) if alternate else case.weight_before_norm
        gg, ww, ii, nn, oo = tensors
        mf.moe_finalize_rmsnorm(gg, ww, ii, nn, oo, eps=case.eps, gain_center=case.gain_center,
                                weight_before_norm=before, variant=variant)

    chosen = (mf.select_finalize_variant(T, case.hidden, case.top_k) if variant == "auto"
              else variant)
    kernel = mf.finalize_kernel_name(T, case.hidden, case.top_k, variant)
    job = Job(case.name, T, si.algorithmic_bytes_tp(T, case.hidden, case.top_k, wbytes), kernel,
              launch, case, {"variant": chosen})
    job.device_tensors = (g, w, idx, nw, out)
    return job


def make_beam_job(torch, mf, case: si.BeamCase, device, variant: str) -> Job:
    cap, K, H = case.expert_outputs.shape
    x = _dev_bf16(torch, case.expert_outputs, device)
    w = torch.from_numpy(case.weights).to(device)
    pw = _dev_bf16(torch, case.post_weight, device) if case.post_weight is not None else None
    out = torch.empty((case.live_tokens, H), dtype=torch.bfloat16, device=device)

    def launch(step: int, tensors=(x, w, pw, out)):
        xx, ww, pp, oo = tensors
        mf.beam_moe_finalize(xx, ww, oo, case.routed_scale, pp, case.post_eps, variant=variant)

    chosen = mf.select_beam_variant(case.live_tokens, K, H) if variant == "auto" else variant
    kernel = mf.beam_kernel_name(case.live_tokens, K, H, variant)
    job = Job(case.name, case.live_tokens, si.algorithmic_bytes_beam(case.live_tokens, H, K),
              kernel, launch, case, {"variant": chosen})
    job.device_tensors = (x, w, pw, out)
    return job


def make_beam_residual_job(torch, mf, case: si.BeamCase, device) -> Job:
    """Beam finalize + residual add + next RMSNorm over the live rows."""
    cap, K, H = case.expert_outputs.shape
    T = case.live_tokens
    x = _dev_bf16(torch, case.expert_outputs.reshape(cap * K, H), device)
    w = torch.from_numpy(case.weights).to(device)
    pw = _dev_bf16(torch, case.post_weight, device)
    res = _dev_bf16(torch, case.meta["residual"], device)
    nw = _dev_bf16(torch, case.meta["next_weight"], device)
    hid = torch.empty((T, H), dtype=torch.bfloat16, device=device)
    nrm = torch.empty((T, H), dtype=torch.bfloat16, device=device)

    def launch(step: int, tensors=(x, w, res, pw, nw, hid, nrm)):
        xx, ww, rr, pp, nn, hh, oo = tensors
        mf.beam_moe_finalize_norm_residual_norm(xx, ww, rr, pp, case.post_eps, nn, 1e-6, None,
                                                case.routed_scale, hidden=hh, normalized=oo)

    job = Job(case.name + "_residual", T, si.algorithmic_bytes_beam_residual(T, H, K, True),
              mf.beam_kernel_name(T, K, H, "auto", residual=True), launch, case,
              {"variant": "bulk"})
    job.device_tensors = (x, w, res, pw, nw, hid, nrm)
    job.n_outputs = 2
    return job


def workload_case(name: str, tokens: int | None, seed_rank: int, args_hidden: int = 4096,
                  args_top_k: int = 8, args_weights: str = "fp32"):
    """Host inputs of a named workload (rank-dependent seed for N > 1)."""
    if name == "roofline":
        c = si.finalize_32768_tokens(False) if seed_rank == 0 else si.tp_case(
            "finalize_T32768", si.ROOFLINE_TOKENS, indexed_rows=si.ROOFLINE_INDEXED_ROWS,
            padding_rows=si.ROOFLINE_PADDING_ROWS, sigma=2.0, invalid_frac=0.01,
            weights_dtype="fp32", gain_center=1.0, eps=1e-6, seed=seed_rank)
        desc = ("finalize+RMSNorm num_tokens=32768 hidden=4096 top_k=8 gemm2=[288358,4096] "
                "~N(0,2) 1% invalid fp32 weights gain_center=1.0 eps=1e-6, "
                "weight_before_norm alternating per step")
        return "tp", c, desc
    if name == "padded":
        return "tp", si.finalize_4096_tokens_padded(poison_padding=False), (
            "finalize+RMSNorm num_tokens=4096 gemm2=[36864,4160] stride 4160, bf16 weights, "
            "2% invalid, eps=1e-5, weight_before_norm=true")
    if name == "small":
        return "tp", si.finalize_16_tokens(), "finalize+RMSNorm num_tokens=16 gemm2=[128,4096]"
    if name == "decode":
        T = tokens or 1
        return "tp", si.finalize_decode(T), f"finalize+RMSNorm decode num_tokens={T} rows={10 * T}"
    if name == "custom":
        T, H, K = tokens or 8192, args_hidden, args_top_k
        c = si.tp_case(f"finalize_T{T}_H{H}_K{K}_{args_weights}", T, hidden=H, top_k=K,
                       indexed_rows=T * K, invalid_frac=0.01, weights_dtype=args_weights,
                       gain_center=1.0, eps=1e-6, seed=seed_rank)
        return "tp", c, (f"finalize+RMSNorm num_tokens={T} hidden={H} top_k={K} "
                         f"{args_weights} weights, 1% invalid, rows={T * K} ~N(0,1)")
    if name == "beam_custom":
        T, H, K = tokens or 8192, args_hidden, args_top_k
        c = si.beam_case(f"beam_T{T}_H{H}_K{K}", T, K, H, T, routed_scale=2.5, post_weight=True,
                         post_eps=1e-6, seed=seed_rank)
        return "beam", c, (f"Beam finalize capacity=live={T} top_k={K} hidden={H} "
                           "routed_scale=2.5 post-RMSNorm")
    if name == "beam_residual":
        c = si.beam_8000_live(poison_dead_rows=False)
        c.meta["residual"] = si.normal_bf16((c.live_tokens, 7168), 1.0, 7, 1)
        c.meta["next_weight"] = si.normal_bf16((7168,), 0.1, 8, 1, mu=1.0)
        return "beam_residual", c, (
            "Beam finalize + residual add + next RMSNorm: capacity=8192 top_k=8 hidden=7168 "
            "tokens=8000 routed_scale=2.5 post-RMSNorm, residual ~N(0,1), next_weight "
            "~1+N(0,0.1), next_eps=1e-6")
    if name == "beam":
        return "beam", si.beam_8000_live(poison_dead_rows=False), (
            "Beam finalize capacity=8192 top_k=8 hidden=7168 live_tokens=8000 routed_scale=2.5 "
            "post-RMSNorm")
    raise SystemExit(f"unknown workload {name}")


# ---------------------------------------------------------------------------
# CPU oracle timing (the reference arm and the cpu_baseline key)

def time_oracle(kind: str, case, token_lo: int, token_hi: int, threads: int,
                before: bool | None = None) -> float:
    """Wall seconds for the oracle over tokens [lo, hi) split across threads."""
    import oracle
    n = token_hi - token_lo
    chunks = max(1, min(threads, n))
    bounds = [token_lo + (n * i) // chunks for i in range(chunks + 1)]

    def work(i):
        lo, hi = bounds[i], bounds[i + 1]
        if hi <= lo:
            return
        if kind == "tp":
            oracle.moe_finalize_rmsnorm(
                case.gemm2, np.ascontiguousarray(case.weights[lo:hi]),
                np.ascontiguousarray(case.idx[lo:hi]), case.norm_weight, eps=case.eps,
                gain_center=case.gain_center,
                weight_before_norm=case.weight_before_norm if before is None else before,
                hidden=case.hidden)
        elif kind == "beam_residual":
            oracle.beam_moe_finalize_norm_residual_norm(
                np.ascontiguousarray(case.expert_outputs[lo:hi]),
                np.ascontiguousarray(case.weights[lo:hi]),
                np.ascontiguousarray(case.meta["residual"][lo:hi]),
                routed_scale=case.routed_scale, post_weight=case.post_weight,
                post_eps=case.post_eps, next_weight=case.meta["next_weight"], next_eps=1e-6)
        else:
            oracle.beam_moe_finalize(
                np.ascontiguousarray(case.expert_outputs[lo:hi]),
                np.ascontiguousarray(case.weights[lo:hi]), hi - lo,
                routed_scale=case.routed_scale, post_weight=case.post_weight,
                post_eps=case.post_eps)

    t0 = time.perf_counter()
    with ThreadPoolExecutor(chunks) as ex:
        list(ex.map(work, range(chunks)))
    return time.perf_counter() - t0


def host_cpu() -> str:
    """CPU model and architecture of the host (for the baseline's record)."""
    import platform
    model = ""
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key = line.split(":")[0].strip().lower()
                if key in ("model name", "cpu part", "processor name"):
                    model = line.split(":", 1)[1].strip()
                    break
    except OSError:
        pass
    return f"{platform.machine()} {model}".strip()


def total_tokens(kind, case):
    return case.num_tokens if kind == "tp" else case.live_tokens


def bytes_per_token(kind, case) -> float:
    """Algorithmic bytes per token of the workload (the roofline's count)."""
    if kind == "tp":
        return si.algorithmic_bytes_tp(1, case.hidden, case.top_k, case.weights.dtype.itemsize)
    _, K, H = case.expert_outputs.shape
    if kind == "beam_residual":
        return si.algorithmic_bytes_beam_residual(1, H, K, True)
    return si.algorithmic_bytes_beam(1, H, K)


def run_reference(args) -> None:
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if rank != 0:
        return
    import oracle
    oracle.build()
    kind, case, desc = workload_case(args.workload, args.tokens, 0, args.hidden, args.top_k,
                                     args.weights)
    threads = os.cpu_count() or 1
    T = total_tokens(kind, case)
    # size each step so the whole run stays within about a minute of wall time
    probe = min(T, max(threads, 64))
    per_token = time_oracle(kind, case, 0, probe, threads) / probe
    budget_s = 60.0
    sample = int(max(1, min(T, budget_s / max(per_token, 1e-9) / max(args.steps + args.warmup, 1))))
    lo = 0

    def step(i):
        nonlocal lo
        if lo + sample > T:
            lo = 0
        before = (i % 2 == 1) if args.workload == "roofline" else None
        s = time_oracle(kind, case, lo, lo + sample, threads, before)
        lo += sample
        return s

    for i in range(args.warmup):
        step(i)
    secs = sum(step(i) for i in range(args.steps))
    value = sample * args.steps / secs
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": secs / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        # the same keys, with the same meaning, as the GPU arm's config: the
        # tokens one step finalizes and how the job is laid out
        "config": {"workload": desc, "global_batch": sample,
                   "parallelism": "single GPU" if world == 1 else
                   f"rank 0 of {world} (the other ranks idle)"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                         "sample": f"{sample} consecutive tokens of the batch per step, "
                                   f"{threads} threads",
                         "host_gbs": value * bytes_per_token(kind, case) / 1e9, "cpu": host_cpu()},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# the CUDA path

def per_launch_pass(torch, launch, stream, n: int, alternating: bool) -> dict:
    """Distribution of single-launch times, from a pass after the timed region
    with an event pair around every launch.  The event records between
    launches make each launch wait for the one before it to drain and expose
    its start-up, so these read a few microseconds above the back-to-back
    average; the headline figures do not use them."""
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(n)]
    for i in range(n):
        ev[i][0].record(stream)
        launch(i)
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    ms = [a.elapsed_time(b) for a, b in ev]
    out = {"launches": n,
           "us_p10_p50_p90": [float(np.percentile(ms, q)) * 1e3 for q in (10, 50, 90)]}
    if alternating and n > 1:
        out["us_mean_by_ordering"] = {"weight_before_norm=false": statistics.fmean(ms[0::2]) * 1e3,
                                      "weight_before_norm=true": statistics.fmean(ms[1::2]) * 1e3}
    return out


def run_ours(args) -> None:
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world != args.gpus:
        raise SystemExit(f"--gpus {args.gpus} but WORLD_SIZE={world}")
    torch.cuda.set_device(local_rank)
    device = torch.device("cuda", local_rank)
    if world > 1:
        dist.init_process_group("nccl", device_id=device)

    from moe_finalize_rmsnorm_gb300.build import build
    if rank == 0:
        build()
    if world > 1:
        dist.barrier()
    import moe_finalize_rmsnorm_gb300 as mf
    mf.set_programmatic_launch(not args.no_pdl)

    kind, case, desc = workload_case(args.workload, args.tokens, rank_seed(0, rank) if rank else 0,
                                     args.hidden, args.top_k, args.weights)
    if kind == "tp":
        job = make_tp_job(torch, mf, case, device, args.variant,
                          alternate=args.workload == "roofline")
    elif kind == "beam_residual":
        job = make_beam_residual_job(torch, mf, case, device)
    else:
        job = make_beam_job(torch, mf, case, device, args.variant)
    stream = torch.cuda.current_stream(device)
    # inputs of a few L2 sizes only: rotate among copies so that no launch finds
    # the previous launch's rows in L2 (one copy for the default workload)
    n_copies = 1 if (args.cold or args.graph) else input_copies(job.bytes_per_launch)
    sets = [tuple(job.device_tensors)] + [
        tuple(None if t is None else _same_layout_copy(torch, t) for t in job.device_tensors)
        for _ in range(n_copies - 1)]

    def launch(i):
        if n_copies == 1:
            job.launch(i)
        else:
            job.launch(i, tensors=sets[i % n_copies])

    # warm-up
    for i in range(args.warmup):
        launch(i)
    torch.cuda.synchronize(device)
    if mf.device_status(clear=True) != 0:
        raise SystemExit("device wait timeout during warm-up")

    uuid = gpu_uuid(local_rank)
    clocks = ClockSampler(uuid)
    nvml = NvmlClock(uuid)
    inwin: list = []  # NVML samples taken while the timed launches run
    clocks.start()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(device)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    cold_ms = None
    if args.cold:
        # a write of twice the L2 size before every launch evicts the inputs and
        # the previous output; each launch is timed between its own event pair
        scratch = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
        t_wall0 = time.time()
        start.record(stream)
        for i in range(args.steps):
            scratch.fill_(i & 0xFF)
            ev[i][0].record(stream)
            job.launch(i)
            ev[i][1].record(stream)
        end.record(stream)
        nvml.poll(end, inwin)
        torch.cuda.synchronize(device)
        t_wall1 = time.time()
        cold_ms = [a.elapsed_time(b) for a, b in ev]
        del scratch
    elif args.graph:
        # decode sizes: the K launches replay from one CUDA graph, so the timed
        # region holds no host launch gaps (the per-launch figure is the mean)
        graph = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(device)
        cap.wait_stream(stream)
        with torch.cuda.stream(cap), torch.cuda.graph(graph, stream=cap):
            for i in range(args.steps):
                job.launch(i)
        torch.cuda.synchronize(device)
        graph.replay()  # one untimed replay
        torch.cuda.synchronize(device)
        t_wall0 = time.time()
        start.record(stream)
        graph.replay()
        end.record(stream)
        nvml.poll(end, inwin)
        torch.cuda.synchronize(device)
        t_wall1 = time.time()
    else:
        # the K launches back to back, as a caller issues them: nothing else on the
        # stream between them, so the region's length / K is the average launch
        t_wall0 = time.time()
        start.record(stream)
        for i in range(args.steps):
            launch(i)
        end.record(stream)
        nvml.poll(end, inwin)
        torch.cuda.synchronize(device)
        t_wall1 = time.time()
    if world > 1:
        dist.barrier()
    clocks.stop()
    if mf.device_status(clear=True) != 0:
        raise SystemExit("device wait timeout in the timed region")

    # the timed work: the K launches (with --cold, the launches alone, not the flushes)
    elapsed_ms = reduce_max(sum(cold_ms) if cold_ms is not None else start.elapsed_time(end))
    avg_launch_ms = elapsed_ms / args.steps
    units = job.units_per_step * args.steps * world
    value = units / (elapsed_ms / 1e3)
    hbm_gbs = job.bytes_per_launch * args.steps / (elapsed_ms / 1e3) / 1e9
    peak, peak_src = measured_peaks()
    achieved = job.bytes_per_launch / (avg_launch_ms / 1e3) / 1e9
    traffic = recorded_traffic(job.kernel, job.name)
    extra = {}
    if cold_ms is not None:
        extra["cold_launch_us_p10_p50_p90"] = [float(np.percentile(cold_ms, q)) * 1e3
                                               for q in (10, 50, 90)]
    elif not args.graph:
        extra["per_launch_events"] = per_launch_pass(torch, launch, stream, min(args.steps, 400),
                                                     args.workload == "roofline")
        if mf.device_status(clear=True) != 0:
            raise SystemExit("device wait timeout in the per-launch pass")

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": elapsed_ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": desc, "global_batch": job.units_per_step * world,
                   "l2": (f"flushed before every launch ({L2_FLUSH_BYTES / 1e6:.0f} MB scratch "
                          "write, not timed)") if args.cold else
                         (f"{n_copies} copies of the inputs, launch i reads copy i mod "
                          f"{n_copies}: each launch's rows were last read at least 4 x L2 of "
                          "traffic earlier") if n_copies > 1 else
                         ("no flush: every step reads its inputs from HBM "
                          f"({job.bytes_per_launch / 1e9:.3f} GB per launch, L2 is 0.13 GB)"
                          if job.bytes_per_launch >= 4 * L2_BYTES else
                          "inputs smaller than L2 (warm)"),
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "timing": "one CUDA graph of all timed launches" if args.graph
                   else ("an event pair around each launch, summed" if args.cold
                         else "one CUDA event pair around the K back-to-back launches"),
                   "programmatic_dependent_launch": not args.no_pdl,
                   **job.describe},
        "hbm_gbs": hbm_gbs,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic, "kernel": job.kernel,
                     "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)"
                     if peak_src == "measured" else "fallback 6.8 TB/s",
                     "algorithmic_bytes_per_launch": job.bytes_per_launch},
        "gpu_launches": args.steps,
        "clocks": clock_record(clocks.summary(t_wall0, t_wall1), nvml, inwin),
        **extra,
    }

    if not args.no_e2e:
        line["e2e"] = run_e2e(torch, mf, job, kind, case, device, args.e2e_steps)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        threads = os.cpu_count() or 1
        T = total_tokens(kind, case)
        n = min(T, args.cpu_tokens)
        # passes over the same tokens until about a second of wall time (some
        # 10-20 s of CPU work on a 16-core host), at most 16
        secs, passes = time_oracle(kind, case, 0, n, threads), 1
        while secs < 1.0 and passes < 16:
            secs += time_oracle(kind, case, 0, n, threads)
            passes += 1
        n1 = min(n, max(1, n // 8))
        secs1 = time_oracle(kind, case, 0, n1, 1)
        line["cpu_baseline"] = {"value": n * passes / secs, "unit": "tokens/s", "cores": threads,
                                "kind": "oracle",
                                "sample": f"the first {n} tokens of the same batch, {passes} "
                                          f"passes, {threads} threads ({secs:.2f} s wall)",
                                "single_thread_value": n1 / secs1,
                                "single_thread_sample": f"the first {n1} tokens, 1 thread",
                                "host_gbs": n * passes / secs * bytes_per_token(kind, case)
                                / 1e9,
                                "cpu": host_cpu()}
    if (rank == 0 and world == 1 and kind == "tp" and case.hidden == 4096 and case.top_k == 8
            and case.num_tokens >= 1024 and not (args.cold or args.graph)):
        line["data_movement"] = run_data_movement(torch, mf, job, sets, device)
    if rank == 0 and world == 1 and args.workload == "roofline" and not (
            args.cold or args.graph or args.no_other_configs):
        line["other_configs"] = run_other_configs(torch, mf, device, nvml)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_data_movement(torch, mf, job: Job, sets, device, rounds: int = 5,
                      launches: int = 100) -> dict:
    """The finalize against its own bytes moved with no arithmetic
    (mf.finalize_data_movement: route, valid rows and output row, one staged CTA
    per token) on the same buffers.  Blocks of back-to-back launches between one
    event pair each, the two kernels alternating block by block (launch i reads
    input copy i mod len(sets), as in the timed region); medians over the rounds."""
    stream = torch.cuda.current_stream(device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def finalize(i):
        job.launch(i, tensors=sets[i % len(sets)])

    def data_movement(i):
        g, w, idx, _nw, out = sets[i % len(sets)]
        mf.finalize_data_movement(g, w, idx, out)

    def block(fn) -> float:
        e0.record(stream)
        for i in range(launches):
            fn(i)
        e1.record(stream)
        torch.cuda.synchronize(device)
        return e0.elapsed_time(e1) * 1e3 / launches

    for fn in (finalize, data_movement):  # untimed
        fn(0)
    torch.cuda.synchronize(device)
    fin, dm = [], []
    for _ in range(rounds):
        fin.append(block(finalize))
        dm.append(block(data_movement))
    if mf.device_status(clear=True) != 0:
        raise SystemExit("device wait timeout in the data-movement comparison")
    fin_us, dm_us = float(np.median(fin)), float(np.median(dm))
    return {"kernel": "tp_data_movement_kernel", "finalize_kernel": job.kernel,
            "rounds": rounds, "launches_per_block": launches,
            "finalize_us": fin_us, "data_movement_us": dm_us,
            "data_movement_gbs": job.bytes_per_launch / (dm_us * 1e-6) / 1e9,
            "finalize_speed_vs_data_movement": dm_us / fin_us,
            "what": "the finalize's algorithmic bytes moved by a staged kernel with no "
                    "arithmetic, timed in alternating blocks with the finalize on the same "
                    "buffers"}


def input_copies(bytes_per_launch: int) -> int:
    """Copies of a workload's device buffers to rotate through, so that each
    launch's rows were last read at least 4 x L2 of traffic ago (1: a single
    launch already moves that much)."""
    b = max(int(bytes_per_launch), 1)
    if b >= 4 * L2_BYTES or b < L2_BYTES:  # cold by size, or warm by design (decode sizes)
        return 1
    return 1 + -(-4 * L2_BYTES // b)


def _same_layout_copy(torch, t):
    """A copy with the same strides (a padded row stride stays padded)."""
    c = torch.empty_strided(t.shape, t.stride(), dtype=t.dtype, device=t.device)
    return c.copy_(t)


def _timed_back_to_back(torch, job: Job, stream, device, launches: int, nvml: NvmlClock,
                        sets=None):
    """Average launch (ms) of `launches` back-to-back launches between one event
    pair, after five untimed ones; NVML samples taken while they run.  With
    `sets` (copies of the job's device buffers) launch i uses copy i mod n."""
    sets = sets or [None]

    def go(i):
        t = sets[i % len(sets)]
        if t is None:
            job.launch(i)
        else:
            job.launch(i, tensors=t)
    for i in range(5):
        go(i)
    torch.cuda.synchronize(device)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    inwin: list = []
    start.record(stream)
    for i in range(launches):
        go(i)
    end.record(stream)
    nvml.poll(end, inwin)
    torch.cuda.synchronize(device)
    return start.elapsed_time(end) / launches, inwin


def _timed_graph(torch, job: Job, device, launches: int, nvml: NvmlClock):
    """Average launch (ms) of `launches` launches replayed from one CUDA graph
    (warm: the inputs stay in L2), after one untimed replay."""
    for i in range(3):
        job.launch(i)
    torch.cuda.synchronize(device)
    graph = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream(device)
    cap.wait_stream(torch.cuda.current_stream(device))
    with torch.cuda.stream(cap), torch.cuda.graph(graph, stream=cap):
        for i in range(launches):
            job.launch(i)
    torch.cuda.synchronize(device)
    graph.replay()
    torch.cuda.synchronize(device)
    stream = torch.cuda.current_stream(device)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    inwin: list = []
    start.record(stream)
    graph.replay()
    end.record(stream)
    nvml.poll(end, inwin)
    torch.cuda.synchronize(device)
    return start.elapsed_time(end) / launches, inwin


def _timed_cold(torch, job: Job, stream, device, launches: int, nvml: NvmlClock, scratch):
    """Per-launch times (ms) with the L2 flushed before every launch (a write of
    twice its size, not timed) and an event pair around each launch."""
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(launches)]
    end = torch.cuda.Event()
    inwin: list = []
    for i in range(launches):
        scratch.fill_(i & 0xFF)
        ev[i][0].record(stream)
        job.launch(i)
        ev[i][1].record(stream)
    end.record(stream)
    nvml.poll(end, inwin)
    torch.cuda.synchronize(device)
    return [a.elapsed_time(b) for a, b in ev], inwin


def run_other_configs(torch, mf, device, nvml: NvmlClock) -> dict:
    """The other workloads of the path, timed on the same GPU after the
    headline: finalize of 16 tokens and the decode sizes (warm from one CUDA
    graph, and cold), finalize of 4096 tokens with padded rows, Beam of 8000
    live tokens and the residual op (back to back; inputs larger than L2)."""
    stream = torch.cuda.current_stream(device)
    peak, _ = measured_peaks()
    out: dict = {}

    def bandwidth_entry(job, launches, desc):
        # consecutive launches read different copies of the inputs: a workload of
        # a few L2 sizes would otherwise find part of its rows still in L2
        n = input_copies(job.bytes_per_launch)
        sets = [tuple(job.device_tensors)] + [
            tuple(None if t is None else _same_layout_copy(torch, t) for t in job.device_tensors)
            for _ in range(n - 1)]
        ms, inwin = _timed_back_to_back(torch, job, stream, device, launches, nvml, sets)
        del sets
        gbs = job.bytes_per_launch / (ms / 1e3) / 1e9
        return {"workload": desc, "kernel": job.kernel, "us_per_launch": ms * 1e3,
                "tokens_per_s": job.units_per_step / (ms / 1e3), "achieved_gbs": gbs,
                "frac": gbs / peak, "algorithmic_bytes_per_launch": job.bytes_per_launch,
                "traffic": recorded_traffic(job.kernel, job.name), "launches": launches,
                "timing": "one CUDA event pair around the back-to-back launches",
                "l2": (f"{n} copies of the inputs, launch i reads copy i mod {n}: each launch's "
                       "rows were last read at least 4 x L2 of traffic earlier") if n > 1 else
                      ("no flush: every launch reads its inputs from HBM "
                       f"({job.bytes_per_launch / 1e9:.3f} GB per launch, L2 is 0.13 GB)"),
                "clocks": nvml.summary(inwin)}

    scratch = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)

    def latency_entry(job, desc):
        warm_ms, win1 = _timed_graph(torch, job, device, 200, nvml)
        cold, win2 = _timed_cold(torch, job, stream, device, 30, nvml, scratch)
        return {"workload": desc, "kernel": job.kernel,
                "warm_us_per_launch": warm_ms * 1e3,
                "warm_timing": "200 launches replayed from one CUDA graph, inputs in L2",
                "cold_us_p10_p50_p90": [float(np.percentile(cold, q)) * 1e3 for q in (10, 50, 90)],
                "cold_timing": (f"L2 flushed before each of 30 launches ({L2_FLUSH_BYTES / 1e6:.0f}"
                                " MB scratch write, not timed), an event pair around each"),
                "algorithmic_bytes_per_launch": job.bytes_per_launch,
                "clocks": nvml.summary(win1 + win2)}

    kind, case, desc = workload_case("small", None, 0)
    out["finalize_T16"] = latency_entry(make_tp_job(torch, mf, case, device, "auto", False), desc)
    for T in si.DECODE_TOKENS:
        kind, case, desc = workload_case("decode", T, 0)
        out[f"decode_T{T}"] = latency_entry(make_tp_job(torch, mf, case, device, "auto", False),
                                            desc)
    del scratch

    kind, case, desc = workload_case("padded", None, 0)
    job = make_tp_job(torch, mf, case, device, "auto", False)
    out["finalize_T4096_stride4160"] = bandwidth_entry(job, 500, desc)
    del job

    kind, case, desc = workload_case("beam", None, 0)
    job = make_beam_job(torch, mf, case, device, "auto")
    out["beam_live8000"] = bandwidth_entry(job, 200, desc)
    del job
    kind, case, desc = workload_case("beam_residual", None, 0)
    job = make_beam_residual_job(torch, mf, case, device)
    out["beam_residual_live8000"] = bandwidth_entry(job, 200, desc)
    del job
    torch.cuda.synchronize(device)
    if mf.device_status(clear=True) != 0:
        raise SystemExit("device wait timeout while timing the other workloads")
    return out


def run_e2e(torch, mf, job: Job, kind: str, case, device, steps: int) -> dict:
    """Same metric through the public API with host buffers: every step copies
    its inputs from pinned host memory and reads its results back.  Steps are
    pipelined over two sets of device buffers: the upload of step i+1 runs
    while step i computes and downloads (uploads and downloads use separate
    streams; the host link is full duplex)."""
    n_out = getattr(job, "n_outputs", 1)
    dev0 = list(job.device_tensors)
    ins_idx = [i for i, t in enumerate(dev0[:-n_out]) if t is not None]
    outs_idx = list(range(len(dev0) - n_out, len(dev0)))
    # pinned host buffers: inputs hold the step's data, outputs receive the results
    host = {i: torch.empty(dev0[i].shape, dtype=dev0[i].dtype).pin_memory()
            for i in ins_idx + outs_idx}
    for i in ins_idx:
        host[i].copy_(dev0[i].cpu())
    dev1 = [None if t is None else torch.empty(t.shape, dtype=t.dtype, device=device) for t in dev0]
    sets = [dev0, dev1]
    h2d = sum(host[i].numel() * host[i].element_size() for i in ins_idx)
    d2h = sum(host[i].numel() * host[i].element_size() for i in outs_idx)
    s_in, s_cmp, s_out = (torch.cuda.Stream(device) for _ in range(3))
    main = torch.cuda.current_stream(device)
    in_done = [torch.cuda.Event() for _ in range(2)]
    cmp_done = [torch.cuda.Event() for _ in range(2)]
    out_done = [torch.cuda.Event() for _ in range(2)]

    def step(i):
        b = i % 2
        d = sets[b]
        if i >= 2:
            s_in.wait_event(cmp_done[b])      # step i-2 no longer reads this set
        with torch.cuda.stream(s_in):
            for k in ins_idx:
                d[k].copy_(host[k], non_blocking=True)
            in_done[b].record(s_in)
        s_cmp.wait_event(in_done[b])
        if i >= 2:
            s_cmp.wait_event(out_done[b])     # step i-2's results have been read back
        with torch.cuda.stream(s_cmp):
            job.launch(i, tensors=tuple(d))
            cmp_done[b].record(s_cmp)
        s_out.wait_event(cmp_done[b])
        with torch.cuda.stream(s_out):
            for k in outs_idx:
                host[k].copy_(d[k], non_blocking=True)
            out_done[b].record(s_out)

    for i in range(2):  # untimed: both buffer sets touched once
        step(i)
    torch.cuda.synchronize(device)
    # the host link on its own: one plain upload of the largest input (context
    # for the e2e figure, which the uploads bound)
    big = max(ins_idx, key=lambda k: host[k].numel() * host[k].element_size())
    nbytes = host[big].numel() * host[big].element_size()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(main)
    dev1[big].copy_(host[big], non_blocking=True)
    e1.record(main)
    torch.cuda.synchronize(device)
    link_gbs = nbytes / (e0.elapsed_time(e1) / 1e3) / 1e9
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(main)
    for st in (s_in, s_cmp, s_out):
        st.wait_stream(main)
    for i in range(steps):
        step(i)
    for st in (s_in, s_cmp, s_out):
        main.wait_stream(st)
    end.record(main)
    torch.cuda.synchronize(device)
    ms = reduce_max(start.elapsed_time(end))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    return {"value": job.units_per_step * steps * world / (ms / 1e3), "unit": "tokens/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps,
            "ms_per_step": ms / steps,
            "h2d_link_gbs": link_gbs,
            "pipeline": "uploads, launches and downloads on three streams, two buffer sets"}


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=("ours", "reference"), default="ours")
    p.add_argument("--workload", default="roofline",
                   choices=("roofline", "padded", "beam", "beam_residual", "small", "decode",
                            "custom", "beam_custom"))
    p.add_argument("--tokens", type=int, default=None,
                   help="token count of --workload decode / custom / beam_custom")
    p.add_argument("--hidden", type=int, default=4096, help="hidden size of --workload custom")
    p.add_argument("--top-k", type=int, default=8, help="top-k of --workload custom")
    p.add_argument("--weights", default="fp32", choices=("fp32", "bf16", "packed"),
                   help="routing weight storage of --workload custom")
    p.add_argument("--variant", default="auto", choices=("auto", "token_cta", "bulk", "cluster"))
    p.add_argument("--graph", action="store_true",
                   help="replay the timed launches from one CUDA graph (decode sizes)")
    p.add_argument("--no-pdl", action="store_true",
                   help="launch without programmatic dependent launch")
    p.add_argument("--cold", action="store_true",
                   help="before every timed launch write a scratch buffer of twice the L2 "
                        "size, and time each launch alone (cold-cache latency at small sizes)")
    p.add_argument("--e2e-steps", type=int, default=8)
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-other-configs", action="store_true",
                   help="skip the other workloads timed after the headline (default run only)")
    p.add_argument("--cpu-tokens", type=int, default=32768,
                   help="tokens of the batch the CPU oracle baseline processes")
    a = p.parse_args(argv)
    a.warmup = max(3, a.warmup)  # at least three untimed warm-up steps
    if a.cold and a.graph:
        p.error("--cold times every launch alone; it cannot be combined with --graph")
    return a


def main(argv=None) -> None:
    args = parse_args(argv)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
