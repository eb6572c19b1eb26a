"""Benchmark of the heterogeneous multi-LoRA linear layer on GB300.

One step = one lora_linear call (decode: stream-K GEMM with the fused shrink, then
the finishing pass with the expand; prefill: segment build, shrink, GEMM with the
fused expand) over one batch of synthetic seeded bf16 input. The headline is the
Llama-2-7B q_proj decode workload (T=64, 4096 -> 4096, 200 resident rank-16
adapters, alpha 32, ids uniform over 0..199); the same JSON line carries a record
per other workload under "configs": the tiny layer, a Llama-3-8B decoder layer's
seven target modules in one grouped call, the mixed-rank prefill (plain and
zero-padded to rank 64), the rank-16 prefill, the 2000-adapter Zipf pool at
T=256, and the specified hot-swap stream (1000 calls, 50 unload+reload cycles).

Timing. Inputs are resident in HBM. The K steps of a workload run back to back
from one CUDA graph over R "layers", each with its own W and adapter pool, step k
on layer k mod R; the layers together hold more than 3x the L2 size, so every
step reads its weights and adapter pages from HBM (no flush needed). The K-step
graph is replayed until at least 100 ms have been timed (at least 3 replays),
each replay bracketed by CUDA events on the launching stream; ms_per_step is the
median replay over K. Clocks are sampled during those replays.

Kernel times come from a device-side span trace (lora_pool_set_trace): every
CTA of every kernel of every step stamps the global timer at entry and exit, so
one kernel's launch duration is its last exit minus its first entry, measured
inside the same back-to-back graph with programmatic dependent launch intact.
roofline = the dominant kernel's algorithmic bytes (or flops) per launch over
that duration, against MEASURED_PEAKS.json; step_roofline = the whole step's
algorithmic bytes (or flops) over ms_per_step.

e2e = the same metric through lora_linear_host (pinned host X and ids in, host
Y out, copies and the final sync inside the measured time, L2 flushed before
each call). cpu_baseline = the fp64 CPU oracle on a bounded sample of the same
workload, on all host cores and on one core.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME|all]
  python bench.py --impl reference ...   (the oracle as the reference arm)
Multi-GPU (torchrun, one rank per GPU): replicas, no data-path collective; the
headline workload only.
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import lora_inputs as L  # noqa: E402

METRIC = ("LoRA-linear tokens/s, overhead vs base-only GEMM, adapter-path HBM GB/s "
          "(1×GB300)")
UNIT = "tokens/s"
GEMM_SRC = os.path.join(ROOT, "adapter_linear_gb300", "csrc", "gemm_decode.cu")
PROFILE = os.path.join(ROOT, "profiles", "gemm_decode_q_proj_T64.md")
KERNEL_SLOTS = ("segment_build", "shrink", "base_gemm", "finish_expand")
MIN_TIMED_MS = 100.0


# ----------------------------------------------------------------- workloads

def workload(name: str):
    """(Problem, config description) of a single-layer workload."""
    if name == "q_proj_decode":
        p = L.q_proj_decode()
        return p, {"workload": "Llama-2-7B q_proj decode", "T": 64, "d_in": 4096, "d_out": 4096,
                   "adapters": 200, "rank": 16, "alpha": 32, "ids": "uniform 0..199"}
    if name == "q_proj_decode_q4":
        p = L.q_proj_decode()
        return p, {"workload": "Llama-2-7B q_proj decode over a 4-bit base", "T": 64, "d_in": 4096,
                   "d_out": 4096, "adapters": 200, "rank": 16, "alpha": 32, "ids": "uniform 0..199",
                   "base": "4-bit codes, bf16 scale and 4-bit zero point per 128 inputs per row "
                           "(AWQ-INT4 layout); bf16 adapters"}
    if name == "hotswap_T256":
        p, _ = L.hotswap()
        return p, {"workload": "q_proj decode, 2000 paged adapters, Zipf ids", "T": 256,
                   "d_in": 4096, "d_out": 4096, "adapters": 2000, "rank": 16, "alpha": 32,
                   "ids": "Zipf(s=1) over 2000"}
    if name in ("prefill_mixed", "prefill_mixed_padded"):
        padded = name.endswith("padded")
        p = L.prefill_mixed(padded=padded)
        return p, {"workload": "gate_proj prefill, 8x2048 tokens, ranks 8..64" +
                   (", every adapter zero-padded to rank 64" if padded else ""),
                   "T": 16384, "d_in": 4096, "d_out": 14336, "adapters": 8,
                   "rank": "64 (padded from 8,8,16,16,32,32,64,64)" if padded else "8,8,16,16,32,32,64,64",
                   "alpha": "2*rank"}
    if name == "prefill_zipf":
        p = L.prefill_zipf()
        return p, {"workload": "q_proj-shaped prefill, 4096 tokens spread over 2000 adapters", "T": 4096,
                   "d_in": 4096, "d_out": 4096, "adapters": 2000, "rank": 16, "alpha": 32,
                   "ids": "Zipf(s=1) over 2000"}
    if name == "prefill_r16":  # the same prefill with every adapter at rank 16 (alpha 32)
        p = L.prefill_mixed(ranks=[16])
        return p, {"workload": "gate_proj prefill, 8x2048 tokens, rank 16", "T": 16384,
                   "d_in": 4096, "d_out": 14336, "adapters": 8, "rank": 16, "alpha": 32}
    if name == "prefill_small":  # same kernels and ranks, 8 x 512 tokens (for profiling)
        p = L.prefill_mixed(seq_len=512)
        return p, {"workload": "gate_proj prefill, 8x512 tokens, ranks 8..64", "T": 4096,
                   "d_in": 4096, "d_out": 14336, "adapters": 8, "rank": "8,8,16,16,32,32,64,64"}
    if name.startswith("llama3_") and name != "llama3_layer":
        mod = name[len("llama3_"):]
        (p,) = L.llama3_7mod(modules=[mod])
        return p, {"workload": f"Llama-3-8B {mod} decode", "T": 32, "d_in": p.d_in,
                   "d_out": p.d_out, "adapters": 32, "rank": 16, "alpha": 32}
    if name == "tiny":
        p = L.tiny()
        return p, {"workload": "tiny single linear", "T": 64, "d_in": 256, "d_out": 256,
                   "adapters": 4, "rank": 8, "alpha": 16, "ids": "uniform over {-1,0,1,2,3}"}
    raise SystemExit(f"unknown workload {name}")


def q4_base(p):
    """The 4-bit base of a q4 workload: codes, scales, zero points (weight std 1/64)."""
    return L.q4_weight(p.seed, p.d_out, p.d_in, 1.0 / 64)


def algorithmic_bytes(p, q4=False):
    """Bytes the layer must move once: X, W, Y, ids and the distinct adapters' A and B.
    A 4-bit W is its codes (half a byte per weight) and one bf16 scale and one byte of
    zero point per 128 weights."""
    T = p.T
    distinct = set(int(i) for i in p.ids if i >= 0)
    w = p.d_out * p.d_in // 2 + (p.d_in // 128) * p.d_out * 3 if q4 else p.d_out * p.d_in * 2
    return {
        "x": T * p.d_in * 2, "w": w, "y": T * p.d_out * 2, "ids": T * 4,
        "adapters": sum(p.adapters[i].rank * (p.d_in + p.d_out) * 2 for i in distinct),
        "adapter_A": sum(p.adapters[i].rank * p.d_in * 2 for i in distinct),
        "adapter_B": sum(p.adapters[i].rank * p.d_out * 2 for i in distinct),
    }


def step_bytes(ab):
    return ab["w"] + ab["x"] + ab["y"] + ab["ids"] + ab["adapters"]


def algorithmic_flops(p):
    lora = sum(2 * p.adapters[int(i)].rank * (p.d_in + p.d_out) for i in p.ids if i >= 0)
    return 2 * p.T * p.d_in * p.d_out + lora


# ------------------------------------------------------------------- clocks

class NvmlClockSampler:
    """SM clock and clock-event reasons read through NVML (read-only queries) every
    half millisecond while the timed region runs."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, torch_device):
        import ctypes
        self.ok = False
        self.samples = []
        self.max_mhz = None
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                return
            import torch
            props = torch.cuda.get_device_properties(torch_device)
            bus = f"{props.pci_domain_id:08X}:{props.pci_bus_id:02X}:{props.pci_device_id:02X}.0"
            h = ctypes.c_void_p()
            if nv.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(h)) != 0:
                return
            mx = ctypes.c_uint()
            if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = float(mx.value)
            self.reason_fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                nv.nvmlDeviceGetCurrentClocksThrottleReasons
            self.nv, self.h, self.ctypes = nv, h, ctypes
            self.ok = True
        except (OSError, AttributeError, ImportError):
            self.ok = False

    def _run(self):
        c = self.ctypes
        mhz, reasons = c.c_uint(), c.c_ulonglong()
        while not self.stop:
            if self.nv.nvmlDeviceGetClockInfo(self.h, 1, c.byref(mhz)) == 0 and \
                    self.reason_fn(self.h, c.byref(reasons)) == 0:
                self.samples.append((float(mhz.value), int(reasons.value)))
            time.sleep(0.0005)

    def __enter__(self):
        if self.ok:
            self.stop = False
            self.thread = threading.Thread(target=self._run, daemon=True)
            self.thread.start()
        return self

    def __exit__(self, *exc):
        if self.ok:
            self.stop = True
            self.thread.join(timeout=5)

    def summary(self):
        if not self.samples:
            return None
        reasons = sorted({name for _, r in self.samples for bit, name in self.REASONS.items()
                          if r & bit})
        return {"sm_mhz": statistics.median(s for s, _ in self.samples),
                "sm_max_mhz": self.max_mhz, "reasons": reasons, "samples": len(self.samples),
                "source": "nvml"}


class ClockSampler:
    """nvidia-smi samples every 200 ms while the timed region runs (a fall-back when NVML
    cannot be loaded)."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                mx = float(f[1])
            except ValueError:
                continue
            for n, v in zip(names, f[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": 0,
                    "source": "nvidia-smi"}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm), "source": "nvidia-smi"}


class Clocks:
    """NVML samples, or nvidia-smi ones when NVML is unavailable."""

    def __init__(self, dev):
        self.nvml = NvmlClockSampler(dev)
        self.smi = None if self.nvml.ok else ClockSampler(dev.index or 0)

    def __enter__(self):
        (self.nvml if self.smi is None else self.smi).__enter__()
        return self

    def __exit__(self, *exc):
        (self.nvml if self.smi is None else self.smi).__exit__(*exc)

    def summary(self):
        return self.nvml.summary() if self.smi is None else self.smi.summary()


# --------------------------------------------------------------- profile data

def source_digest(path=GEMM_SRC) -> str:
    h = hashlib.sha256()
    for f in (path, os.path.join(os.path.dirname(path), "device_common.cuh")):
        h.update(open(f, "rb").read())
    return h.hexdigest()[:16]


def profiled_traffic(workload_name: str):
    """DRAM bytes per launch of the decode GEMM from the committed ncu summary, if it was
    taken on this workload (the default q_proj decode) with the current kernel source
    (else None)."""
    if workload_name != "q_proj_decode" or not os.path.exists(PROFILE):
        return None
    text = open(PROFILE).read()
    m_src = re.search(r"source_digest:\s*([0-9a-f]+)", text)
    m_bytes = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not m_src or not m_bytes or m_src.group(1) != source_digest():
        return None
    return float(m_bytes.group(1))


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return {"hbm_gbs": d.get("hbm_gbs"), "bf16_tflops": d.get("bf16_tflops"),
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


# --------------------------------------------------------------- cpu oracle

def cpu_oracle_rate(p, seconds: float, max_tokens: int):
    """tokens/s of the fp64 oracle on the first `n` tokens of the batch, repeated until
    `seconds` of wall time."""
    import oracle
    ads = oracle.problem_adapters(p)
    n = min(max_tokens, p.T)
    X, ids = p.X[:n], p.ids[:n]
    done, t0 = 0, time.perf_counter()
    while True:
        oracle.lora_linear(X, p.W, ids, ads, p.max_adapters)
        done += n
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    return done / el, oracle.num_threads(), f"{n} of {p.T} tokens per pass, {done} tokens in {el:.1f} s"


def cpu_oracle_one_core(name: str, seconds: float, max_tokens: int):
    """The same measurement in a child process with OpenMP held to one thread."""
    env = dict(os.environ, OMP_NUM_THREADS="1")
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--cpu-probe", name,
           "--cpu-seconds", str(seconds), "--cpu-tokens", str(max_tokens)]
    r = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=600)
    if r.returncode != 0:
        return None
    return json.loads(r.stdout.strip().splitlines()[-1])


def cpu_baselines(name: str, p, seconds: float, tokens: int, one_core_seconds: float,
                  one_core_tokens: int):
    rate, cores, sample = cpu_oracle_rate(p, seconds, tokens)
    out = {"value": rate, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample}
    one = cpu_oracle_one_core(name, one_core_seconds, one_core_tokens)
    if one is not None:
        out["one_core"] = {"value": one["value"], "unit": UNIT, "cores": one["cores"],
                           "sample": one["sample"] + " (tokens/s of a sample extrapolate to the "
                                                     "whole batch: the work is the same per token)"}
    return out


# ------------------------------------------------------------- measurement kit

class Kit:
    """Device, stream, helpers shared by the workload measurements."""

    def __init__(self, args):
        import torch
        import adapter_linear_gb300 as al
        self.torch, self.al, self.args = torch, al, args
        ws, rank, local = dist_env()
        self.ws, self.rank = ws, rank
        if ws > 1:
            import torch.distributed as dist
            torch.cuda.set_device(local)
            dist.init_process_group("nccl")
        self.dev = torch.device("cuda", local if ws > 1 else 0)
        torch.cuda.set_device(self.dev)
        self.stream = torch.cuda.current_stream(self.dev)
        self.l2 = torch.cuda.get_device_properties(self.dev).L2_cache_size
        self.flush = torch.empty(2 * self.l2 // 4 + 1024, dtype=torch.float32, device=self.dev)
        self.peaks = measured_peaks()
        self.graphs = []

    def t(self, a):
        torch = self.torch
        if a.dtype == np.uint16:
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(self.dev)
        return torch.from_numpy(np.ascontiguousarray(a)).to(self.dev)

    def barrier(self):
        if self.ws > 1:
            self.torch.distributed.barrier()
        self.torch.cuda.synchronize(self.dev)

    def capture(self, step, n):
        """n consecutive steps captured as one CUDA graph; returns its replay."""
        torch = self.torch
        if self.args.no_graph:
            return lambda: [step(k) for k in range(n)]
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for k in range(n):
                step(k)
        self.graphs.append(g)
        return g.replay

    def time_once(self, prog):
        torch = self.torch
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(self.stream)
        prog()
        e1.record(self.stream)
        torch.cuda.synchronize(self.dev)
        return e0.elapsed_time(e1)

    def time_replays(self, prog, min_ms=MIN_TIMED_MS, min_reps=3):
        """Replays of one K-step program, each timed on its own, until min_ms in all."""
        out = []
        while len(out) < min_reps or sum(out) < min_ms:
            self.barrier()
            out.append(self.time_once(prog))
        return out

    def spans(self, calls_of_pools, capture_fn, K, R, replays=3):
        """Per-kernel times from the span trace of one K-step program.

        calls_of_pools: the pools that carry the trace, one per layer (step k uses layer
        k mod R); capture_fn(): captures the K-step program. For every step after the
        first, each kernel gets
          share: its last CTA exit minus the last exit of the kernel before it in the
                 stream (the previous step's last kernel for the first one): the
                 kernels' shares of a step add up to the step period exactly;
          span:  its last exit minus its first CTA entry (under programmatic dependent
                 launch a kernel's CTAs enter, and stream weights, while the kernel
                 before it still runs, so spans overlap and can exceed the step);
          active: its last exit minus the first moment a CTA got past its wait.
        Returns the means over the steps (ms) of each, per kernel slot."""
        torch = self.torch
        W = 4  # words per kernel slot
        per_layer = [len(range(j, K, R)) for j in range(R)]
        buf = torch.zeros((R, max(per_layer), len(KERNEL_SLOTS), W), dtype=torch.int64,
                          device=self.dev)
        for j, pool in enumerate(calls_of_pools):
            if per_layer[j] > 0:
                pool.set_trace(buf[j], per_layer[j])
        prog = capture_fn()
        for pool in calls_of_pools:
            pool.set_trace(None)
        share = {s: [] for s in KERNEL_SLOTS}
        span = {s: [] for s in KERNEL_SLOTS}
        active = {s: [] for s in KERNEL_SLOTS}
        windows = []
        periods = {}  # step index -> its periods (last exit minus the step before's), ms
        step_share = {}  # step index -> {kernel slot -> its shares}
        big = 2 ** 63 - 1
        for _ in range(replays):
            buf[..., 0].fill_(big)
            buf[..., 1].fill_(0)
            buf[..., 2].fill_(big)
            buf[..., 3].fill_(0)
            self.barrier()
            prog()
            self.barrier()
            b = buf.cpu().numpy()

            def used(k):
                e = b[k % R, k // R]
                return e, [si for si in range(len(KERNEL_SLOTS)) if e[si, 1] > 0]

            for k in range(1, K):
                ep, up = used(k - 1)
                e, u = used(k)
                if not u or not up:
                    continue
                prev_exit = ep[up[-1], 1]
                periods.setdefault(k, []).append((e[u[-1], 1] - prev_exit) * 1e-6)
                for si in u:
                    name = KERNEL_SLOTS[si]
                    share[name].append((e[si, 1] - prev_exit) * 1e-6)
                    step_share.setdefault(k, {}).setdefault(name, []).append((e[si, 1] - prev_exit) * 1e-6)
                    span[name].append((e[si, 1] - e[si, 0]) * 1e-6)
                    active[name].append((e[si, 1] - e[si, 2]) * 1e-6)
                    prev_exit = e[si, 1]
                windows.append((e[u[-1], 1] - e[u, 0].min()) * 1e-6)

        def means(d):
            return {s: (statistics.mean(v) if v else 0.0) for s, v in d.items()}
        return {"share": means(share), "span": means(span), "active": means(active),
                "step_window": statistics.mean(windows) if windows else 0.0, "periods": periods,
                "step_share": step_share}

    def paired_overhead(self, pools, capture_alt, K, R):
        """LoRA overhead from one graph whose steps alternate base-only (even k) and LoRA
        (odd k) calls: every step's period comes from the span trace, so both kinds are
        measured under the same clocks (a long prefill run lowers them under the power
        cap). Returns (LoRA / base - 1, mean LoRA period, mean base period) in ms."""
        tr = self.spans(pools, capture_alt, K, R, replays=5)
        lo = [v for k, vs in tr["periods"].items() if k % 2 == 1 for v in vs]
        ba = [v for k, vs in tr["periods"].items() if k % 2 == 0 for v in vs]
        if not lo or not ba:
            return None, None, None, {}
        ml, mb = statistics.mean(lo), statistics.mean(ba)

        def by_kernel(parity):
            acc = {}
            for k, d in tr["step_share"].items():
                if k % 2 == parity:
                    for name, vs in d.items():
                        acc.setdefault(name, []).extend(vs)
            return {name: statistics.mean(vs) for name, vs in acc.items()}
        return ml / mb - 1.0, ml, mb, {"lora": by_kernel(1), "base": by_kernel(0)}

    def replay_overhead(self, base_prog, lora_prog, min_ms=MIN_TIMED_MS):
        """LoRA and base-only K-step graphs replayed in the order base, LoRA, LoRA, base
        until min_ms of LoRA time (decode steps overlap their neighbours under
        programmatic dependent launch, so their periods cannot be paired step by step;
        they are short enough not to move the clocks). Returns mean ms per replay."""
        b, l_ = [], []
        base_prog()
        while len(l_) < 4 or sum(l_) < min_ms:
            b.append(self.time_once(base_prog))
            l_.append(self.time_once(lora_prog))
            l_.append(self.time_once(lora_prog))
            b.append(self.time_once(base_prog))
        return sum(l_) / len(l_), sum(b) / len(b)

    def iso_call(self, one_step, n):
        prog = self.capture(lambda k: one_step(), 1)
        iso = []
        for i in range(n):
            self.flush.fill_(float(i))
            iso.append(self.time_once(prog))
        return statistics.median(iso)


def roofline_decode(ab, gemm_ms, peaks, traffic, kernel="gemm_decode_kernel"):
    gemm_bytes = ab["w"] + ab["x"] + ab["adapter_A"]
    achieved = gemm_bytes / (gemm_ms * 1e-3) / 1e9 if gemm_ms > 0 else None
    return {"kernel": kernel, "bound": "hbm", "achieved": achieved,
            "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": achieved / peaks["hbm_gbs"] if achieved else None, "traffic": traffic,
            "algorithmic_bytes": gemm_bytes,
            "per_unit": "W + X + the distinct adapters' A pages (the kernel also runs the shrink)",
            "launch_ms": gemm_ms,
            "timing": "the kernel's critical-path share of the back-to-back step (span trace): "
                      "its last CTA exit minus the finishing pass's last exit of the step before; "
                      "its W prefetch before the wait overlaps that pass, as the pass's B loads "
                      "overlap this kernel",
            "peak_source": peaks["source"]}


def roofline_prefill(p, gemm_ms, peaks, kname):
    flops = 2.0 * p.T * p.d_in * p.d_out
    achieved = flops / (gemm_ms * 1e-3) / 1e12 if gemm_ms > 0 else None
    return {"kernel": kname, "bound": "tensor", "achieved": achieved,
            "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
            "frac": achieved / peaks["bf16_tflops"] if achieved else None,
            "frac_of_sustained": achieved / peaks["bf16_tflops_sustained"]
            if achieved and peaks.get("bf16_tflops_sustained") else None,
            "traffic": None, "algorithmic_flops": flops,
            "per_unit": "2 * T * d_in * d_out (the base product; the fused expand is not counted)",
            "launch_ms": gemm_ms,
            "timing": "the kernel's critical-path share of the back-to-back step (span trace): "
                      "its last CTA exit minus the shrink kernel's last exit",
            "peak_source": peaks["source"]}


# ------------------------------------------------------- single-layer workloads

def measure_layer(kit: Kit, name: str, K: int, with_e2e=True, headline=False):
    """A record for one single-layer workload (one lora_linear call per step)."""
    torch, al, args = kit.torch, kit.al, kit.args
    p, cfg = workload(name)
    q4 = name.endswith("_q4")
    if q4:
        with_e2e = False  # the host-buffer entry point takes a bf16 base
    A_dev = {s: kit.t(ad.A) for s, ad in p.adapters.items()}
    B_dev = {s: kit.t(ad.B) for s, ad in p.adapters.items()}

    def new_layer(W):
        pool = al.LoraPool(p.max_adapters, p.max_rank, p.d_in, p.d_out)
        for slot, ad in p.adapters.items():
            pool.load_adapter(slot, A_dev[slot], B_dev[slot], ad.rank, ad.alpha)
        pool.reserve(p.T)
        return pool, W

    # R layers, each its own W and adapter pool (like the layers of a model): the
    # layers' footprint is more than 3x L2, so no flush is needed between steps
    W0 = tuple(kit.t(a) for a in q4_base(p)) if q4 else (kit.t(p.W),)
    layers = [new_layer(W0)]
    layer_bytes = sum(t.numel() * t.element_size() for t in W0) + layers[0][0].stats()["bytes_held"]
    R = max(2, min(32, -(-3 * kit.l2 // layer_bytes)))
    while len(layers) < R:
        layers.append(new_layer(tuple(t.clone() for t in W0)))
    del A_dev, B_dev
    X, ids = kit.t(p.X), kit.t(p.ids)
    Y = torch.empty((p.T, p.d_out), dtype=torch.bfloat16, device=kit.dev)

    def lora_step(k):
        pool, W = layers[k % R]
        if q4:
            pool.linear_q4(X, *W, ids, Y)
        else:
            pool.linear(X, W[0], ids, Y)

    def base_step(k):
        pool, W = layers[k % R]
        if q4:
            pool.base_linear_q4(X, *W, Y)
        else:
            pool.base_linear(X, W[0], Y)

    for k in range(max(args.warmup, R)):
        lora_step(k)
        base_step(k)
    kit.barrier()
    lora_prog = kit.capture(lora_step, K)
    kit.capture(lora_step, args.warmup)()
    kit.barrier()

    # ---- timed: replays of exactly K back-to-back steps, >= 100 ms in all
    clocks = Clocks(kit.dev)
    with clocks:
        reps = kit.time_replays(lora_prog)
    reps = [max_over_ranks(r, kit.ws, kit.dev) for r in reps]
    total_ms = statistics.median(reps)
    value = job_tokens_per_s(p.T * K, kit.ws, total_ms)

    def alt_step(k):  # even steps base-only, odd steps LoRA
        (base_step if k % 2 == 0 else lora_step)(k)

    decode = p.T <= 256
    Kp = max(K, 20)
    paired_kernels = None
    if decode:
        base_prog = kit.capture(base_step, K)
        lora_rep, base_rep = kit.replay_overhead(base_prog, lora_prog)
        lora_ms, base_ms = lora_rep / K, base_rep / K
        overhead = lora_ms / base_ms - 1.0
        overhead_how = ("base-only, LoRA, LoRA, base-only replays of the K-step graphs, repeated "
                        f"to >= {MIN_TIMED_MS:.0f} ms of LoRA time")
    else:
        overhead, lora_ms, base_ms, paired_kernels = kit.paired_overhead(
            [pool for pool, _ in layers], lambda: kit.capture(alt_step, Kp), Kp, R)
        overhead_how = (f"one graph of {Kp} steps alternating base-only and LoRA calls (5 "
                        "replays); each step's period from the span trace, so both kinds run "
                        "under the same clocks")
    tr = kit.spans([pool for pool, _ in layers], lambda: kit.capture(lora_step, K), K, R)
    base_tr = kit.spans([pool for pool, _ in layers], lambda: kit.capture(base_step, K), K, R)
    iso_ms = kit.iso_call(lambda: lora_step(0), min(K, 50))

    e2e = None
    if with_e2e:
        pool0, (W,) = layers[0]
        Xh = torch.from_numpy(p.X.view(np.int16)).view(torch.bfloat16).pin_memory()
        idh = torch.from_numpy(p.ids).pin_memory()
        Yh = torch.empty((p.T, p.d_out), dtype=torch.bfloat16).pin_memory()
        for _ in range(3):
            pool0.linear_host(Xh, W, idh, Yh)
        n_e2e = max(3, min(K, 200 if p.T <= 256 else 10))
        e2e_s = 0.0
        for i in range(n_e2e):
            kit.flush.fill_(float(i))
            torch.cuda.synchronize(kit.dev)
            t0 = time.perf_counter()
            pool0.linear_host(Xh, W, idh, Yh)
            e2e_s += time.perf_counter() - t0
        ab0 = algorithmic_bytes(p)
        e2e = {"value": p.T * n_e2e * kit.ws / e2e_s, "unit": UNIT,
               "h2d_bytes_per_step": ab0["x"] + ab0["ids"], "d2h_bytes_per_step": ab0["y"],
               "calls": n_e2e}
    for pool, _ in layers:
        assert pool.check_errors() == al.LORA_OK
    kit.barrier()

    ab = algorithmic_bytes(p, q4)
    step_ms = total_ms / K
    gemm_share = tr["share"]["base_gemm"]
    if decode:
        roof = roofline_decode(ab, gemm_share, kit.peaks,
                               profiled_traffic(name) if headline else None,
                               "gemm_decode_q4_kernel" if q4 else "gemm_decode_kernel")
        sb = step_bytes(ab)
        step_roof = {"bound": "hbm", "achieved": sb / (step_ms * 1e-3) / 1e9, "unit": "GB/s",
                     "peak": kit.peaks["hbm_gbs"],
                     "frac": sb / (step_ms * 1e-3) / 1e9 / kit.peaks["hbm_gbs"],
                     "algorithmic_bytes": sb,
                     "per_unit": "W + X + Y + ids + the distinct adapters' A and B, per step"}
    else:
        kname = "gemm_prefill_pair_kernel" if p.T > 128 else "gemm_prefill_kernel"
        roof = roofline_prefill(p, gemm_share, kit.peaks, kname)
        fl = algorithmic_flops(p)
        step_roof = {"bound": "tensor", "achieved": fl / (step_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                     "peak": kit.peaks["bf16_tflops"],
                     "frac": fl / (step_ms * 1e-3) / 1e12 / kit.peaks["bf16_tflops"],
                     "algorithmic_flops": fl,
                     "per_unit": "2 T d_in d_out + the low-rank flops of every adapter token"}
    extra_ms = lora_ms - base_ms
    rec = {
        "metric": METRIC, "value": value, "unit": UNIT, "ms_per_step": step_ms,
        "tokens_per_step": p.T,
        "config": dict(cfg, layers=R,
                       l2=f"inputs larger than L2: {R} layers, each its own W and adapter pool "
                          f"({R * layer_bytes / 1e6:.0f} MB cycled), step k uses layer k mod {R}",
                       launch="direct" if args.no_graph else "one CUDA graph of the K steps"),
        "timing": {"replays": len(reps), "replay_ms_min": min(reps), "replay_ms_median": total_ms,
                   "replay_ms_max": max(reps),
                   "rule": f"median of replays of the K-step graph, >= {MIN_TIMED_MS:.0f} ms timed"},
        "overhead_vs_base": overhead,
        "overhead_floor": (ab["adapters"] / (ab["w"] + ab["x"] + ab["y"]) if decode
                           else (algorithmic_flops(p) - 2.0 * p.T * p.d_in * p.d_out) /
                           (2.0 * p.T * p.d_in * p.d_out)),
        "overhead_floor_kind": "adapter bytes / base bytes" if decode else "LoRA flops / base flops",
        "base_only_ms_per_step": base_ms,
        "lora_ms_per_step_in_overhead_run": lora_ms,
        "overhead_measured_on": overhead_how,
        "paired_kernel_ms": paired_kernels,
        "isolated_call_ms": iso_ms,
        "adapter_path_gbs": ab["adapters"] / (extra_ms * 1e-3) / 1e9 if (decode and extra_ms > 0) else None,
        "kernel_ms": {k: v for k, v in tr["share"].items() if v > 0},
        "kernel_span_ms": {k: v for k, v in tr["span"].items() if v > 0},
        "kernel_active_ms": {k: v for k, v in tr["active"].items() if v > 0},
        "kernel_timing": "span trace inside the back-to-back graph; kernel_ms = each kernel's "
                         "critical-path share of the step (its last CTA exit minus the last exit "
                         "of the kernel before it in the stream; the shares add up to the step); "
                         "span = last exit - first entry (overlaps the neighbours under "
                         "programmatic dependent launch); active = last exit - first release "
                         "from the wait on the previous kernel",
        "base_only_kernel_ms": {k: v for k, v in base_tr["share"].items() if v > 0},
        "step_window_ms": tr["step_window"],
        "roofline": roof,
        "step_roofline": step_roof,
        "tflops": algorithmic_flops(p) / (step_ms * 1e-3) / 1e12,
        "clocks": clocks.summary(),
        "e2e": e2e,
        "gpu_launches": (2 if decode else 3) * K,
    }
    for pool, _ in layers:
        pool.close()
    del layers
    torch.cuda.empty_cache()
    return rec, p


# ------------------------------------------------------- grouped layer (7 modules)

def measure_grouped_layer(kit: Kit, K: int):
    """A Llama-3-8B decoder layer's seven target modules (q,k,v,o,gate,up,down; T = 32,
    32 adapters r16 per module, one id vector) per step: one lora_linear_grouped call,
    against seven separate lora_linear calls and the grouped base-only call."""
    torch, al, args = kit.torch, kit.al, kit.args
    probs = L.llama3_7mod()
    T = probs[0].T
    Xs = [kit.t(p.X) for p in probs]
    ids = kit.t(probs[0].ids)
    Ys = [torch.empty((T, p.d_out), dtype=torch.bfloat16, device=kit.dev) for p in probs]

    def new_layer():
        pools, Ws = [], []
        for p in probs:
            pool = al.LoraPool(p.max_adapters, p.max_rank, p.d_in, p.d_out)
            for slot, ad in p.adapters.items():
                pool.load_adapter(slot, kit.t(ad.A), kit.t(ad.B), ad.rank, ad.alpha)
            pool.reserve(T)
            pools.append(pool)
            Ws.append(kit.t(p.W))
        return pools, Ws

    layers = [new_layer()]
    layer_bytes = sum(w.numel() * 2 for w in layers[0][1]) + \
        sum(pl.stats()["bytes_held"] for pl in layers[0][0])
    R = max(2, -(-3 * kit.l2 // layer_bytes))
    while len(layers) < R:
        layers.append(new_layer())
    no_ids = torch.full_like(ids, -1)

    def grouped_step(k):
        pools, Ws = layers[k % R]
        al.LoraPool.linear_grouped(pools, Xs, Ws, ids, Ys)

    def separate_step(k):
        pools, Ws = layers[k % R]
        for m, pool in enumerate(pools):
            pool.linear(Xs[m], Ws[m], ids, Ys[m])

    def grouped_base_step(k):  # the same grouped call with every token on the base path
        pools, Ws = layers[k % R]
        al.LoraPool.linear_grouped(pools, Xs, Ws, no_ids, Ys)

    for k in range(max(args.warmup, R)):
        grouped_step(k)
        separate_step(k)
        grouped_base_step(k)
    kit.barrier()
    g_prog = kit.capture(grouped_step, K)
    s_prog = kit.capture(separate_step, K)
    kit.capture(grouped_step, args.warmup)()
    kit.barrier()

    clocks = Clocks(kit.dev)
    with clocks:
        reps = kit.time_replays(g_prog)
    total_ms = statistics.median(reps)
    sep_ms = statistics.median(kit.time_replays(s_prog))
    gb_prog = kit.capture(grouped_base_step, K)
    lora_rep, base_rep = kit.replay_overhead(gb_prog, g_prog)
    lora_ms, base_ms = lora_rep / K, base_rep / K
    overhead = lora_ms / base_ms - 1.0
    tr = kit.spans([pools[0] for pools, _ in layers], lambda: kit.capture(grouped_step, K), K, R)

    # e2e: pinned host inputs copied in, the grouped call, outputs copied back
    Xh = [x.cpu().pin_memory() for x in Xs]
    idh = ids.cpu().pin_memory()
    Yh = [torch.empty(y.shape, dtype=y.dtype).pin_memory() for y in Ys]
    Xd = [torch.empty_like(x) for x in Xs]
    idd = torch.empty_like(ids)
    pools0, Ws0 = layers[0]

    def e2e_once():
        for a, b in zip(Xd, Xh):
            a.copy_(b, non_blocking=True)
        idd.copy_(idh, non_blocking=True)
        al.LoraPool.linear_grouped(pools0, Xd, Ws0, idd, Ys)
        for a, b in zip(Yh, Ys):
            a.copy_(b, non_blocking=True)
        torch.cuda.synchronize(kit.dev)

    for _ in range(3):
        e2e_once()
    n_e2e = max(3, min(K, 100))
    e2e_s = 0.0
    for _ in range(n_e2e):
        kit.flush.fill_(1.0)
        torch.cuda.synchronize(kit.dev)
        t0 = time.perf_counter()
        e2e_once()
        e2e_s += time.perf_counter() - t0
    for pools, _ in layers:
        for pool in pools:
            assert pool.check_errors() == al.LORA_OK

    abs_ = [algorithmic_bytes(p) for p in probs]
    w_b = sum(a["w"] for a in abs_)
    x_b = sum(a["x"] for a in abs_)
    y_b = sum(a["y"] for a in abs_)
    ad_a = sum(a["adapter_A"] for a in abs_)
    ad_all = sum(a["adapters"] for a in abs_)
    gemm_bytes = w_b + x_b + ad_a
    step_ms = total_ms / K
    gemm_ms = tr["share"]["base_gemm"]
    sb = w_b + x_b + y_b + T * 4 + ad_all
    rec = {
        "metric": METRIC, "value": T * K / (total_ms / 1e3), "unit": UNIT,
        "value_note": "tokens/s of the layer (each token through all seven modules)",
        "ms_per_step": step_ms, "tokens_per_step": T,
        "config": {"workload": "Llama-3-8B decoder layer, 7 target modules in one grouped call",
                   "T": T, "modules": [p.name.split("/")[1] for p in probs], "adapters": 32,
                   "rank": 16, "alpha": 32, "base_only_tokens": "4 of 32", "layers": R,
                   "l2": f"inputs larger than L2: {R} layers of 7 modules, each its own W and "
                         f"pools ({R * layer_bytes / 1e6:.0f} MB cycled)",
                   "launch": "one CUDA graph of the K steps"},
        "timing": {"replays": len(reps), "replay_ms_median": total_ms,
                   "rule": f"median of replays of the K-step graph, >= {MIN_TIMED_MS:.0f} ms timed"},
        "separate_calls_ms_per_step": sep_ms / K,
        "base_only_ms_per_step": base_ms,
        "overhead_vs_base": overhead,
        "overhead_measured_on": "grouped base-only, LoRA, LoRA, base-only replays of the K-step "
                                f"graphs, repeated to >= {MIN_TIMED_MS:.0f} ms of LoRA time",
        "overhead_floor": ad_all / (w_b + x_b + y_b),
        "overhead_floor_kind": "adapter bytes / base bytes",
        "kernel_ms": {k: v for k, v in tr["share"].items() if v > 0},
        "kernel_span_ms": {k: v for k, v in tr["span"].items() if v > 0},
        "kernel_active_ms": {k: v for k, v in tr["active"].items() if v > 0},
        "step_window_ms": tr["step_window"],
        "roofline": {"kernel": "gemm_decode_kernel (7-layer problem table)", "bound": "hbm",
                     "achieved": gemm_bytes / (gemm_ms * 1e-3) / 1e9 if gemm_ms else None,
                     "peak": kit.peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": gemm_bytes / (gemm_ms * 1e-3) / 1e9 / kit.peaks["hbm_gbs"] if gemm_ms else None,
                     "traffic": None, "algorithmic_bytes": gemm_bytes,
                     "per_unit": "the seven W + X + the distinct adapters' A pages",
                     "launch_ms": gemm_ms, "peak_source": kit.peaks["source"]},
        "step_roofline": {"bound": "hbm", "achieved": sb / (step_ms * 1e-3) / 1e9, "unit": "GB/s",
                          "peak": kit.peaks["hbm_gbs"],
                          "frac": sb / (step_ms * 1e-3) / 1e9 / kit.peaks["hbm_gbs"],
                          "algorithmic_bytes": sb},
        "clocks": clocks.summary(),
        "e2e": {"value": T * n_e2e / e2e_s, "unit": UNIT, "h2d_bytes_per_step": x_b + T * 4,
                "d2h_bytes_per_step": y_b, "calls": n_e2e},
        "gpu_launches": 2 * K,
    }
    for pools, _ in layers:
        for pool in pools:
            pool.close()
    del layers
    torch.cuda.empty_cache()
    return rec


# ------------------------------------------------- hot-swap stream (as specified)

def measure_hotswap_stream(kit: Kit):
    """1000 calls of 256 tokens over 2000 r16 adapters with Zipf ids (a new id vector
    every call), with one unload + reload of a slot in every block of 20 calls (50
    cycles), all through the public API; the same 1000 calls without the swaps give
    the swap cost."""
    torch, al, args = kit.torch, kit.al, kit.args
    p, sched = L.hotswap()
    pool = al.LoraPool(p.max_adapters, p.max_rank, p.d_in, p.d_out)
    for slot, ad in p.adapters.items():
        pool.load_adapter(slot, kit.t(ad.A), kit.t(ad.B), ad.rank, ad.alpha)
    pool.reserve(p.T)
    pool.set_path(al.LORA_PATH_DECODE)
    X, W = kit.t(p.X), kit.t(p.W)
    ids = kit.t(sched.ids)                                 # [calls, T]
    Y = torch.empty((p.T, p.d_out), dtype=torch.bfloat16, device=kit.dev)
    swaps = {c: (slot, gen) for c, slot, gen in sched.swaps}
    fresh = {}
    for c, (slot, gen) in swaps.items():
        ad = L.make_adapter(p.seed, slot, p.d_in, p.d_out, 16, 32.0, generation=gen)
        fresh[c] = (kit.t(ad.A), kit.t(ad.B))
    old = {c: (kit.t(p.adapters[slot].A), kit.t(p.adapters[slot].B)) for c, (slot, _) in swaps.items()}

    def run(with_swaps, restore):
        for c in range(sched.calls):
            pool.linear(X, W, ids[c], Y)
            if with_swaps and c in swaps:
                slot, _ = swaps[c]
                pool.unload_adapter(slot)
                A, B = (old if restore else fresh)[c]
                pool.load_adapter(slot, A, B, 16, 32.0)

    for _ in range(args.warmup):
        pool.linear(X, W, ids[0], Y)
    torch.cuda.synchronize(kit.dev)

    def timed(fn):
        torch.cuda.synchronize(kit.dev)
        t0 = time.perf_counter()
        fn()
        torch.cuda.synchronize(kit.dev)
        return time.perf_counter() - t0

    clocks = Clocks(kit.dev)
    swap_s, nosw_s = [], []
    with clocks:
        for _ in range(3):
            swap_s.append(timed(lambda: run(True, False)))
            timed(lambda: run(True, True))                 # put the first generation back
            nosw_s.append(timed(lambda: run(False, False)))
    assert pool.check_errors() == al.LORA_OK
    sw, ns = statistics.median(swap_s), statistics.median(nosw_s)
    n_tok = p.T * sched.calls
    rec = {
        "metric": METRIC, "value": n_tok / sw, "unit": UNIT,
        "ms_per_step": 1e3 * sw / sched.calls, "tokens_per_step": p.T,
        "config": {"workload": "hot-swap stream: 1000 calls x 256 tokens, 2000 x r16 adapters, "
                               "Zipf ids, 50 unload+reload cycles", "T": p.T, "d_in": p.d_in,
                   "d_out": p.d_out, "adapters": p.max_adapters, "rank": 16, "alpha": 32,
                   "launch": "direct calls; a swap orders itself after the calls enqueued before "
                             "it on the GPU, with no device-wide synchronisation",
                   "l2": "one W (33.5 MB) stays in L2 across calls; the 2000 adapters' pages "
                         "(524 MB) do not"},
        "timing": {"rule": "median of 3 passes of the 1000-call stream, host wall clock around "
                           "each (synchronised before and after)"},
        "no_swap_ms_per_step": 1e3 * ns / sched.calls,
        "swap_cost_per_call": sw / ns - 1.0,
        "swap_cycle_ms": 1e3 * (sw - ns) / max(1, len(swaps)),
        "clocks": clocks.summary(),
        "gpu_launches": 2 * sched.calls + len(swaps),
    }
    pool.close()
    torch.cuda.empty_cache()
    return rec


# --------------------------------------------------------------------- main

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(ms: float, ws: int, device=None) -> float:
    """The timed region's length as the slowest rank saw it (replicas: every rank runs
    the same steps on its own GPU; the job takes as long as its slowest rank)."""
    if ws <= 1:
        return ms
    import torch
    import torch.distributed as dist
    tt = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(tt, op=dist.ReduceOp.MAX)
    return float(tt.item())


def job_tokens_per_s(tokens_per_rank: int, ws: int, ms: float) -> float:
    """Whole-job throughput: the tokens all ranks processed over the slowest rank's time."""
    return tokens_per_rank * ws / (ms / 1e3)


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    p, cfg = workload(args.workload if args.workload != "all" else "q_proj_decode")
    import oracle
    ads = oracle.problem_adapters(p)
    n = min(args.ref_tokens, p.T)
    X, ids = p.X[:n], p.ids[:n]
    for _ in range(args.warmup):
        oracle.lora_linear(X, p.W, ids, ads, p.max_adapters)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.lora_linear(X, p.W, ids, ads, p.max_adapters)
    el = time.perf_counter() - t0
    value = n * args.steps / el
    cores = oracle.num_threads()
    cfg = dict(cfg, sample=f"{n} of {p.T} tokens per step")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": cfg,
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"{n} of {p.T} tokens per step, {args.steps} steps"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def run_profile_calls(args):
    """N plain calls of one single-layer workload and nothing else: a short program for
    a profiler to attach to (ncu -k <kernel> -s <skip> -c <count> ...)."""
    import torch
    import adapter_linear_gb300 as al
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    name = "q_proj_decode" if args.workload == "all" else args.workload
    p, _ = workload(name)

    def t(a):
        if a.dtype == np.uint16:
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    pool = al.LoraPool(p.max_adapters, p.max_rank, p.d_in, p.d_out)
    for slot, ad in p.adapters.items():
        pool.load_adapter(slot, t(ad.A), t(ad.B), ad.rank, ad.alpha)
    pool.reserve(p.T)
    X, ids = t(p.X), t(p.ids)
    Y = torch.empty((p.T, p.d_out), dtype=torch.bfloat16, device=dev)
    if name.endswith("_q4"):
        Wq = tuple(t(a) for a in q4_base(p))
        for _ in range(args.profile):
            pool.linear_q4(X, *Wq, ids, Y)
    else:
        W = t(p.W)
        for _ in range(args.profile):
            pool.linear(X, W, ids, Y)
    torch.cuda.synchronize(dev)
    assert pool.check_errors() == al.LORA_OK
    pool.close()
    print(json.dumps({"profile_calls": args.profile, "workload": name}), flush=True)


def run_cpu_probe(args):
    """Child process of the one-core CPU baseline (OMP_NUM_THREADS set by the parent)."""
    p, _ = workload(args.cpu_probe)
    rate, cores, sample = cpu_oracle_rate(p, args.cpu_seconds, args.cpu_tokens)
    print(json.dumps({"value": rate, "cores": cores, "sample": sample}), flush=True)


CONFIG_ORDER = ("tiny", "llama3_layer", "q_proj_decode_q4", "prefill_mixed", "prefill_mixed_padded", "prefill_r16",
                "prefill_zipf",
                "hotswap_T256", "hotswap_stream")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--workload", default="all",
                    help="all (the headline q_proj decode line with every other workload under "
                         "'configs'), or one workload name alone")
    ap.add_argument("--cpu-seconds", type=float, default=8.0)
    ap.add_argument("--cpu-tokens", type=int, default=16)
    ap.add_argument("--cpu-probe", default=None, help=argparse.SUPPRESS)
    ap.add_argument("--profile", type=int, default=0,
                    help="run this many plain calls of --workload and exit (for profilers)")
    ap.add_argument("--ref-tokens", type=int, default=8)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", action="store_true",
                    help="launch the kernels directly instead of replaying a captured CUDA graph")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    if args.cpu_probe:
        return run_cpu_probe(args)
    if args.profile > 0:
        return run_profile_calls(args)
    if args.impl == "reference":
        return run_reference(args)

    kit = Kit(args)
    K = args.steps
    headline_name = "q_proj_decode" if args.workload == "all" else args.workload
    if headline_name == "llama3_layer":
        rec, p = measure_grouped_layer(kit, K), None
    elif headline_name == "hotswap_stream":
        rec, p = measure_hotswap_stream(kit), None
    else:
        rec, p = measure_layer(kit, headline_name, K, headline=True)

    configs = {}
    if args.workload == "all" and kit.ws == 1:
        for name in CONFIG_ORDER:
            try:
                if name == "llama3_layer":
                    configs[name] = measure_grouped_layer(kit, K)
                elif name == "hotswap_stream":
                    configs[name] = measure_hotswap_stream(kit)
                else:
                    configs[name], _ = measure_layer(kit, name, K)
            except Exception as e:  # one workload's failure must not hide the others
                configs[name] = {"error": f"{type(e).__name__}: {e}"}
                kit.torch.cuda.synchronize(kit.dev)

    if kit.rank != 0:
        if kit.ws > 1:
            kit.torch.distributed.destroy_process_group()
        return

    cpu = None
    if not args.no_cpu_baseline and p is not None:
        cpu = cpu_baselines(headline_name, p, args.cpu_seconds, args.cpu_tokens,
                            args.cpu_seconds / 2, args.cpu_tokens)
        if "prefill_mixed" in configs:
            pm, _ = workload("prefill_mixed")
            c4 = cpu_baselines("prefill_mixed", pm, 1.0, 256, 1.0, 256)
            c4["sample"] += "; a 256-row subsample of the 16384-token batch"
            configs["prefill_mixed"]["cpu_baseline"] = c4

    out = {
        "metric": METRIC, "value": rec["value"], "unit": UNIT, "n_gpus": kit.ws, "steps": K,
        "warmup": args.warmup, "ms_per_step": rec["ms_per_step"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": dict(rec["config"],
                       parallelism=f"replicas x{kit.ws}" if kit.ws > 1 else "single GPU"),
    }
    for k, v in rec.items():
        if k not in out and k not in ("metric", "value", "unit", "config"):
            out[k] = v
    out["cpu_baseline"] = cpu
    if configs:
        out["configs"] = configs
    print(json.dumps(out), flush=True)
    if kit.ws > 1:
        kit.torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
