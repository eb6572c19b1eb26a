"""Benchmark of the heterogeneous multi-LoRA linear layer on GB300.

One step = one lora_linear call (segment build, shrink, base GEMM, expand)
over one batch of the Llama-2-7B q_proj decode workload: T=64 tokens,
d_in=d_out=4096, 200 resident rank-16 adapters (alpha 32), ids uniform over
0..199, synthetic seeded bf16 data. Inputs are resident in HBM when the timed
region starts. The K steps run back to back (one CUDA graph) over R "layers",
each with its own W and adapter pool, step k on layer k mod R; the layers
together hold more than 3x the L2 size, so every step reads its weights and
adapter pages from HBM. An isolated call (L2 flushed before it) is reported
beside it.

Prints ONE JSON line (rank 0). value = tokens/s over all ranks; e2e = the
same metric through lora_linear_host (pinned host X/ids in, host Y out,
copies and the final sync inside the measured time); roofline = the
dominant kernel (the base GEMM) against the measured HBM copy bandwidth;
cpu_baseline = the fp64 CPU oracle on a bounded sample of the same workload.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   (the oracle as the reference arm)
Multi-GPU (torchrun, one rank per GPU): replicas, no data-path collective.
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


# ----------------------------------------------------------------- workloads

def workload(name: str):
    if name == "q_proj_decode":
        p = L.q_proj_decode()
        return p, {"workload": "Llama-2-7B q_proj decode", "T": 64, "d_in": 4096, "d_out": 4096,
                   "adapters": 200, "rank": 16, "alpha": 32, "ids": "uniform 0..199"}
    if name == "hotswap_T256":
        p, _ = L.hotswap()
        return p, {"workload": "q_proj decode, 2000 paged adapters, Zipf ids", "T": 256,
                   "d_in": 4096, "d_out": 4096, "adapters": 2000, "rank": 16}
    if name == "prefill_mixed":
        p = L.prefill_mixed()
        return p, {"workload": "gate_proj prefill, 8x2048 tokens, ranks 8..64", "T": 16384,
                   "d_in": 4096, "d_out": 14336, "adapters": 8, "rank": "8,8,16,16,32,32,64,64"}
    if name == "prefill_r16":  # the same prefill with every adapter at rank 16 (alpha 32)
        p = L.prefill_mixed(ranks=[16])
        return p, {"workload": "gate_proj prefill, 8x2048 tokens, rank 16", "T": 16384,
                   "d_in": 4096, "d_out": 14336, "adapters": 8, "rank": 16, "alpha": 32}
    if name == "prefill_small":  # same kernels and ranks, 8 x 512 tokens (for profiling)
        p = L.prefill_mixed(seq_len=512)
        return p, {"workload": "gate_proj prefill, 8x512 tokens, ranks 8..64", "T": 4096,
                   "d_in": 4096, "d_out": 14336, "adapters": 8, "rank": "8,8,16,16,32,32,64,64"}
    if name.startswith("llama3_"):
        mod = name[len("llama3_"):]
        (p,) = L.llama3_7mod(modules=[mod])
        return p, {"workload": f"Llama-3-8B {mod} decode", "T": 32, "d_in": p.d_in,
                   "d_out": p.d_out, "adapters": 32, "rank": 16}
    if name == "tiny":
        p = L.tiny()
        return p, {"workload": "tiny", "T": 64, "d_in": 256, "d_out": 256, "adapters": 4, "rank": 8}
    raise SystemExit(f"unknown workload {name}")


def algorithmic_bytes(p):
    """Bytes the layer must move once: X, W, Y, ids and the distinct adapters' A and B."""
    T = p.T
    distinct = set(int(i) for i in p.ids if i >= 0)
    ad_bytes = sum(p.adapters[i].rank * (p.d_in + p.d_out) * 2 for i in distinct)
    return {
        "x": T * p.d_in * 2, "w": p.d_out * p.d_in * 2, "y": T * p.d_out * 2, "ids": T * 4,
        "adapters": ad_bytes,
        "adapter_A": sum(p.adapters[i].rank * p.d_in * 2 for i in distinct),
        "adapter_B": sum(p.adapters[i].rank * p.d_out * 2 for i in distinct),
    }


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
    """nvidia-smi samples every 200 ms while the timed region runs."""
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
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


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
        return d.get("hbm_gbs"), d.get("bf16_tflops"), "measured"
    return 6800.0, 1900.0, "fallback"


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


# ------------------------------------------------------- grouped layer (7 modules)

def run_grouped_layer(args):
    """A Llama-3-8B decoder layer's seven target modules (q,k,v,o,gate,up,down; T = 32,
    32 adapters r16 per module, one id vector) per step: one lora_linear_grouped call,
    against seven lora_linear calls and seven base-only calls of the same layer."""
    import torch
    import adapter_linear_gb300 as al

    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if ws > 1 else 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    probs = L.llama3_7mod()
    T = probs[0].T

    def t(a):
        if a.dtype == np.uint16:
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    Xs = [t(p.X) for p in probs]
    ids = t(probs[0].ids)
    Ys = [torch.empty((T, p.d_out), dtype=torch.bfloat16, device=dev) for p in probs]

    def new_layer():
        pools, Ws = [], []
        for p in probs:
            pool = al.LoraPool(p.max_adapters, p.max_rank, p.d_in, p.d_out)
            for slot, ad in p.adapters.items():
                pool.load_adapter(slot, t(ad.A), t(ad.B), ad.rank, ad.alpha)
            pool.reserve(T)
            pools.append(pool)
            Ws.append(t(p.W))
        return pools, Ws

    layers = [new_layer()]
    layer_bytes = sum(w.numel() * 2 for w in layers[0][1]) + \
        sum(pl.stats()["bytes_held"] for pl in layers[0][0])
    R = max(2, -(-3 * l2 // layer_bytes))
    while len(layers) < R:
        layers.append(new_layer())

    def grouped_step(k):
        pools, Ws = layers[k % R]
        al.LoraPool.linear_grouped(pools, Xs, Ws, ids, Ys)

    def separate_step(k):
        pools, Ws = layers[k % R]
        for m, pool in enumerate(pools):
            pool.linear(Xs[m], Ws[m], ids, Ys[m])

    def base_step(k):
        pools, Ws = layers[k % R]
        for m, pool in enumerate(pools):
            pool.base_linear(Xs[m], Ws[m], Ys[m])

    no_ids = torch.full_like(ids, -1)

    def grouped_base_step(k):  # the same grouped call with every token on the base path
        pools, Ws = layers[k % R]
        al.LoraPool.linear_grouped(pools, Xs, Ws, no_ids, Ys)

    graphs = []

    def program(step, n, timing=False):
        for pools, _ in layers:
            for pool in pools:
                pool.enable_timing(timing)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for k in range(n):
                step(k)
        for pools, _ in layers:
            for pool in pools:
                pool.enable_timing(False)
        graphs.append(g)
        return g.replay

    def time_program(prog):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        prog()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1)

    for k in range(max(args.warmup, R)):
        grouped_step(k)
        separate_step(k)
        base_step(k)
        grouped_base_step(k)
    torch.cuda.synchronize(dev)
    g_prog = program(grouped_step, args.steps)
    gb_prog = program(grouped_base_step, args.steps)
    s_prog = program(separate_step, args.steps)
    b_prog = program(base_step, args.steps)
    program(grouped_step, args.warmup)()
    torch.cuda.synchronize(dev)

    nvml = NvmlClockSampler(dev)
    with ClockSampler(dev.index or 0) as clocks, nvml:
        torch.cuda.synchronize(dev)
        total_ms = time_program(g_prog)
        torch.cuda.synchronize(dev)
    total_ms = max_over_ranks(total_ms, ws, dev)
    sep_ms = time_program(s_prog)
    base_ms = time_program(b_prog)
    # the overhead against the grouped base-only call: base, LoRA, LoRA, base (same
    # clocks on average)
    b1 = time_program(gb_prog)
    l1 = time_program(g_prog)
    l2 = time_program(g_prog)
    b2 = time_program(gb_prog)
    g_il, gb_il = l1 + l2, b1 + b2
    gbase_ms = gb_il / 2

    # per-kernel device time of the grouped call (events of the first module's pool)
    kprog = program(grouped_step, R, timing=True)
    kts = []
    for _ in range(max(1, -(-args.steps // R))):
        kprog()
        torch.cuda.synchronize(dev)
        kts += [pools[0].kernel_times() for pools, _ in layers]
    gemm_ms = statistics.mean(k["base_gemm"] for k in kts)
    finish_ms = statistics.mean(k["finish_expand"] for k in kts)

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
        torch.cuda.synchronize(dev)

    for _ in range(3):
        e2e_once()
    e2e_s = 0.0
    for _ in range(args.steps):
        t0 = time.perf_counter()
        e2e_once()
        e2e_s += time.perf_counter() - t0
    for pools, _ in layers:
        for pool in pools:
            assert pool.check_errors() == al.LORA_OK

    if rank != 0:
        if ws > 1:
            torch.distributed.destroy_process_group()
        return

    abs_ = [algorithmic_bytes(p) for p in probs]
    w_b = sum(a["w"] for a in abs_)
    x_b = sum(a["x"] for a in abs_)
    y_b = sum(a["y"] for a in abs_)
    ad_a = sum(a["adapter_A"] for a in abs_)
    ad_all = sum(a["adapters"] for a in abs_)
    hbm_peak, _, peak_src = measured_peaks()
    gemm_bytes = w_b + x_b + ad_a
    achieved = gemm_bytes / (gemm_ms * 1e-3) / 1e9
    cpu = None
    if not args.no_cpu_baseline:
        import oracle
        n, done, t0 = 2, 0, time.perf_counter()
        ads = [oracle.problem_adapters(p) for p in probs]
        while time.perf_counter() - t0 < args.cpu_seconds:
            for p, a in zip(probs, ads):
                oracle.lora_linear(p.X[:n], p.W, p.ids[:n], a, p.max_adapters)
            done += n
        el = time.perf_counter() - t0
        cpu = {"value": done / el, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
               "sample": f"{n} of {T} tokens through all 7 modules per pass, {done} tokens in {el:.1f} s"}
    clk = nvml.summary() or dict(clocks.summary(), source="nvidia-smi")
    out = {
        "metric": METRIC, "value": job_tokens_per_s(T * args.steps, ws, total_ms), "unit": UNIT,
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": total_ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "Llama-3-8B decoder layer, 7 target modules in one grouped call",
                   "T": T, "modules": [p.name.split("/")[1] for p in probs], "adapters": 32,
                   "rank": 16, "layers": R,
                   "l2": f"inputs larger than L2: {R} layers of 7 modules, each its own W and "
                         f"pools ({R * layer_bytes / 1e6:.0f} MB cycled)",
                   "launch": "one CUDA graph of the K steps",
                   "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU"},
        "separate_calls_ms_per_step": sep_ms / args.steps,
        "base_only_ms_per_step": gbase_ms / args.steps,
        "base_only_separate_calls_ms_per_step": base_ms / args.steps,
        "overhead_vs_base": g_il / gb_il - 1.0,
        "overhead_measured_on": "K grouped base-only, 2K grouped LoRA, K grouped base-only calls in that order",
        "overhead_floor": ad_all / (w_b + x_b + y_b),
        "kernel_ms": {"base_gemm": gemm_ms, "finish_expand": finish_ms},
        "roofline": {"kernel": "gemm_decode_kernel", "bound": "hbm", "achieved": achieved,
                     "peak": hbm_peak, "unit": "GB/s", "frac": achieved / hbm_peak,
                     "traffic": None, "algorithmic_bytes": gemm_bytes, "peak_source": peak_src},
        "clocks": clk,
        "e2e": {"value": T * args.steps * ws / e2e_s, "unit": UNIT, "h2d_bytes_per_step": x_b + T * 4,
                "d2h_bytes_per_step": y_b},
        "gpu_launches": 2 * args.steps,
        "cpu_baseline": cpu,
    }
    print(json.dumps(out), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


# ------------------------------------------------- hot-swap stream (config 5 as specified)

def run_hotswap_stream(args):
    """1000 calls of 256 tokens over 2000 r16 adapters with Zipf ids (a new id vector
    every call), with one unload + reload of a slot in every block of 20 calls (50
    cycles), all through the public API; the same 1000 calls without the swaps give
    the swap cost."""
    import torch
    import adapter_linear_gb300 as al

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    p, sched = L.hotswap()

    def t(a):
        if a.dtype == np.uint16:
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    pool = al.LoraPool(p.max_adapters, p.max_rank, p.d_in, p.d_out)
    for slot, ad in p.adapters.items():
        pool.load_adapter(slot, t(ad.A), t(ad.B), ad.rank, ad.alpha)
    pool.reserve(p.T)
    pool.set_path(al.LORA_PATH_DECODE)
    X, W = t(p.X), t(p.W)
    ids = t(sched.ids)                                 # [calls, T]
    Y = torch.empty((p.T, p.d_out), dtype=torch.bfloat16, device=dev)
    swaps = {c: (slot, gen) for c, slot, gen in sched.swaps}
    fresh = {}
    for c, (slot, gen) in swaps.items():
        ad = L.make_adapter(p.seed, slot, p.d_in, p.d_out, 16, 32.0, generation=gen)
        fresh[c] = (t(ad.A), t(ad.B))
    old = {c: (t(p.adapters[slot].A), t(p.adapters[slot].B)) for c, (slot, _) in swaps.items()}

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
    torch.cuda.synchronize(dev)

    def timed(fn):
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        fn()
        torch.cuda.synchronize(dev)
        return time.perf_counter() - t0

    nvml = NvmlClockSampler(dev)
    with ClockSampler(dev.index or 0) as clocks, nvml:
        swap_s = timed(lambda: run(True, False))
    nosw_s = timed(lambda: run(False, False))
    timed(lambda: run(True, True))                     # put the first generation back
    assert pool.check_errors() == al.LORA_OK
    n_tok = p.T * sched.calls
    clk = nvml.summary() or dict(clocks.summary(), source="nvidia-smi")
    out = {
        "metric": METRIC, "value": n_tok / swap_s, "unit": UNIT, "n_gpus": 1,
        "steps": sched.calls, "warmup": args.warmup,
        "ms_per_step": 1e3 * swap_s / sched.calls, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "hot-swap stream: 1000 calls x 256 tokens, 2000 x r16 adapters, "
                               "Zipf ids, 50 unload+reload cycles", "T": p.T, "d_in": p.d_in,
                   "d_out": p.d_out, "adapters": p.max_adapters, "rank": 16,
                   "launch": "direct calls (a swap synchronises the device)",
                   "l2": "one W (33.5 MB) stays in L2 across calls; the 2000 adapters' pages "
                         "(524 MB) do not",
                   "parallelism": "single GPU"},
        "no_swap_ms_per_step": 1e3 * nosw_s / sched.calls,
        "swap_cycle_ms": 1e3 * (swap_s - nosw_s) / max(1, len(swaps)),
        "clocks": clk,
        "e2e": {"value": n_tok / swap_s, "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 2 * sched.calls + len(swaps),
        "cpu_baseline": None,
    }
    print(json.dumps(out), flush=True)


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
    p, cfg = workload(args.workload)
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


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    # 1000 q_proj decode steps are ~16 ms of timed work: enough for a clock record
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--workload", default="q_proj_decode")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--ref-tokens", type=int, default=8)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", action="store_true",
                    help="launch the kernels directly instead of replaying a captured CUDA graph")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    if args.impl == "reference":
        return run_reference(args)
    if args.workload == "llama3_layer":
        return run_grouped_layer(args)
    if args.workload == "hotswap_stream":
        return run_hotswap_stream(args)

    import torch
    import adapter_linear_gb300 as al

    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if ws > 1 else 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)

    p, cfg = workload(args.workload)

    def t(a):
        if a.dtype == np.uint16:
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    props = torch.cuda.get_device_properties(dev)
    l2 = props.L2_cache_size
    A_dev = {s: t(ad.A) for s, ad in p.adapters.items()}
    B_dev = {s: t(ad.B) for s, ad in p.adapters.items()}

    def new_layer(W):
        pool = al.LoraPool(p.max_adapters, p.max_rank, p.d_in, p.d_out)
        for slot, ad in p.adapters.items():
            pool.load_adapter(slot, A_dev[slot], B_dev[slot], ad.rank, ad.alpha)
        pool.reserve(p.T)
        return pool, W

    # R layers, each with its own W and its own adapter pool (like the layers of a
    # model): step k runs layer k mod R, so every step reads its weights and adapter
    # pages from HBM -- the layers' footprint is more than 3x L2, no flush needed.
    W0 = t(p.W)
    layers = [new_layer(W0)]
    layer_bytes = W0.numel() * 2 + layers[0][0].stats()["bytes_held"]
    R = max(2, min(32, -(-3 * l2 // layer_bytes)))
    while len(layers) < R:
        layers.append(new_layer(W0.clone()))
    X, ids = t(p.X), t(p.ids)
    Y = torch.empty((p.T, p.d_out), dtype=torch.bfloat16, device=dev)
    flush = torch.empty(2 * l2 // 4 + 1024, dtype=torch.float32, device=dev)

    def barrier():
        if ws > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(dev)

    def lora_step(k):
        pool, W = layers[k % R]
        pool.linear(X, W, ids, Y)

    def base_step(k):
        pool, W = layers[k % R]
        pool.base_linear(X, W, Y)

    def program(step, n, timing=False):
        """n consecutive steps captured as one CUDA graph (or a plain loop)."""
        for pool, _ in layers:
            pool.enable_timing(timing)
        run = lambda: [step(k) for k in range(n)]  # noqa: E731
        if args.no_graph:
            return run
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            run()
        for pool, _ in layers:
            pool.enable_timing(False)
        graphs.append(g)
        return g.replay

    def time_program(prog):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        prog()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1)

    # warm-up: W plain steps of each kind (scratch, tensor maps, modules, graphs)
    for k in range(max(args.warmup, R)):
        lora_step(k)
        base_step(k)
    barrier()
    graphs = []
    lora_prog = program(lora_step, args.steps)
    base_prog = program(base_step, args.steps)
    warm_prog = program(lora_step, args.warmup)
    warm_prog()
    barrier()

    # ---- timed region: exactly K lora_linear steps, back to back
    nvml = NvmlClockSampler(dev)
    with ClockSampler(dev.index or 0) as clocks, nvml:
        barrier()
        total_ms = time_program(lora_prog)
        barrier()
    total_ms = max_over_ranks(total_ms, ws, dev)
    value = job_tokens_per_s(p.T * args.steps, ws, total_ms)

    # ---- LoRA overhead against the base-only product, same structure: K base-only and
    # K LoRA steps in the order base, LoRA, LoRA, base, so that both kinds see the same
    # clocks on average (a long compute-bound run heats the GPU and lowers its clock)
    base_prog()
    b1 = time_program(base_prog)
    l1 = time_program(lora_prog)
    l2 = time_program(lora_prog)
    b2 = time_program(base_prog)
    lora_il, base_il = l1 + l2, b1 + b2
    base_step_ms = base_il / (2 * args.steps)
    lora_il_step_ms = lora_il / (2 * args.steps)

    # ---- per-kernel device time: one step per layer with the library's timing events
    def kernel_samples(step):
        prog = program(step, R, timing=True)
        out = []
        for _ in range(max(1, -(-args.steps // R))):
            prog()
            torch.cuda.synchronize(dev)
            out += [pool.kernel_times() for pool, _ in layers]
        return out[:args.steps]
    kts = kernel_samples(lora_step)
    base_kts = kernel_samples(base_step)

    # ---- an isolated call: L2 flushed before it, one call per replay
    iso_prog = program(lambda k: lora_step(0), 1)
    iso = []
    for i in range(args.steps):
        flush.fill_(float(i))
        iso.append(time_program(iso_prog))
    iso_ms = statistics.median(iso)

    # ---- e2e through the host entry point (pinned buffers, copies + sync inside)
    pool0, W = layers[0]
    Xh = torch.from_numpy(p.X.view(np.int16)).view(torch.bfloat16).pin_memory()
    idh = torch.from_numpy(p.ids).pin_memory()
    Yh = torch.empty((p.T, p.d_out), dtype=torch.bfloat16).pin_memory()
    for _ in range(3):
        pool0.linear_host(Xh, W, idh, Yh)
    e2e_s = 0.0
    for i in range(args.steps):
        flush.fill_(float(i))
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        pool0.linear_host(Xh, W, idh, Yh)
        e2e_s += time.perf_counter() - t0
    e2e_value = p.T * args.steps * ws / e2e_s
    for pool, _ in layers:
        assert pool.check_errors() == al.LORA_OK
    barrier()

    if rank != 0:
        if ws > 1:
            torch.distributed.destroy_process_group()
        return

    def mean_of(kts, key):
        return statistics.mean(k[key] for k in kts) if kts else 0.0

    gemm_ms = mean_of(kts, "base_gemm")
    shrink_ms = mean_of(kts, "shrink")
    finish_ms = mean_of(kts, "finish_expand")
    seg_ms = mean_of(kts, "segment_build")
    ab = algorithmic_bytes(p)
    hbm_peak, tf_peak, peak_src = measured_peaks()
    decode = p.T <= 256
    # the decode GEMM kernel also runs the shrink: it reads the distinct adapters' A pages
    gemm_bytes = ab["w"] + ab["x"] + ab["adapter_A"]
    if decode:
        achieved = gemm_bytes / (gemm_ms * 1e-3) / 1e9
        roof = {"kernel": "gemm_decode_kernel", "bound": "hbm", "achieved": achieved,
                "peak": hbm_peak, "unit": "GB/s", "frac": achieved / hbm_peak,
                "traffic": profiled_traffic(args.workload), "algorithmic_bytes": gemm_bytes,
                "peak_source": peak_src}
    else:
        gemm_flops = 2.0 * p.T * p.d_in * p.d_out
        achieved = gemm_flops / (gemm_ms * 1e-3) / 1e12
        # above 128 tokens the prefill path runs the CTA-pair kernel
        kname = "gemm_prefill_pair_kernel" if p.T > 128 else "gemm_prefill_kernel"
        roof = {"kernel": kname, "bound": "tensor", "achieved": achieved,
                "peak": tf_peak, "unit": "TFLOP/s", "frac": achieved / tf_peak, "traffic": None,
                "algorithmic_flops": gemm_flops, "peak_source": peak_src}
    # adapter path: the distinct adapters' A and B bytes over the time the adapters add to
    # a step (LoRA step minus base-only step, both back to back)
    extra_ms = lora_il_step_ms - base_step_ms
    adapter_gbs = ab["adapters"] / (extra_ms * 1e-3) / 1e9 if extra_ms > 0 else None
    overhead = lora_il / base_il - 1.0
    floor = ab["adapters"] / (ab["w"] + ab["x"] + ab["y"])

    cpu = None
    if not args.no_cpu_baseline and ws >= 1:
        rate, cores, sample = cpu_oracle_rate(p, args.cpu_seconds, max_tokens=16)
        cpu = {"value": rate, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample}

    clk = nvml.summary() or dict(clocks.summary(), source="nvidia-smi")
    out = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": dict(cfg, layers=R,
                       l2=f"inputs larger than L2: {R} layers, each its own W and adapter pool "
                          f"({R * layer_bytes / 1e6:.0f} MB cycled), step k uses layer k mod {R}",
                       launch="direct" if args.no_graph else "one CUDA graph of the K steps",
                       parallelism=f"replicas x{ws}" if ws > 1 else "single GPU"),
        "overhead_vs_base": overhead,
        "overhead_floor": floor,
        "base_only_ms_per_step": base_step_ms,
        "overhead_measured_on": f"K base-only, 2K LoRA, K base-only steps in that order (LoRA "
                                f"{lora_il_step_ms:.5f} ms per step there)",
        "isolated_call_ms": iso_ms,
        "adapter_path_gbs": adapter_gbs,
        # the whole step's algorithmic bytes (W, X, Y, ids, the distinct adapters) over
        # the back-to-back step time: both kernels, with the next call's W overlapping
        "step_hbm_gbs": (ab["w"] + ab["x"] + ab["y"] + ab["ids"] + ab["adapters"]) / (total_ms / args.steps * 1e-3) / 1e9,
        "kernel_ms": {"segment_build": seg_ms, "shrink": shrink_ms, "base_gemm": gemm_ms,
                      "finish_expand": finish_ms},
        "base_only_kernel_ms": {"base_gemm": mean_of(base_kts, "base_gemm"),
                                "finish": mean_of(base_kts, "finish_expand")},
        "roofline": roof,
        "tflops": algorithmic_flops(p) / (total_ms / args.steps * 1e-3) / 1e12,
        "clocks": clk,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": ab["x"] + ab["ids"],
                "d2h_bytes_per_step": ab["y"]},
        "gpu_launches": (2 if decode else 3) * args.steps,
        "cpu_baseline": cpu,
    }
    print(json.dumps(out), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
