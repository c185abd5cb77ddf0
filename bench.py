"""Benchmark of the NVFP4 rollout linear layer on one GB300 (or N replicas).

Workload (one step): a Qwen2.5-7B-shaped decoder layer in W4A16 decode --
hidden 3584; q/o 3584x3584, gate/up 18944x3584, down 3584x18944 bf16 weights
~N(0, 0.02) with 1% outlier columns x8; M = 64 bf16 tokens; LoRA r = 32 on every
linear; AQN sigma schedule 1e-2 -> 5e-4 over K = 10. One step runs every stage of
the path on that layer:
  1. AQN sigma_k (host) and RMSNorm-AQN of the 64 tokens (input norm), then again
     (post-attention norm);
  2. the rollout weight refresh: the tensor amax and the NVFP4 encoding (codes,
     E4M3 block scales, fp32 g) of all five weights, in one nvfp4_quantize_batch call;
  3. the five W4A16 LoRA linears at M = 64.
Inputs are synthetic, generated on the device from a seed, and larger than L2:
every step streams the five bf16 weights (458 MB) and their NVFP4 codes (122 MB).

Prints one JSON line. `value` is algorithmic bytes per step (what the method must
move, each tensor once) over the device time of a step, summed over ranks.
`--impl reference` times the CPU oracle on a bounded sample of the same
workload instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "NVFP4 LoRA-linear TFLOP/s & HBM GB/s (% roofline); quantize GB/s, 1×GB300"
WORKLOAD = ("qwen2.5-7b-shaped decode layer, W4A16: hidden 3584, q/o 3584x3584, gate/up 18944x3584, "
            "down 3584x18944, M=64 tokens, LoRA r=32 s=2, AQN sigma 1e-2->5e-4 over K=10, "
            "weight refresh (amax + NVFP4 encode) of all five weights each step")
HIDDEN, INTER, M_TOK, RANK, S_LORA = 3584, 18944, 64, 32, 2.0
LINEARS = [("q", 3584, 3584), ("o", 3584, 3584), ("gate", 18944, 3584), ("up", 18944, 3584), ("down", 3584, 18944)]
SIGMA0, SIGMAK, KSCHED = 1e-2, 5e-4, 10


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


# ----------------------------------------------------------------------------- byte / flop counts

def bytes_rmsnorm(M, H):
    return M * H * 2 * 2 + H * 8


def bytes_quantize(n):
    return n * (2 + 0.5 + 0.0625)


def bytes_linear(M, N, K, r):
    return N * K * 0.5625 + 2 * M * K + 2 * M * N + 2 * r * (K + N)


def flops_linear(M, N, K, r):
    return 2 * M * N * K + 2 * M * r * (K + N)


def step_bytes():
    b = 2 * bytes_rmsnorm(M_TOK, HIDDEN)
    b += sum(bytes_quantize(n * k) for _, n, k in LINEARS)
    b += sum(bytes_linear(M_TOK, n, k, RANK) for _, n, k in LINEARS)
    return b


# ----------------------------------------------------------------------------- replicas (N > 1)

def max_over_ranks(ms, device, world, dist_mod):
    """The slowest replica's time: the job's N replicas have all finished only then."""
    if world <= 1:
        return float(ms)
    import torch
    t = torch.tensor([float(ms)], device=device, dtype=torch.float64)
    dist_mod.all_reduce(t, op=dist_mod.ReduceOp.MAX)
    return float(t.item())


def job_throughput(bytes_per_replica_step, world, ms_per_step):
    """Whole-job GB/s: every replica moves the same bytes per step (weak scaling)."""
    return bytes_per_replica_step * world / (ms_per_step / 1e3) / 1e9


def reference_runs_here(rank, world):
    """Under torchrun the CPU reference arm runs and prints on rank 0 only."""
    return world <= 1 or rank == 0


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    """Samples the SM clock and the clock-event (throttle) reasons of one GPU in the background,
    through NVML (read-only queries), falling back to nvidia-smi when NVML cannot be loaded."""

    REASONS = {0x2: "applications_clocks_setting", 0x4: "sw_power_cap", 0x8: "hw_slowdown",
               0x10: "sync_boost", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown", 0x100: "display_clock_setting"}

    def __init__(self, pci_bus_id: str, period_s: float = 0.002):
        self.pci = pci_bus_id
        self.period = period_s
        self.samples = []
        self.max_mhz = None
        self._stop = threading.Event()
        self._t = None
        self._nvml = None
        self._h = None
        try:
            import ctypes
            L = ctypes.CDLL("libnvidia-ml.so.1")
            if L.nvmlInit_v2() == 0:
                h = ctypes.c_void_p()
                if L.nvmlDeviceGetHandleByPciBusId_v2(self.pci.encode(), ctypes.byref(h)) == 0:
                    self._nvml, self._h = L, h
                    mx = ctypes.c_uint()
                    if L.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
                        self.max_mhz = float(mx.value)
        except Exception:
            self._nvml = None

    def _sample_nvml(self):
        import ctypes
        L, h = self._nvml, self._h
        clk, rs = ctypes.c_uint(), ctypes.c_ulonglong()
        if L.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) != 0:
            return None
        fn = getattr(L, "nvmlDeviceGetCurrentClocksEventReasons", None) or L.nvmlDeviceGetCurrentClocksThrottleReasons
        if fn(h, ctypes.byref(rs)) != 0:
            return None
        return float(clk.value), int(rs.value)

    def _sample_smi(self):
        out = subprocess.run(["nvidia-smi", "--id=" + self.pci, "--query-gpu=clocks.sm,clocks.max.sm,clocks_event_reasons.active",
                              "--format=csv,noheader,nounits"], capture_output=True, text=True, timeout=5)
        parts = [q.strip() for q in out.stdout.strip().split(",")]
        if len(parts) != 3:
            return None
        self.max_mhz = float(parts[1])
        return float(parts[0]), int(parts[2], 16)

    def _run(self):
        while not self._stop.is_set():
            try:
                s = self._sample_nvml() if self._nvml else self._sample_smi()
                if s:
                    self.samples.append(s)
            except Exception:
                pass
            self._stop.wait(self.period if self._nvml else 0.2)

    def __enter__(self):
        self._t = threading.Thread(target=self._run, daemon=True)
        self._t.start()
        return self

    def __exit__(self, *a):
        self._stop.set()
        if self._t:
            self._t.join(timeout=10)

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": ["unsampled"], "samples": 0}
        sm = [s[0] for s in self.samples]
        mask = 0
        for s in self.samples:
            mask |= s[1]
        reasons = [name for bit, name in self.REASONS.items() if mask & bit]
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": self.max_mhz, "reasons": reasons,
                "samples": len(sm), "source": "nvml" if self._nvml else "nvidia-smi"}


# ----------------------------------------------------------------------------- GPU arm

def source_hash(*files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel):
    """DRAM bytes per launch from a committed ncu summary, if the kernel's source is unchanged since."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)[kernel]
        if d.get("source_hash") != source_hash(*d["sources"]):
            return None
        return d
    except Exception:
        return None


def run_gpu(args):
    import torch
    import torch.distributed as dist
    import nvfp4_quantized_rl_gb300 as nv

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)

    gen = torch.Generator(device=dev)
    gen.manual_seed(1234 + rank)

    def randn(*shape, std=1.0):
        return torch.randn(*shape, generator=gen, device=dev, dtype=torch.float32).mul_(std)

    # weights: bf16 ~N(0, 0.02), 1% of the input columns x8
    W = {}
    for name, n, k in LINEARS:
        w = randn(n, k, std=0.02)
        cols = torch.randperm(k, generator=gen, device=dev)[: round(0.01 * k)]
        w[:, cols] *= 8
        W[name] = w.to(torch.bfloat16)
        del w
    lora = {name: (randn(RANK, k, std=0.02).to(torch.bfloat16), randn(n, RANK, std=0.02).to(torch.bfloat16))
            for name, n, k in LINEARS}
    x_in = randn(M_TOK, HIDDEN).to(torch.bfloat16)
    x_res = randn(M_TOK, HIDDEN).to(torch.bfloat16)
    attn = randn(M_TOK, HIDDEN).to(torch.bfloat16)
    act = randn(M_TOK, INTER).to(torch.bfloat16)
    w1, w2 = (1 + randn(HIDDEN, std=0.1)), (1 + randn(HIDDEN, std=0.1))
    eps = [randn(HIDDEN) for _ in range(KSCHED + 1)]

    # outputs and workspaces, allocated once
    Q = {name: (torch.empty(n, k // 2, dtype=torch.uint8, device=dev), torch.empty(n, k // 16, dtype=torch.uint8, device=dev),
                torch.empty(1, dtype=torch.float32, device=dev), torch.empty(1, dtype=torch.float32, device=dev))
         for name, n, k in LINEARS}
    Y = {name: torch.empty(M_TOK, n, dtype=torch.bfloat16, device=dev) for name, n, k in LINEARS}
    h1 = torch.empty(M_TOK, HIDDEN, dtype=torch.bfloat16, device=dev)
    h2 = torch.empty_like(h1)
    ws_bytes = max(nv.workspace_bytes(nv.OP_LINEAR_W4A16, M_TOK, n, k, RANK) for _, n, k in LINEARS)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    wsq = torch.empty(nv.workspace_bytes(nv.OP_QUANTIZE_BATCH, len(LINEARS), 0, 0), dtype=torch.uint8, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    refresh_args = ([W[n] for n, _, _ in LINEARS], [Q[n][0] for n, _, _ in LINEARS], [Q[n][1] for n, _, _ in LINEARS],
                    [Q[n][2] for n, _, _ in LINEARS])
    for name, _, _ in LINEARS:  # each weight's amax, the input of the single-op encode (quantize_<w>)
        nv.nvfp4_amax(W[name], out=Q[name][3])
    inputs = {"q": h1, "o": attn, "gate": h2, "up": h2, "down": act}
    stream = torch.cuda.current_stream(dev)

    # per-op CUDA events (all launches go to the current stream)
    ops = ["rmsnorm_aqn", "rmsnorm_aqn_2", "weight_refresh"] + [f"linear_{n}" for n, _, _ in LINEARS]
    # single-op mode only (not part of the step): the per-weight amax and encode kernels alone
    solo_ops = [f"amax_{n}" for n, _, _ in LINEARS] + [f"quantize_{n}" for n, _, _ in LINEARS]

    def step(k, ev=None, only=None):
        st = torch.cuda.current_stream(dev)

        def mark(name, fn):
            if only is not None and name not in only:
                return
            if ev is None:
                fn()
                return
            a, b = ev[name]
            a.record(st)
            fn()
            b.record(st)
        sigma = nv.aqn_sigma(SIGMA0, SIGMAK, k, KSCHED)
        mark("rmsnorm_aqn", lambda: nv.rmsnorm_aqn(x_in, w1, eps[k], sigma, 1e-6, out=h1))
        mark("weight_refresh", lambda: nv.nvfp4_quantize_batch(refresh_args[0], codes=refresh_args[1],
                                                               scales=refresh_args[2], g=refresh_args[3], workspace=wsq))
        if only is not None:
            for name, n, kk in LINEARS:
                c, s, g, a = Q[name]
                if f"amax_{name}" in only:
                    nv.nvfp4_amax(W[name], out=a)
                if f"quantize_{name}" in only:
                    nv.nvfp4_quantize(W[name], amax_in=a, codes=c, scales=s, g=g)
        mark("rmsnorm_aqn_2", lambda: nv.rmsnorm_aqn(x_res, w2, eps[k], sigma, 1e-6, out=h2))
        for name, n, kk in LINEARS:
            c, s, g, _ = Q[name]
            A, B = lora[name]
            mark(f"linear_{name}", lambda: nv.nvfp4_lora_linear(inputs[name], c, s, g, A, B, S_LORA, out=Y[name],
                                                                 workspace=ws))

    # eager warm-up (initialises the library), then one CUDA graph per noise-schedule index k:
    # a step replays the library's launches without host overhead between kernels
    for i in range(2):
        step(i % (KSCHED + 1))
    torch.cuda.synchronize()
    if args.op:
        return run_ops(args, torch, step, ops + solo_ops, flush, stream, rank)
    graphs, ev_graphs = [], []
    launches_per_step = None
    for k in range(KSCHED + 1):
        g = torch.cuda.CUDAGraph()
        l0 = nv.kernel_launches()
        with torch.cuda.graph(g):
            step(k)
        if launches_per_step is None:
            launches_per_step = nv.kernel_launches() - l0
        graphs.append(g)
        # the same step with CUDA events around every op, replayed only for the per-op breakdown
        ev = {name: (torch.cuda.Event(enable_timing=True, external=True),
                     torch.cuda.Event(enable_timing=True, external=True)) for name in ops}
        ge = torch.cuda.CUDAGraph()
        with torch.cuda.graph(ge):
            step(k, ev)
        ev_graphs.append((ge, ev))
    torch.cuda.synchronize()
    for i in range(args.warmup):
        graphs[i % (KSCHED + 1)].replay()
    torch.cuda.synchronize()

    bounds = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    props = torch.cuda.get_device_properties(dev)
    pci = f"{props.pci_domain_id:08x}:{props.pci_bus_id:02x}:{props.pci_device_id:02x}.0"
    # Steps run back to back: every step streams 458 MB of bf16 weights and 122 MB of codes,
    # several times the 129 MB L2, so nothing one step leaves in L2 serves the next.
    with ClockSampler(pci) as clocks:
        for i in range(args.steps):
            bounds[i][0].record(stream)
            graphs[i % (KSCHED + 1)].replay()
            bounds[i][1].record(stream)
        torch.cuda.synchronize()
    step_ms = [a.elapsed_time(b) for a, b in bounds]
    # per-op breakdown (not part of the timed region): event-instrumented replays
    op_samples = {name: [] for name in ops}
    for i in range(max(3, min(args.steps, 10))):
        ge, ev = ev_graphs[i % (KSCHED + 1)]
        ge.replay()
        torch.cuda.synchronize()
        for name in ops:
            op_samples[name].append(ev[name][0].elapsed_time(ev[name][1]))
    launches = launches_per_step * args.steps
    if world > 1:
        dist.barrier()
    total_ms = float(sum(step_ms))
    op_ms = {name: float(np.mean(v)) for name, v in op_samples.items()}
    total_ms = max_over_ranks(total_ms, dev, world, dist)
    ms_per_step = total_ms / args.steps

    # ---- end to end: host buffers in, host result out, through the same public API
    e2e = run_e2e(args, nv, torch, dev, W, lora, x_in, x_res, attn, act, w1, w2, eps, Q, Y, h1, h2, ws, flush,
                  inputs, world)

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return
    hbm, bf16_tf, peak_src = peaks()
    sb = step_bytes()
    value = job_throughput(sb, world, total_ms / args.steps)

    # parts
    q_bytes = sum(bytes_quantize(n * k) for _, n, k in LINEARS)
    q_ms = op_ms["weight_refresh"]
    l_bytes = sum(bytes_linear(M_TOK, n, k, RANK) for _, n, k in LINEARS)
    l_flops = sum(flops_linear(M_TOK, n, k, RANK) for _, n, k in LINEARS)
    l_ms = sum(op_ms[f"linear_{n}"] for n, _, _ in LINEARS)
    r_ms = op_ms["rmsnorm_aqn"] + op_ms["rmsnorm_aqn_2"]
    parts = {
        "rmsnorm_aqn": {"us": r_ms * 1e3, "GB/s": 2 * bytes_rmsnorm(M_TOK, HIDDEN) / r_ms / 1e6},
        "weight_refresh": {"us": q_ms * 1e3, "GB/s": q_bytes / q_ms / 1e6,
                           "note": "amax + NVFP4 encode of the five weights, one nvfp4_quantize_batch call; bytes: each "
                                   "weight read once, codes and scales written (the amax pass reads each weight again)"},
        "lora_linear_w4a16": {"us": l_ms * 1e3, "GB/s": l_bytes / l_ms / 1e6, "TFLOP/s": l_flops / l_ms / 1e9,
                              "frac_hbm": l_bytes / l_ms / 1e6 / hbm},
        "per_linear_us": {n: op_ms[f"linear_{n}"] * 1e3 for n, _, _ in LINEARS},
    }
    # dominant kernel by device time
    groups = {"weight_refresh": q_ms, "lora_linear_w4a16": l_ms, "rmsnorm_aqn_kernel": op_ms["rmsnorm_aqn"]}
    dom = max(groups, key=groups.get)
    if dom == "weight_refresh":
        ach = q_bytes / q_ms / 1e6
        per_launch_bytes = q_bytes
    elif dom == "lora_linear_w4a16":
        ach = l_bytes / l_ms / 1e6
        per_launch_bytes = l_bytes / len(LINEARS)
    else:
        ach = parts["rmsnorm_aqn"]["GB/s"]
        per_launch_bytes = bytes_rmsnorm(M_TOK, HIDDEN)
    tr = recorded_traffic(dom)
    roofline = {"kernel": dom, "bound": "hbm", "achieved": ach, "peak": hbm, "unit": "GB/s", "frac": ach / hbm,
                "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured" else "fallback",
                "algorithmic_bytes_per_launch": per_launch_bytes,
                "traffic": None if tr is None else tr["dram_bytes_per_launch"]}
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded, generated on device)",
        "config": {"workload": WORKLOAD, "l2": "inputs larger than L2: each step streams 458 MB of bf16 weights and 122 MB of NVFP4 codes (L2 129 MB); no flush",
                   "replicas": world, "algorithmic_bytes_per_step": sb},
        "parts": parts, "roofline": roofline, "e2e": e2e, "gpu_launches": int(launches),
        "clocks": clocks.summary(),
    }
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline(args.cpu_seconds)
    print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


def select_ops(spec, ops):
    """--op names: op names of the step (e.g. linear_gate, weight_refresh, rmsnorm_aqn), the single-weight
    amax_<w> / quantize_<w> (the per-tensor amax and encode kernels alone; not part of the step) or the
    groups linears, refresh, rmsnorm, amax, quantize, all (= the step's ops); comma-separated."""
    groups = {"linears": [o for o in ops if o.startswith("linear_")], "refresh": ["weight_refresh"],
              "rmsnorm": [o for o in ops if "rmsnorm" in o], "amax": [o for o in ops if o.startswith("amax_")],
              "quantize": [o for o in ops if o.startswith("quantize_")],
              "all": [o for o in ops if not o.startswith(("amax_", "quantize_"))]}
    out = []
    for part in spec.split(","):
        part = part.strip()
        sel = groups.get(part, [part] if part in ops else None)
        if sel is None:
            raise SystemExit(f"unknown op {part!r}; ops: {', '.join(ops)}; groups: {', '.join(groups)}")
        out += [o for o in sel if o not in out]
    return out


def run_ops(args, torch, step, ops, flush, stream, rank):
    """Single-op timing (eager launches; before every op a 256 MB read evicts L2): W warm-up and K timed runs of
    each selected op of the step; one JSON line of per-op device microseconds. Serves per-kernel
    measurement and profiler captures of one op on the step's full-size inputs."""
    sel = select_ops(args.op, ops)
    flush64 = flush.view(torch.int64)

    def evict():  # read a buffer twice the L2 size: L2 then holds clean lines only (no write-backs later)
        flush64.sum()

    res = {}
    for name in sel:
        for i in range(args.warmup):
            evict()
            step(i % (KSCHED + 1), only={name})
        torch.cuda.synchronize()
        ts = []
        for i in range(args.steps):
            evict()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            step(i % (KSCHED + 1), only={name})
            b.record(stream)
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b) * 1e3)
        res[name] = {"us_median": float(np.median(ts)), "us_min": float(np.min(ts)), "runs": len(ts)}
    if rank == 0:
        print(json.dumps({"mode": "ops", "workload": WORKLOAD, "steps": args.steps, "warmup": args.warmup, "ops": res}))


def run_suite(args):
    """Secondary measurements of the other configurations on the path (not the headline step):
    W4A4 prefill (7B shapes, 4096 tokens; 32B gate, 8192 tokens), W4A16 at 256 tokens on the 32B
    shapes, the grouped MoE layer (128 experts, 32768 routed rows), the NVFP4 encode of one 32B
    layer (per tensor and batched), the guided encode, and RMSNorm-AQN at prefill sizes. One JSON line per case: device time per call through the public API (eager, a 256 MB
    read evicts L2 before each call), achieved TFLOP/s and GB/s, and the fraction of the binding
    roof (FP4 tensor peak = the measured bf16 peak x 6, the nominal 13.5 / 2.25 ratio)."""
    import torch
    import nvfp4_quantized_rl_gb300 as nv
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    gen = torch.Generator(device=dev)
    gen.manual_seed(4321)
    hbm, bf16_tf, src = peaks()
    fp4_tf = bf16_tf * 6.0
    flush64 = torch.empty(256 << 20, dtype=torch.uint8, device=dev).view(torch.int64)

    def randn(*shape, std=1.0):
        return torch.randn(*shape, generator=gen, device=dev, dtype=torch.float32).mul_(std)

    def weight(n, k, std=0.02):
        w = randn(n, k, std=std)
        cols = torch.randperm(k, generator=gen, device=dev)[: round(0.01 * k)]
        w[:, cols] *= 8
        return w.to(torch.bfloat16)

    def activations(m, k, heavy=True):
        x = randn(m, k)
        if heavy:  # 1% of the channels Student-t(4)
            ch = torch.randperm(k, generator=gen, device=dev)[: max(1, round(0.01 * k))]
            z = randn(m, ch.numel())
            chi = (randn(m, ch.numel()) ** 2 + randn(m, ch.numel()) ** 2 + randn(m, ch.numel()) ** 2 +
                   randn(m, ch.numel()) ** 2) / 4
            x[:, ch] = z / chi.sqrt()
        return x.to(torch.bfloat16)

    def timed(fn, reps):
        for _ in range(max(3, args.warmup)):
            fn()
        torch.cuda.synchronize()
        ts = []
        for _ in range(reps):
            # two passes over the 256 MB buffer: L2 is evicted, and the GPU stays busy (~80 us) while
            # the host enqueues the call, so the events time the call's kernels, not the host's
            # argument checks and launches
            flush64.sum()
            flush64.sum()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b) * 1e3)
        return float(np.median(ts))

    def emit(case, us, flops, nbytes, bound, extra=None):
        tf = flops / us / 1e6 if flops else None
        gbs = nbytes / us / 1e3
        if bound == "fp4":
            roof = {"bound": "tensor", "dtype": "fp4", "achieved": tf, "peak": fp4_tf, "unit": "TFLOP/s",
                    "frac": tf / fp4_tf, "peak_source": f"{src} bf16 x 6 (nominal fp4/bf16 ratio)"}
        elif bound == "bf16":
            roof = {"bound": "tensor", "dtype": "bf16", "achieved": tf, "peak": bf16_tf, "unit": "TFLOP/s",
                    "frac": tf / bf16_tf, "peak_source": src}
        else:
            roof = {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": gbs / hbm,
                    "peak_source": src}
        line = {"mode": "suite", "case": case, "us": us, "TFLOP/s": tf, "GB/s": gbs, "roofline": roof}
        if extra:
            line.update(extra)
        print(json.dumps(line), flush=True)

    r = RANK
    cases = set((args.suite or "all").split(","))

    def want(name):
        return "all" in cases or name in cases

    # ---- W4A4 prefill, 7B shapes, 4096 tokens (LoRA r = 32)
    if want("w4a4_7b"):
        M = 4096
        for name, n, k in [("q", 3584, 3584), ("gate", 18944, 3584), ("down", 3584, 18944)]:
            W = weight(n, k)
            c, sc, g = nv.nvfp4_quantize(W)
            del W
            x = activations(M, k)
            A, B = randn(r, k, std=0.02).to(torch.bfloat16), randn(n, r, std=0.02).to(torch.bfloat16)
            y = torch.empty(M, n, dtype=torch.bfloat16, device=dev)
            ws = torch.empty(nv.workspace_bytes(nv.OP_LINEAR_W4A4, M, n, k, r), dtype=torch.uint8, device=dev)
            us = timed(lambda: nv.nvfp4_lora_linear_w4a4(x, c, sc, g, A, B, S_LORA, out=y, workspace=ws), 10)
            emit(f"w4a4_7b_{name}_m{M}", us, flops_linear(M, n, k, r),
                 n * k * 0.5625 + 2 * M * k + 2 * M * n + 2 * r * (k + n), "fp4",
                 {"shape": [M, n, k], "note": "full API: activation amax + NVFP4 encode, LoRA down, FP4 GEMM + LoRA up"})
            del c, sc, g, x, A, B, y, ws
            torch.cuda.empty_cache()
    # ---- 32B shapes: W4A16 at 256 tokens (r = 64), W4A4 gate at 8192 tokens
    if want("w4a16_32b") or want("w4a4_32b"):
        r32 = 64
        for name, n, k in [("q", 5120, 5120), ("gate", 27648, 5120), ("down", 5120, 27648)]:
            W = weight(n, k, 0.015)
            c, sc, g = nv.nvfp4_quantize(W)
            del W
            A, B = randn(r32, k, std=0.02).to(torch.bfloat16), randn(n, r32, std=0.02).to(torch.bfloat16)
            if want("w4a16_32b"):
                M = 256
                x = activations(M, k, heavy=False)
                y = torch.empty(M, n, dtype=torch.bfloat16, device=dev)
                ws = torch.empty(nv.workspace_bytes(nv.OP_LINEAR_W4A16, M, n, k, r32), dtype=torch.uint8, device=dev)
                us = timed(lambda: nv.nvfp4_lora_linear(x, c, sc, g, A, B, S_LORA, out=y, workspace=ws), 10)
                emit(f"w4a16_32b_{name}_m{M}", us, flops_linear(M, n, k, r32),
                     n * k * 0.5625 + 2 * M * k + 2 * M * n + 2 * r32 * (k + n), "bf16", {"shape": [M, n, k]})
                del x, y, ws
            if want("w4a4_32b") and name == "gate":
                M = 8192
                x = activations(M, k)
                y = torch.empty(M, n, dtype=torch.bfloat16, device=dev)
                ws = torch.empty(nv.workspace_bytes(nv.OP_LINEAR_W4A4, M, n, k, r32), dtype=torch.uint8, device=dev)
                us = timed(lambda: nv.nvfp4_lora_linear_w4a4(x, c, sc, g, A, B, S_LORA, out=y, workspace=ws), 5)
                emit(f"w4a4_32b_{name}_m{M}", us, flops_linear(M, n, k, r32),
                     n * k * 0.5625 + 2 * M * k + 2 * M * n + 2 * r32 * (k + n), "fp4", {"shape": [M, n, k]})
                del x, y, ws
            del c, sc, g, A, B
            torch.cuda.empty_cache()
    # ---- MoE layer: 128 experts, H = 2048, I = 768, 4096 tokens x top-8 = 32768 rows, grouped W4A4
    if want("moe"):
        E, H, I, T, TOPK = 128, 2048, 768, 4096, 8
        logits = randn(T, E)
        top = torch.topk(torch.softmax(logits, dim=1), TOPK, dim=1).indices.reshape(-1)
        counts = torch.bincount(top, minlength=E)
        offsets = torch.zeros(E + 1, dtype=torch.int32, device=dev)
        offsets[1:] = torch.cumsum(counts, 0).to(torch.int32)
        rows = int(offsets[-1].item())
        for name, n, k in [("gate", I, H), ("down", H, I)]:
            codes = torch.empty(E, n, k // 2, dtype=torch.uint8, device=dev)
            scales = torch.empty(E, n, k // 16, dtype=torch.uint8, device=dev)
            gs = torch.empty(E, dtype=torch.float32, device=dev)
            for e in range(E):
                W = (randn(n, k, std=0.02)).to(torch.bfloat16)
                nv.nvfp4_quantize(W, codes=codes[e], scales=scales[e], g=gs[e:e + 1])
            x = activations(rows, k, heavy=False)
            y = torch.empty(rows, n, dtype=torch.bfloat16, device=dev)
            ws = torch.empty(nv.workspace_bytes(nv.OP_LINEAR_W4A4, rows, n, k, 0, E), dtype=torch.uint8, device=dev)
            us = timed(lambda: nv.nvfp4_lora_linear_w4a4(x, codes, scales, gs, group_offsets=offsets, num_groups=E,
                                                         out=y, workspace=ws), 10)
            emit(f"moe_{name}_rows{rows}", us, 2 * rows * n * k, E * n * k * 0.5625 + 2 * rows * k + 2 * rows * n,
                 "hbm", {"shape": [rows, n, k], "experts": E})
            del codes, scales, gs, x, y, ws
            torch.cuda.empty_cache()
    # ---- NVFP4 encode of one 32B layer's weights (q, k, v, o, gate, up, down; bf16)
    if want("quantize_32b"):
        tot_us, tot_bytes = 0.0, 0.0
        for name, n, k in [("q", 5120, 5120), ("k", 1024, 5120), ("v", 1024, 5120), ("o", 5120, 5120),
                           ("gate", 27648, 5120), ("up", 27648, 5120), ("down", 5120, 27648)]:
            W = weight(n, k, 0.015)
            c = torch.empty(n, k // 2, dtype=torch.uint8, device=dev)
            sc = torch.empty(n, k // 16, dtype=torch.uint8, device=dev)
            g = torch.empty(1, dtype=torch.float32, device=dev)
            wsq = torch.empty(nv.workspace_bytes(nv.OP_QUANTIZE, 0, 0, 0), dtype=torch.uint8, device=dev)
            us = timed(lambda: nv.nvfp4_quantize(W, codes=c, scales=sc, g=g, workspace=wsq), 5)
            tot_us += us
            tot_bytes += bytes_quantize(n * k)
            del W, c, sc, g
            torch.cuda.empty_cache()
        emit("quantize_32b_layer", tot_us, 0, tot_bytes, "hbm",
             {"note": "amax + encode of the seven weights, each call timed separately and summed; bytes count each "
                      "element once (2 B in, 0.5625 B out)"})
    # ---- the same seven 32B weights in one nvfp4_quantize_batch call (the weight refresh)
    if want("quantize_batch_32b"):
        shapes = [(5120, 5120), (1024, 5120), (1024, 5120), (5120, 5120), (27648, 5120), (27648, 5120), (5120, 27648)]
        Ws = [weight(n, k, 0.015) for n, k in shapes]
        cs = [torch.empty(n, k // 2, dtype=torch.uint8, device=dev) for n, k in shapes]
        ss = [torch.empty(n, k // 16, dtype=torch.uint8, device=dev) for n, k in shapes]
        gs = [torch.empty(1, dtype=torch.float32, device=dev) for _ in shapes]
        wsb = torch.empty(nv.workspace_bytes(nv.OP_QUANTIZE_BATCH, len(shapes), 0, 0), dtype=torch.uint8, device=dev)
        us = timed(lambda: nv.nvfp4_quantize_batch(Ws, codes=cs, scales=ss, g=gs, workspace=wsb), 5)
        emit("quantize_batch_32b_layer", us, 0, sum(bytes_quantize(n * k) for n, k in shapes), "hbm",
             {"note": "amax + encode of the seven weights in one nvfp4_quantize_batch call; bytes count each element "
                      "once (2 B in, 0.5625 B out)"})
        del Ws, cs, ss, gs, wsb
        torch.cuda.empty_cache()
    # ---- guided encode (a 1-bit mask per element picks the rounding direction) of the 7B gate weight
    if want("quantize_guided"):
        n, k = 18944, 3584
        W = weight(n, k)
        mask = torch.randint(-2 ** 31, 2 ** 31 - 1, ((n * k + 31) // 32,), generator=gen, device=dev,
                             dtype=torch.int64).to(torch.int32)  # Bernoulli(1/2) bits
        c = torch.empty(n, k // 2, dtype=torch.uint8, device=dev)
        sc = torch.empty(n, k // 16, dtype=torch.uint8, device=dev)
        g = torch.empty(1, dtype=torch.float32, device=dev)
        wsq = torch.empty(nv.workspace_bytes(nv.OP_QUANTIZE, 0, 0, 0), dtype=torch.uint8, device=dev)
        us_g = timed(lambda: nv.nvfp4_quantize_guided(W, mask, codes=c, scales=sc, g=g, workspace=wsq), 10)
        emit("quantize_guided_7b_gate", us_g, 0, n * k * (2 + 0.5625 + 0.125), "hbm",
             {"shape": [n, k], "note": "amax + guided encode; bytes: 2 B in, 0.5625 B out, 0.125 B of mask per element"})
        us_p = timed(lambda: nv.nvfp4_quantize(W, codes=c, scales=sc, g=g, workspace=wsq), 10)
        emit("quantize_plain_7b_gate", us_p, 0, n * k * (2 + 0.5625), "hbm",
             {"shape": [n, k], "note": "amax + plain encode, same weight"})
        rec = torch.empty((n * k + 31) // 32, dtype=torch.int32, device=dev)
        us_r = timed(lambda: nv.nvfp4_quantize_record(W, codes=c, scales=sc, g=g, record=rec, workspace=wsq), 10)
        emit("quantize_record_7b_gate", us_r, 0, n * k * (2 + 0.5625 + 0.125), "hbm",
             {"shape": [n, k], "note": "TRACE rollout side: amax + plain encode + the rounding-direction record; "
                                       "bytes: 2 B in, 0.5625 B out, 0.125 B of record per element"})
        c2 = torch.empty_like(c)
        us_c = timed(lambda: nv.nvfp4_quantize_cached(W, rec, sc, g, codes=c2), 10)
        emit("quantize_cached_7b_gate", us_c, 0, n * k * (2 + 0.125 + 0.0625 + 0.5), "hbm",
             {"shape": [n, k], "note": "TRACE training side: one pass from the cached record, scales and g; "
                                       "bytes: 2 B in, 0.125 B record + 0.0625 B scales in, 0.5 B codes out"})
        del W, mask, c, sc, g, rec, c2
        torch.cuda.empty_cache()
    # ---- RMSNorm-AQN fused with the NVFP4 quantization of its output (the W4A4 activation operand)
    if want("rmsnorm_quantize"):
        m, h = 4096, 3584
        x = activations(m, h)
        w = (1.0 + randn(h, std=0.1)).float()
        z = randn(h)
        y = torch.empty(m, h, dtype=torch.bfloat16, device=dev)
        c = torch.empty(m, h // 2, dtype=torch.uint8, device=dev)
        sc = torch.empty(m, h // 16, dtype=torch.uint8, device=dev)
        g = torch.empty(1, dtype=torch.float32, device=dev)
        wsq = torch.empty(nv.workspace_bytes(nv.OP_RMSNORM_QUANTIZE, 0, 0, 0), dtype=torch.uint8, device=dev)
        us_f = timed(lambda: nv.rmsnorm_aqn_quantize(x, w, z, 0.01, 1e-6, out=y, codes=c, scales=sc, g=g,
                                                     workspace=wsq), 10)
        fused_bytes = m * h * (2 + 2 + 0.5625)  # x in; y, codes and scales out
        emit(f"rmsnorm_quantize_m{m}_h{h}", us_f, 0, fused_bytes, "hbm",
             {"shape": [m, h], "note": "rmsnorm_aqn_quantize: one cooperative kernel keeps y on chip"})

        def separate():
            nv.rmsnorm_aqn(x, w, z, 0.01, 1e-6, out=y)
            nv.nvfp4_quantize(y, codes=c, scales=sc, g=g, workspace=wsq)
        us_s = timed(separate, 10)
        emit(f"rmsnorm_then_quantize_m{m}_h{h}", us_s, 0, fused_bytes, "hbm",
             {"shape": [m, h], "note": "rmsnorm_aqn, then nvfp4_quantize of y (amax pass + encode pass): same bytes "
                                       "counted, for comparison"})
        del x, w, z, y, c, sc, g, wsq
        torch.cuda.empty_cache()
    # ---- decode attention over an NVFP4 KV cache (Qwen2.5-7B heads: 28 query / 4 KV, 128 dims)
    if want("kv_attention"):
        B_, Hq_, Hkv_, D_, L_ = 64, 28, 4, 128, 8192
        gen = torch.Generator(device=dev).manual_seed(35)
        kc_ = torch.randint(0, 256, (B_, L_, Hkv_, D_ // 2), generator=gen, device=dev, dtype=torch.int32).to(torch.uint8)
        vc_ = torch.randint(0, 256, (B_, L_, Hkv_, D_ // 2), generator=gen, device=dev, dtype=torch.int32).to(torch.uint8)
        ks_ = torch.randint(0x28, 0x40, (B_, L_, Hkv_, D_ // 16), generator=gen, device=dev,
                            dtype=torch.int32).to(torch.uint8)
        vs_ = torch.randint(0x28, 0x40, (B_, L_, Hkv_, D_ // 16), generator=gen, device=dev,
                            dtype=torch.int32).to(torch.uint8)
        lens_h = np.random.default_rng(35).integers(4096, L_ + 1, B_).astype(np.int32)
        lens_d = torch.from_numpy(lens_h).to(dev)
        q_ = (torch.randn(B_, Hq_, D_, generator=gen, device=dev)).to(torch.bfloat16)
        g_ = torch.tensor([1.0 / 64], dtype=torch.float32, device=dev)
        out_ = torch.empty(B_, Hq_, D_, dtype=torch.bfloat16, device=dev)
        ws_ = torch.empty(max(16, nv.workspace_bytes(nv.OP_KV_ATTENTION, B_, Hkv_, L_)), dtype=torch.uint8, device=dev)
        us_k = timed(lambda: nv.nvfp4_kv_decode_attention(q_, kc_, ks_, g_, vc_, vs_, g_, lens_d, 1.0 / np.sqrt(D_),
                                                          out=out_, workspace=ws_), 10)
        kv_bytes = int(lens_h.sum()) * Hkv_ * (D_ // 2 + D_ // 16) * 2 + 2 * B_ * Hq_ * D_ * 2
        emit("kv_decode_attention_7b_b64_l8192", us_k, 0, kv_bytes, "hbm",
             {"shape": {"B": B_, "Hq": Hq_, "Hkv": Hkv_, "D": D_, "Lmax": L_, "tokens": int(lens_h.sum())},
              "note": "nvfp4_kv_decode_attention: random valid NVFP4 cache bytes, lengths 4096..8192; bytes: "
                      "the attended K and V rows (codes + scales), q and out"})
        del kc_, vc_, ks_, vs_, q_, out_, ws_
        torch.cuda.empty_cache()
    # ---- AIS mixing coefficient and rectified weights of a GRPO training batch (~4 M tokens)
    if want("ais"):
        import synth
        bcfg = synth.GRPO_BATCH
        lr_h, lt_h, adv_h = synth.grpo_token_batch(bcfg["prompts"], bcfg["group"], bcfg["mean_len"], 22,
                                                   max_tokens=bcfg["tokens"])
        lr_d, lt_d, adv_d = (torch.from_numpy(a).to(dev) for a in (lr_h, lt_h, adv_h))
        n_tok = lr_h.size
        w_d = torch.empty(n_tok, dtype=torch.float32, device=dev)
        st_d = torch.empty(8, dtype=torch.float64, device=dev)
        ws_a = torch.empty(nv.workspace_bytes(nv.OP_AIS, 0, 0, 0), dtype=torch.uint8, device=dev)
        us_a = timed(lambda: nv.ais_mixing(lr_d, lt_d, adv_d, 2.0, 0.05, 0.5, 1.0, w_out=w_d, stats=st_d,
                                           workspace=ws_a), 10)
        emit(f"ais_grpo_{n_tok}_tokens", us_a, 0, n_tok * 16, "hbm",
             {"tokens": n_tok, "note": "ais_mixing: one cooperative kernel; bytes: 3 fp32 inputs read and the "
                                        "rectified weight written per token (the second read of the log-probs, "
                                        "from L2, is not counted)"})
        del lr_d, lt_d, adv_d, w_d, st_d, ws_a
        torch.cuda.empty_cache()
    # ---- RMSNorm-AQN at prefill sizes (HBM-bound there; M = 64 in the step is bound by launch latency)
    if want("rmsnorm_prefill"):
        for m, h in [(4096, 3584), (8192, 5120)]:
            x = activations(m, h, heavy=False)
            w = (1.0 + randn(h, std=0.1)).float()
            z = randn(h)
            y = torch.empty(m, h, dtype=torch.bfloat16, device=dev)
            us = timed(lambda: nv.rmsnorm_aqn(x, w, z, 0.01, 1e-6, out=y), 10)
            emit(f"rmsnorm_aqn_m{m}_h{h}", us, 0, bytes_rmsnorm(m, h), "hbm", {"shape": [m, h]})
            del x, w, z, y
            torch.cuda.empty_cache()


def run_e2e(args, nv, torch, dev, W, lora, x_in, x_res, attn, act, w1, w2, eps, Q, Y, h1, h2, ws, flush, inputs,
            world):
    """Same step through the public API, with each step's inputs copied from pinned host memory and every
    output read back to pinned host memory inside the timed region. The copies are the step's bound (462 MB
    over the host link), so they run on a copy stream, largest weights first, and each weight is quantized
    (nvfp4_quantize: amax + encode) and its linear run as soon as it has landed; the step ends when the last
    output is back in host memory."""
    host_in = {name: W[name].cpu().pin_memory() for name, _, _ in LINEARS}
    host_x = {"x_in": x_in.cpu().pin_memory(), "x_res": x_res.cpu().pin_memory(), "attn": attn.cpu().pin_memory(),
              "act": act.cpu().pin_memory()}
    dev_x = {"x_in": x_in, "x_res": x_res, "attn": attn, "act": act}
    host_out = {name: torch.empty(Y[name].shape, dtype=torch.bfloat16).pin_memory() for name, _, _ in LINEARS}
    h2d = sum(t.numel() * t.element_size() for t in host_in.values()) + \
        sum(t.numel() * t.element_size() for t in host_x.values())
    d2h = sum(t.numel() * t.element_size() for t in host_out.values())
    stream = torch.cuda.current_stream(dev)
    copy_stream = torch.cuda.Stream(dev)
    inputs_e2e = {"q": h1, "o": dev_x["attn"], "gate": h2, "up": h2, "down": dev_x["act"]}
    wsq_e2e = torch.empty(nv.workspace_bytes(nv.OP_QUANTIZE, 0, 0, 0), dtype=torch.uint8, device=dev)
    order = [name for name, n, k in sorted(LINEARS, key=lambda t: -t[1] * t[2])]  # largest first
    ev_x = torch.cuda.Event()
    ev_w = {name: torch.cuda.Event() for name in order}
    done = torch.cuda.Event()
    done.record(stream)

    def step(k):
        # inputs: the copy stream may overwrite them once the previous step has read them
        copy_stream.wait_event(done)
        with torch.cuda.stream(copy_stream):
            for key in host_x:
                dev_x[key].copy_(host_x[key], non_blocking=True)
            ev_x.record(copy_stream)
            for name in order:
                W[name].copy_(host_in[name], non_blocking=True)
                ev_w[name].record(copy_stream)
        stream.wait_event(ev_x)
        sigma = nv.aqn_sigma(SIGMA0, SIGMAK, k, KSCHED)
        nv.rmsnorm_aqn(dev_x["x_in"], w1, eps[k], sigma, 1e-6, out=h1)
        nv.rmsnorm_aqn(dev_x["x_res"], w2, eps[k], sigma, 1e-6, out=h2)
        for name in order:
            stream.wait_event(ev_w[name])
            c, s, g, _ = Q[name]
            nv.nvfp4_quantize(W[name], codes=c, scales=s, g=g, workspace=wsq_e2e)
            A, B = lora[name]
            nv.nvfp4_lora_linear(inputs_e2e[name], c, s, g, A, B, S_LORA, out=Y[name], workspace=ws)
            host_out[name].copy_(Y[name], non_blocking=True)
        done.record(stream)

    for i in range(max(1, args.warmup)):
        step(i % (KSCHED + 1))
    torch.cuda.synchronize()
    n = max(1, args.steps)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    done.record(stream)  # the first step's copies start after the timed region has begun
    for i in range(n):
        step(i % (KSCHED + 1))
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / n
    if world > 1:
        import torch.distributed as dist
        ms = max_over_ranks(ms, dev, world, dist)
    return {"value": job_throughput(step_bytes(), world, ms), "unit": "GB/s", "ms_per_step": ms,
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)}


# ----------------------------------------------------------------------------- CPU oracle arm

def oracle_sample(den: int):
    """A bounded sample of the same step, run by the CPU oracle: RMSNorm of all 64 tokens twice, the NVFP4
    encoding of 1/den of each weight's rows, and every linear's outputs for those 1/den of its output rows
    (all 64 tokens). Returns (algorithmic bytes of the sample, seconds, threads)."""
    import oracle
    import synth
    t_total, bytes_total = 0.0, 0.0
    nthreads = oracle.threads()
    x = synth.activation_bf16(M_TOK, HIDDEN, 9, 0)
    w = synth.aqn_weight(HIDDEN, 9, 1)
    e = synth.aqn_eps(HIDDEN, 9, 2)
    t0 = time.perf_counter()
    oracle.rmsnorm_aqn(x, w, e, np.float32(SIGMA0), 1e-6)
    oracle.rmsnorm_aqn(x, w, e, np.float32(SIGMA0), 1e-6)
    t_total += time.perf_counter() - t0
    bytes_total += 2 * bytes_rmsnorm(M_TOK, HIDDEN)
    for i, (name, n, k) in enumerate(LINEARS):
        rows = n // den
        Wb = synth.weight_bf16(rows, k, 0.02, 9, 10 + i, outlier_frac=0.01)
        t0 = time.perf_counter()
        codes, scales, g = oracle.quantize(Wb)
        t_total += time.perf_counter() - t0
        bytes_total += bytes_quantize(rows * k)
        A, B = synth.lora_factors(RANK, k, rows, 9, 20 + i)
        xi = synth.activation_bf16(M_TOK, k, 9, 30 + i)
        t0 = time.perf_counter()
        oracle.lora_linear_w4a16(xi, codes, scales, g, A, B, S_LORA)
        t_total += time.perf_counter() - t0
        bytes_total += bytes_linear(M_TOK, rows, k, RANK)
    return bytes_total, t_total, nthreads


def sample_den(seconds_budget: float) -> int:
    """The smallest sampling denominator (1/den of every weight) whose oracle run fits the budget,
    extrapolated from a 1/64 probe run."""
    _, t64, _ = oracle_sample(64)
    for den in (1, 2, 4, 8, 16, 32):
        if t64 * 64 / den <= seconds_budget:
            return den
    return 64


def sample_desc(den: int) -> str:
    frac = "all" if den == 1 else f"1/{den}"
    return (f"RMSNorm-AQN of the 64x3584 tokens twice; NVFP4 encoding of {frac} of each weight's rows; "
            f"each LoRA linear on those rows' outputs for all 64 tokens (fp64 oracle)")


def cpu_baseline(seconds_budget=20.0):
    den = sample_den(seconds_budget)
    b, t, th = oracle_sample(den)
    return {"value": b / t / 1e9, "unit": "GB/s", "cores": th, "kind": "oracle", "sample": sample_desc(den),
            "sample_seconds": t}


def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if not reference_runs_here(rank, world):
        return
    # each step is a sample sized so that warm-up and timed steps together take about two minutes
    den = sample_den(120.0 / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        oracle_sample(den)
    tot_b, tot_t, th = 0.0, 0.0, 1
    for _ in range(args.steps):
        b, t, th = oracle_sample(den)
        tot_b += b
        tot_t += t
    v = tot_b / tot_t / 1e9
    desc = sample_desc(den)
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "GB/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": tot_t / max(1, args.steps) * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
        "config": {"workload": WORKLOAD, "sample": desc},
        "cpu_baseline": {"value": v, "unit": "GB/s", "cores": th, "kind": "oracle", "sample": desc},
        "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=20.0)
    ap.add_argument("--op", default=None, help="time single ops of the step instead (see select_ops)")
    ap.add_argument("--suite", default=None, nargs="?", const="all",
                    help="secondary measurements instead: all or any of w4a4_7b,w4a16_32b,w4a4_32b,moe,quantize_32b")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    elif args.suite:
        run_suite(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
