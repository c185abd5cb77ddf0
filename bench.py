"""Benchmark of the NVFP4 rollout linear layer on one GB300 (or N replicas).

Default workload (one step): 12 Qwen2.5-32B-shaped decoder layers, each with its own
weights -- hidden 5120; q/o 5120x5120, k/v 1024x5120, gate/up 27648x5120,
down 5120x27648 bf16 weights ~N(0, 0.015); LoRA r = 64, s = 2, on every linear;
AQN sigma schedule 1e-2 -> 5e-4 over K = 10. Per layer the step runs every stage of
the path:
  1. the rollout weight refresh: the tensor amax and the NVFP4 encoding (codes, E4M3
     block scales, fp32 g) of all seven weights, one nvfp4_quantize_batch call;
  2. decode, M = 256 tokens: RMSNorm-AQN of the input and of the residual stream,
     then the seven W4A16 LoRA linears;
  3. prefill, M = 8192 tokens: RMSNorm-AQN fused with the NVFP4 encoding of its output
     (rmsnorm_aqn_quantize) for the input and the residual stream, then the seven W4A4 LoRA
     linears (block-scaled FP4 MMA): q/k/v and gate/up on those shared NVFP4 activations
     (nvfp4_lora_linear_w4a4_quantized), o and down quantizing theirs on the fly.
One refresh thus serves 256 decode and 8192 prefill tokens per layer. `--config
qwen7b-decode` runs the Qwen2.5-7B-shaped decode layer instead (M = 64, W4A16 only).
Inputs are synthetic, generated on the device from a seed, and larger than L2: a
step streams 37 GB of bf16 weights and 10 GB of NVFP4 codes.

Prints one JSON line. For the 32B step `value` is the LoRA-linear TFLOP/s of the whole
step (every linear's 2MNK + 2Mr(K+N) over the device time of the step, including the
refresh and the norms), summed over replicas; for the 7B decode step it is algorithmic
GB/s. `--impl reference` times the CPU oracle on a bounded sample of the same workload.
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
S_LORA = 2.0
SIGMA0, SIGMAK, KSCHED = 1e-2, 5e-4, 10
FP4_PER_BF16 = 6.0  # nominal dense FP4 / BF16 tensor rate (13.5 / 2.25 PFLOP/s)

LINEARS_32B = [("q", 5120, 5120), ("k", 1024, 5120), ("v", 1024, 5120), ("o", 5120, 5120), ("gate", 27648, 5120),
               ("up", 27648, 5120), ("down", 5120, 27648)]
LINEARS_7B = [("q", 3584, 3584), ("o", 3584, 3584), ("gate", 18944, 3584), ("up", 18944, 3584),
              ("down", 3584, 18944)]

CONFIGS = {
    "qwen32b": {
        "workload": "qwen2.5-32b-shaped decoder layers, decode + prefill: hidden 5120, q/o 5120x5120, k/v 1024x5120, "
                    "gate/up 27648x5120, down 5120x27648 bf16 weights ~N(0,0.015); per layer: weight refresh (amax + "
                    "NVFP4 encode) of all seven weights, RMSNorm-AQN x2 + W4A16 LoRA linears at M=256, RMSNorm-AQN->NVFP4 "
                    "x2 + W4A4 LoRA linears at M=8192 (q/k/v, gate/up on the shared NVFP4 activations); LoRA r=64 "
                    "s=2; AQN sigma 1e-2->5e-4 over K=10",
        "hidden": 5120, "inter": 27648, "linears": LINEARS_32B, "std": 0.015, "outliers": 0.0, "rank": 64,
        "decode_m": 256, "prefill_m": 8192, "layers": 12, "unit": "TFLOP/s", "probe_den": 256,
    },
    "qwen7b-decode": {
        "workload": "qwen2.5-7b-shaped decode layer, W4A16: hidden 3584, q/o 3584x3584, gate/up 18944x3584, "
                    "down 3584x18944 bf16 weights ~N(0,0.02) with 1% outlier columns x8, M=64 tokens, LoRA r=32 s=2, "
                    "AQN sigma 1e-2->5e-4 over K=10, weight refresh (amax + NVFP4 encode) of all five weights each step",
        "hidden": 3584, "inter": 18944, "linears": LINEARS_7B, "std": 0.02, "outliers": 0.01, "rank": 32,
        "decode_m": 64, "prefill_m": 0, "layers": 1, "unit": "GB/s", "probe_den": 64,
    },
}

# Which activation feeds each linear: q/k/v the normed input, o the attention output, gate/up the
# normed residual stream, down the MLP activation (M x intermediate).
INPUT_OF = {"q": "h1", "k": "h1", "v": "h1", "o": "attn", "gate": "h2", "up": "h2", "down": "act"}


def peaks():
    """(hbm GB/s, bf16 burst TFLOP/s, bf16 sustained TFLOP/s, source) from MEASURED_PEAKS.json, else the
    fallback figures."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        bf = float(d["bf16_tflops"])
        return float(d["hbm_gbs"]), bf, float(d.get("bf16_tflops_sustained", bf)), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


# ----------------------------------------------------------------------------- byte / flop counts

def bytes_rmsnorm(M, H):
    return M * H * 2 * 2 + H * 8


def bytes_quantize(n):
    return n * (2 + 0.5 + 0.0625)


def bytes_linear(M, N, K, r):
    return N * K * 0.5625 + 2 * M * K + 2 * M * N + 2 * r * (K + N)


def bytes_linear_w4a4(M, N, K, r):
    # the activation codes and scales written once by the on-the-fly quantizer and read by the GEMM
    return bytes_linear(M, N, K, r) + 0.5625 * M * K


def flops_linear(M, N, K, r):
    return 2 * M * N * K + 2 * M * r * (K + N)


def layer_counts(cfg):
    """Algorithmic bytes and flops of one layer of the step, per part."""
    H, r = cfg["hidden"], cfg["rank"]
    md, mp = cfg["decode_m"], cfg["prefill_m"]
    lin = cfg["linears"]
    c = {
        "refresh_bytes": sum(bytes_quantize(n * k) for _, n, k in lin),
        "rms_d_bytes": 2 * bytes_rmsnorm(md, H),
        "w4a16_bytes": sum(bytes_linear(md, n, k, r) for _, n, k in lin),
        "w4a16_flops": sum(flops_linear(md, n, k, r) for _, n, k in lin),
        "rms_p_bytes": 2 * (bytes_rmsnorm(mp, H) + 0.5625 * mp * H) if mp else 0.0,
        "w4a4_bytes": sum(bytes_linear_w4a4(mp, n, k, r) for _, n, k in lin) if mp else 0.0,
        "w4a4_flops": sum(flops_linear(mp, n, k, r) for _, n, k in lin) if mp else 0.0,
    }
    c["bytes"] = c["refresh_bytes"] + c["rms_d_bytes"] + c["w4a16_bytes"] + c["rms_p_bytes"] + c["w4a4_bytes"]
    c["flops"] = c["w4a16_flops"] + c["w4a4_flops"]
    return c


def step_units(cfg, layers):
    """Units of the step's metric (flops for TFLOP/s, bytes for GB/s) and the divisor to that unit."""
    c = layer_counts(cfg)
    if cfg["unit"] == "TFLOP/s":
        return c["flops"] * layers, 1e12
    return c["bytes"] * layers, 1e9


# ----------------------------------------------------------------------------- replicas (N > 1)

def max_over_ranks(ms, device, world, dist_mod):
    """The slowest replica's time: the job's N replicas have all finished only then."""
    if world <= 1:
        return float(ms)
    import torch
    t = torch.tensor([float(ms)], device=device, dtype=torch.float64)
    dist_mod.all_reduce(t, op=dist_mod.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_replica_step, world, ms_per_step, scale=1e9):
    """Whole-job throughput (units / s / scale): every replica does the same work per step (weak scaling)."""
    return units_per_replica_step * world / (ms_per_step / 1e3) / scale


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


class Workload:
    """Device buffers of the step: per-layer weights, their NVFP4 outputs and LoRA factors; activations,
    outputs and workspaces per phase (decode / prefill), shared by the layers."""

    def __init__(self, nv, torch, dev, cfg, layers, seed):
        self.cfg, self.layers = cfg, layers
        gen = torch.Generator(device=dev)
        gen.manual_seed(seed)

        def randn(*shape, std=1.0):
            return torch.randn(*shape, generator=gen, device=dev, dtype=torch.float32).mul_(std)

        H, I, r = cfg["hidden"], cfg["inter"], cfg["rank"]
        self.W, self.Q, self.lora = [], [], []
        for _ in range(layers):
            W, Q, lora = {}, {}, {}
            for name, n, k in cfg["linears"]:
                w = randn(n, k, std=cfg["std"])
                if cfg["outliers"]:  # a seeded 1% of the input columns x8
                    cols = torch.randperm(k, generator=gen, device=dev)[: round(cfg["outliers"] * k)]
                    w[:, cols] *= 8
                W[name] = w.to(torch.bfloat16)
                del w
                Q[name] = (torch.empty(n, k // 2, dtype=torch.uint8, device=dev),
                           torch.empty(n, k // 16, dtype=torch.uint8, device=dev),
                           torch.empty(1, dtype=torch.float32, device=dev))
                lora[name] = (randn(r, k, std=0.02).to(torch.bfloat16), randn(n, r, std=0.02).to(torch.bfloat16))
            self.W.append(W)
            self.Q.append(Q)
            self.lora.append(lora)
        self.w1, self.w2 = (1 + randn(H, std=0.1)), (1 + randn(H, std=0.1))
        self.eps = [randn(H) for _ in range(KSCHED + 1)]
        self.phases = {}
        for phase, M, w4a4 in (("d", cfg["decode_m"], False), ("p", cfg["prefill_m"], True)):
            if not M:
                continue
            b = {"x_in": randn(M, H).to(torch.bfloat16), "x_res": randn(M, H).to(torch.bfloat16),
                 "attn": randn(M, H).to(torch.bfloat16), "act": randn(M, I).to(torch.bfloat16),
                 "h1": torch.empty(M, H, dtype=torch.bfloat16, device=dev),
                 "h2": torch.empty(M, H, dtype=torch.bfloat16, device=dev)}
            if w4a4:  # the normed inputs in NVFP4 as well (rmsnorm_aqn_quantize), shared by their linears
                for h in ("h1", "h2"):
                    b[h + "q"] = (torch.empty(M, H // 2, dtype=torch.uint8, device=dev),
                                  torch.empty(M, H // 16, dtype=torch.uint8, device=dev),
                                  torch.empty(1, dtype=torch.float32, device=dev))
            Y = {name: torch.empty(M, n, dtype=torch.bfloat16, device=dev) for name, n, k in cfg["linears"]}
            op = nv.OP_LINEAR_W4A4 if w4a4 else nv.OP_LINEAR_W4A16
            wsb = max(nv.workspace_bytes(op, M, n, k, r) for _, n, k in cfg["linears"])
            self.phases[phase] = {"M": M, "w4a4": w4a4, "buf": b, "Y": Y,
                                  "ws": torch.empty(wsb, dtype=torch.uint8, device=dev)}
        self.wsq = torch.empty(nv.workspace_bytes(nv.OP_QUANTIZE_BATCH, len(cfg["linears"]), 0, 0),
                               dtype=torch.uint8, device=dev)
        self.wsa = torch.empty(nv.workspace_bytes(nv.OP_QUANTIZE, 0, 0, 0), dtype=torch.uint8, device=dev)
        self.wsr = torch.empty(nv.workspace_bytes(nv.OP_RMSNORM_QUANTIZE, 0, 0, 0), dtype=torch.uint8, device=dev)
        self.amax = {name: torch.empty(1, dtype=torch.float32, device=dev) for name, _, _ in cfg["linears"]}

    def ops(self):
        """Names of the step's ops, per layer (the events of the per-op breakdown)."""
        names = ["weight_refresh"]
        for phase, P in self.phases.items():
            kind = "w4a4" if P["w4a4"] else "w4a16"
            names += [f"rmsnorm_{phase}"] + [f"{kind}_{n}" for n, _, _ in self.cfg["linears"]]
        return names

    def step(self, nv, k, ev=None, only=None, layer_sel=None, grp=None):
        """One step at noise-schedule index k. ev: {(layer, op): (start, end)} events recorded around the ops
        it names; grp: {(layer, "linears_<phase>"): (start, end)} events around all linears of a phase;
        only: run just these op names (single-op mode, layer 0 unless layer_sel)."""
        sigma = nv.aqn_sigma(SIGMA0, SIGMAK, k, KSCHED)
        lin = self.cfg["linears"]
        for l in (range(self.layers) if layer_sel is None else layer_sel):
            def mark(name, fn):
                if only is not None and name not in only:
                    return
                if ev is None or (l, name) not in ev:
                    fn()
                    return
                a, b = ev[(l, name)]
                a.record()
                fn()
                b.record()
            W, Q, lora = self.W[l], self.Q[l], self.lora[l]
            mark("weight_refresh", lambda: nv.nvfp4_quantize_batch(
                [W[n] for n, _, _ in lin], codes=[Q[n][0] for n, _, _ in lin], scales=[Q[n][1] for n, _, _ in lin],
                g=[Q[n][2] for n, _, _ in lin], workspace=self.wsq))
            if only is not None:  # the single-weight amax and encode kernels (not part of the step)
                for name, _, _ in lin:
                    c, s, g = Q[name]
                    if f"amax_{name}" in only:
                        nv.nvfp4_amax(W[name], out=self.amax[name])
                    if f"quantize_{name}" in only:
                        nv.nvfp4_quantize(W[name], amax_in=self.amax[name], codes=c, scales=s, g=g)
            for phase, P in self.phases.items():
                b = P["buf"]

                def norms():
                    for src, w, h in (("x_in", self.w1, "h1"), ("x_res", self.w2, "h2")):
                        if P["w4a4"]:  # W4A4: RMSNorm-AQN and the NVFP4 encoding of its output in one call
                            nv.rmsnorm_aqn_quantize(b[src], w, self.eps[k], sigma, 1e-6, out=b[h], codes=b[h + "q"][0],
                                                    scales=b[h + "q"][1], g=b[h + "q"][2], workspace=self.wsr)
                        else:
                            nv.rmsnorm_aqn(b[src], w, self.eps[k], sigma, 1e-6, out=b[h])
                mark(f"rmsnorm_{phase}", norms)
                kind = "w4a4" if P["w4a4"] else "w4a16"
                span = grp.get((l, f"linears_{phase}")) if grp else None
                if span:
                    span[0].record()
                for name, _, _ in lin:
                    c, s, g = Q[name]
                    A, B = lora[name]
                    src = INPUT_OF[name]
                    if not P["w4a4"]:
                        fn = lambda: nv.nvfp4_lora_linear(b[src], c, s, g, A, B, S_LORA, out=P["Y"][name],
                                                          workspace=P["ws"])
                    elif src + "q" in b:  # activations already in NVFP4 (q/k/v, gate/up)
                        xc, xs, xg = b[src + "q"]
                        fn = lambda: nv.nvfp4_lora_linear_w4a4_quantized(b[src], xc, xs, xg, c, s, g, A, B, S_LORA,
                                                                         out=P["Y"][name], workspace=P["ws"])
                    else:  # o and down: quantized on the fly
                        fn = lambda: nv.nvfp4_lora_linear_w4a4(b[src], c, s, g, A, B, S_LORA, out=P["Y"][name],
                                                               workspace=P["ws"])
                    mark(f"{kind}_{name}", fn)
                if span:
                    span[1].record()


def run_gpu(args):
    import torch
    import torch.distributed as dist
    import nvfp4_quantized_rl_gb300 as nv

    cfg = CONFIGS[args.config]
    layers = args.layers or cfg["layers"]
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    wl = Workload(nv, torch, dev, cfg, layers, 1234 + rank)
    for name, _, _ in cfg["linears"]:  # each weight's amax, the input of the single-op encode (quantize_<w>)
        nv.nvfp4_amax(wl.W[0][name], out=wl.amax[name])
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    ops = wl.ops()

    # eager warm-up (initialises the library), then one CUDA graph per noise-schedule index k: a step
    # replays the library's launches without host overhead between kernels
    for i in range(2):
        wl.step(nv, i % (KSCHED + 1))
    torch.cuda.synchronize()
    if args.op:
        return run_ops(args, torch, nv, wl, ops, flush, stream, rank)
    graphs, ev_graphs = [], []
    launches_per_step = None
    n_graphs = KSCHED + 1
    for k in range(n_graphs):
        g = torch.cuda.CUDAGraph()
        l0 = nv.kernel_launches()
        with torch.cuda.graph(g):
            wl.step(nv, k)
        if launches_per_step is None:
            launches_per_step = nv.kernel_launches() - l0
        graphs.append(g)
    # the same step with CUDA events around every op of every layer, replayed only for the per-op
    # breakdown (two noise indices suffice: the launches do not depend on k)
    for k in range(2):
        ev = {(l, name): (torch.cuda.Event(enable_timing=True, external=True),
                          torch.cuda.Event(enable_timing=True, external=True)) for l in range(layers) for name in ops}
        ge = torch.cuda.CUDAGraph()
        with torch.cuda.graph(ge):
            wl.step(nv, k, ev)
        ev_graphs.append((ge, ev))
    # and with events only at the ends of each op group (the refresh, each phase's RMSNorms, each
    # phase's linears as one span): the parts' times, free of the per-call event boundaries
    group_names = ["weight_refresh"] + [f"rmsnorm_{p}" for p in wl.phases] + [f"linears_{p}" for p in wl.phases]
    evg = {(l, name): (torch.cuda.Event(enable_timing=True, external=True),
                       torch.cuda.Event(enable_timing=True, external=True)) for l in range(layers) for name in group_names}
    gg = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gg):
        wl.step(nv, 0, ev={key: v for key, v in evg.items() if not key[1].startswith("linears_")},
                grp={key: v for key, v in evg.items() if key[1].startswith("linears_")})
    torch.cuda.synchronize()
    for i in range(args.warmup):
        graphs[i % n_graphs].replay()
    torch.cuda.synchronize()

    bounds = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    props = torch.cuda.get_device_properties(dev)
    pci = f"{props.pci_domain_id:08x}:{props.pci_bus_id:02x}:{props.pci_device_id:02x}.0"
    # Steps run back to back: every step streams each layer's bf16 weights and NVFP4 codes (several
    # times the 129 MB L2 per layer), so nothing one step leaves in L2 serves the next.
    with ClockSampler(pci) as clocks:
        for i in range(args.steps):
            bounds[i][0].record(stream)
            graphs[i % n_graphs].replay()
            bounds[i][1].record(stream)
        torch.cuda.synchronize()
    step_ms = [a.elapsed_time(b) for a, b in bounds]
    # per-op breakdown (not part of the timed region): event-instrumented replays
    op_samples = {name: [] for name in ops}
    for i in range(3):
        ge, ev = ev_graphs[i % 2]
        ge.replay()
        torch.cuda.synchronize()
        for name in ops:
            op_samples[name].append(sum(ev[(l, name)][0].elapsed_time(ev[(l, name)][1]) for l in range(layers)))
    group_samples = {name: [] for name in group_names}
    for i in range(3):
        gg.replay()
        torch.cuda.synchronize()
        for name in group_names:
            group_samples[name].append(sum(evg[(l, name)][0].elapsed_time(evg[(l, name)][1]) for l in range(layers)))
    group_ms = {name: float(np.median(v)) for name, v in group_samples.items()}
    launches = launches_per_step * args.steps
    if world > 1:
        dist.barrier()
    total_ms = float(sum(step_ms))
    op_ms = {name: float(np.median(v)) for name, v in op_samples.items()}  # per step (all layers)
    total_ms = max_over_ranks(total_ms, dev, world, dist)
    ms_per_step = total_ms / args.steps

    # ---- end to end: host buffers in, host result out, through the same public API
    e2e = run_e2e(args, nv, torch, dev, wl, world)

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return
    units, scale = step_units(cfg, layers)
    value = job_throughput(units, world, ms_per_step, scale)
    line = summarize(args, cfg, layers, world, value, ms_per_step, step_ms, op_ms, group_ms, launches, clocks, e2e)
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline(cfg, args.cpu_seconds)
    print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


def summarize(args, cfg, layers, world, value, ms_per_step, step_ms, op_ms, group_ms, launches, clocks, e2e):
    """The bench's JSON line: the step's throughput, the per-part breakdown with each part's fraction of its
    binding roof, and the roofline of the op that takes the most device time. Part times come from the
    replays with events only at the group ends (group_ms); per_linear_us from the replays with events
    around every call (op_ms)."""
    hbm, bf16_burst, bf16_sus, src = peaks()
    fp4_sus = bf16_sus * FP4_PER_BF16
    c = layer_counts(cfg)
    lin = cfg["linears"]
    L = layers
    sus_note = f"{src} bf16_tflops_sustained (MEASURED_PEAKS.json): the op runs inside a long step"
    parts, groups = {}, {}
    q_ms = group_ms["weight_refresh"]
    parts["weight_refresh"] = {
        "us": q_ms * 1e3, "GB/s": c["refresh_bytes"] * L / q_ms / 1e6, "frac_hbm": c["refresh_bytes"] * L / q_ms / 1e6 / hbm,
        "note": "amax + NVFP4 encode of every weight of every layer, one nvfp4_quantize_batch call per layer; bytes: "
                "each weight read once, codes and scales written (the amax pass reads each weight again)"}
    groups["weight_refresh"] = q_ms
    for phase in ("d", "p"):
        if f"rmsnorm_{phase}" not in op_ms:
            continue
        M = cfg["decode_m"] if phase == "d" else cfg["prefill_m"]
        kind = "w4a16" if phase == "d" else "w4a4"
        r_ms = group_ms[f"rmsnorm_{phase}"]
        rb = c["rms_d_bytes" if phase == "d" else "rms_p_bytes"] * L
        parts[f"rmsnorm_aqn_m{M}"] = {"us": r_ms * 1e3, "GB/s": rb / r_ms / 1e6, "frac_hbm": rb / r_ms / 1e6 / hbm}
        l_ms = group_ms[f"linears_{phase}"]
        fl, by = c[f"{kind}_flops"] * L, c[f"{kind}_bytes"] * L
        tf = fl / l_ms / 1e9
        part = {"us": l_ms * 1e3, "TFLOP/s": tf, "GB/s": by / l_ms / 1e6, "frac_hbm": by / l_ms / 1e6 / hbm,
                "per_linear_us": {n: op_ms[f"{kind}_{n}"] * 1e3 / L for n, _, _ in lin}}
        if kind == "w4a16":
            part["frac_bf16_tensor"] = tf / bf16_sus
            part["note"] = ("fractions against the sustained bf16 tensor peak and the HBM copy rate; us: the phase's "
                            "linears as one span; per_linear_us: per layer (LoRA-down + w4a16_tc_kernel), with events "
                            "around every call (each call boundary then adds its own gap)")
            groups["lora_linear_w4a16"] = l_ms
        else:
            part["frac_fp4_tensor"] = tf / fp4_sus
            part["note"] = (f"us: the phase's linears as one span; per_linear_us: events around every call; "
                            f"the full calls: LoRA-down and the block-scaled GEMM; q/k/v and gate/up read the NVFP4 "
                            f"activations rmsnorm_aqn_quantize wrote (timed under rmsnorm), o and down quantize theirs "
                            f"(amax + encode) in the call; fraction of the dense FP4 peak = {FP4_PER_BF16:g} x "
                            f"sustained bf16 (the nominal 13.5 / 2.25 ratio)")
            groups["lora_linear_w4a4"] = l_ms
        parts[f"lora_linear_{kind}_m{M}"] = part
    rms_ms = sum(group_ms[f"rmsnorm_{p}"] for p in ("d", "p") if f"rmsnorm_{p}" in group_ms)
    groups["rmsnorm_aqn"] = rms_ms
    dom = max(groups, key=groups.get)
    n_lin = len(lin) * L
    if dom == "lora_linear_w4a4":
        ach = c["w4a4_flops"] * L / groups[dom] / 1e9
        roofline = {"kernel": dom, "bound": "tensor", "dtype": "fp4", "achieved": ach, "peak": fp4_sus,
                    "unit": "TFLOP/s", "frac": ach / fp4_sus,
                    "peak_source": f"{FP4_PER_BF16:g} x {sus_note}",
                    "algorithmic_flops_per_launch": c["w4a4_flops"] * L / n_lin, "launches_per_step": n_lin}
    elif dom == "lora_linear_w4a16" and cfg["unit"] == "TFLOP/s":
        ach = c["w4a16_flops"] * L / groups[dom] / 1e9
        roofline = {"kernel": dom, "bound": "tensor", "dtype": "bf16", "achieved": ach, "peak": bf16_sus,
                    "unit": "TFLOP/s", "frac": ach / bf16_sus, "peak_source": sus_note,
                    "algorithmic_flops_per_launch": c["w4a16_flops"] * L / n_lin, "launches_per_step": n_lin}
    else:
        key = {"weight_refresh": "refresh_bytes", "lora_linear_w4a16": "w4a16_bytes"}.get(dom)
        nb = c[key] * L if key else c["rms_d_bytes"] * L + c["rms_p_bytes"] * L
        per = L if dom == "weight_refresh" else (n_lin if dom == "lora_linear_w4a16" else 2 * L * len(
            [p for p in ("d", "p") if f"rmsnorm_{p}" in op_ms]))
        ach = nb / groups[dom] / 1e6
        roofline = {"kernel": dom, "bound": "hbm", "achieved": ach, "peak": hbm, "unit": "GB/s", "frac": ach / hbm,
                    "peak_source": f"{src} (MEASURED_PEAKS.json hbm_gbs)" if src == "measured" else "fallback",
                    "algorithmic_bytes_per_launch": nb / per, "launches_per_step": per}
    tr = recorded_traffic(f"{args.config}:{dom}")
    roofline["traffic"] = None if tr is None else tr["dram_bytes_per_launch"]
    units, _ = step_units(cfg, layers)
    return {
        "metric": METRIC, "value": value, "unit": cfg["unit"], "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step,
        "ms_per_step_p10_p50_p90": [float(np.percentile(step_ms, q)) for q in (10, 50, 90)],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded, generated on device)",
        "config": {"workload": cfg["workload"], "layers_per_step": layers,
                   "l2": "inputs larger than L2: every layer streams its own bf16 weights and NVFP4 codes (far more "
                         "than the 129 MB L2); no flush",
                   "replicas": world, "algorithmic_bytes_per_step": c["bytes"] * layers,
                   "linear_flops_per_step": c["flops"] * layers,
                   "tokens_per_refresh": {"decode": cfg["decode_m"], "prefill": cfg["prefill_m"]}},
        "parts": parts, "roofline": roofline, "e2e": e2e, "gpu_launches": int(launches),
        "clocks": clocks.summary(),
    }


def select_ops(spec, ops):
    """--op names: op names of the step (weight_refresh, rmsnorm_d, w4a16_<w>, rmsnorm_p, w4a4_<w>), the
    single-weight amax_<w> / quantize_<w> (the per-tensor amax and encode kernels alone; not part of the
    step) or the groups w4a16, w4a4, linears, refresh, rmsnorm, amax, quantize, all (= the step's ops);
    comma-separated. Single ops run on layer 0."""
    groups = {"w4a16": [o for o in ops if o.startswith("w4a16_")], "w4a4": [o for o in ops if o.startswith("w4a4_")],
              "linears": [o for o in ops if o.startswith(("w4a16_", "w4a4_"))], "refresh": ["weight_refresh"],
              "rmsnorm": [o for o in ops if o.startswith("rmsnorm")], "amax": [o for o in ops if o.startswith("amax_")],
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


def run_ops(args, torch, nv, wl, ops, flush, stream, rank):
    """Single-op timing (eager launches on layer 0; before every op a 256 MB read evicts L2): W warm-up and
    K timed runs of each selected op; one JSON line of per-op device microseconds. Serves per-kernel
    measurement and profiler captures of one op on the step's full-size inputs."""
    solo = [f"amax_{n}" for n, _, _ in wl.cfg["linears"]] + [f"quantize_{n}" for n, _, _ in wl.cfg["linears"]]
    sel = select_ops(args.op, ops + solo)
    flush64 = flush.view(torch.int64)

    def evict():  # read a buffer twice the L2 size: L2 then holds clean lines only (no write-backs later)
        flush64.sum()

    res = {}
    for name in sel:
        for i in range(args.warmup):
            evict()
            wl.step(nv, i % (KSCHED + 1), only={name}, layer_sel=[0])
        torch.cuda.synchronize()
        ts = []
        for i in range(args.steps):
            evict()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            wl.step(nv, i % (KSCHED + 1), only={name}, layer_sel=[0])
            b.record(stream)
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b) * 1e3)
        res[name] = {"us_median": float(np.median(ts)), "us_min": float(np.min(ts)), "runs": len(ts)}
    if rank == 0:
        print(json.dumps({"mode": "ops", "workload": wl.cfg["workload"], "steps": args.steps, "warmup": args.warmup,
                          "ops": res}))


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
    hbm, bf16_tf, _, src = peaks()
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

    r = 32  # LoRA rank of the 7B cases
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
    # ---- plain encode of the 7B gate weight with its amax given (the single encode pass alone)
    if want("quantize_amax_given"):
        n, k = 18944, 3584
        W = weight(n, k)
        am = W.float().abs().amax().reshape(1)
        c = torch.empty(n, k // 2, dtype=torch.uint8, device=dev)
        sc = torch.empty(n, k // 16, dtype=torch.uint8, device=dev)
        g = torch.empty(1, dtype=torch.float32, device=dev)
        wsq = torch.empty(nv.workspace_bytes(nv.OP_QUANTIZE, 0, 0, 0), dtype=torch.uint8, device=dev)
        us_a = timed(lambda: nv.nvfp4_quantize(W, amax_in=am, codes=c, scales=sc, g=g, workspace=wsq), 10)
        emit("quantize_amax_given_7b_gate", us_a, 0, n * k * (2 + 0.5625), "hbm",
             {"shape": [n, k], "note": "one encode pass, amax given (nvfp4_quantize amax_in); bytes: 2 B in, "
                                       "0.5625 B out per element"})
        mask = torch.randint(-2 ** 31, 2 ** 31 - 1, ((n * k + 31) // 32,), generator=gen, device=dev,
                             dtype=torch.int64).to(torch.int32)  # Bernoulli(1/2) bits
        us_ga = timed(lambda: nv.nvfp4_quantize_guided(W, mask, amax_in=am, codes=c, scales=sc, g=g, workspace=wsq),
                      10)
        emit("quantize_guided_amax_given_7b_gate", us_ga, 0, n * k * (2 + 0.5625 + 0.125), "hbm",
             {"shape": [n, k], "note": "one guided encode pass, amax given; bytes: 2 B in, 0.5625 B out, 0.125 B "
                                       "of mask per element"})
        rec = torch.empty((n * k + 31) // 32, dtype=torch.int32, device=dev)
        us_ra = timed(lambda: nv.nvfp4_quantize_record(W, amax_in=am, codes=c, scales=sc, g=g, record=rec,
                                                       workspace=wsq), 10)
        emit("quantize_record_amax_given_7b_gate", us_ra, 0, n * k * (2 + 0.5625 + 0.125), "hbm",
             {"shape": [n, k], "note": "one record encode pass, amax given; bytes: 2 B in, 0.5625 B out, 0.125 B "
                                       "of record per element"})
        del W, c, sc, g, wsq, mask, rec
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



def run_e2e(args, nv, torch, dev, wl, world):
    """The same step through the public API, with its inputs copied from pinned host memory and its result
    read back to pinned host memory inside the timed region. Inputs: every layer's bf16 weights (the
    refresh's input; one pinned host copy per weight shape is sent to every layer) and the step's
    activations; the result: the outputs of every linear as they stand at the end of the step (the last
    layer's). The copies are the bound (the host link), so they run on a copy stream, layer by layer, and
    each layer is refreshed and run as soon as its weights have landed."""
    cfg, L = wl.cfg, wl.layers
    lin = cfg["linears"]
    host_w = {name: wl.W[0][name].cpu().pin_memory() for name, _, _ in lin}
    host_x, dev_x = {}, {}
    for phase, P in wl.phases.items():
        for key in ("x_in", "x_res", "attn", "act"):
            host_x[(phase, key)] = P["buf"][key].cpu().pin_memory()
            dev_x[(phase, key)] = P["buf"][key]
    host_out = {(phase, name): torch.empty(P["Y"][name].shape, dtype=torch.bfloat16).pin_memory()
                for phase, P in wl.phases.items() for name, _, _ in lin}
    h2d = L * sum(t.numel() * t.element_size() for t in host_w.values()) + \
        sum(t.numel() * t.element_size() for t in host_x.values())
    d2h = sum(t.numel() * t.element_size() for t in host_out.values())
    stream = torch.cuda.current_stream(dev)
    copy_stream = torch.cuda.Stream(dev)
    ev_x = torch.cuda.Event()
    ev_w = [torch.cuda.Event() for _ in range(L)]
    read_w = [torch.cuda.Event() for _ in range(L)]  # layer l's weights have been read by its refresh
    done = torch.cuda.Event()
    for e in read_w:
        e.record(stream)
    done.record(stream)

    def step(k):
        with torch.cuda.stream(copy_stream):
            copy_stream.wait_event(done)  # the previous step has read its activations
            for key, h in host_x.items():
                dev_x[key].copy_(h, non_blocking=True)
            ev_x.record(copy_stream)
            for l in range(L):
                copy_stream.wait_event(read_w[l])
                for name, _, _ in lin:
                    wl.W[l][name].copy_(host_w[name], non_blocking=True)
                ev_w[l].record(copy_stream)
        stream.wait_event(ev_x)
        for l in range(L):
            stream.wait_event(ev_w[l])
            wl.step(nv, k, only={"weight_refresh"}, layer_sel=[l])
            read_w[l].record(stream)
            wl.step(nv, k, only=set(wl.ops()) - {"weight_refresh"}, layer_sel=[l])
        for (phase, name), h in host_out.items():
            h.copy_(wl.phases[phase]["Y"][name], non_blocking=True)
        done.record(stream)

    for i in range(max(1, min(args.warmup, 2))):
        step(i % (KSCHED + 1))
    torch.cuda.synchronize()
    n = max(1, min(args.steps, args.e2e_steps))
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
    units, scale = step_units(cfg, L)
    return {"value": job_throughput(units, world, ms, scale), "unit": cfg["unit"], "ms_per_step": ms, "steps": n,
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)}


# ----------------------------------------------------------------------------- CPU oracle arm

_SAMPLE_INPUTS = {}


def _sample_input(key, make):
    """Seeded sample inputs, generated once per process (their generation is not part of the timing)."""
    if key not in _SAMPLE_INPUTS:
        _SAMPLE_INPUTS[key] = make()
    return _SAMPLE_INPUTS[key]


def oracle_sample(cfg, den: int):
    """A bounded sample of one layer of the step, run by the CPU oracle: RMSNorm-AQN of 1/den of each
    phase's tokens (twice), the NVFP4 encoding of 1/den of each weight's rows, and each linear's outputs
    for those rows: W4A16 on every decode token, W4A4 on 1/32 of the prefill tokens (g_x over all of
    them). Returns (metric units of the sample, seconds, threads, description)."""
    import oracle
    import synth
    H, r = cfg["hidden"], cfg["rank"]
    md, mp = cfg["decode_m"], cfg["prefill_m"]
    t_total, flops, nbytes = 0.0, 0.0, 0.0
    nthreads = oracle.threads()
    w = synth.aqn_weight(H, 9, 1)
    e = synth.aqn_eps(H, 9, 2)
    for phase, M in (("d", md), ("p", mp)):
        if not M:
            continue
        mr = max(1, M // den)
        x = _sample_input(("x", mr, H, M), lambda: synth.activation_bf16(mr, H, 9, 3, M))
        t0 = time.perf_counter()
        oracle.rmsnorm_aqn(x, w, e, np.float32(SIGMA0), 1e-6)
        oracle.rmsnorm_aqn(x, w, e, np.float32(SIGMA0), 1e-6)
        t_total += time.perf_counter() - t0
        nbytes += 2 * bytes_rmsnorm(mr, H)
    for i, (name, n, k) in enumerate(cfg["linears"]):
        rows = max(1, n // den)
        Wb = _sample_input(("w", rows, k, cfg["std"], cfg["outliers"], i),
                           lambda: synth.weight_bf16(rows, k, cfg["std"], 9, 10 + i, outlier_frac=cfg["outliers"]))
        t0 = time.perf_counter()
        codes, scales, g = oracle.quantize(Wb)
        t_total += time.perf_counter() - t0
        nbytes += bytes_quantize(rows * k)
        A, B = _sample_input(("lora", r, k, rows, i), lambda: synth.lora_factors(r, k, rows, 9, 20 + i))
        xi = _sample_input(("d", md, k), lambda: synth.activation_bf16(md, k, 9, 30, k))
        t0 = time.perf_counter()
        oracle.lora_linear_w4a16(xi, codes, scales, g, A, B, S_LORA)
        t_total += time.perf_counter() - t0
        flops += flops_linear(md, rows, k, r)
        nbytes += bytes_linear(md, rows, k, r)
        if mp:
            xp = _sample_input(("p", mp, k), lambda: synth.heavy_tail_activation_bf16(mp, k, 9, 31, k))
            sel = np.arange(0, mp, 32)
            t0 = time.perf_counter()
            oracle.lora_linear_w4a4(xp, codes, scales, g, A, B, S_LORA, rows=sel)
            t_total += time.perf_counter() - t0
            flops += flops_linear(len(sel), rows, k, r)
            nbytes += bytes_linear_w4a4(len(sel), rows, k, r)
    frac = "all" if den == 1 else f"1/{den}"
    desc = (f"one layer: RMSNorm-AQN of {frac} of the tokens twice; NVFP4 encoding of {frac} of each weight's rows; "
            f"each LoRA linear on those rows' outputs for all {md} decode tokens (W4A16)"
            + (f" and 1/32 of the {mp} prefill tokens (W4A4, g_x over all of them)" if mp else "") + " (fp64 oracle)")
    units = flops if cfg["unit"] == "TFLOP/s" else nbytes
    return units, t_total, nthreads, desc


def sample_den(cfg, seconds_budget: float) -> int:
    """The smallest sampling denominator whose oracle run fits the budget: two probe runs (at the config's
    probe denominator and half of it) fit t(den) = a + b / den (a: the work that does not shrink with den,
    such as the activation amax over all tokens), which is then extrapolated."""
    probe = cfg["probe_den"]
    _, t1, _, _ = oracle_sample(cfg, probe)
    _, t2, _, _ = oracle_sample(cfg, probe // 2)
    b = max(0.0, (t2 - t1) * probe)
    a = max(0.0, t1 - b / probe)
    if b == 0.0:  # timing noise: proportional extrapolation from the larger probe
        a, b = 0.0, t2 * probe / 2
    den = 1
    while den < probe and a + b / den > seconds_budget:
        den *= 2
    return den


def cpu_baseline(cfg, seconds_budget=20.0):
    den = sample_den(cfg, seconds_budget)
    u, t, th, desc = oracle_sample(cfg, den)
    scale = 1e12 if cfg["unit"] == "TFLOP/s" else 1e9
    return {"value": u / t / scale, "unit": cfg["unit"], "cores": th, "kind": "oracle", "sample": desc,
            "sample_seconds": t}


def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if not reference_runs_here(rank, world):
        return
    cfg = CONFIGS[args.config]
    # each step is a sample sized so that warm-up and timed steps together take about two minutes
    den = sample_den(cfg, 120.0 / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        oracle_sample(cfg, den)
    tot_u, tot_t, th, desc = 0.0, 0.0, 1, ""
    for _ in range(args.steps):
        u, t, th, desc = oracle_sample(cfg, den)
        tot_u += u
        tot_t += t
    scale = 1e12 if cfg["unit"] == "TFLOP/s" else 1e9
    v = tot_u / tot_t / scale
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": cfg["unit"], "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": tot_t / max(1, args.steps) * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
        "config": {"workload": cfg["workload"], "sample": desc},
        "cpu_baseline": {"value": v, "unit": cfg["unit"], "cores": th, "kind": "oracle", "sample": desc},
        "e2e": {"value": v, "unit": cfg["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--config", default="qwen32b", choices=sorted(CONFIGS))
    ap.add_argument("--layers", type=int, default=0, help="layers per step (default: the config's)")
    ap.add_argument("--e2e-steps", type=int, default=3, help="timed steps of the end-to-end measurement")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=20.0)
    ap.add_argument("--op", default=None, help="time single ops of the step instead (see select_ops)")
    ap.add_argument("--suite", default=None, nargs="?", const="all",
                    help="secondary measurements instead: all or any of w4a4_7b,w4a16_32b,w4a4_32b,moe,quantize_32b,"
                         "quantize_batch_32b,quantize_guided,rmsnorm_quantize,kv_attention,ais,rmsnorm_prefill")
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
