"""Throughput of the fused MoE expert layer on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

One "step" is one pass of the whole layer (route, permute, gate/up + SiLU-and-
mul, down projection with the route weight, ordered top-k reduce) over one
batch of synthetic input resident in HBM.  The default workload is the decode
sweep: the layer at T = 1, 8, 32 and 64 tokens (K=4096, I=1536, E=128,
top_k=8, bf16), all four passes forming one step.  Other workloads (prefill,
mxfp8, mxfp8_act, batched, batched_tokens, tiny) can be selected with --workload.

Rank 0 prints ONE JSON line.  After the headline workload, every other
configuration is timed in the same process on the same GPU (`configs`: value,
ms_per_step, the roofline of its dominant kernel, the whole-layer roofline
fraction and the clocks of its own timed region; --configs picks a subset,
--no-configs none).  `sweep` gives each pass of the headline workload its GEMM 1
and whole-layer time.

--gpus N runs N independent replicas, one per GPU (the layer has no exchange
step): under torchrun each rank is one replica; without a launcher bench.py
starts N local ranks itself.  A barrier brackets the timed region, the max time
over ranks is used, and value = routed tokens of all ranks / that time.

--impl reference times the CPU oracle (the plain fp64 C reference) on a bounded
sample of the same workload on all host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "routed tokens/s per MoE layer on 1 GB300; % of HBM (decode) / tensor (prefill) roofline"
UNIT = "routed tokens/s"
FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS = 6800.0, 1900.0


# ----------------------------------------------------------------------------
# workloads
# ----------------------------------------------------------------------------

def workload_list(name):
    from mixture_experts_layer_permute_gb300 import workloads as wl
    if name == "decode":
        return [wl.decode(T) for T in (1, 8, 32, 64)]
    if name.startswith("decode"):
        return [wl.decode(int(name[len("decode"):]))]
    return [{"prefill": wl.prefill, "mxfp8": wl.mxfp8, "mxfp8_act": wl.mxfp8_act, "batched": wl.batched,
             "batched_tokens": wl.batched_tokens, "tiny": wl.tiny}[name]()]


def describe(name, ws):
    if name == "decode":
        return "decode bf16 sweep T in {1,8,32,64}: K=4096, I=1536, E=128, top_k=8, contiguous, swap-AB tiles"
    w = ws[0]
    act = f"{w.act} quantised to mxfp8 on the fly" if w.act_quant else w.act
    return (f"{w.name}: T={w.T}, K={w.K}, I={w.I}, E={w.E}, top_k={w.top_k}, act={act}, weights={w.weight}, "
            f"layout={w.layout}, block_m={w.block_m}, max_tokens={w.max_tokens}")


def read_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", 0.0)), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


class Instance:
    """Device inputs and the layer object of one workload."""

    def __init__(self, w, seed, device, fused=True, tiled=True, weights=None, impl=None):
        import torch
        import mixture_experts_layer_permute_gb300 as m
        from mixture_experts_layer_permute_gb300 import workloads as wl
        self.w = w
        self.m = m
        dev = torch.device(device)
        self.routes_fixed = None
        if w.layout == "batched":
            self.xb, self.counts, self.rw = wl.batched_inputs(w, seed, dev)
            self.W1 = wl.expert_weights(w, "W1", seed, dev)
            self.W2 = wl.expert_weights(w, "W2", seed, dev)
            self.layer = m.MoELayer(0, w.K, w.I, w.E, 1, layout=m.MOE_LAYOUT_BATCHED, max_tokens=w.max_tokens,
                                    device=dev, impl=m.MOE_IMPL_AUTO if impl is None else impl)
            self.s1 = self.s2 = None
            self.W1r, self.W2r, self.w1_layout = self.W1, self.W2, w.w1_layout
            self.routes = int(self.counts.sum().item())
            self.used_experts = int((self.counts > 0).sum().item())
            if tiled and impl in (None, m.MOE_IMPL_AUTO, m.MOE_IMPL_TCGEN05_PAIR) and self._pair_plan():
                self._tile_weights()
            return
        self.x = wl.activations(w, seed, dev)
        if w.routing == "affine":
            self.ids, self.tw = [t.to(dev) for t in wl.affine_routing(w)]
            self.logits = None
        else:
            self.logits = wl.router_logits(w, seed, dev)
        if w.weight == "mxfp8" and weights is not None:   # the same draw, quantised once by another instance
            self.W1, self.s1, self.W2, self.s2 = weights
        elif w.weight == "mxfp8":
            self.W1, self.s1 = self._mxfp8(w, "W1", seed, dev)
            self.W2, self.s2 = self._mxfp8(w, "W2", seed, dev)
        else:
            self.W1 = wl.expert_weights(w, "W1", seed, dev)
            self.W2 = wl.expert_weights(w, "W2", seed, dev)
            self.s1 = self.s2 = None
        if w.layout == "batched_tokens":
            self.layer = m.MoELayer(w.T, w.K, w.I, w.E, w.top_k, act_dtype=self.x.dtype,
                                    layout=m.MOE_LAYOUT_BATCHED, max_tokens=w.max_tokens, device=dev,
                                    impl=m.MOE_IMPL_AUTO if impl is None else impl)
        else:
            self.layer = m.MoELayer(w.T, w.K, w.I, w.E, w.top_k, act_dtype=self.x.dtype, block_m=w.block_m,
                                    act_quant=w.act_quant, fused_experts=fused, device=dev,
                                    impl=m.MOE_IMPL_AUTO if impl is None else impl)
        # weights as the kernels stream them: row-major, or re-laid out once into the tile-contiguous layout by
        # moe_tile_weights (bf16 on the fused decode launch and CTA-pair tiles; MXFP8 codes with an interleave-16
        # W1 on swap-AB tiles) -- weight preparation, outside every timed region
        self.W1r, self.W2r, self.w1_layout = self.W1, self.W2, w.w1_layout
        self.forward()
        torch.cuda.synchronize()
        codes_tileable = (w.weight == "mxfp8" and w.layout == "contiguous" and w.w1_layout == m.MOE_W1_INTERLEAVE16
                          and impl in (None, m.MOE_IMPL_AUTO, m.MOE_IMPL_TCGEN05_SWAP_AB))
        if tiled and (codes_tileable or (w.weight == "bf16" and (
                (w.layout == "contiguous" and self.fused())
                or (impl in (None, m.MOE_IMPL_AUTO, m.MOE_IMPL_TCGEN05_PAIR) and self._pair_plan())))):
            self._tile_weights()
            self.forward()
            torch.cuda.synchronize()
        ids = self.layer.ids if self.logits is not None else self.ids
        kept = self.layer.route_row >= 0      # batched: routes beyond the capacity are dropped
        self.routes = int(kept.sum().item())
        self.used_experts = int(torch.unique(ids[kept]).numel())

    def _pair_plan(self):
        """True where the layer's GEMMs run on CTA-pair tiles (bf16, many rows per expert)."""
        return "CTA-pair" in gemm1_kernel(self)

    def _tile_weights(self):
        """Weights re-laid out once into the tile-contiguous layout the kernels stream (moe_tile_weights): weight
        preparation, outside every timed region."""
        m = self.m
        self.W1r = m.moe_tile_weights(self.W1, 1, self.w.w1_layout)
        self.W2r = m.moe_tile_weights(self.W2, 2)
        self.w1_layout = m.MOE_W_TILED

    def _mxfp8(self, w, which, seed, dev):
        import torch
        from mixture_experts_layer_permute_gb300 import workloads as wl
        rows, cols = (2 * w.I, w.K) if which == "W1" else (w.K, w.I)
        codes = torch.empty((w.E, rows, cols), dtype=torch.uint8, device=dev)
        scales = torch.empty((w.E, rows, cols // 32), dtype=torch.uint8, device=dev)
        for e in range(w.E):
            self.m.mxfp8_quantize_block32(wl.expert_weights(w, which, seed, dev, experts=[e])[0], codes=codes[e],
                                          scales=scales[e])
        return codes, scales

    def forward(self, x=None, logits=None, gemm1_events=None):
        L = self.layer
        w1_layout = self.w1_layout
        if self.w.layout == "batched":
            return L.forward(self.xb, self.W1r, self.W2r, expert_num_tokens=self.counts, row_weights=self.rw,
                             w1_layout=w1_layout, gemm1_events=gemm1_events)
        x = self.x if x is None else x
        if self.logits is not None:
            lg = self.logits if logits is None else logits
            return L.forward(x, self.W1r, self.W2r, logits=lg, w1_scale=self.s1, w2_scale=self.s2,
                             w1_layout=w1_layout, gemm1_events=gemm1_events)
        return L.forward(x, self.W1r, self.W2r, topk_ids=self.ids, topk_weights=self.tw, w1_scale=self.s1,
                         w2_scale=self.s2, w1_layout=w1_layout, gemm1_events=gemm1_events)

    def launches(self):
        return self.layer.launches_per_forward()

    # algorithmic bytes / FLOPs (touched weights + scales + activations in + output; 6 K I flops per route)
    def gemm1_bytes(self):
        w = self.w
        wb = 2 * w.I * w.K * (1 if w.weight == "mxfp8" else 2)
        sb = (2 * w.I * w.K // 32) if w.weight == "mxfp8" else 0
        act = 2 if w.act == "bf16" else 4
        if w.act_quant:   # MXFP8 rows in, MXFP8 h out (E4M3 codes + one scale byte per 32)
            return int(self.used_experts * (wb + sb) + self.routes * (w.K + w.I) * 33 // 32)
        return self.used_experts * (wb + sb) + self.routes * (w.K + w.I) * act

    def layer_bytes(self):
        w = self.w
        per_w = 3 * w.I * w.K * (1 if w.weight == "mxfp8" else (4 if w.weight == "f32" else 2))
        if w.weight == "mxfp8":
            per_w += 3 * w.I * w.K // 32
        act = 2 if w.act == "bf16" else 4
        if w.layout == "batched":
            return self.used_experts * per_w + 2 * self.routes * w.K * act
        return self.used_experts * per_w + 2 * w.T * w.K * act

    def layer_flops(self):
        return 6.0 * self.w.K * self.w.I * self.routes

    def gemm2_bytes(self):
        w = self.w
        return self.used_experts * w.K * w.I * 2 + self.routes * (w.I + w.K) * 2

    def fused(self):
        return any(name == "gemm1" and fn is self.layer.lib.moe_experts_fused for fn, _, name in (self.layer._plan or []))

    def gemm1_flops(self):
        return 4.0 * self.w.K * self.w.I * self.routes


# ----------------------------------------------------------------------------
# clocks
# ----------------------------------------------------------------------------

class ClockSampler:
    """Samples SM clock and clock-event reasons of one GPU while the timed region runs.

    Polls NVML (libnvidia-ml, loaded with ctypes) every 2 ms from a thread, so
    that even a timed region of a few tens of milliseconds gets many samples;
    falls back to `nvidia-smi -lms 100` when NVML cannot be loaded.  Reads only.
    """
    # clock-event reason bits of nvmlDeviceGetCurrentClocksEventReasons
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown"}

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.samples = []
        self.max_mhz = None
        self._stop = None
        self._thread = None
        self._smi = None

    def _nvml(self):
        import ctypes
        for name in ("libnvidia-ml.so.1", "libnvidia-ml.so"):
            try:
                lib = ctypes.CDLL(name)
                break
            except OSError:
                lib = None
        if lib is None or lib.nvmlInit_v2() != 0:
            return None
        h = ctypes.c_void_p()
        ok = False
        try:   # the CUDA device's PCI address (NVML numbers GPUs its own way)
            import torch
            pr = torch.cuda.get_device_properties(self.gpu)
            bus = f"{pr.pci_domain_id:08x}:{pr.pci_bus_id:02x}:{pr.pci_device_id:02x}.0".encode()
            ok = lib.nvmlDeviceGetHandleByPciBusId_v2(ctypes.c_char_p(bus), ctypes.byref(h)) == 0
        except (AttributeError, RuntimeError):
            ok = False
        if not ok and lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.gpu), ctypes.byref(h)) != 0:
            return None
        return lib, h

    def __enter__(self):
        import ctypes
        import threading
        nv = self._nvml()
        if nv is None:
            fd, self._path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            try:
                self._smi = subprocess.Popen(
                    ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=clocks.sm,clocks.max.sm,"
                     "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                     "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap",
                     "--format=csv,noheader,nounits", "-lms", "100"],
                    stdout=open(self._path, "w"), stderr=subprocess.DEVNULL)
            except OSError:
                self._smi = None
            return self
        lib, h = nv
        mx = ctypes.c_uint()
        if lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:   # NVML_CLOCK_SM = 1
            self.max_mhz = float(mx.value)
        self._stop = threading.Event()

        def poll():
            clk = ctypes.c_uint()
            rs = ctypes.c_ulonglong()
            while not self._stop.is_set():
                ok1 = lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0
                ok2 = lib.nvmlDeviceGetCurrentClocksEventReasons(h, ctypes.byref(rs)) == 0
                if ok1:
                    self.samples.append((float(clk.value), int(rs.value) if ok2 else 0))
                time.sleep(0.002)

        self._thread = threading.Thread(target=poll, daemon=True)
        self._thread.start()
        return self

    def __exit__(self, *exc):
        if self._thread is not None:
            self._stop.set()
            self._thread.join(timeout=2)
        if self._smi is not None:
            self._smi.terminate()
            try:
                self._smi.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self._smi.kill()
            try:
                with open(self._path) as f:
                    for line in f:
                        parts = [p.strip() for p in line.split(",")]
                        if len(parts) >= 6 and parts[0].replace(".", "").isdigit():
                            bits = 0
                            for b, v in zip((0x8, 0x40, 0x20, 0x4), parts[2:6]):
                                if v.lower().startswith("active"):
                                    bits |= b
                            self.samples.append((float(parts[0]), bits))
                            if parts[1].replace(".", "").isdigit():
                                self.max_mhz = float(parts[1])
                os.remove(self._path)
            except OSError:
                pass

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": ["unsampled"], "samples": 0}
        bits = 0
        for _, b in self.samples:
            bits |= b
        reasons = sorted(name for b, name in self.REASONS.items() if bits & b)
        return {"sm_mhz": statistics.median(c for c, _ in self.samples), "sm_max_mhz": self.max_mhz,
                "reasons": reasons, "samples": len(self.samples),
                "source": "nvml" if self._smi is None else "nvidia-smi"}


# ----------------------------------------------------------------------------
# traffic from the committed ncu summary (valid only for the kernel source it was taken on)
# ----------------------------------------------------------------------------

def kernel_source_hash(name="gemm_tc.cu"):
    """Hash of a kernel source's code: comments, trailing blanks and empty lines are left out, so that a record
    taken on a kernel stays valid across edits of its comments only."""
    import re
    p = os.path.join(ROOT, "mixture_experts_layer_permute_gb300", "csrc", name)
    with open(p) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)            # block comments
    text = re.sub(r"//[^\n]*", "", text)                          # line comments (none sit inside strings here)
    code = "\n".join(line.rstrip() for line in text.splitlines() if line.strip())
    return hashlib.sha256(code.encode()).hexdigest()[:16]


def recorded_traffic(workload, fused=False, tiled=False):
    """GEMM 1 DRAM bytes per launch from the committed ncu summary, if taken on this kernel source.

    profiles/gemm_{tc,mx,pair}_traffic_<workload>.txt holds `source <file>`, `source_sha <hash>` (or the older
    `gemm_tc_sha`), `workload` and `gemm1_traffic_bytes` lines."""
    tag = "decode_sweep" if workload == "decode" else workload
    for kind in ("tc", "mx", "pair"):
        p = os.path.join(ROOT, "profiles", f"gemm_{kind}_traffic_{tag}.txt")
        fields = {}
        try:
            with open(p) as f:
                for line in f:
                    line = line.strip()
                    if line and not line.startswith("#"):
                        k, _, v = line.partition(" ")
                        fields[k] = v.split()
        except OSError:
            continue
        src = fields.get("source", ["gemm_tc.cu"])[0]
        sha = (fields.get("source_sha") or fields.get("gemm_tc_sha") or [None])[0]
        if sha != kernel_source_hash(src) or fields.get("workload", [None])[0] != workload:
            continue
        if fields.get("experts", ["split"])[0] != ("fused" if fused else "split"):
            continue
        if fields.get("weights", ["stored"])[0] != ("tiled" if tiled else "stored"):
            continue
        vals = [int(v) for v in fields.get("gemm1_traffic_bytes", [])]
        if vals:
            return vals
    return None


def aggregate_over_ranks(ms_total, routes, world, device):
    """Whole-job figures of N replicas: the slowest rank's time (max) and every rank's routes (sum)."""
    if world <= 1:
        return float(ms_total), float(routes)
    import torch
    import torch.distributed as dist
    tt = torch.tensor([float(ms_total)], dtype=torch.float64, device=device)
    dist.all_reduce(tt, op=dist.ReduceOp.MAX)
    rr = torch.tensor([float(routes)], dtype=torch.float64, device=device)
    dist.all_reduce(rr, op=dist.ReduceOp.SUM)
    return float(tt.item()), float(rr.item())


# ----------------------------------------------------------------------------
# our arm
# ----------------------------------------------------------------------------

def measure(insts, args, stream, world=1, flush=None):
    """Times K steps of the passes in `insts` (one step = one forward of each, in order).

    Graph mode (default): the K steps are captured in one CUDA graph with no event node inside and one replay
    is timed with events on the stream around it (barriers on both sides for N > 1), while the SM clocks are
    sampled; four more replays and one eager run of the same steps give the spread.  A second graph of the same
    K steps with CUDA events around every GEMM 1 launch (or fused experts launch) gives the launch durations
    behind the roofline, and for more than one pass a graph of K steps of each pass alone gives that pass's
    whole-layer time.  `flush` (a device buffer larger than L2): for inputs that fit in L2, the buffer is
    rewritten before every step and the timed quantity is the sum of CUDA events around each forward.
    """
    import numpy as np
    import torch
    import torch.distributed as dist
    K = args.steps
    ext = not args.eager

    def ev():
        return torch.cuda.Event(enable_timing=True, external=ext), torch.cuda.Event(enable_timing=True, external=ext)
    gev = [[ev() for _ in range(K)] for _ in insts]      # GEMM 1 (or fused experts) launches
    lev = [[ev() for _ in range(K)] for _ in insts]      # whole forwards (flush mode)

    def step(s=None, gemm=False):
        for n, inst in enumerate(insts):
            inst.forward(gemm1_events=gev[n][s] if gemm else None)

    def step_flush(s):
        flush.fill_(s & 127)
        cur = torch.cuda.current_stream()     # the capture stream while a graph is being recorded
        for n, inst in enumerate(insts):
            lev[n][s][0].record(cur)
            inst.forward()
            lev[n][s][1].record(cur)

    timed = step_flush if flush is not None else (lambda s: step(s))
    for s in range(args.warmup):
        timed(s % K)
    torch.cuda.synchronize()

    def graph_of(fn):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for s in range(K):
                fn(s)
        g.replay()                    # untimed: uploads the graph
        torch.cuda.synchronize()
        return g

    mode = "eager" if args.eager else "cuda_graph"
    g_main = g_gemm = None
    g_pass = []
    if not args.eager:
        try:
            g_main = graph_of(timed)
            g_gemm = graph_of(lambda s: step(s, gemm=True))
            if len(insts) > 1 and flush is None:
                g_pass = [graph_of(lambda s, i=inst: i.forward()) for inst in insts]
        except Exception as exc:      # capture unavailable: time the same launches eagerly
            print(f"bench: graph capture failed ({exc}); timing eagerly", file=sys.stderr)
            g_main = g_gemm = None
            g_pass = []
            mode = "eager (capture failed)"
            gev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
                   for _ in insts]
            lev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
                   for _ in insts]

    def run_main():
        if g_main is not None:
            g_main.replay()
        else:
            for s in range(K):
                timed(s)

    def once():
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        run_main()
        b.record(stream)
        torch.cuda.synchronize()
        if flush is not None:
            return sum(x.elapsed_time(y) for e in lev for x, y in e)
        return a.elapsed_time(b)

    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(torch.cuda.current_device()) as clk:
        ms_total = once()
        if world > 1:
            dist.barrier()
    reps = [ms_total / K] + [once() / K for _ in range(4 if g_main is not None else 0)]
    eager_ms = reps[0]
    if g_main is not None:
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for s in range(K):
            timed(s)
        b.record(stream)
        torch.cuda.synchronize()
        eager_ms = (sum(x.elapsed_time(y) for e in lev for x, y in e) if flush is not None
                    else a.elapsed_time(b)) / K
    stats = {"ms_per_step_replays": [round(x, 4) for x in reps], "median": round(statistics.median(reps), 4),
             "p10": round(float(np.percentile(reps, 10)), 4), "p90": round(float(np.percentile(reps, 90)), 4),
             "eager_ms_per_step": round(eager_ms, 4)}
    # the GEMM launch durations, from the same K steps again with their events
    if g_gemm is not None:
        g_gemm.replay()
    else:
        for s in range(K):
            step(s, gemm=True)
    torch.cuda.synchronize()
    g1_ms = [sum(a.elapsed_time(b) for a, b in e) / K for e in gev]
    # whole-layer time of each pass
    if flush is not None:
        layer_ms = [sum(a.elapsed_time(b) for a, b in e) / K for e in lev]
    elif g_pass:
        layer_ms = []
        for g in g_pass:
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            g.replay()
            b.record(stream)
            torch.cuda.synchronize()
            layer_ms.append(a.elapsed_time(b) / K)
    else:
        layer_ms = [ms_total / K]
    return {"ms_total": ms_total, "clocks": clk.summary(), "timing_stats": stats, "g1_ms": g1_ms,
            "layer_ms": layer_ms, "mode": mode}


def gemm_roofline(insts, g1_ms, peaks, tensor_bound):
    """Roofline of the dominant kernel (GEMM 1, or GEMM 1 + GEMM 2 where one launch runs both): algorithmic
    bytes (HBM bound) or flops (tensor bound) per launch over its average launch duration."""
    hbm, tf_burst, _tf_sust, peak_kind = peaks
    g1_bytes = [i.gemm1_bytes() + (i.gemm2_bytes() if i.fused() else 0) for i in insts]
    g1_flops = [i.gemm1_flops() for i in insts]
    if tensor_bound:
        achieved = sum(g1_flops) / (sum(g1_ms) / 1e3) / 1e12
        roof = {"bound": "tensor", "achieved": round(achieved, 2), "peak": tf_burst, "unit": "TFLOP/s",
                "frac": round(achieved / tf_burst, 4)}
    else:
        achieved = sum(g1_bytes) / (sum(g1_ms) / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                "frac": round(achieved / hbm, 4)}
    roof["kernel"] = gemm1_kernel(insts[0])
    roof["peak_source"] = (f"MEASURED_PEAKS.json ({peak_kind}), " +
                           ("bf16_tflops (burst: the GEMM runs inside a timed replay of milliseconds)"
                            if tensor_bound else "hbm_gbs"))
    roof["algorithmic_per_launch"] = [int(b) for b in (g1_flops if tensor_bound else g1_bytes)]
    roof["launch_ms"] = [round(x, 4) for x in g1_ms]
    roof["timing"] = "CUDA events around each GEMM launch, in a replay of the same K steps right after the timed one"
    return roof


def gemm1_kernel(inst):
    """The kernel behind the timed GEMM 1 launch, by the library's MOE_IMPL_AUTO rule: block-scaled MXFP8 for
    quantised activations, the fused experts launch in the decode regime, swap-AB tiles for E4M3 weights or
    few rows per expert, CTA-pair tiles otherwise (bf16)."""
    w, L = inst.w, inst.layer
    if w.act_quant:
        return "gemm_mx_kernel (moe_gemm1_swiglu)"
    if inst.fused():
        return "gemm_tc_kernel (moe_experts_fused: GEMM 1 + GEMM 2 in one launch)"
    if w.weight == "f32":
        return "gemm_simt_kernel (moe_gemm1_swiglu)"
    per_expert = (L.max_tokens // 2) if w.layout != "contiguous" else L.rows_cap // max(1, w.E)
    if w.weight == "mxfp8" or per_expert < 64:
        return "gemm_tc_kernel (moe_gemm1_swiglu, swap-AB tiles)"
    return "gemm_pair_kernel (moe_gemm1_swiglu, CTA-pair tiles)"


def layer_sweep(insts, m, peaks):
    """Per pass: routes, touched experts, algorithmic bytes and flops, GEMM 1 and whole-layer time, and the
    layer's roofline time max(flops / tensor peak, bytes / HBM peak)."""
    hbm, tf_burst = peaks[0], peaks[1]
    out = []
    for n, inst in enumerate(insts):
        t_roof = max(inst.layer_flops() / (tf_burst * 1e12), inst.layer_bytes() / (hbm * 1e9)) * 1e3
        out.append({"workload": inst.w.name, "routes": inst.routes, "experts_touched": inst.used_experts,
                    "layer_bytes": inst.layer_bytes(), "layer_flops": inst.layer_flops(),
                    "gemm1_ms": round(m["g1_ms"][n], 4), "layer_ms": round(m["layer_ms"][n], 4),
                    "roofline_ms": round(t_roof, 4), "layer_frac": round(t_roof / m["layer_ms"][n], 4)})
    return out


def run_ours(args, rank, world, local_rank):
    import torch

    torch.cuda.set_device(local_rank)
    dev = f"cuda:{local_rank}"
    ws = workload_list(args.workload)
    if args.experts or args.tokens:
        from mixture_experts_layer_permute_gb300 import workloads as wl
        ws = [wl.scaled(w, E=args.experts or w.E, T=args.tokens or w.T) for w in ws]
    import mixture_experts_layer_permute_gb300 as m
    impl = {"auto": m.MOE_IMPL_AUTO, "tcgen05": m.MOE_IMPL_TCGEN05, "swap_ab": m.MOE_IMPL_TCGEN05_SWAP_AB,
            "pair": m.MOE_IMPL_TCGEN05_PAIR, "mixed": m.MOE_IMPL_TCGEN05_MIXED, "simt": m.MOE_IMPL_SIMT}[args.gemm_impl]
    insts = [Instance(w, args.seed, dev, fused=not args.split_experts, tiled=not args.row_major_weights, impl=impl)
             for w in ws]
    stream = torch.cuda.current_stream()
    peaks = read_peaks()
    flush = l2_flush_buffer(insts, dev)
    m = measure(insts, args, stream, world, flush)
    routes_per_step = sum(i.routes for i in insts)
    t_max, total_routes = aggregate_over_ranks(m["ms_total"], routes_per_step * args.steps, world, dev)
    value = total_routes / (t_max / 1e3)
    prefill = args.workload == "prefill"
    roof = gemm_roofline(insts, m["g1_ms"], peaks, tensor_bound=prefill)
    roof["traffic"] = recorded_traffic(args.workload, any(i.fused() for i in insts),
                                       any(i.w1_layout == i.m.MOE_W_TILED for i in insts))
    sweep = layer_sweep(insts, m, peaks)
    del flush

    configs = None
    if world == 1 and rank == 0 and not args.no_configs:
        configs = run_configs(args, dev, stream, peaks, skip=args.workload)
    e2e = None if args.no_e2e else run_e2e(args, insts, dev)
    launches = sum(i.launches() for i in insts) * args.steps
    cpu = cpu_baseline(args, insts) if (rank == 0 and world == 1 and not args.no_cpu_baseline) else None
    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(t_max / args.steps, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": insts[0].w.act, "data": "synthetic",
            "config": {"workload": describe(args.workload, ws), "parallelism": f"replicas x{world}",
                       "launch": m["mode"],
                       "weights": ("tile-contiguous (moe_tile_weights, prepared once, untimed)"
                                   if any(i.w1_layout == i.m.MOE_W_TILED for i in insts) else "as stored"),
                       "l2": l2_note(insts),
                       "routes_per_step": routes_per_step},
            "roofline": roof, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches, "clocks": m["clocks"],
            "timing_stats": m["timing_stats"], "sweep": sweep, "configs": configs,
        }
        print(json.dumps(line), flush=True)


L2_BYTES = 129 * 2 ** 20


def l2_flush_buffer(insts, dev):
    """A 512 MiB device buffer rewritten between steps when one step's touched bytes fit in L2 (else None)."""
    import torch
    if sum(i.layer_bytes() for i in insts) > 2 * L2_BYTES:
        return None
    return torch.empty(512 * 2 ** 20, dtype=torch.uint8, device=dev)


def l2_note(insts):
    if sum(i.layer_bytes() for i in insts) > 2 * L2_BYTES:
        return "inputs larger than L2 (the touched expert weights of every step exceed 129 MB)"
    return "L2 flushed between steps (512 MiB write, outside the timed forwards)"


# the other configurations, timed in the same process after the headline workload
CONFIG_WORKLOADS = ("tiny", "prefill", "mxfp8", "mxfp8_act", "batched", "batched_tokens")


def run_configs(args, dev, stream, peaks, skip=None):
    """Every other configuration, one at a time on the same GPU: value, ms_per_step, roofline of the dominant
    kernel, whole-layer roofline fraction and the clocks seen while it was timed."""
    import gc
    import torch
    out = {}
    shared = None   # the quantised MXFP8 weights, drawn once for mxfp8 and mxfp8_act
    chosen = [c for c in args.configs.split(",") if c]
    for c in chosen:
        if c not in CONFIG_WORKLOADS:
            raise SystemExit(f"bench.py: unknown configuration {c!r} (known: {', '.join(CONFIG_WORKLOADS)})")
    for name in CONFIG_WORKLOADS:
        if name == skip or name not in chosen:
            continue
        w = workload_list(name)[0]
        inst = Instance(w, args.seed, dev, weights=shared if w.weight == "mxfp8" else None)
        if w.weight == "mxfp8":
            shared = (inst.W1, inst.s1, inst.W2, inst.s2)
        flush = l2_flush_buffer([inst], dev)
        m = measure([inst], args, stream, 1, flush)
        roof = gemm_roofline([inst], m["g1_ms"], peaks, tensor_bound=(name == "prefill"))
        tiled = inst.w1_layout == inst.m.MOE_W_TILED
        roof["traffic"] = recorded_traffic(name, inst.fused(), tiled)
        sw = layer_sweep([inst], m, peaks)[0]
        out[name] = {"workload": describe(name, [w]), "value": round(inst.routes * args.steps / (m["ms_total"] / 1e3), 1),
                     "unit": UNIT, "ms_per_step": round(m["ms_total"] / args.steps, 4),
                     "routes_per_step": inst.routes, "experts_touched": inst.used_experts,
                     "weights": ("tile-contiguous (moe_tile_weights, prepared once, untimed)" if tiled
                                 else "as stored"),
                     "layer_roofline_ms": sw["roofline_ms"], "layer_frac": sw["layer_frac"],
                     "roofline": roof, "clocks": m["clocks"], "timing_stats": m["timing_stats"],
                     "gpu_launches": inst.launches() * args.steps, "l2": l2_note([inst]), "launch": m["mode"]}
        del inst, flush, m
        if name == "mxfp8_act" or (w.weight == "mxfp8" and ("mxfp8_act" == skip or "mxfp8_act" not in chosen)):
            shared = None
        gc.collect()
        torch.cuda.empty_cache()
    return out


def run_e2e(args, insts, dev):
    """Same metric through the public API with host buffers: every step copies its inputs (x and router logits
    of every pass, packed in one pinned staging buffer: one H2D copy) to the device, runs the layer (MoELayer.forward
    per pass) and reads each pass's output back to pinned host memory."""
    import torch
    # staging: the inputs of all passes back to back (256-byte aligned views), on the host (pinned) and device
    parts = []
    for inst in insts:
        src_x = inst.x if inst.w.layout != "batched" else inst.xb
        lg = getattr(inst, "logits", None)
        parts.append((src_x, lg))
    off, offs = 0, []
    for src_x, lg in parts:
        ox = off
        off += (src_x.numel() * src_x.element_size() + 255) // 256 * 256
        ol = None
        if lg is not None:
            ol = off
            off += (lg.numel() * lg.element_size() + 255) // 256 * 256
        offs.append((ox, ol))
    hstage = torch.empty(off, dtype=torch.uint8, pin_memory=True)
    dstage = torch.empty(off, dtype=torch.uint8, device=dev)

    def view(buf, o, like):
        n = like.numel() * like.element_size()
        return buf[o:o + n].view(like.dtype).view(like.shape)

    host = []
    for inst, (src_x, lg), (ox, ol) in zip(insts, parts, offs):
        view(hstage, ox, src_x).copy_(src_x.cpu())
        if lg is not None:
            view(hstage, ol, lg).copy_(lg.cpu())
        dx = view(dstage, ox, src_x)
        dl = view(dstage, ol, lg) if lg is not None else None
        ho = torch.empty(inst.layer.out.shape, dtype=inst.layer.out.dtype, pin_memory=True)
        host.append((ho, dx, dl))

    def kwargs_of(inst, dl):
        if inst.w.layout == "batched":
            return dict(expert_num_tokens=inst.counts, row_weights=inst.rw, w1_layout=inst.w1_layout)
        if dl is not None:
            return dict(logits=dl, w1_scale=inst.s1, w2_scale=inst.s2, w1_layout=inst.w1_layout)
        return dict(topk_ids=inst.ids, topk_weights=inst.tw, w1_scale=inst.s1, w2_scale=inst.s2,
                    w1_layout=inst.w1_layout)

    def h2d():
        dstage.copy_(hstage, non_blocking=True)

    def d2h_of(inst, ho):
        return lambda: ho.copy_(inst.layer.out, non_blocking=True)

    # one CUDA graph per step: the step's H2D copy, then the passes; each pass's output is read back on a side
    # stream while the next pass computes, and the side stream rejoins before the step ends
    side = torch.cuda.Stream(device=dev)

    def body():
        cur = torch.cuda.current_stream()
        h2d()
        for inst, (ho, dx, dl) in zip(insts, host):
            inst.layer.forward(dx, inst.W1r, inst.W2r, **kwargs_of(inst, dl))
            side.wait_stream(cur)
            with torch.cuda.stream(side):
                d2h_of(inst, ho)()
        cur.wait_stream(side)

    graph = None
    if not args.eager:
        try:
            body()                    # eager once: builds each layer's call plan for these tensors
            torch.cuda.synchronize()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                body()
        except RuntimeError as exc:
            print(f"bench: e2e graph capture failed ({exc}); e2e runs eagerly", file=sys.stderr)
            graph = None

    def step():
        if graph is not None:
            graph.replay()
        else:
            body()

    for _ in range(max(1, args.warmup)):
        step()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    routes = sum(i.routes for i in insts) * args.steps
    d2h = sum(h[0].numel() * h[0].element_size() for h in host)
    return {"value": round(routes / dt, 1), "unit": UNIT, "h2d_bytes_per_step": int(hstage.numel()),
            "d2h_bytes_per_step": d2h}


# ----------------------------------------------------------------------------
# CPU oracle (baseline / reference arm)
# ----------------------------------------------------------------------------

def oracle_sample(ws, seed, device_inputs=None):
    """Host inputs for a bounded oracle sample: one token of each pass of the workload (every route of it)."""
    import numpy as np
    import torch
    import oracle
    from mixture_experts_layer_permute_gb300 import workloads as wl
    samples = []
    for n, w in enumerate(ws):
        if w.layout == "batched":
            if device_inputs is not None:
                inst = device_inputs[n]
                e = int(torch.argmax(inst.counts).item())
                xb = wl.to_numpy(inst.xb[e:e + 1, :1])
                W1 = wl.to_numpy(inst.W1[e:e + 1])
                W2 = wl.to_numpy(inst.W2[e:e + 1])
            else:
                g = wl.scaled(w, E=1, max_tokens=1)
                xb = wl.to_numpy(wl._normal((1, 1, w.K), 1.0, seed, "xb", 0, "cpu", torch.bfloat16))
                W1 = wl.to_numpy(wl.expert_weights(g, "W1", seed))
                W2 = wl.to_numpy(wl.expert_weights(g, "W2", seed))
            samples.append(("batched", xb, W1, W2, None, None, 1))
            continue
        if device_inputs is not None:
            inst = device_inputs[n]
            x = wl.to_numpy(inst.x[:1])
            if inst.logits is not None:
                ids, wts = oracle.topk_route(inst.logits[:1].cpu().numpy(), w.top_k)
            else:
                ids, wts = inst.ids[:1].cpu().numpy(), inst.tw[:1].cpu().numpy()
            used = sorted({int(e) for e in ids.reshape(-1)})
            sel = torch.tensor(used, device=inst.W1.device)
            W1 = wl.to_numpy(inst.W1.index_select(0, sel))
            W2 = wl.to_numpy(inst.W2.index_select(0, sel))
            S1 = None if inst.s1 is None else wl.to_numpy(inst.s1.index_select(0, sel))
            S2 = None if inst.s2 is None else wl.to_numpy(inst.s2.index_select(0, sel))
        else:
            x = wl.to_numpy(wl.activations(wl.scaled(w, T=1), seed))
            if w.routing == "affine":
                it, iw = wl.affine_routing(wl.scaled(w, T=1))
                ids, wts = it.numpy(), iw.numpy()
            else:
                ids, wts = oracle.topk_route(wl.router_logits(wl.scaled(w, T=1), seed).numpy(), w.top_k)
            used = sorted({int(e) for e in ids.reshape(-1)})
            W1t = wl.expert_weights(w, "W1", seed, experts=used)
            W2t = wl.expert_weights(w, "W2", seed, experts=used)
            if w.weight == "mxfp8":
                W1, S1 = oracle.mxfp8_quantize(W1t.numpy())
                W2, S2 = oracle.mxfp8_quantize(W2t.numpy())
            else:
                W1, W2, S1, S2 = wl.to_numpy(W1t), wl.to_numpy(W2t), None, None
        remap = {e: i for i, e in enumerate(used)}
        cids = np.vectorize(lambda e: remap[int(e)])(ids).astype(np.int32)
        samples.append(("contig", x, W1, W2, (cids, wts, S1, S2, w.w1_layout, w.act_quant), None, int(ids.size)))
    return samples


def run_oracle_samples(samples):
    import oracle
    routes = 0
    for kind, x, W1, W2, extra, _, n in samples:
        if kind == "batched":
            oracle.moe_layer_batched(x, [1], None, W1, W2)
        else:
            cids, wts, S1, S2, w1l, aq = extra
            oracle.moe_layer(x, cids, wts, W1, W2, w1_scale=S1, w2_scale=S2, w1_layout=w1l, quant_x=aq,
                             quant_h="bf16" if aq else False)
        routes += n
    return routes


def host_cores():
    """Host cores this process may run on (the affinity mask; os.cpu_count() where that is unavailable)."""
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def time_oracle(samples, seconds, threads):
    """Routes per second of the oracle on `samples` (one token each) for about `seconds`: `threads` host threads
    each run whole oracle calls, one sample at a time (the oracle's C calls release the GIL); the oracle itself
    is unchanged."""
    from concurrent.futures import ThreadPoolExecutor
    t0 = time.perf_counter()
    routes, reps = 0, 0
    with ThreadPoolExecutor(max_workers=threads) as ex:
        while True:
            # one round: every thread gets len(samples) calls
            tasks = [[sm] for sm in samples] * threads
            routes += sum(ex.map(run_oracle_samples, tasks))
            reps += 1
            if time.perf_counter() - t0 > seconds or reps >= 50:
                break
    dt = time.perf_counter() - t0
    return routes / dt, routes, dt, reps


def cpu_baseline(args, insts):
    import oracle
    oracle.build()
    samples = oracle_sample([i.w for i in insts], args.seed, insts)
    n = host_cores()
    v1, r1, t1, k1 = time_oracle(samples, args.cpu_seconds / 2, 1)
    vn, rn, tn, kn = time_oracle(samples, args.cpu_seconds / 2, n)
    return {"value": round(vn, 3), "unit": UNIT, "cores": n, "kind": "oracle",
            "sample": f"one token of each pass of the workload (all its routes) per oracle call, fp64 C oracle; "
                      f"{n} host threads: {rn} routes in {tn:.1f} s; 1 thread: {r1} routes in {t1:.1f} s",
            "single_thread": {"value": round(v1, 3), "cores": 1},
            "nproc": os.cpu_count()}


def run_reference(args, rank):
    if rank != 0:
        return
    from concurrent.futures import ThreadPoolExecutor
    import oracle
    oracle.build()
    ws = workload_list(args.workload)
    samples = oracle_sample(ws, args.seed)
    n = host_cores()
    # each step: one oracle call per host thread, each on one token (all its routes) of one pass of the
    # workload, passes in rotation
    calls = 0

    def one_step(ex):
        nonlocal calls
        tasks = [[samples[(calls + i) % len(samples)]] for i in range(n)]
        calls += n
        return sum(ex.map(run_oracle_samples, tasks))

    with ThreadPoolExecutor(max_workers=n) as ex:
        for _ in range(args.warmup):
            one_step(ex)
        t0 = time.perf_counter()
        routes = 0
        for _ in range(args.steps):
            routes += one_step(ex)
        dt = time.perf_counter() - t0
    value = routes / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3 / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": describe(args.workload, ws),
                   "sample": f"each step: {n} oracle calls on {n} host threads, each one token (all its routes) of "
                             "one pass of the workload, passes in rotation"},
        "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": n, "kind": "oracle",
                         "sample": f"{n} tokens per step, one per host thread, fp64 C oracle"},
        "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def replica_launch(args, env):
    """How `bench.py --gpus N` runs: None when this process is one rank of a launch of N ranks (or N = 1 without
    a launcher), else the torchrun command that starts N local ranks, one replica per GPU.  A launcher whose
    world size differs from --gpus is an error."""
    world = env.get("WORLD_SIZE")
    if world is not None:
        if int(world) != args.gpus:
            raise SystemExit(f"bench.py: --gpus {args.gpus} but the launcher started {world} ranks")
        return None
    if args.gpus <= 1:
        return None
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    return [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={args.gpus}",
            "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.abspath(__file__)] + sys.argv[1:]


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="decode")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="time only the selected workload (by default every other configuration is timed after it, "
                         "in the line's `configs`)")
    ap.add_argument("--configs", default=",".join(CONFIG_WORKLOADS),
                    help="comma-separated configurations timed after the headline workload")
    ap.add_argument("--eager", action="store_true", help="issue the timed steps from Python, not as a CUDA graph")
    ap.add_argument("--split-experts", action="store_true",
                    help="run GEMM 1 and GEMM 2 as two launches even where the plan uses swap-AB tiles (by default "
                         "they are one launch, moe_experts_fused)")
    ap.add_argument("--row-major-weights", action="store_true",
                    help="stream the weights as stored (E, rows, cols); by default the fused decode plan reads them "
                         "re-laid out once by moe_tile_weights")
    ap.add_argument("--gemm-impl", default="auto", choices=["auto", "tcgen05", "swap_ab", "pair", "mixed", "simt"],
                    help="GEMM implementation of the headline workload's contiguous layer (default: the library's "
                         "choice)")
    ap.add_argument("--experts", type=int, default=0,
                    help="profiling only: fewer experts than the workload (a small case for ncu)")
    ap.add_argument("--tokens", type=int, default=0,
                    help="profiling only: another token count than the workload (with --experts, the routed rows "
                         "per expert of the full workload at a small size)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    cmd = replica_launch(args, os.environ)
    if cmd is not None:   # --gpus N without a launcher: N local ranks, one replica of the workload per GPU
        sys.exit(subprocess.call(cmd))
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    try:
        run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
