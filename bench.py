#!/usr/bin/env python3
"""Benchmark of the theta-bundle reconstruction linear on GB300.

Headline (one "step"): the Gemma-3-1B-shaped decode stack -- 26 layers x 7 projection
families in the pages' production-path form (q/k/v batched through aq_linear_qkv, gate and
up batched through aq_linear_multi, o and down through aq_linear: 4 calls per layer),
r = 16, one pass at each of M = 1, 4 and 16 tokens -- captured once into a CUDA graph
and replayed. Each layer reads its own physical copy of the family W0 (1.40 GB per pass,
well above the 129 MB L2), so W0 streams from HBM: value = algorithmic bytes / time (x of
a batched call counted once).

Also measured in the same run (extra keys): the same step with gate and up as separate
calls; the same stack with one shared W0 per family
as served at G = 1 (W0 stays in L2; effective GB/s, not an HBM figure); prefill TFLOP/s
on Gemma-3-1B shapes (r = 64, M = 8192) and on the 31B-class projection (21504 x 5376,
r = 128, M = 8192); W_eff precompute GB/s over the 60-layer 31B-class stack with G = 4.

--impl reference times the fp64 CPU oracle on a bounded sample of the same workload.
--sweep times the rank/shape sweep (gate-like and down-like projections, r = 0..256,
M = 1..4096) against the roofline; --case times one call for profiler captures.
"""
from __future__ import annotations

import os

_CORES = os.cpu_count() or 1
for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, str(_CORES))

import argparse  # noqa: E402
import json  # noqa: E402
import statistics  # noqa: E402
import sys  # noqa: E402
import time  # noqa: E402

import numpy as np  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from rank_weight_reconstruction_gb300 import synth  # noqa: E402

METRIC = "decode GB/s & prefill TFLOP/s of s⊙W0x+U(Vᵀx) on 1 GB300, % of roofline"
FAMS = synth.GEMMA3_1B_FAMILIES
LAYERS = synth.GEMMA3_1B_LAYERS
DECODE_MS = (1, 4, 16)
DECODE_RANK = 16


# ----------------------------------------------------------------------------------
# work accounting (algorithmic bytes / flops; dense work the method avoids is not counted)
# ----------------------------------------------------------------------------------
def linear_bytes(out, inp, r, M):
    return 2 * (out * inp + r * (out + inp) + out + M * (inp + out))


def qkv_bytes(shapes, r, M):
    inp = shapes[0][1]
    return 2 * (sum(o * inp + r * (o + inp) + o + M * o for o, _ in shapes) + M * inp)


def linear_flops(out, inp, r, M):
    return 2 * M * (out * inp + r * (out + inp)) + M * out


def precompute_bytes(out, inp, r):
    return 2 * (2 * out * inp + r * (out + inp) + out)


def nvfp4_bytes(out, inp, r):
    """Read W0, U, V, s once; write the E2M1 codes, the E4M3 scales and the global scale."""
    return 2 * out * inp + 2 * r * (out + inp) + 2 * out + out * inp // 2 + out * inp // 16 + 4


def gate_up_bytes(r, M):
    """gate and up over one x in one batched call: x counted once, like Q/K/V."""
    (og, ig), (ou, iu) = FAMS["gate_proj"], FAMS["up_proj"]
    return linear_bytes(og, ig, r, M) + linear_bytes(ou, iu, r, M) - 2 * M * ig


def decode_config():
    """The headline workload, shared by both arms of the benchmark."""
    return {"workload": "gemma3-1b-shaped decode stack: 26 layers x 7 projection families "
                        "(q 1024x1152, k/v 256x1152, o 1152x1024, gate/up 6912x1152, down 1152x6912), "
                        "r=16, one pass each at M=1,4,16; q/k/v batched via aq_linear_qkv and gate/up via "
                        "aq_linear_multi (the pages' production-path fusion, 4 calls per layer)",
            "layers": LAYERS, "rank": DECODE_RANK, "M": list(DECODE_MS),
            "algorithmic_bytes_per_step": step_bytes()}


def step_bytes(fuse_gateup=True):
    """Algorithmic bytes of one decode step. fuse_gateup: gate and up of a layer are one
    batched call (the pages' production path), so their shared x is read once."""
    qkv_shapes = [FAMS[f] for f in ("q_proj", "k_proj", "v_proj")]
    total = 0
    for M in DECODE_MS:
        per_layer = qkv_bytes(qkv_shapes, DECODE_RANK, M)
        for f in ("o_proj", "down_proj"):
            per_layer += linear_bytes(*FAMS[f], DECODE_RANK, M)
        if fuse_gateup:
            per_layer += gate_up_bytes(DECODE_RANK, M)
        else:
            per_layer += sum(linear_bytes(*FAMS[f], DECODE_RANK, M) for f in ("gate_proj", "up_proj"))
        total += LAYERS * per_layer
    return total


# ----------------------------------------------------------------------------------
# distributed plumbing (independent replicas, one per GPU)
# ----------------------------------------------------------------------------------
class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None

    def init(self, backend):
        if self.world > 1:
            import torch.distributed as dist
            dist.init_process_group(backend=backend)
            self.pg = dist

    def barrier(self):
        if self.pg is not None:
            self.pg.barrier()

    def max(self, v: float, device) -> float:
        if self.pg is None:
            return v
        import torch
        t = torch.tensor([v], dtype=torch.float64, device=device)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg is not None:
            self.pg.destroy_process_group()


# ----------------------------------------------------------------------------------
# clocks sampled during the timed region
# ----------------------------------------------------------------------------------
class ClockSampler:
    """Samples the SM clock and the clock-event (throttle) reasons of one GPU while the
    timed region runs: read-only NVML queries every millisecond from a background thread.
    Nothing about the GPU's settings is changed."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, torch_device_index: int):
        self.idx = torch_device_index
        self.samples = []
        self.max_mhz = None
        self._stop = False
        self._thread = None
        self._nvml = None
        self._handle = None

    def _open_nvml(self):
        import ctypes
        import torch
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        h = ctypes.c_void_p()
        uuid = getattr(torch.cuda.get_device_properties(self.idx), "uuid", None)
        ok = False
        if uuid is not None:
            ok = lib.nvmlDeviceGetHandleByUUID(("GPU-" + str(uuid)).encode(), ctypes.byref(h)) == 0
        if not ok and lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.idx), ctypes.byref(h)) != 0:
            raise OSError("no NVML handle")
        self._nvml, self._handle = lib, h
        mx = ctypes.c_uint()
        if lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
            self.max_mhz = float(mx.value)
        self._reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons")

    def _poll(self):
        import ctypes
        mhz = ctypes.c_uint()
        rs = ctypes.c_ulonglong()
        while not self._stop:
            if self._nvml.nvmlDeviceGetClockInfo(self._handle, 1, ctypes.byref(mhz)) == 0 and \
                    self._reasons_fn(self._handle, ctypes.byref(rs)) == 0:
                self.samples.append((float(mhz.value), int(rs.value)))
            time.sleep(0.001)

    def __enter__(self):
        import threading
        try:
            self._open_nvml()
            self._thread = threading.Thread(target=self._poll, daemon=True)
            self._thread.start()
        except (OSError, AttributeError):
            self._nvml = None
        return self

    def __exit__(self, *exc):
        self._stop = True
        if self._thread is not None:
            self._thread.join(timeout=2)

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": ["unsampled"], "samples": 0}
        reasons = set()
        for _, bits in self.samples:
            for b, name in self.REASONS.items():
                if bits & b:
                    reasons.add(name)
        return {"sm_mhz": statistics.median(m for m, _ in self.samples), "sm_max_mhz": self.max_mhz,
                "reasons": sorted(reasons), "samples": len(self.samples), "source": "nvml"}


# ----------------------------------------------------------------------------------
# helpers
# ----------------------------------------------------------------------------------
def dev_bits(bits, device):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


KERNEL_SOURCES = ("aq_decode.cu", "aq_decode2.cu", "aq_kernels.cu", "aq_host.cu", "aq_internal.h", "aq_ptx.cuh")


def kernel_source_hash():
    """sha256 over the CUDA sources: a profiler figure counts only for the code it measured."""
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "rank_weight_reconstruction_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def captured_traffic(key):
    """DRAM bytes (read + write) of one launch of `key` from the committed profiler summary
    profiles/dram_traffic.json, or None when that capture predates the current sources."""
    try:
        with open(os.path.join(ROOT, "profiles", "dram_traffic.json")) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None, "no capture"
    ent = rec.get("launches", {}).get(key)
    if ent is None:
        return None, "no capture of this call type"
    if rec.get("source_hash") != kernel_source_hash():
        return None, "capture predates the current kernel sources"
    return int(ent["dram_bytes"]), f"ncu capture ({ent.get('command', '')})"


def time_graph(g, reps, stream=None):
    """Average milliseconds of one replay of graph g over `reps` back-to-back replays."""
    import torch
    s = torch.cuda.Event(enable_timing=True)
    e = torch.cuda.Event(enable_timing=True)
    g.replay()
    torch.cuda.synchronize()
    s.record()
    for _ in range(reps):
        g.replay()
    e.record()
    torch.cuda.synchronize()
    return s.elapsed_time(e) / reps


# ----------------------------------------------------------------------------------
# the decode stack
# ----------------------------------------------------------------------------------
class DecodeStack:
    """26 layers x 7 families. ``copies=True`` gives every layer its own physical W0
    buffer (same values: G = 1 semantics, L2-cold streaming); ``copies=False`` shares one
    W0 per family as served at G = 1."""

    def __init__(self, device, copies: bool, seed_tag="bench"):
        import torch
        from rank_weight_reconstruction_gb300 import Theta
        self.device = device
        self.layers = []
        w0_host = {f: synth.make_w0((seed_tag, "W0", f), o, i) for f, (o, i) in FAMS.items()}
        w0_base = {f: dev_bits(w0_host[f], device) for f in FAMS}
        for layer in range(LAYERS):
            ths = {}
            for f, (o, i) in FAMS.items():
                th = synth.make_theta((seed_tag, f, layer), o, i, DECODE_RANK, W0=w0_host[f])
                W0 = w0_base[f].clone() if copies else w0_base[f]
                ths[f] = Theta(W0=W0[:, :i], s=dev_bits(th.s, device), U=dev_bits(th.U, device)[:, :DECODE_RANK],
                               V=dev_bits(th.V, device)[:, :DECODE_RANK])
            self.layers.append(ths)
        # activations: x per (M, layer, input) and outputs per call, in two flat buffers
        self.x_views, self.y_views = [], []
        x_sizes, y_sizes = [], []
        for M in DECODE_MS:
            for layer in range(LAYERS):
                x_sizes += [M * 1152, M * 1024, M * 1152, M * 6912]
                y_sizes += [M * o for o, _ in (FAMS[f] for f in FAMS)]
        self.X = torch.empty(sum(x_sizes), dtype=torch.bfloat16, device=device)
        self.Y = torch.empty(sum(y_sizes), dtype=torch.bfloat16, device=device)
        xh = synth.make_x((seed_tag, "x"), 1, sum(x_sizes))[0, :sum(x_sizes)]
        self.X_host = torch.from_numpy(xh.view(np.int16)).view(torch.bfloat16).pin_memory()
        self.Y_host = torch.empty(self.Y.numel(), dtype=torch.bfloat16).pin_memory()
        self.X.copy_(self.X_host)
        xo = yo = 0
        for M in DECODE_MS:
            for layer in range(LAYERS):
                xv = {}
                for key, inp in (("qkv", 1152), ("o", 1024), ("mlp", 1152), ("down", 6912)):
                    xv[key] = self.X[xo:xo + M * inp].view(M, inp)
                    xo += M * inp
                yv = {}
                for f, (o, _) in FAMS.items():
                    yv[f] = self.Y[yo:yo + M * o].view(M, o)
                    yo += M * o
                self.x_views.append((M, layer, xv))
                self.y_views.append(yv)
        import rank_weight_reconstruction_gb300 as aq
        ws = 0
        for M in DECODE_MS:
            th0 = self.layers[0]
            ws = max(ws, aq.aq_linear_workspace_bytes([th0["q_proj"], th0["k_proj"], th0["v_proj"]], M))
            for f in ("o_proj", "gate_proj", "up_proj", "down_proj"):
                ws = max(ws, aq.aq_linear_workspace_bytes(th0[f], M))
            ws = max(ws, aq.aq_linear_workspace_bytes([th0["gate_proj"], th0["up_proj"]], M))
        self.ws = torch.zeros(max(ws, 256), dtype=torch.uint8, device=device)   # sync part must start at 0

    def calls(self, only=None, fuse_gateup=False):
        """List of (family key, callable) in step order. fuse_gateup: gate and up of a layer
        go through one aq_linear_multi call (the pages' gate-up fusion)."""
        import rank_weight_reconstruction_gb300 as aq
        out = []
        for (M, layer, xv), yv in zip(self.x_views, self.y_views):
            th = self.layers[layer]
            if only in (None, "qkv"):
                out.append(("qkv", M, lambda th=th, xv=xv, yv=yv: aq.aq_linear_qkv(
                    [th["q_proj"], th["k_proj"], th["v_proj"]], xv["qkv"],
                    ys=[yv["q_proj"], yv["k_proj"], yv["v_proj"]], workspace=self.ws)))
            fams = (("o_proj", "o"), ("gate_proj", "mlp"), ("up_proj", "mlp"), ("down_proj", "down"))
            for f, key in fams:
                if fuse_gateup and f == "up_proj":
                    continue
                if fuse_gateup and f == "gate_proj":
                    if only in (None, "gate_up"):
                        out.append(("gate_up", M, lambda th=th, xv=xv, yv=yv: aq.aq_linear_multi(
                            [th["gate_proj"], th["up_proj"]], xv["mlp"], ys=[yv["gate_proj"], yv["up_proj"]],
                            workspace=self.ws)))
                    continue
                if only in (None, f):
                    out.append((f, M, lambda th=th, f=f, key=key, xv=xv, yv=yv: aq.aq_linear(
                        th[f], xv[key], y=yv[f], workspace=self.ws)))
        return out

    def capture(self, only=None, M=None, fuse_gateup=False):
        import torch
        import rank_weight_reconstruction_gb300 as aq
        calls = [c for c in self.calls(only, fuse_gateup) if M is None or c[1] == M]
        for _, _, fn in calls:          # eager warm-up: device set-up happens outside capture
            fn()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        launches = 0
        with torch.cuda.graph(g):
            for _, _, fn in calls:
                fn()
                launches += aq.aq_last_launch_count()
        return g, launches, calls


def call_bytes(key, M):
    if key == "gate_up":
        return gate_up_bytes(DECODE_RANK, M)
    if key == "qkv":
        return qkv_bytes([FAMS[f] for f in ("q_proj", "k_proj", "v_proj")], DECODE_RANK, M)
    return linear_bytes(*FAMS[key], DECODE_RANK, M)


# ----------------------------------------------------------------------------------
# our arm
# ----------------------------------------------------------------------------------
def run_ours(args, dist: Dist):
    import torch
    import rank_weight_reconstruction_gb300 as aq
    from rank_weight_reconstruction_gb300 import build_lib

    torch.cuda.set_device(dist.local_rank)
    device = torch.device("cuda", dist.local_rank)
    dist.init("nccl")
    build_lib.build()
    aq.load()
    pk = peaks()

    stack = DecodeStack(device, copies=True)
    g, launches, calls = stack.capture(fuse_gateup=True)
    B = step_bytes()
    assert B == sum(call_bytes(k, M) for k, M, _ in calls)
    for _ in range(args.warmup):
        g.replay()
    torch.cuda.synchronize()
    if args.profile:
        # kernel-profiler mode: the eager warm-up (one launch per call), W warm-up
        # replays and K replays of the step, nothing else
        for _ in range(args.steps):
            g.replay()
        torch.cuda.synchronize()
        return {"profile": True, "launches_per_step": launches, "warmup": args.warmup, "steps": args.steps,
                "status": aq.aq_device_status()}
    dist.barrier()
    torch.cuda.synchronize()
    ev_s, ev_e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(dist.local_rank) as clk:
        t0 = time.perf_counter()
        ev_s.record()
        for _ in range(args.steps):
            g.replay()
        ev_e.record()
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
    dist.barrier()
    torch.cuda.synchronize()
    ms = dist.max(ev_s.elapsed_time(ev_e), device)
    ms_step = ms / args.steps
    value = dist.world * B / (ms_step * 1e-3) / 1e9
    status = aq.aq_device_status()
    if status != aq.AQ_OK:
        raise RuntimeError(f"device status {status} after the timed region")

    result = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": dist.world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic: seeded splitmix64 + Box-Muller draws rounded to bf16; W0~N(0,0.02^2), "
                "s~U(0.9,1.1), U,V~N(0,0.01^2), x~N(0,1); shapes only, no trained weights",
        "config": decode_config(),
        "setup": {"calls_per_step": len(calls),
                  "w0_storage": "G=1 values, one physical W0 copy per layer (1.40 GB streamed per M pass)",
                  "l2": "inputs larger than L2 (each pass streams 1.40 GB of W0 against a 129 MB L2)",
                  "timing": "CUDA graph of the whole step, CUDA events on the replay stream, max over ranks",
                  "parallelism": f"replicas x{dist.world}"},
        "gpu_launches": launches * args.steps,
        "wall_s_timed": round(wall, 4),
        "peaks": pk,
    }
    result["clocks"] = clk.summary()

    # ---- per-call timing of the dominant call type (roofline) ----
    # (the step's own call types, plus gate and up as single calls for comparison)
    step_types = ("gate_up", "down_proj", "o_proj", "qkv")
    per_type = {}
    for key in step_types + ("gate_proj", "up_proj"):
        for M in DECODE_MS:
            gk, nl, ck = stack.capture(only=key, M=M, fuse_gateup=key == "gate_up")
            t = time_graph(gk, max(3, args.steps))
            per_type[(key, M)] = {"ms_per_call": t / len(ck), "bytes_per_call": call_bytes(key, M),
                                  "launches_per_call": nl / len(ck)}
            del gk
    total = {k: v["ms_per_call"] * LAYERS for k, v in per_type.items() if k[0] in step_types}
    dom = max(total, key=total.get)
    d = per_type[dom]
    ach = d["bytes_per_call"] / (d["ms_per_call"] * 1e-3) / 1e9
    traffic, traffic_src = captured_traffic(f"decode:{dom[0]}:M{dom[1]}")
    result["roofline"] = {
        "bound": "hbm",
        "kernel": f"aq_decode2_kernel ({dom[0]}, M={dom[1]}): clusters split over K, TMA W0 ring, mma.sync with "
                  "t = V^T x in the same loop, partial sums pushed through distributed shared memory, fused s "
                  "scale and U t",
        "achieved": round(ach, 1), "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": round(ach / pk["hbm_gbs"], 4),
        "peak_source": f"{pk['source']} copy bandwidth (burst)", "traffic": traffic, "traffic_source": traffic_src,
        "note": "algorithmic bytes of one call / average time per call over 26 back-to-back calls, each on its "
                "own W0 copy (L2-cold)"}
    result["decode_calls"] = {f"{k}@M{M}": {"GB_s": round(v["bytes_per_call"] / (v["ms_per_call"] * 1e-3) / 1e9, 1),
                                            "us_per_call": round(v["ms_per_call"] * 1e3, 3),
                                            "frac_hbm": round(v["bytes_per_call"] / (v["ms_per_call"] * 1e-3) / 1e9
                                                              / pk["hbm_gbs"], 4)}
                              for (k, M), v in per_type.items()}

    # ---- e2e: host buffers, copies inside the timed region ----
    h2d = stack.X.numel() * 2
    d2h = stack.Y.numel() * 2
    for _ in range(2):
        stack.X.copy_(stack.X_host, non_blocking=True)
        g.replay()
        stack.Y_host.copy_(stack.Y, non_blocking=True)
    torch.cuda.synchronize()
    dist.barrier()
    e_s, e_e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.perf_counter()
    e_s.record()
    for _ in range(args.steps):
        stack.X.copy_(stack.X_host, non_blocking=True)
        g.replay()
        stack.Y_host.copy_(stack.Y, non_blocking=True)
    e_e.record()
    torch.cuda.synchronize()
    e2e_wall = time.perf_counter() - t0
    e2e_ms = dist.max(e2e_wall * 1e3 / args.steps, device)
    result["e2e"] = {"value": round(dist.world * B / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                     "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                     "ms_per_step": round(e2e_ms, 5),
                     "how": "per step: pinned-host -> device copy of all x, the captured aq_* calls, device -> "
                            "pinned-host copy of all y; host wall clock around K steps"}
    del g
    if not args.decode_only:
        extras(result, args, dist, stack, device, pk)
    del stack
    torch.cuda.empty_cache()
    if dist.rank == 0 and not args.no_cpu_baseline and dist.world == 1:
        result["cpu_baseline"] = cpu_baseline(args, budget_s=args.cpu_seconds)
    elif dist.rank == 0:
        result["cpu_baseline"] = None
    status = aq.aq_device_status()
    if status != aq.AQ_OK:
        raise RuntimeError(f"device status {status} after the extra phases")
    return result


def extras(result, args, dist, stack, device, pk):
    import torch
    import rank_weight_reconstruction_gb300 as aq
    from rank_weight_reconstruction_gb300 import Theta

    # ---- the same step with gate and up of each layer as two aq_linear calls ----
    gf, lf, _ = stack.capture(fuse_gateup=False)
    t = time_graph(gf, max(3, args.steps))
    result["decode_gateup_separate"] = {"GB_s": round(step_bytes(fuse_gateup=False) / (t * 1e-3) / 1e9, 1),
                                        "ms_per_step": round(t, 4), "launches_per_step": lf,
                                        "note": "same outputs, gate and up of a layer as separate calls (5 calls per "
                                                "layer; x of the MLP read twice)"}
    del gf
    torch.cuda.empty_cache()

    # ---- as served at G = 1: one shared W0 per family (L2-resident) ----
    shared = DecodeStack(device, copies=False, seed_tag="bench")
    gs, _, calls = shared.capture(fuse_gateup=True)
    t = time_graph(gs, max(3, args.steps))
    result["decode_g1_as_served"] = {"effective_GB_s": round(step_bytes() / (t * 1e-3) / 1e9, 1),
                                     "ms_per_step": round(t, 4),
                                     "note": "same step, one W0 per family shared by all 26 layers (53.7 MB, "
                                             "L2-resident): effective rate, not an HBM figure"}
    del gs, shared
    torch.cuda.empty_cache()

    # ---- prefill: Gemma-3-1B shapes, r = 64, M = 8192, x rows scaled by U(0.5, 2) ----
    M, r = 8192, 64
    xs = {inp: dev_bits(synth.make_x(("bench-prefill", inp), M, inp, row_scale=(0.5, 2.0)), device)[:, :inp]
          for inp in (1152, 1024, 6912)}
    nl = 2
    layers = []
    for layer in range(nl):
        ths = {}
        for f, (o, i) in FAMS.items():
            th = synth.make_theta(("bench-prefill", f, layer), o, i, r)
            ths[f] = Theta(W0=dev_bits(th.W0, device)[:, :i], s=dev_bits(th.s, device),
                           U=dev_bits(th.U, device)[:, :r], V=dev_bits(th.V, device)[:, :r])
        layers.append(ths)
    ys = {f: torch.empty(M, o, dtype=torch.bfloat16, device=device) for f, (o, _) in FAMS.items()}
    ws = torch.zeros(max(aq.aq_linear_workspace_bytes([layers[0]["q_proj"], layers[0]["k_proj"],
                                                        layers[0]["v_proj"]], M),
                         aq.aq_linear_workspace_bytes([layers[0]["gate_proj"], layers[0]["up_proj"]], M),
                         aq.aq_linear_workspace_bytes(layers[0]["down_proj"], M)), dtype=torch.uint8, device=device)

    def prefill_layer(ths, fuse_gateup):
        aq.aq_linear_qkv([ths["q_proj"], ths["k_proj"], ths["v_proj"]], xs[1152],
                         ys=[ys["q_proj"], ys["k_proj"], ys["v_proj"]], workspace=ws)
        aq.aq_linear(ths["o_proj"], xs[1024], y=ys["o_proj"], workspace=ws)
        if fuse_gateup:
            aq.aq_linear_multi([ths["gate_proj"], ths["up_proj"]], xs[1152], ys=[ys["gate_proj"], ys["up_proj"]],
                               workspace=ws)
        else:
            aq.aq_linear(ths["gate_proj"], xs[1152], y=ys["gate_proj"], workspace=ws)
            aq.aq_linear(ths["up_proj"], xs[1152], y=ys["up_proj"], workspace=ws)
        aq.aq_linear(ths["down_proj"], xs[6912], y=ys["down_proj"], workspace=ws)

    flops_layer = sum(linear_flops(o, i, r, M) for o, i in FAMS.values())
    pre = {}
    # the pages' production-path form (Q/K/V and gate/up batched), then gate and up apart
    for key, fuse in (("gemma3_1b_M8192_r64", True), ("gemma3_1b_M8192_r64_gateup_separate", False)):
        for ths in layers:
            prefill_layer(ths, fuse)
        torch.cuda.synchronize()
        gp = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gp):
            for ths in layers:
                prefill_layer(ths, fuse)
        t = time_graph(gp, max(3, args.steps))
        tf = nl * flops_layer / (t * 1e-3) / 1e12
        pre[key] = {"TFLOP_s": round(tf, 1), "frac_bf16_peak": round(tf / pk["bf16_tflops"], 4),
                    "ms_per_layer": round(t / nl, 4), "flops_per_layer": flops_layer,
                    "calls_per_layer": 4 if fuse else 5}
        del gp
    # per family at M = 8192 (gate is the largest)
    fam_t = {}
    for f in ("gate_proj", "down_proj", "o_proj"):
        gf = torch.cuda.CUDAGraph()
        aq.aq_linear(layers[0][f], xs[FAMS[f][1]], y=ys[f], workspace=ws)
        with torch.cuda.graph(gf):
            for ths in layers:
                aq.aq_linear(ths[f], xs[FAMS[f][1]], y=ys[f], workspace=ws)
        tt = time_graph(gf, max(3, args.steps)) / nl
        fl = linear_flops(*FAMS[f], r, M)
        fam_t[f] = {"TFLOP_s": round(fl / (tt * 1e-3) / 1e12, 1), "us": round(tt * 1e3, 2)}
        del gf
    pre["gemma3_1b_M8192_r64"]["per_family"] = fam_t
    del layers, xs, ys, ws
    torch.cuda.empty_cache()

    # ---- 31B-class projection at M = 8192 (r = 128) ----
    out, inp = synth.CLASS31B_SHAPES["wide"]
    th = synth.make_theta(("bench-31b",), out, inp, 128)
    T = Theta(W0=dev_bits(th.W0, device)[:, :inp], s=dev_bits(th.s, device), U=dev_bits(th.U, device)[:, :128],
              V=dev_bits(th.V, device)[:, :128])
    x = dev_bits(synth.make_x(("bench-31b",), 8192, inp), device)[:, :inp]
    y = torch.empty(8192, out, dtype=torch.bfloat16, device=device)
    ws = torch.zeros(max(aq.aq_linear_workspace_bytes(T, m) for m in (1, 32, 8192)), dtype=torch.uint8,
                     device=device)
    aq.aq_linear(T, x, y=y, workspace=ws)
    torch.cuda.synchronize()
    g31 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g31):
        aq.aq_linear(T, x, y=y, workspace=ws)
    t = time_graph(g31, max(3, args.steps))
    fl = linear_flops(out, inp, 128, 8192)
    tf = fl / (t * 1e-3) / 1e12
    pre["31b_21504x5376_M8192_r128"] = {"TFLOP_s": round(tf, 1), "frac_bf16_peak": round(tf / pk["bf16_tflops"], 4),
                                        "ms": round(t, 4)}
    # decode on the same projection (M = 1 and 32): one 231 MB W0 read per call. Steady
    # state of consecutive layers: a graph of CHAIN calls back to back, each on its own
    # physical copy of W0 (so every call streams from HBM); `us_isolated` is one call per
    # graph replay, launch latency included.
    CHAIN = 4
    Ts = [T] + [Theta(W0=T.W0.clone(), s=T.s, U=T.U, V=T.V) for _ in range(CHAIN - 1)]
    for Md in (1, 32):
        xd = x[:Md]
        yd = y[:Md]
        aq.aq_linear(T, xd, y=yd, workspace=ws)
        gd = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gd):
            aq.aq_linear(T, xd, y=yd, workspace=ws)
        t_iso = time_graph(gd, max(5, args.steps))
        del gd
        gc = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gc):
            for Tc in Ts:
                aq.aq_linear(Tc, xd, y=yd, workspace=ws)
        td = time_graph(gc, max(5, args.steps)) / CHAIN
        gb = linear_bytes(out, inp, 128, Md) / (td * 1e-3) / 1e9
        result.setdefault("decode_31b", {})[f"M{Md}"] = {
            "GB_s": round(gb, 1), "frac_hbm": round(gb / pk["hbm_gbs"], 4), "us": round(td * 1e3, 2),
            "us_isolated": round(t_iso * 1e3, 2),
            "how": f"per call in a graph of {CHAIN} back-to-back calls, each on its own W0 copy (L2-cold)"}
        del gc
    del Ts
    result["prefill"] = pre
    del g31, T, x, y, ws
    torch.cuda.empty_cache()

    # ---- precompute: 60-layer 31B-class stack, G = 4, r = 128 ----
    if args.skip_precompute:
        return
    nb, L, r = 4, synth.CLASS31B_LAYERS, 128
    shapes = synth.CLASS31B_SHAPES
    w0h = {k: synth.make_w0(("bench-pre", k), o, i) for k, (o, i) in shapes.items()}
    w0d = {k: [dev_bits(w0h[k], device)[:, :shapes[k][1]] for _ in range(nb)] for k in shapes}
    thetas = []
    for layer in range(L):
        b = layer * nb // L
        for k, (o, i) in shapes.items():
            th = synth.make_theta(("bench-pre", k, layer), o, i, r, W0=w0h[k])
            thetas.append((k, Theta(W0=w0d[k][b], s=dev_bits(th.s, device), U=dev_bits(th.U, device)[:, :r],
                                    V=dev_bits(th.V, device)[:, :r])))
    outs = {k: [torch.empty(o, i, dtype=torch.bfloat16, device=device) for _ in range(2)] for k, (o, i) in shapes.items()}
    Bp = sum(precompute_bytes(*shapes[k], r) for k, _ in thetas)
    for j, (k, T) in enumerate(thetas[:2]):
        aq.aq_precompute(T, W_eff=outs[k][j % 2])
    torch.cuda.synchronize()
    gpc = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gpc):
        for j, (k, T) in enumerate(thetas):
            aq.aq_precompute(T, W_eff=outs[k][(j // 2) % 2])
    t = time_graph(gpc, max(2, args.steps // 2))
    gb = Bp / (t * 1e-3) / 1e9
    result["precompute"] = {"workload": "W_eff for 60 layers x (21504x5376 + 5376x5376), r=128, G=4",
                            "GB_s": round(gb, 1), "frac_hbm": round(gb / pk["hbm_gbs"], 4), "ms": round(t, 3),
                            "algorithmic_bytes": Bp}
    # single largest call as the precompute roofline point
    gq = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gq):
        aq.aq_precompute(thetas[0][1], W_eff=outs["wide"][0])
    tq = time_graph(gq, 10)
    gbq = precompute_bytes(*shapes["wide"], r) / (tq * 1e-3) / 1e9
    result["precompute"]["wide_single"] = {"GB_s": round(gbq, 1), "us": round(tq * 1e3, 1),
                                           "frac_hbm": round(gbq / pk["hbm_gbs"], 4)}
    del gpc, gq, outs
    torch.cuda.empty_cache()

    # ---- the same stack quantized to NVFP4 in the precompute epilogue (128x4 scales) ----
    qs = {k: [(torch.empty(o, i // 2, dtype=torch.uint8, device=device),
               torch.empty(aq.binding.nvfp4_scale_bytes(o, i, aq.AQ_SF_128X4), dtype=torch.uint8, device=device))
              for _ in range(2)] for k, (o, i) in shapes.items()}
    gsc = torch.ones(len(thetas), dtype=torch.float32, device=device)
    wsn = torch.empty(aq.binding.load().aq_precompute_nvfp4_workspace_bytes(), dtype=torch.uint8, device=device)

    def nvfp4_call(j, k, T, given):
        qq, ss = qs[k][(j // 2) % 2]
        aq.aq_precompute_nvfp4(T, sf_layout=aq.AQ_SF_128X4, global_scale=gsc[j:j + 1], scale_given=given,
                               q=qq, sf=ss, workspace=wsn)

    Bn = sum(nvfp4_bytes(*shapes[k], r) for k, _ in thetas)
    nv = {"workload": "NVFP4 W_eff (E2M1 codes, E4M3 scales in the 128x4 layout) for the same 60 layers",
          "algorithmic_bytes": Bn,
          "bytes_rule": "W0, U, V, s read once; codes (1/2 B per weight), scales (1/16 B) and g written"}
    for given in (False, True):
        for j, (k, T) in enumerate(thetas[:2]):
            nvfp4_call(j, k, T, given)
        torch.cuda.synchronize()
        gn = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gn):
            for j, (k, T) in enumerate(thetas):
                nvfp4_call(j, k, T, given)
        tn = time_graph(gn, max(2, args.steps // 2))
        gbn = Bn / (tn * 1e-3) / 1e9
        g1 = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g1):
            nvfp4_call(0, thetas[0][0], thetas[0][1], given)
        t1 = time_graph(g1, 10)
        gb1 = nvfp4_bytes(*shapes["wide"], r) / (t1 * 1e-3) / 1e9
        nv["given_scale" if given else "scale_from_amax"] = {
            "GB_s": round(gbn, 1), "frac_hbm": round(gbn / pk["hbm_gbs"], 4), "ms": round(tn, 3),
            "launches_per_layer_matrix": 1 if given else 2,
            "wide_single": {"GB_s": round(gb1, 1), "us": round(t1 * 1e3, 1), "frac_hbm": round(gb1 / pk["hbm_gbs"], 4)}}
        del gn, g1
    result["precompute_nvfp4"] = nv
    del thetas, w0d, qs
    torch.cuda.empty_cache()


# ----------------------------------------------------------------------------------
# CPU oracle timing (the oracle as it stands, on the host cores)
# ----------------------------------------------------------------------------------
def cpu_baseline(args, budget_s=15.0, steps=1):
    """Times oracle.linear / linear_qkv over a bounded sample of the decode step: whole
    layers (all 7 families at M = 1, 4, 16) until about budget_s seconds have passed.
    Returns GB/s of algorithmic bytes processed by the sample."""
    import oracle
    w0 = {f: synth.bf16_bits_to_f64(synth.make_w0(("bench", "W0", f), o, i))[:, :i] for f, (o, i) in FAMS.items()}
    done_bytes, spent, layers_done = 0, 0.0, 0
    layer = 0
    while spent < budget_s and layer < LAYERS * steps:
        l = layer % LAYERS
        th = {}
        for f, (o, i) in FAMS.items():
            t = synth.make_theta(("bench", f, l), o, i, DECODE_RANK, W0=np.zeros((1, 1), dtype=np.uint16))
            th[f] = (w0[f], synth.bf16_bits_to_f64(t.s), synth.bf16_bits_to_f64(t.U)[:, :DECODE_RANK],
                     synth.bf16_bits_to_f64(t.V)[:, :DECODE_RANK])
        xs = {M: {i: synth.bf16_bits_to_f64(synth.make_x(("bench-cpu", l, M, i), M, i))[:, :i]
                  for i in (1152, 1024, 6912)} for M in DECODE_MS}
        t0 = time.perf_counter()
        for M in DECODE_MS:
            oracle.linear_qkv([th["q_proj"], th["k_proj"], th["v_proj"]], xs[M][1152])
            for f in ("o_proj", "gate_proj", "up_proj", "down_proj"):
                oracle.linear(*th[f], xs[M][FAMS[f][1]])
        spent += time.perf_counter() - t0
        for M in DECODE_MS:
            done_bytes += sum(call_bytes(k, M) for k in ("qkv", "o_proj", "gate_up", "down_proj"))
        layers_done += 1
        layer += 1
    return {"value": round(done_bytes / spent / 1e9, 3), "unit": "GB/s", "cores": int(os.environ["OPENBLAS_NUM_THREADS"]),
            "kind": "oracle", "sample": f"{layers_done} of 26 layers of the decode step (7 families x M=1,4,16), "
                                        f"fp64 numpy, {spent:.2f} s",
            "seconds": round(spent, 3)}


def run_case(args, dist: Dist):
    """One aq_* call repeated: W eager warm-up calls, then K timed calls back to back on
    one stream (the single-kernel workload that kernel-profiler captures use).

    ``linear:out,in,r,M`` times aq_linear on a seeded theta bundle and x [M, in];
    ``gateup:out,in,r,M`` times aq_linear_multi over two such bundles sharing x (the batched
    gate and up projections); ``precompute:out,in,r`` times aq_precompute. Prints one JSON line with the average
    microseconds per call and its algorithmic bytes or flops."""
    import torch
    import rank_weight_reconstruction_gb300 as aq
    from rank_weight_reconstruction_gb300 import build_lib, synth

    if dist.rank != 0:
        return None
    kind, _, dims = args.case.partition(":")
    vals = [int(v) for v in dims.split(",")]
    device = torch.device("cuda", dist.local_rank)
    torch.cuda.set_device(device)
    build_lib.build()
    aq.load()
    aq.aq_set_path({"auto": aq.AQ_PATH_AUTO, "decode": aq.AQ_PATH_DECODE, "midm": aq.AQ_PATH_MIDM,
                    "prefill": aq.AQ_PATH_PREFILL}[args.path])
    out, inp, r = vals[:3] if kind != "qkv" else (vals[0], vals[2], vals[3])
    th = synth.make_theta(("case", out, inp, r), out, inp, r)
    theta = aq.Theta(W0=dev_bits(th.W0, device)[:, :inp], s=dev_bits(th.s, device),
                     U=dev_bits(th.U, device)[:, :r] if r else None, V=dev_bits(th.V, device)[:, :r] if r else None)
    if kind == "linear":
        M = vals[3]
        x = dev_bits(synth.make_x(("case", M), M, inp), device)[:, :inp]
        y = torch.empty(M, (out + 7) // 8 * 8, dtype=torch.bfloat16, device=device)[:, :out]
        ws = aq.new_workspace(aq.aq_linear_workspace_bytes(theta, M), device)
        run = lambda: aq.aq_linear(theta, x, y=y, workspace=ws)
        work = {"bytes": linear_bytes(out, inp, r, M), "flops": linear_flops(out, inp, r, M)}
    elif kind == "gateup":
        M = vals[3]
        th2 = synth.make_theta(("case", "up", out, inp, r), out, inp, r)
        theta2 = aq.Theta(W0=dev_bits(th2.W0, device)[:, :inp], s=dev_bits(th2.s, device),
                          U=dev_bits(th2.U, device)[:, :r] if r else None,
                          V=dev_bits(th2.V, device)[:, :r] if r else None)
        x = dev_bits(synth.make_x(("case", M), M, inp), device)[:, :inp]
        ys = [torch.empty(M, (out + 7) // 8 * 8, dtype=torch.bfloat16, device=device)[:, :out] for _ in range(2)]
        ws = aq.new_workspace(aq.aq_linear_workspace_bytes([theta, theta2], M), device)
        run = lambda: aq.aq_linear_multi([theta, theta2], x, ys=ys, workspace=ws)
        work = {"bytes": 2 * linear_bytes(out, inp, r, M) - 2 * M * inp,
                "flops": 2 * linear_flops(out, inp, r, M)}
    elif kind == "qkv":
        # q/k/v of one layer over one x: qkv:out_q,out_kv,in,r,M (the k and v families have out_kv rows)
        out_q, out_kv, inp, r, M = vals
        ths = [synth.make_theta(("case", "qkv", j, o, inp, r), o, inp, r) for j, o in enumerate((out_q, out_kv, out_kv))]
        thetas = [aq.Theta(W0=dev_bits(t.W0, device)[:, :inp], s=dev_bits(t.s, device),
                           U=dev_bits(t.U, device)[:, :r] if r else None, V=dev_bits(t.V, device)[:, :r] if r else None)
                  for t in ths]
        x = dev_bits(synth.make_x(("case", M), M, inp), device)[:, :inp]
        Y = torch.empty(M, out_q + 2 * out_kv, dtype=torch.bfloat16, device=device)
        ys = [Y[:, :out_q], Y[:, out_q:out_q + out_kv], Y[:, out_q + out_kv:]]
        ws = aq.new_workspace(aq.aq_linear_workspace_bytes(thetas, M), device)
        run = lambda: aq.aq_linear_qkv(thetas, x, ys=ys, workspace=ws)
        work = {"bytes": qkv_bytes([(out_q, inp), (out_kv, inp), (out_kv, inp)], r, M),
                "flops": sum(linear_flops(o, inp, r, M) for o in (out_q, out_kv, out_kv))}
        vals = [out_q, inp, r, M]
    elif kind == "precompute":
        W = torch.empty(out, (inp + 7) // 8 * 8, dtype=torch.bfloat16, device=device)[:, :inp]
        run = lambda: aq.aq_precompute(theta, W_eff=W)
        work = {"bytes": precompute_bytes(out, inp, r)}
    elif kind == "nvfp4":
        # nvfp4:out,in,r[,given]: NVFP4 precompute, 128x4 scales; given=1 takes g as input
        given = len(vals) > 3 and vals[3] != 0
        qq = torch.empty(out, inp // 2, dtype=torch.uint8, device=device)
        ss = torch.empty(aq.binding.nvfp4_scale_bytes(out, inp, aq.AQ_SF_128X4), dtype=torch.uint8, device=device)
        gg = torch.full((1,), 1e-4, dtype=torch.float32, device=device)
        wsn = torch.empty(aq.binding.load().aq_precompute_nvfp4_workspace_bytes(), dtype=torch.uint8, device=device)
        run = lambda: aq.aq_precompute_nvfp4(theta, sf_layout=aq.AQ_SF_128X4, global_scale=gg, scale_given=given,
                                             q=qq, sf=ss, workspace=wsn)
        work = {"bytes": nvfp4_bytes(out, inp, r)}
        kind = "precompute"
    else:
        raise SystemExit(f"unknown --case kind {kind!r} (linear:out,in,r,M, gateup:out,in,r,M, "
                         "qkv:out_q,out_kv,in,r,M, precompute:out,in,r or nvfp4:out,in,r[,given])")
    for _ in range(args.warmup):
        run()
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    for _ in range(args.steps):
        run()
    e.record()
    torch.cuda.synchronize()
    us = s.elapsed_time(e) * 1e3 / max(1, args.steps)
    res = {"case": args.case, "us_per_call": round(us, 3), "steps": args.steps, "warmup": args.warmup,
           "status": aq.aq_device_status(), **work}
    res["GB_s" if kind == "precompute" or vals[3] <= 32 else "TFLOP_s"] = round(
        (work["bytes"] / us * 1e-3) if (kind == "precompute" or vals[3] <= 32) else (work["flops"] / us * 1e-6), 1)
    return res


SWEEP_SHAPES = {"gate-like": (6912, 1152), "down-like": (1152, 6912)}
SWEEP_RANKS = (0, 4, 16, 64, 256)
SWEEP_MS = (1, 8, 64, 512, 4096)
SWEEP_COPIES = 16   # W0 copies per point: 255 MB, about twice the L2


def run_sweep(args, dist: Dist):
    """The rank/shape sweep on gate-like and down-like projections (50 points): per point
    the average time of one aq_linear call in a graph of SWEEP_COPIES back-to-back calls,
    each on its own copy of W0 (L2-cold), the path the dispatcher took, and the fraction of
    the roofline time T* = max(B / HBM, F / bf16 peak) on the measured peaks."""
    import torch
    import rank_weight_reconstruction_gb300 as aq
    from rank_weight_reconstruction_gb300 import Theta, build_lib

    if dist.rank != 0:
        return None
    device = torch.device("cuda", dist.local_rank)
    torch.cuda.set_device(device)
    build_lib.build()
    aq.load()
    pk = peaks()
    names = {aq.AQ_PATH_DECODE: "decode", aq.AQ_PATH_MIDM: "midm", aq.AQ_PATH_PREFILL: "prefill"}
    forced = {"auto": aq.AQ_PATH_AUTO, "decode": aq.AQ_PATH_DECODE, "midm": aq.AQ_PATH_MIDM,
              "prefill": aq.AQ_PATH_PREFILL}[args.path]
    aq.aq_set_path(forced)
    points = []
    for sname, (out, inp) in SWEEP_SHAPES.items():
        xs = {M: dev_bits(synth.make_x(("sweep", M, inp), M, inp), device)[:, :inp] for M in SWEEP_MS}
        for r in SWEEP_RANKS:
            th = synth.make_theta(("sweep", out, inp, r), out, inp, r)
            w0 = dev_bits(th.W0, device)
            s_ = dev_bits(th.s, device)
            U, V = (dev_bits(th.U, device), dev_bits(th.V, device)) if r else (None, None)
            thetas = [Theta(W0=(w0 if c == 0 else w0.clone())[:, :inp], s=s_, U=U[:, :r] if r else None,
                            V=V[:, :r] if r else None) for c in range(SWEEP_COPIES)]
            for M in SWEEP_MS:
                if forced == aq.AQ_PATH_DECODE and M > aq.aq_decode_max_m():
                    continue
                x = xs[M]
                y = torch.empty(M, out, dtype=torch.bfloat16, device=device)
                ws = aq.new_workspace(aq.aq_linear_workspace_bytes(thetas[0], M), device)
                for T in thetas:
                    aq.aq_linear(T, x, y=y, workspace=ws)
                path = names.get(aq.aq_last_path(), str(aq.aq_last_path()))
                torch.cuda.synchronize()
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g):
                    for T in thetas:
                        aq.aq_linear(T, x, y=y, workspace=ws)
                us = time_graph(g, max(3, min(args.steps, 20))) * 1e3 / SWEEP_COPIES
                del g
                B, F = linear_bytes(out, inp, r, M), linear_flops(out, inp, r, M)
                t_star = max(B / (pk["hbm_gbs"] * 1e9), F / (pk["bf16_tflops"] * 1e12)) * 1e6
                points.append({"shape": sname, "out": out, "in": inp, "r": r, "M": M, "path": path,
                               "us": round(us, 3), "GB_s": round(B / us * 1e-3, 1), "TFLOP_s": round(F / us * 1e-6, 1),
                               "bound": "hbm" if B / (pk["hbm_gbs"] * 1e9) >= F / (pk["bf16_tflops"] * 1e12)
                               else "tensor", "frac_roofline": round(t_star / us, 4)})
            del thetas, w0
            torch.cuda.empty_cache()
    aq.aq_set_path(aq.AQ_PATH_AUTO)
    return {"sweep": "rank/shape sweep, gate-like 6912x1152 and down-like 1152x6912", "path": args.path, "peaks": pk,
            "copies_per_point": SWEEP_COPIES, "status": aq.aq_device_status(), "points": points}


FP64_NOMINAL_TFLOPS = 1.25   # GB300 fp64 FMA rate, nominal (no measured figure exists for it)


def mlp_bytes(M, r=DECODE_RANK):
    """Algorithmic bytes of one fused MLP call over the step's gate, up and down families: the
    three weight bundles (W0, U, V, s), x and y; the gated activation is the call's own."""
    w = lambda o, i: 2 * (o * i + r * (o + i) + o)
    g, u, d = FAMS["gate_proj"], FAMS["up_proj"], FAMS["down_proj"]
    return w(*g) + w(*u) + w(*d) + 2 * M * g[1] + 2 * M * d[0]


def rsvd_flops(m, n, k, q):
    """fp64 flops of the randomized SVD's dense products: A Omega, then q rounds of A^T Q and
    A Q', then Q^T A (each 2 m n k), the CholeskyQR2 Gram products (2 x 2 m k^2 per
    orthonormalisation) and U = Q W (2 m k^2); the k x k eigen-solve is not counted."""
    return 2 * m * n * k * (2 + 2 * q) + 4 * m * k * k * (2 + 2 * q) + 2 * m * k * k


def run_extras(args, dist: Dist):
    """The fused MLP and the decomposition, measured.

    * aq_mlp (gate and up batched, the activation, down) for every layer of the Gemma-3-1B-shaped
      stack at M = 1, 4, 16: a graph of 26 calls, each layer on its own W0 copies (L2-cold).
    * The decomposition of one band of four Gemma-3-1B o_proj-shaped layers (1152 x 1024):
      band mean, then per layer the stored scale with its fp64 residual and the randomized SVD
      (r = 16, k = 24, q = 0 and 1), eager calls timed with CUDA events (the SVD synchronises
      its stream)."""
    import torch
    import rank_weight_reconstruction_gb300 as aq
    from rank_weight_reconstruction_gb300 import build_lib

    if dist.rank != 0:
        return None
    device = torch.device("cuda", dist.local_rank)
    torch.cuda.set_device(device)
    build_lib.build()
    aq.load()
    pk = peaks()
    stack = DecodeStack(device, copies=True, seed_tag="extras")
    th0 = stack.layers[0]
    ws_bytes = max(aq.aq_mlp_workspace_bytes(th0["gate_proj"], th0["up_proj"], th0["down_proj"], M) for M in DECODE_MS)
    ws = torch.zeros(max(ws_bytes, 256), dtype=torch.uint8, device=device)
    mlp = {}
    for M in DECODE_MS:
        views = [(lay, xv, yv) for (m, lay, xv), yv in zip(stack.x_views, stack.y_views) if m == M]
        call = lambda lay, xv, yv: aq.aq_mlp(stack.layers[lay]["gate_proj"], stack.layers[lay]["up_proj"],
                                             stack.layers[lay]["down_proj"], xv["mlp"], y=yv["down_proj"],
                                             workspace=ws)
        for v in views:
            call(*v)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        launches = 0
        with torch.cuda.graph(g):
            for v in views:
                call(*v)
                launches += aq.aq_last_launch_count()
        for _ in range(max(3, args.warmup)):
            g.replay()
        us = time_graph(g, max(5, min(args.steps, 50))) * 1e3 / len(views)
        del g
        B = mlp_bytes(M)
        mlp[f"M{M}"] = {"us_per_call": round(us, 3), "GB_s": round(B / us * 1e-3, 1),
                        "frac_hbm": round(B / us * 1e-3 / pk["hbm_gbs"], 4), "launches_per_call": launches // len(views),
                        "algorithmic_bytes": B}
    status_mlp = aq.aq_device_status()
    del stack
    torch.cuda.empty_cache()

    out, inp, L, r, k = 1152, 1024, 4, 16, 24
    ws_host = [synth.make_w0(("extras", "band", l), out, inp) for l in range(L)]
    weights = [dev_bits(w, device)[:, :inp] for w in ws_host]
    omega = torch.from_numpy(synth.normal_f64(synth.stream_seed("extras", "omega"), inp * k).reshape(inp, k)).to(device)
    ev = lambda: torch.cuda.Event(enable_timing=True)

    def timed(fn, reps=5):
        fn()
        torch.cuda.synchronize()
        a, b = ev(), ev()
        a.record()
        for _ in range(reps):
            fn()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) / reps

    W0 = aq.aq_band_mean(weights)
    t_band = timed(lambda: aq.aq_band_mean(weights, W0=W0))
    s_, resid = aq.aq_ls_residual(weights[0], W0)
    t_ls = timed(lambda: aq.aq_ls_residual(weights[0], W0, s=s_, resid=resid))
    t_svd = {q: timed(lambda q=q: aq.aq_randomized_svd(resid, r, omega, power_iters=q)) for q in (0, 1)}
    band_b = 2 * L * out * inp + 2 * out * inp
    ls_b = out * inp * (2 + 2 + 8) + 2 * out
    dec = {"workload": f"one band of {L} layers of {out}x{inp} (Gemma-3-1B o_proj shape), r={r}, k={k}",
           "band_mean": {"ms": round(t_band, 4), "GB_s": round(band_b / t_band * 1e-6, 1),
                         "frac_hbm": round(band_b / t_band * 1e-6 / pk["hbm_gbs"], 4)},
           "ls_residual_per_layer": {"ms": round(t_ls, 4), "GB_s": round(ls_b / t_ls * 1e-6, 1),
                                     "frac_hbm": round(ls_b / t_ls * 1e-6 / pk["hbm_gbs"], 4)},
           "randomized_svd_per_layer": {f"q{q}": {"ms": round(t, 4), "fp64_TFLOP_s": round(rsvd_flops(out, inp, k, q) / t * 1e-9, 3),
                                                  "frac_fp64_nominal": round(rsvd_flops(out, inp, k, q) / t * 1e-9 / FP64_NOMINAL_TFLOPS, 4)}
                                        for q, t in t_svd.items()},
           "band_total_ms_q1": round(t_band + L * (t_ls + t_svd[1]), 3)}
    return {"extras": "fused MLP over the decode stack and the GPU decomposition of one band", "peaks": pk,
            "fp64_peak_tflops": {"value": FP64_NOMINAL_TFLOPS, "source": "nominal"},
            "mlp": mlp, "decomposition": dec, "status": [status_mlp, aq.aq_device_status()]}


def run_reference(args, dist: Dist):
    if dist.rank != 0:
        return None
    per_step_budget = max(2.0, min(20.0, 150.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        cpu_baseline(args, budget_s=per_step_budget)
    vals = [cpu_baseline(args, budget_s=per_step_budget) for _ in range(args.steps)]
    v = statistics.median([x["value"] for x in vals])
    B = step_bytes()
    cb = dict(vals[0])
    cb["value"] = v
    return {"metric": METRIC, "impl": "reference", "value": v, "unit": "GB/s", "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(B / (v * 1e9) * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (same seeded inputs)",
            "config": decode_config(),
            "setup": {"timing": "each step: the fp64 oracle over a bounded sample of whole layers of the "
                                "step on the host cores, host wall clock",
                      "parallelism": "host cores"},
            "cpu_baseline": cb, "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--decode-only", action="store_true", help="time only the headline decode step")
    ap.add_argument("--skip-precompute", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--profile", action="store_true",
                    help="run only the captured decode step (for kernel-profiler launch lists)")
    ap.add_argument("--sweep", action="store_true",
                    help="the rank/shape sweep (gate-like and down-like, r in 0..256, M in 1..4096)")
    ap.add_argument("--extras", action="store_true",
                    help="the fused MLP over the decode stack and the GPU decomposition of one band")
    ap.add_argument("--path", choices=["auto", "decode", "midm", "prefill"], default="auto",
                    help="--sweep / --case: force one path (aq_set_path) to map where the paths cross")
    ap.add_argument("--case", default=None,
                    help="time one call instead: linear:out,in,r,M, gateup:out,in,r,M, qkv:out_q,out_kv,in,r,M "
                         "or precompute:out,in,r (profiler captures)")
    args = ap.parse_args()
    if args.warmup < 3:
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    dist = Dist()
    if args.impl == "reference":
        res = run_reference(args, dist)
    elif args.case:
        res = run_case(args, dist)
    elif args.sweep:
        res = run_sweep(args, dist)
    elif args.extras:
        res = run_extras(args, dist)
    else:
        res = run_ours(args, dist)
    if dist.rank == 0 and res is not None:
        print(json.dumps(res))
    dist.close()


if __name__ == "__main__":
    main()
