"""Benchmark of the FORGE hot path on one GB300: input gradient + fused
weight-gradient / optimizer step of one Llama-3.1-8B linear layer.

Default workload (the headline configuration): the MLP up-projection,
W 14336 x 4096 fp32 master weights with fp32 AdamW moments, BT = 512
tokens of bf16 activations X and upstream gradients dY. One step = one
forge_backward_step call: the input gradient dX = dY W_old and the fused
weight-gradient / AdamW step, in one pass over W where the layer allows it
(BT <= 768, fp32 / bf16 state), else its split path: the input gradient
(forge_dgrad_ws's kernel, given the workspace) followed by the step. The state (1.4 GB) is far larger than L2 and L2 is
also flushed between timed steps. The two-kernel split path is timed as
well and reported beside the headline (split_* keys).

Prints one JSON line (see the keys below). ``--impl reference`` times the
CPU oracle instead (a bounded row sample, extrapolated).
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "fused wgrad+AdamW µs/step, GB/s & % roofline at Llama-8B linear shapes"
UNIT = "us/step"

WORKLOADS = {
    # name: (D_out, D_in, BT, W storage, moment storage)
    "llama31_8b_up_proj_bt512_f32state": (14336, 4096, 512, "f32", "f32"),
    "llama31_8b_up_proj_bt512_bf16state_sr": (14336, 4096, 512, "bf16", "bf16"),
    "llama31_8b_up_proj_bt2048_bf16state_sr": (14336, 4096, 2048, "bf16", "bf16"),
    "llama31_8b_up_proj_bt8192_bf16state_sr": (14336, 4096, 8192, "bf16", "bf16"),
    "llama31_8b_up_proj_bt512_q8state": (14336, 4096, 512, "f32", "q8"),
}
DEFAULT = "llama31_8b_up_proj_bt512_f32state"
# Exact gradient accumulation: micro-batches of BT tokens into an fp32
# accumulator, the step fired once at the last one (name: (micro-batches, BT)).
ACCUM = {"llama31_8b_up_proj_accum4x512_f32state": (4, 512)}
# The full Llama-3.1-8B linear stack (32 layers x 7 linears, BT = 512).
STACKS = {f"llama31_8b_stack_{o}_{st}": (o, st) for o in ("adamw", "lion", "sgdm") for st in ("f32state", "bf16state")}
STACK_HYPER = {"adamw": dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01),
               "lion": dict(lr=3e-6, beta1=0.9, beta2=0.99, eps=0.0, weight_decay=1.0),
               "sgdm": dict(lr=2e-5, beta1=0.9, beta2=0.0, eps=0.0, weight_decay=1e-2)}
HYPER = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)


def state_bytes_per_param(w, st):
    wb = 4 if w == "f32" else 2
    mb = {"f32": 4, "bf16": 2, "q8": 1 + 4 / 128}[st]
    return 2 * wb + 2 * 2 * mb   # W read + write, m and v read + write


def algorithmic_bytes(d_out, d_in, bt, w, st):
    """State read + written once, X and dY read once (no re-reads, no G)."""
    return int(round(d_out * d_in * state_bytes_per_param(w, st))) + 2 * bt * (d_in + d_out)


def backward_algorithmic_bytes(d_out, d_in, bt, w, st):
    """The fused backward pass: the step's bytes plus the bf16 dX written once."""
    return algorithmic_bytes(d_out, d_in, bt, w, st) + 2 * bt * d_in


def fused_path(bt, st):
    """Whether forge_backward_step can take the one-pass path for this workload."""
    return 1 <= bt <= 768 and st != "q8"


def dgrad_algorithmic_bytes(d_out, d_in, bt, w):
    return d_out * d_in * (4 if w == "f32" else 2) + 2 * bt * d_out + 2 * bt * d_in


KERNEL_SOURCES = ["wgrad_tc.cuh", "wgrad_tc_dispatch.cuh", "wgrad_tc_adamw.cu", "forge_math.cuh", "forge_ptx.cuh",
                  "forge_params.h", "dx_reduce.cu"]


def kernel_source_hash() -> str:
    """Hash of the sources that define the fused kernel (ties an ncu capture to this code)."""
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "backward_gemm_optimizer_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def load_traffic(workload: str):
    """DRAM bytes per launch of the fused kernel from the committed ncu capture, if it
    was taken on the current kernel sources (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None, None
    with open(p) as f:
        d = json.load(f).get(workload)
    if not d or d.get("kernel_source_hash") != kernel_source_hash():
        return None, None
    return d.get("dram_bytes_per_launch"), d.get("units_scale", 1.0)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d.get("hbm_gbs", 6800.0), d.get("bf16_tflops", 1900.0), "measured"
    return 6800.0, 1900.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 100 ms in the background."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.f = None

    def start(self):
        try:
            self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.flush()
        self.f.seek(0)
        rows = [r.split(",") for r in self.f.read().strip().splitlines() if r.strip()]
        os.unlink(self.f.name)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1])); mx.append(float(r[2]))
            except ValueError:
                continue
            for n, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------- the other configurations


CONFIG_LAYERS = {
    # name: (D_out, D_in, BT, W storage, moment storage, zero-gradient row share)
    "up_proj_bt512_bf16state_sr": (14336, 4096, 512, "bf16", "bf16", 0.0),
    "up_proj_bt2048_bf16state_sr": (14336, 4096, 2048, "bf16", "bf16", 0.0),
    "up_proj_bt8192_bf16state_sr": (14336, 4096, 8192, "bf16", "bf16", 0.0),
    "up_proj_bt512_q8state_zero30": (14336, 4096, 512, "f32", "q8", 0.3),
}


def device_layer(d_out, d_in, bt, w, st, dev, seed, zero_frac=0.0):
    """One layer's backward-pass inputs and state, drawn on the device (the
    distributions of the host generator: X, dY ~ N(0, 1), W ~ N(0, 0.02),
    m ~ N(0, 1e-3), v = |N(0, 1e-6)|; 8-bit state as codes with one scale per
    block; zero rows get zero dY columns and zero state)."""
    import torch
    from backward_gemm_optimizer_gb300 import synthetic as S
    f = lambda shape, dt, std, sid, absolute=False: S.device_normal_(  # noqa: E731
        torch.empty(shape, dtype=dt, device=dev), std, seed, sid, absolute)
    wdt = torch.float32 if w == "f32" else torch.bfloat16
    s = {"X": f((bt, d_in), torch.bfloat16, 1.0, S.STREAM_X), "dY": f((bt, d_out), torch.bfloat16, 1.0, S.STREAM_DY),
         "W": f((d_out, d_in), wdt, 0.02, S.STREAM_W),
         "dX": torch.empty((bt, d_in), dtype=torch.bfloat16, device=dev)}
    if st == "q8":
        g = torch.Generator(device=dev)
        g.manual_seed(seed * 1000003 + S.STREAM_M_CODES)
        s["m"] = torch.randn((d_out, d_in), device=dev, generator=g).mul_(42.0).round_().clamp_(-127, 127).to(torch.int8)
        s["v"] = torch.randint(1, 256, (d_out, d_in), device=dev, generator=g, dtype=torch.int32).to(torch.uint8)
        s["m_scale"] = torch.full((d_in // 128, d_out), 3e-3 / 127.0, dtype=torch.float32, device=dev)
        s["v_scale"] = torch.full((d_in // 128, d_out), 2e-3 / 255.0, dtype=torch.float32, device=dev)
    else:
        mdt = torch.float32 if st == "f32" else torch.bfloat16
        s["m"] = f((d_out, d_in), mdt, 1e-3, S.STREAM_M)
        s["v"] = f((d_out, d_in), mdt, 1e-6, S.STREAM_V, True)
    if zero_frac > 0.0:
        zr = torch.from_numpy(S.zero_row_mask(d_out, zero_frac, seed)).to(dev)
        s["dY"][:, zr] = 0
        s["m"][zr] = 0
        s["v"][zr] = 0
        if st == "q8":
            s["m_scale"][:, zr] = 0
            s["v_scale"][:, zr] = 0
    return s


def measure_configs(F, dev, K, warm, hbm, tflops):
    """Time the other configurations the benchmark is quoted on, each as one
    backward pass per step through the public API (library path policy, L2
    flushed between steps), and the 224-linear stack per rule and state as a
    replayed CUDA graph. Returns a compact record per configuration."""
    import torch
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    out = {}
    for name, (d_out, d_in, bt, w, st, zf) in CONFIG_LAYERS.items():
        s = device_layer(d_out, d_in, bt, w, st, dev, seed=5, zero_frac=zf)
        ws = torch.empty(max(16, F.workspace_bytes(d_out, d_in, bt)), dtype=torch.uint8, device=dev)
        t = 1
        for _ in range(warm):
            one_step(F, s, w, st, t, stream, ws, 0); t += 1
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
        for i in range(K):
            flush.fill_(float(i))
            ev[i][0].record(stream)
            one_step(F, s, w, st, t, stream, ws, 0); t += 1
            ev[i][1].record(stream)
        torch.cuda.synchronize(dev)
        F.sync_status(stream)
        us = statistics.mean(e0.elapsed_time(e1) for e0, e1 in ev) * 1000.0
        ab = backward_algorithmic_bytes(d_out, d_in, bt, w, st)
        flops = 2.0 * 2.0 * bt * d_out * d_in          # weight gradient + input gradient
        t_roof = max(ab / (hbm * 1e9), flops / (tflops * 1e12)) * 1e6
        out[name] = {"us": round(us, 2), "GBps": round(ab / (us * 1e-6) / 1e9, 1),
                     "TFLOPs": round(flops / (us * 1e-6) / 1e12, 1),
                     "bound": "hbm" if ab / (hbm * 1e9) >= flops / (tflops * 1e12) else "tensor",
                     "frac": round(t_roof / us, 4), "algorithmic_bytes": ab,
                     "path": ("fused input gradient" if fused_path(bt, st) else
                              "split path: dgrad + fused step" +
                              (" (256 x 256 step tiles on CTA pairs)" if bt >= 2048 else ""))}
        del s, ws
    for opt in ("adamw", "lion", "sgdm"):
        for stname in ("f32state", "bf16state"):
            st = build_stack(opt, stname, dev, seed=7)
            layers, order = st["layers"], st["order"]

            def stack_step(t, stream_):
                for layer in reversed(range(len(layers))):
                    for lname, _, _ in order:
                        stack_backward(F, st, layers[layer][lname], t, stream_)

            for t in range(1, warm + 1):
                stack_step(t, stream)
            torch.cuda.synchronize(dev)
            g = torch.cuda.CUDAGraph()
            side = torch.cuda.Stream(dev)
            side.wait_stream(stream)
            with torch.cuda.graph(g, stream=side):
                stack_step(warm + 1, torch.cuda.current_stream(dev))
            g.replay(); torch.cuda.synchronize(dev)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            ks = max(2, min(K, 5))
            e0.record(stream)
            for _ in range(ks):
                g.replay()
            e1.record(stream)
            torch.cuda.synchronize(dev)
            F.sync_status(stream)
            ms = e0.elapsed_time(e1) / ks
            ab = stack_algorithmic_bytes(st)
            out[f"stack_{opt}_{stname}"] = {"ms": round(ms, 3), "GBps": round(ab / (ms * 1e-3) / 1e9, 1),
                                            "bound": "hbm", "frac": round(ab / (ms * 1e-3) / 1e9 / hbm, 4),
                                            "algorithmic_bytes": ab, "timed": f"CUDA graph, {ks} replays"}
            del g, st, layers
            torch.cuda.synchronize(dev)
            torch.cuda.empty_cache()
    return out


# --------------------------------------------------------------------------- CPU oracle arm


def cpu_oracle_step_us(d_out, d_in, bt, w, st, rows):
    """Time the CPU oracle (dgrad + step) on a row sample of W, extrapolated."""
    from backward_gemm_optimizer_gb300 import synthetic as S
    import oracle.forge_oracle as O

    prob = S.linear_problem(rows, d_in, bt, seed=0, x_dtype="bf16", w_dtype=w, state=st)
    Xn = prob.X.float().numpy(); dYn = prob.dY.float().numpy()
    def tonp(t):
        if t is None:
            return None
        import torch
        return t.view(torch.int16).numpy().view(np.uint16) if t.dtype == torch.bfloat16 else t.numpy()
    state = O.State(W=tonp(prob.W), m=tonp(prob.m), v=tonp(prob.v), m_scale=tonp(prob.m_scale),
                    v_scale=tonp(prob.v_scale), w_dtype=w, state=st)
    h = O.Hyper(**HYPER)
    t0 = time.perf_counter()
    O.dgrad_f64(dYn, O.load_w(state))            # this row block's share of dX
    O.step("adamw", Xn, dYn, state, h, 1, seed=1234, sr_w=(w == "bf16"))
    dt = time.perf_counter() - t0
    return dt * 1e6 * (d_out / rows), dt


def run_reference(args, rank, world):
    if rank != 0:
        return
    d_out, d_in, bt, w, st = WORKLOADS[args.workload]
    rows = args.cpu_rows
    vals = []
    t_start = time.perf_counter()
    for i in range(args.warmup + args.steps):
        us, _ = cpu_oracle_step_us(d_out, d_in, bt, w, st, rows)
        if i >= args.warmup:
            vals.append(us)
        if time.perf_counter() - t_start > args.cpu_budget_s:
            break
    v = statistics.median(vals) if vals else us
    cores = os.cpu_count()
    line = {
        "impl": "reference", "metric": METRIC, "value": round(v, 1), "unit": UNIT, "n_gpus": world,
        "steps": len(vals), "warmup": args.warmup, "ms_per_step": round(v / 1000, 3), "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": layer_config(args.workload, world),
        "cpu_baseline": {"value": round(v, 1), "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"rows 0..{rows} of W ({rows}/{d_out} of the layer), dgrad share + step, "
                                   f"float64 numpy, extrapolated x{d_out / rows:.2f}"},
        "e2e": {"value": round(v, 1), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------- ranks (replicas)


def layer_config(workload: str, world: int) -> dict:
    """The ``config`` of a single-layer workload's line (both arms print the same)."""
    d_out, d_in, bt, w, st = WORKLOADS[workload]
    return {"workload": workload, "d_out": d_out, "d_in": d_in, "bt": bt, "w_storage": w,
            "moment_storage": st, "optimizer": "adamw",
            "step": "forge_backward_step, fused input gradient (one pass over W)" if fused_path(bt, st) else
                    "forge_backward_step, split path (dgrad with workspace, then the fused step)",
            "l2": "flushed between steps (256 MB write) and state 1.4 GB > L2",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}


def replica_seed(rank: int) -> int:
    """Each rank steps its own, independently drawn layer (replicas; no data-path collective)."""
    return rank


def barrier(world: int):
    if world > 1:
        import torch
        torch.distributed.barrier()


def max_over_ranks(value: float, world: int, device=None) -> float:
    """The job's time is the slowest rank's (max over ranks)."""
    if world <= 1:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


# --------------------------------------------------------------------------- GPU arm


def make_state(d_out, d_in, bt, w, st, dev, seed=0):
    import torch
    from backward_gemm_optimizer_gb300 import synthetic as S
    prob = S.linear_problem(d_out, d_in, bt, seed=seed, x_dtype="bf16", w_dtype=w, state=st)
    out = {k: t.to(dev) for k, t in prob.tensors().items()}
    out["dX"] = torch.empty((bt, d_in), dtype=torch.bfloat16, device=dev)
    host = {"X": prob.X.pin_memory(), "dY": prob.dY.pin_memory(),
            "dX": torch.empty((bt, d_in), dtype=torch.bfloat16).pin_memory()}
    return out, host


def one_step(F, s, w, st, t, stream, ws, flags):
    """One backward pass of the layer through the public API (8-bit state:
    the descriptors carry their block scales)."""
    F.backward_step("adamw", s["X"], s["dY"], s["W"], s["m"], s["v"], s["dX"], step=t, seed=1234,
                    sr_w=(w == "bf16"), workspace=ws, flags=flags, stream=stream, m_scale=s.get("m_scale"),
                    v_scale=s.get("v_scale"), **HYPER)


def split_step(F, s, w, t, stream, ws, events=None):
    if events is not None:
        events[0].record(stream)
    F.dgrad(s["dY"], s["W"], s["dX"], workspace=ws, stream=stream)   # the split path's input gradient
    if events is not None:
        events[1].record(stream)
    F.wgrad_step_adamw(s["X"], s["dY"], s["W"], s["m"], s["v"], m_scale=s.get("m_scale"),
                       v_scale=s.get("v_scale"), step=t, seed=1234, sr_w=(w == "bf16"), stream=stream, **HYPER)
    if events is not None:
        events[2].record(stream)


def run_gpu(args, rank, world, local_rank):
    import torch
    import backward_gemm_optimizer_gb300 as F

    dev = torch.device(f"cuda:{local_rank}")
    torch.cuda.set_device(dev)
    d_out, d_in, bt, w, st = WORKLOADS[args.workload]
    s, host = make_state(d_out, d_in, bt, w, st, dev, seed=replica_seed(rank))
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)   # 256 MB > L2

    fused = fused_path(bt, st)
    flags = F.FLAG_BACKWARD_FUSED if fused else F.FLAG_BACKWARD_SPLIT
    # the fused pass's dX slabs, or on the split path the balanced dgrad's partial sums
    ws = torch.empty(max(16, F.workspace_bytes(d_out, d_in, bt)), dtype=torch.uint8, device=dev)
    t = 1
    for _ in range(args.warmup):
        one_step(F, s, w, st, t, stream, ws, flags); t += 1
    F.sync_status(stream)

    # ---- the headline: one backward pass per step, inputs resident in HBM
    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    sampler = ClockSampler(local_rank)
    barrier(world)
    torch.cuda.synchronize(dev)
    sampler.start()
    time.sleep(0.3)
    wall0 = time.perf_counter()
    for i in range(K):
        flush.fill_(float(i))                      # evict L2 between steps (not timed)
        ev[i][0].record(stream)
        one_step(F, s, w, st, t, stream, ws, flags)
        ev[i][1].record(stream)
        t += 1
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - wall0
    barrier(world)
    clocks = sampler.stop()
    F.sync_status(stream)
    step_ms = [ev[i][0].elapsed_time(ev[i][1]) for i in range(K)]
    total_ms = max_over_ranks(sum(step_ms), world, dev)

    # ---- the split path (forge_dgrad_ws, then the fused step), for comparison
    KS = max(1, min(K, args.split_steps))
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(KS)]
    for _ in range(3):
        split_step(F, s, w, t, stream, ws); t += 1
    for i in range(KS):
        flush.fill_(float(i))
        split_step(F, s, w, t, stream, ws, evs[i]); t += 1
    torch.cuda.synchronize(dev)
    F.sync_status(stream)
    split_ms = [evs[i][0].elapsed_time(evs[i][2]) for i in range(KS)]
    dgrad_ms = [evs[i][0].elapsed_time(evs[i][1]) for i in range(KS)]
    wstep_ms = [evs[i][1].elapsed_time(evs[i][2]) for i in range(KS)]

    # ---- end to end through the public API, host buffers, copies timed.
    # Serial: upload, step, download and a status read, one after another.
    KE = max(1, min(args.e2e_steps, K))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize(dev)
    e0.record(stream)
    for i in range(KE):
        s["X"].copy_(host["X"], non_blocking=True)
        s["dY"].copy_(host["dY"], non_blocking=True)
        one_step(F, s, w, st, t, stream, ws, flags); t += 1
        host["dX"].copy_(s["dX"], non_blocking=True)
        F.sync_status(stream)                       # reads the status word back each step
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_serial_ms = e0.elapsed_time(e1) / KE
    # Pipelined: step i+1's inputs upload on one stream and step i-1's dX
    # downloads on another while step i runs (double-buffered device buffers;
    # every copy is still inside the timed region). The status word is read
    # once after the loop (it keeps the first failure).
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    bufs = [dict(s), dict(s, X=torch.empty_like(s["X"]), dY=torch.empty_like(s["dY"]), dX=torch.empty_like(s["dX"]))]
    host_dx = [host["dX"], torch.empty_like(host["dX"]).pin_memory()]
    ev = lambda: torch.cuda.Event()  # noqa: E731
    inp, comp, dl = [ev() for _ in range(KE)], [ev() for _ in range(KE)], [ev() for _ in range(KE)]
    barrier(world)
    torch.cuda.synchronize(dev)
    e0.record(stream)
    up.wait_event(e0)
    for i in range(KE):
        b = bufs[i % 2]
        with torch.cuda.stream(up):
            if i >= 2:
                up.wait_event(comp[i - 2])             # buffers of step i-2 no longer read
            b["X"].copy_(host["X"], non_blocking=True)
            b["dY"].copy_(host["dY"], non_blocking=True)
            inp[i].record(up)
        stream.wait_event(inp[i])
        if i >= 2:
            stream.wait_event(dl[i - 2])               # dX of step i-2 downloaded
        one_step(F, b, w, st, t, stream, ws, flags); t += 1
        comp[i].record(stream)
        with torch.cuda.stream(down):
            down.wait_event(comp[i])
            host_dx[i % 2].copy_(b["dX"], non_blocking=True)
            dl[i].record(down)
    stream.wait_event(dl[KE - 1])
    e1.record(stream)
    torch.cuda.synchronize(dev)
    F.sync_status(stream)
    e2e_ms = e0.elapsed_time(e1) / KE
    h2d = host["X"].numel() * 2 + host["dY"].numel() * 2
    d2h = host["dX"].numel() * 2

    if rank != 0:
        return
    hbm, tflops, peak_src = load_peaks()
    us = total_ms * 1000.0 / K
    med_us = statistics.median(step_ms) * 1000.0
    flops = 2.0 * bt * d_out * d_in * (2 if fused else 1)
    if fused:
        abytes = backward_algorithmic_bytes(d_out, d_in, bt, w, st)
        kern_us = statistics.mean(step_ms) * 1000.0
        kernel = "wgrad_step_tc_kernel with the fused input gradient + dx_reduce_kernel (one forge_backward_step)"
    else:
        abytes = algorithmic_bytes(d_out, d_in, bt, w, st)
        kern_us = statistics.mean(wstep_ms) * 1000.0
        kernel = "wgrad_step_tc_kernel (split path: the step after forge_dgrad_ws)"
    achieved = abytes / (kern_us * 1e-6) / 1e9
    tfl = flops / (kern_us * 1e-6) / 1e12
    t_roof = max(abytes / (hbm * 1e9), flops / (tflops * 1e12)) * 1e6
    bound = "hbm" if abytes / (hbm * 1e9) >= flops / (tflops * 1e12) else "tensor"
    traffic, _ = load_traffic(args.workload)
    split_us = statistics.mean(split_ms) * 1000.0
    wstep_us = statistics.mean(wstep_ms) * 1000.0
    sbytes = algorithmic_bytes(d_out, d_in, bt, w, st)
    line = {
        "metric": METRIC, "value": round(us, 2), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(us / 1000.0, 4), "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": layer_config(args.workload, world),
        "step_median_us": round(med_us, 2),
        "roofline_us": round(t_roof, 2), "frac_of_roofline": round(t_roof / kern_us, 4),
        "GBps": round(achieved, 1), "TFLOPs": round(tfl, 1),
        "roofline": {"bound": bound, "achieved": round(achieved, 1) if bound == "hbm" else round(tfl, 1),
                     "peak": hbm if bound == "hbm" else tflops, "unit": "GB/s" if bound == "hbm" else "TFLOP/s",
                     "frac": round((achieved / hbm) if bound == "hbm" else tfl / tflops, 4),
                     "traffic": traffic, "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)"
                     if peak_src == "measured" else peak_src,
                     "algorithmic_bytes": abytes, "kernel": kernel,
                     "kernel_source_hash": kernel_source_hash()},
        "split_step_us": round(split_us, 2), "split_dgrad_us": round(statistics.mean(dgrad_ms) * 1000.0, 2),
        "split_wgrad_step_us": round(wstep_us, 2),
        "split_wgrad_step_frac_of_hbm": round(sbytes / (wstep_us * 1e-6) / 1e9 / hbm, 4),
        "e2e": {"value": round(e2e_ms * 1000.0, 2), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "how": "each step uploads X, dY from pinned host memory and downloads dX, on two copy streams "
                       "overlapping the previous / next step's compute (double-buffered)"},
        "e2e_serial": {"value": round(e2e_serial_ms * 1000.0, 2), "unit": UNIT,
                       "how": "upload, step, download, status read, one after another"},
        "gpu_launches": 2 * K,
        "clocks": clocks,
        "wall_s_timed": round(wall, 3),
    }
    if not args.no_configs and world == 1:
        del s, host, bufs, ws
        torch.cuda.empty_cache()
        cfg_t0 = time.perf_counter()
        line["configs"] = measure_configs(F, dev, max(3, min(K, 20)), 3, hbm, tflops)
        line["configs"]["wall_s"] = round(time.perf_counter() - cfg_t0, 1)
    if not args.no_cpu_baseline:
        try:
            rows = min(args.cpu_rows, d_out)
            vals, spent = [], 0.0
            while spent < args.cpu_min_s or not vals:     # repeat to ~10 s of CPU work
                v, dt = cpu_oracle_step_us(d_out, d_in, bt, w, st, rows)
                vals.append(v); spent += dt
            line["cpu_baseline"] = {"value": round(statistics.median(vals), 1), "unit": UNIT,
                                    "cores": os.cpu_count(), "kind": "oracle",
                                    "sample": f"rows 0..{rows} of W (x{d_out / rows:.2f} to the layer), dgrad share "
                                              f"+ AdamW step, float64 numpy, median of {len(vals)} runs, "
                                              f"{spent:.1f} s of CPU work"}
        except Exception as e:  # report, do not fail the GPU line
            line["cpu_baseline"] = {"value": None, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
                                    "sample": f"failed: {e}"}
    print(json.dumps(line), flush=True)


def run_accum(args, rank, world, local_rank):
    """One step = one accumulation window on the up-projection (fp32 W, m, v):
    every micro-batch but the last runs forge_backward_accumulate (dX and the
    accumulation into G_acc in one pass; the first overwrites G_acc), the last
    forge_dgrad_ws and forge_wgrad_step_accumulated. The same window with
    forge_dgrad_ws + forge_wgrad_accumulate per micro-batch is timed after it
    (split_* keys)."""
    import torch
    import backward_gemm_optimizer_gb300 as F
    from backward_gemm_optimizer_gb300 import synthetic as S

    nmb, bt = ACCUM[args.workload]
    d_out, d_in = 14336, 4096
    dev = torch.device(f"cuda:{local_rank}")
    torch.cuda.set_device(dev)
    seed = replica_seed(rank)
    W = S.device_normal_(torch.empty((d_out, d_in), dtype=torch.float32, device=dev), 0.02, seed, 1)
    m = S.device_normal_(torch.empty_like(W), 1e-3, seed, 2)
    v = S.device_normal_(torch.empty_like(W), 1e-6, seed, 3, absolute=True)
    G = torch.empty_like(W)
    mbs = [(S.device_normal_(torch.empty((bt, d_in), dtype=torch.bfloat16, device=dev), 1.0, seed, 10 + 2 * k),
            S.device_normal_(torch.empty((bt, d_out), dtype=torch.bfloat16, device=dev), 1.0, seed, 11 + 2 * k))
           for k in range(nmb)]
    dX = torch.empty((bt, d_in), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(max(16, F.workspace_bytes(d_out, d_in, bt)), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)

    def window(t, ev=None, split=False):
        for k, (X, dY) in enumerate(mbs):
            last = k == nmb - 1
            if ev is not None:
                ev[k][0].record(stream)
            if last or split:
                F.dgrad(dY, W, dX, workspace=ws, stream=stream)
            if ev is not None:
                ev[k][1].record(stream)
            if last:
                F.wgrad_step_accumulated("adamw", X, dY, G, W, m, v, step=t, stream=stream, **HYPER)
            elif split:
                F.wgrad_accumulate(X, dY, G, overwrite=(k == 0), stream=stream)
            else:
                F.backward_accumulate(X, dY, W, G, dX, overwrite=(k == 0), workspace=ws,
                                      flags=F.FLAG_BACKWARD_FUSED, stream=stream)
            if ev is not None:
                ev[k][2].record(stream)

    def timed(K, split, t):
        evs = [[[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(nmb)] for _ in range(K)]
        barrier(world)
        torch.cuda.synchronize(dev)
        for i in range(K):
            flush.fill_(float(i))
            window(t, evs[i], split); t += 1
        torch.cuda.synchronize(dev)
        return evs, t

    t = 1
    for _ in range(args.warmup):
        window(t); t += 1
        window(t, split=True); t += 1
    F.sync_status(stream)
    K = args.steps
    sampler = ClockSampler(local_rank)
    sampler.start()
    time.sleep(0.3)
    evs, t = timed(K, False, t)
    clocks = sampler.stop()
    F.sync_status(stream)
    total_ms = max_over_ranks(sum(evs[i][0][0].elapsed_time(evs[i][-1][2]) for i in range(K)), world, dev)
    KS = max(1, min(K, args.split_steps))
    sev, t = timed(KS, True, t)
    F.sync_status(stream)
    split_ms = max_over_ranks(sum(sev[i][0][0].elapsed_time(sev[i][-1][2]) for i in range(KS)), world, dev)
    if rank != 0:
        return
    hbm, _, _ = load_peaks()

    def part(e, n, k, a, b):
        return statistics.mean(e[i][k][a].elapsed_time(e[i][k][b]) for i in range(n)) * 1000.0

    params = d_out * d_in
    ops_b = 2 * bt * (d_in + d_out)
    first_b = params * 4 + params * 4 + ops_b + 2 * bt * d_in   # G_acc written, W read, dX written
    acc_b = params * 8 + params * 4 + ops_b + 2 * bt * d_in     # G_acc read + written, W read, dX written
    last_b = params * 28 + ops_b                                # W, m, v read + written, G_acc read
    mid = list(range(1, nmb - 1))
    fa_first = part(evs, K, 0, 1, 2)
    fa_mid = statistics.mean(part(evs, K, k, 1, 2) for k in mid) if mid else None
    s_first = part(sev, KS, 0, 1, 2)
    s_mid = statistics.mean(part(sev, KS, k, 1, 2) for k in mid) if mid else None
    line = {
        "metric": METRIC, "value": round(total_ms * 1000.0 / K, 1), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(total_ms / K, 3), "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": args.workload, "d_out": d_out, "d_in": d_in, "micro_batches": nmb, "bt": bt,
                   "effective_batch": nmb * bt, "optimizer": "adamw", "state": "fp32 W, m, v; fp32 G_acc",
                   "step": f"{nmb - 1} x forge_backward_accumulate (fused), 1 x forge_dgrad_ws + "
                           "forge_wgrad_step_accumulated",
                   "l2": "flushed between windows"},
        "backward_accumulate_first_us": round(fa_first, 2),
        "backward_accumulate_first_frac_of_hbm": round(first_b / (fa_first * 1e-6) / 1e9 / hbm, 4),
        "backward_accumulate_us": round(fa_mid, 2) if fa_mid is not None else None,
        "backward_accumulate_frac_of_hbm": round(acc_b / (fa_mid * 1e-6) / 1e9 / hbm, 4) if mid else None,
        "accumulated_step_us": round(part(evs, K, nmb - 1, 1, 2), 2),
        "accumulated_step_frac_of_hbm": round(last_b / (part(evs, K, nmb - 1, 1, 2) * 1e-6) / 1e9 / hbm, 4),
        "dgrad_us": round(part(evs, K, nmb - 1, 0, 1), 2),
        "split_us_per_window": round(split_ms * 1000.0 / KS, 1),
        "split_accumulate_first_us": round(s_first, 2),
        "split_accumulate_us": round(s_mid, 2) if s_mid is not None else None,
        "split_dgrad_us": round(statistics.mean(part(sev, KS, k, 0, 1) for k in range(nmb)), 2),
        "gpu_launches": 2 * nmb * K, "clocks": clocks,
    }
    print(json.dumps(line), flush=True)


def build_stack(opt, stname, dev, seed, bt=512):
    """The 224 linears of Llama-3.1-8B (32 layers x down, up, gate, o, v, k, q)
    with their state, inputs and one shared dX buffer per D_in and workspace,
    drawn on the device."""
    import torch
    import backward_gemm_optimizer_gb300 as F
    from backward_gemm_optimizer_gb300 import synthetic as S

    wdt = torch.float32 if stname == "f32state" else torch.bfloat16
    mdt = wdt
    two = opt == "adamw"
    order = [x for x in reversed(S.LLAMA31_8B_LINEARS)]
    layers = []
    sid = 0
    for layer in range(S.LLAMA31_8B_LAYERS):
        lin = {}
        for name, d_out, d_in in order:
            sid += 1
            L = {"name": name, "d_out": d_out, "d_in": d_in}
            L["W"] = S.device_normal_(torch.empty((d_out, d_in), dtype=wdt, device=dev), 0.02, seed, 16 * sid)
            L["m"] = S.device_normal_(torch.empty((d_out, d_in), dtype=mdt, device=dev), 1e-3, seed, 16 * sid + 1)
            if two:
                L["v"] = S.device_normal_(torch.empty((d_out, d_in), dtype=mdt, device=dev), 1e-6, seed,
                                          16 * sid + 2, absolute=True)
            L["X"] = S.device_normal_(torch.empty((bt, d_in), dtype=torch.bfloat16, device=dev), 1.0, seed,
                                      16 * sid + 3)
            L["dY"] = S.device_normal_(torch.empty((bt, d_out), dtype=torch.bfloat16, device=dev), 1.0, seed,
                                       16 * sid + 4)
            lin[name] = L
        layers.append(lin)
    dX = {d_in: torch.empty((bt, d_in), dtype=torch.bfloat16, device=dev) for _, _, d_in in order}
    # One workspace serves every linear: the calls run one after another on one stream.
    ws_bytes = max(F.workspace_bytes(d_out, d_in, bt) for _, d_out, d_in in order)
    ws = torch.empty(max(16, ws_bytes), dtype=torch.uint8, device=dev)
    return {"opt": opt, "stname": stname, "layers": layers, "order": order, "dX": dX, "ws": ws, "bt": bt,
            "hp": STACK_HYPER[opt], "sr": stname == "bf16state", "two": two}


def stack_backward(F, st, L, t, stream_, flags=0):
    """One linear's backward pass (dX and the fused step) through the public API."""
    opt, hp, sr, ws = st["opt"], st["hp"], st["sr"], st["ws"]
    dxb = st["dX"][L["d_in"]]
    if opt == "adamw":
        F.backward_step("adamw", L["X"], L["dY"], L["W"], L["m"], L["v"], dxb, step=t, seed=1234, sr_w=sr,
                        workspace=ws, flags=flags, stream=stream_, **hp)
    elif opt == "lion":
        F.backward_step("lion", L["X"], L["dY"], L["W"], L["m"], None, dxb, lr=hp["lr"], beta1=hp["beta1"],
                        beta2=hp["beta2"], weight_decay=hp["weight_decay"], step=t, seed=1234, sr_w=sr,
                        workspace=ws, flags=flags, stream=stream_)
    else:
        F.backward_step("sgdm", L["X"], L["dY"], L["W"], L["m"], None, dxb, lr=hp["lr"], momentum=hp["beta1"],
                        weight_decay=hp["weight_decay"], step=t, seed=1234, sr_w=sr, workspace=ws, flags=flags,
                        stream=stream_)


def stack_algorithmic_bytes(st):
    """Every linear's state read and written once, X and dY read, dX written."""
    eb = 4 if st["stname"] == "f32state" else 2
    sb = 2 * eb * (3 if st["two"] else 2)
    bt = st["bt"]
    return sum(len(st["layers"]) * (d_out * d_in * sb + 2 * bt * (d_out + 2 * d_in))
               for _, d_out, d_in in st["order"])


def run_stack(args, rank, world, local_rank):
    """One step = backward over the 224 linears of Llama-3.1-8B (layer 31 .. 0,
    down, up, gate, o, v, k, q): one forge_backward_step per linear, on the
    path the library picks for each shape (the split path is timed too)."""
    import torch
    import backward_gemm_optimizer_gb300 as F

    opt, stname = STACKS[args.workload]
    dev = torch.device(f"cuda:{local_rank}")
    torch.cuda.set_device(dev)
    st = build_stack(opt, stname, dev, replica_seed(rank))
    layers, order, bt, two = st["layers"], st["order"], st["bt"], st["two"]
    stream = torch.cuda.current_stream(dev)

    def backward(L, t, stream_, flags=0):
        stack_backward(F, st, L, t, stream_, flags)

    def stack_step(t, events=None, flags=0, stream_=None):
        stream_ = stream if stream_ is None else stream_
        i = 0
        for layer in reversed(range(len(layers))):
            for name, _, _ in order:
                L = layers[layer][name]
                if events is not None:
                    events[i][0].record(stream_)
                backward(L, t, stream_, flags)
                if events is not None:
                    events[i][1].record(stream_)
                i += 1

    t = 1
    for _ in range(args.warmup):
        stack_step(t); t += 1
    F.sync_status(stream)
    n_lin = len(layers) * len(order)
    K = args.steps
    # per-linear events for one instrumented pass of each path (per-shape breakdown)
    per_shape = {}
    for key, flags in (("backward_us", 0), ("split_us", F.FLAG_BACKWARD_SPLIT)):
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n_lin)]
        torch.cuda.synchronize(dev)
        stack_step(t, ev, flags); t += 1
        torch.cuda.synchronize(dev)
        i = 0
        for layer in reversed(range(len(layers))):
            for name, d_out, d_in in order:
                a = per_shape.setdefault(name, {"d_out": d_out, "d_in": d_in, "backward_us": 0.0, "split_us": 0.0,
                                                "n": 0})
                a[key] += ev[i][0].elapsed_time(ev[i][1]) * 1000.0
                if key == "backward_us":
                    a["n"] += 1
                i += 1
    hbm, tflops, _ = load_peaks()
    for name, a in per_shape.items():
        for key in ("backward_us", "split_us"):
            a[key] = round(a[key] / a["n"], 2)
        eb = 4 if stname == "f32state" else 2
        sb = 2 * eb * (3 if two else 2)     # W and each moment read + written once
        ab = a["d_out"] * a["d_in"] * sb + 2 * bt * (a["d_out"] + 2 * a["d_in"])   # + X, dY read, dX written
        a["backward_algorithmic_bytes"] = ab
        a["backward_GBps"] = round(ab / (a["backward_us"] * 1e-6) / 1e9, 1)
        a["backward_frac_of_hbm"] = round(a["backward_GBps"] / hbm, 4)

    def timed(flags):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world)
        torch.cuda.synchronize(dev)
        e0.record(stream)
        nonlocal t
        for _ in range(K):
            stack_step(t, None, flags); t += 1
        e1.record(stream)
        torch.cuda.synchronize(dev)
        F.sync_status(stream)
        return max_over_ranks(e0.elapsed_time(e1) / K, world, dev)

    sampler = ClockSampler(local_rank)
    sampler.start()
    time.sleep(0.2)
    eager_ms = timed(0)
    clocks = sampler.stop()
    split_ms = timed(F.FLAG_BACKWARD_SPLIT)
    graph_ms = None
    if args.graph:
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        # capture on a side stream: the library launches on the stream it is given
        with torch.cuda.graph(g, stream=side):
            stack_step(t, None, 0, torch.cuda.current_stream(dev))
        torch.cuda.synchronize(dev)
        g.replay(); torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(K):
            g.replay()     # the same step index each replay (graph parameters are fixed)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        F.sync_status(stream)
        graph_ms = max_over_ranks(e0.elapsed_time(e1) / K, world, dev)
    if rank != 0:
        return
    params = sum(a["d_out"] * a["d_in"] * a["n"] for a in per_shape.values())
    # The whole stack against the measured HBM peak: every linear's state read
    # and written once, X and dY read, dX written (the CUDA-graph time where
    # it was taken, else the eager one).
    stack_bytes = sum(a["backward_algorithmic_bytes"] * a["n"] for a in per_shape.values())
    best_ms = graph_ms if graph_ms is not None else eager_ms
    achieved = stack_bytes / (best_ms * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": round(eager_ms * 1000.0, 1), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(eager_ms, 3), "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": args.workload, "linears": n_lin, "params": params, "bt": bt, "optimizer": opt,
                   "state": stname, "step": "224 x forge_backward_step (library's path choice), layer 31..0",
                   "l2": "state 84 GB (fp32) / 42 GB (bf16) >> L2"},
        "graph_ms_per_step": round(graph_ms, 3) if graph_ms is not None else None,
        "split_ms_per_step": round(split_ms, 3),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(achieved / hbm, 4), "traffic": None, "algorithmic_bytes": stack_bytes,
                     "timed": "CUDA graph" if graph_ms is not None else "eager"},
        "per_shape": per_shape, "gpu_launches": 2 * n_lin * K, "clocks": clocks,
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="forge", choices=["forge", "reference"])
    ap.add_argument("--workload", default=DEFAULT, choices=sorted(WORKLOADS) + sorted(STACKS) + sorted(ACCUM))
    ap.add_argument("--graph", action="store_true", help="stack workloads: also replay the step as a CUDA graph")
    ap.add_argument("--e2e-steps", type=int, default=100)
    ap.add_argument("--split-steps", type=int, default=200, help="steps of the split-path comparison")
    ap.add_argument("--cpu-rows", type=int, default=14336)
    ap.add_argument("--cpu-min-s", type=float, default=10.0)
    ap.add_argument("--cpu-budget-s", type=float, default=120.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the other configurations' compact record (BT sweep, 8-bit, 224-linear stacks)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        import torch
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    try:
        if args.workload in STACKS:
            run_stack(args, rank, world, local_rank)
        elif args.workload in ACCUM:
            run_accum(args, rank, world, local_rank)
        else:
            run_gpu(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
