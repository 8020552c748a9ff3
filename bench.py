"""Decode-step benchmark of the GB300 Q4_0 decoder-layer library.

One step = one new token through every layer of the workload (all steps of the hot path:
norm, Q4_0 QKV, QK-norm, RoPE, KV append, split-K GQA attention, O + residual, norm,
gate/up + gated activation, down + residual).  Default workload: the Qwen3-1.7B-shape
decode step at batch 1 (28 layers, hidden 2048, 16/8 heads of 128, FFN 6144, 4096
cached positions), whose 1.26 GB of weights and KV per step exceed the 129 MB L2, so
nothing is flushed between steps.

Prints one JSON line.  `value` is achieved HBM GB/s over the step's algorithmic bytes
(Q4_0 weights + KV cache read + activations), with inputs resident; `e2e` is the same
metric through the C ABI with the step's input copied from pinned host memory and the
output read back inside the timed region.  --impl reference times the fp64 oracle on the
host cores on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import gem_synth  # noqa: E402
from gem_synth import configs  # noqa: E402

METRIC = "Q4_0 decode GEMV+attn HBM GB/s (% of ~8 TB/s); decode layer-step tok/s at B=1/8"
UNIT = "GB/s"


# ---- helpers ------------------------------------------------------------------------------

def layer_bytes(shape, B: int, T: int) -> dict:
    """Algorithmic bytes of one layer step: every byte the method must move once."""
    def q4(n, k):
        return n * (k // 32) * 18
    w = (q4(shape.n_qkv, shape.H) + q4(shape.H, shape.n_q * shape.d) + 2 * q4(shape.F, shape.H)
         + q4(shape.H, shape.F))
    kv = B * shape.n_kv * T * shape.d * 2 * 2
    kv_write = B * shape.n_kv * shape.d * 2 * 2
    act = 4 * B * (2 * shape.H + shape.n_qkv * 2 + 2 * shape.n_q * shape.d + 3 * shape.F + 4 * shape.H)
    return {"weights": w, "kv": kv + kv_write, "act": act, "total": w + kv + kv_write + act}


def attn_bytes(shape, B, T):
    return B * shape.n_kv * T * shape.d * 2 * 2 + 4 * B * 2 * shape.n_q * shape.d


def gemv_bytes(N, K, B):
    return N * (K // 32) * 18 + 4 * B * (K + N)


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(path))
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def device_record(torch, index: int) -> dict:
    """GPU name, SM count, L2 size and driver version of the measuring device."""
    pr = torch.cuda.get_device_properties(index)
    rec = {"name": pr.name, "sms": pr.multi_processor_count,
           "l2_bytes": getattr(pr, "L2_cache_size", None), "driver": None}
    try:
        out = subprocess.run(["nvidia-smi", "-i", str(index), "--query-gpu=driver_version",
                              "--format=csv,noheader"], capture_output=True, text=True, timeout=20)
        rec["driver"] = out.stdout.strip() or None
    except Exception:
        pass
    return rec


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []   # (wall time, csv line)
        self.t0 = self.t1 = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            deadline = time.time() + 2.0   # the sampler is running before the timed region starts
            while not self.lines and time.time() < deadline:
                time.sleep(0.01)
        except Exception:
            self.proc = None
        self.t0 = time.time()
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def __exit__(self, *a):
        self.t1 = time.time()
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        inside = [ln for t, ln in self.lines if self.t0 is not None and self.t0 <= t <= (self.t1 or t) + 0.15]
        for ln in inside:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = max(mx, float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def traffic_record(kernel_key: str):
    """ncu DRAM traffic per launch, valid only while the kernel source is unchanged."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        rec = json.load(open(path))[kernel_key]
    except Exception:
        return None
    src = os.path.join(ROOT, rec["source"])
    h = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    return rec["bytes_per_launch"] if h == rec["source_sha256_16"] else None


# ---- replicas (N > 1): one independent step per rank, max-over-ranks timing -------------------

def max_over_ranks(dist, torch, ms: float, device) -> float:
    """The slowest rank's step time: every rank contributes its own, all receive the max."""
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(step_bytes: int, world: int, ms: float) -> float:
    """Aggregate algorithmic GB/s of `world` replicas, each streaming step_bytes per step."""
    return step_bytes * world / (ms * 1e-3) / 1e9


# ---- device setup -----------------------------------------------------------------------------

class Model:
    def __init__(self, gem, torch, wl, seed=0):
        self.gem, self.t, self.wl = gem, torch, wl
        self.B = wl.B
        self.layers, self.kc, self.vc, self.ws = [], [], [], []
        for li, (shape, cap) in enumerate(zip(wl.layers, wl.cache_cap)):
            tens = configs.layer_tensors(shape, wl.B, cap, seed, li)
            dl = gem.DeviceLayer(shape, tens)
            self.layers.append(dl)
            self.kc.append(torch.from_numpy(tens.k_cache.view(np.int16)).cuda())
            self.vc.append(torch.from_numpy(tens.v_cache.view(np.int16)).cuda())
            self.ws.append(torch.empty(max(1, gem.decode_layer_workspace(dl, wl.B, cap)),
                                       dtype=torch.uint8, device="cuda"))
            del tens
        H = wl.layers[0].H
        self.x0 = configs.layer_input(H, wl.B, seed)
        self.x = torch.from_numpy(self.x0.copy()).cuda()
        self.pos = torch.full((wl.B,), wl.pos, dtype=torch.int32, device="cuda")

    def step(self):
        for dl, k, v, w in zip(self.layers, self.kc, self.vc, self.ws):
            self.gem.decode_layer(dl, self.x, k, v, self.pos, w)

    def launches_per_step(self):
        n = 0
        for s, cap in zip(self.wl.layers, self.wl.cache_cap):
            fused = s.d <= 256 and s.n_q // s.n_kv <= 4   # QK-norm/RoPE/append inside attention
            n += (5 if fused else 6) + (2 if s.post_norms else 0)
            if self.gem.gqa_decode_attn_workspace(self.B, s.n_q, s.n_kv, s.d, cap, s.window) > 0:
                n += 1
        return n


def capture(torch, fn):
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()  # warm (sets kernel attributes outside capture)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


def time_graph(torch, g, reps, warmup=3):
    for _ in range(warmup):
        g.replay()
    torch.cuda.synchronize()
    st = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(st)
    for _ in range(reps):
        g.replay()
    e1.record(st)
    e1.synchronize()
    return e0.elapsed_time(e1) / reps


# ---- arms -------------------------------------------------------------------------------------

def run_kernel_only(args):
    """A single op on its own (for ncu captures): `gemv` = a 31B FFN projection over --mats
    rotated matrices at --batch (--gemv-shape up: K=5376 -> N=21504; down: K=21504 -> N=5376);
    `attn` = GQA decode attention over the workload's first --layers caches."""
    import torch
    import q4_gemv_gqa_gb300 as gem
    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    res = {"kernel": args.kernel}
    if args.kernel == "gemv":
        B = args.batch
        N, K = (21504, 5376) if args.gemv_shape == "up" else (5376, 21504)
        res["shape"] = {"N": N, "K": K, "B": B}
        mats = [torch.from_numpy(gem_synth.q4_0_matrix(0, 5000 + i, N, K)).cuda()
                for i in range(args.mats)]
        x = torch.from_numpy(gem_synth.normal_f32(0, 6000, (B, K))).cuda()
        y = torch.empty((B, N), device="cuda")

        def run():
            for W in mats:
                gem.q4_0_gemv(W, N, K, x, y)
        b = gemv_bytes(N, K, B)
        n = len(mats)
    else:
        wl = configs.workload(args.workload)
        wl = configs.with_layers(wl, args.layers or 2)
        s0, cap = wl.layers[0], wl.cache_cap[0]
        kcs = [torch.from_numpy(gem_synth.normal_f16_bits(0, 100 + i, (wl.B, s0.n_kv, cap, s0.d)).view(np.int16)).cuda()
               for i in range(len(wl.layers))]
        vcs = [torch.from_numpy(gem_synth.normal_f16_bits(0, 200 + i, (wl.B, s0.n_kv, cap, s0.d)).view(np.int16)).cuda()
               for i in range(len(wl.layers))]
        q = torch.from_numpy(gem_synth.normal_f32(0, 7, (wl.B, s0.n_q * s0.d))).cuda()
        out = torch.empty_like(q)
        pos = torch.full((wl.B,), wl.pos, dtype=torch.int32, device="cuda")
        ws = torch.empty(max(1, gem.gqa_decode_attn_workspace(wl.B, s0.n_q, s0.n_kv, s0.d, cap, s0.window)),
                         dtype=torch.uint8, device="cuda")

        def run():
            for kc, vc in zip(kcs, vcs):
                gem.gqa_decode_attn(q, kc, vc, s0.n_q, s0.n_kv, s0.d, pos, s0.window, float(s0.scale), out, ws)
        T = min(wl.pos + 1, s0.window) if s0.window else wl.pos + 1
        b = attn_bytes(s0, wl.B, T)
        n = len(kcs)
    for _ in range(args.warmup):
        run()
    torch.cuda.synchronize()
    st = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(st)
    for _ in range(args.steps):
        run()
    e1.record(st)
    e1.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / (args.steps * n)
    res.update({"us_per_launch": round(us, 3), "bytes_per_launch": b, "gbs": round(b / us / 1e3, 1)})
    print(json.dumps(res), flush=True)


def run_gem(args):
    import torch
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    import q4_gemv_gqa_gb300 as gem

    wl = configs.workload(args.workload)
    if args.layers:
        wl = configs.with_layers(wl, args.layers)
    T = wl.pos + 1
    model = Model(gem, torch, wl)
    nL = len(wl.layers)
    step_bytes = sum(layer_bytes(s, wl.B, min(T, s.window) if s.window else T)["total"] for s in wl.layers)

    g = capture(torch, model.step)
    for _ in range(args.warmup):
        g.replay()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    st = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        e0.record(st)
        for _ in range(args.steps):
            g.replay()
        e1.record(st)
        e1.synchronize()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / args.steps
    if dist:
        ms = max_over_ranks(dist, torch, ms, "cuda")
        dist.barrier()
    flags = gem.device_status()

    # e2e through the C ABI from pinned host memory: H2D input, the step, D2H output
    hx = torch.from_numpy(model.x0.copy()).pin_memory()
    hpos = torch.full((wl.B,), wl.pos, dtype=torch.int32).pin_memory()
    hout = torch.empty_like(hx).pin_memory()

    def e2e_step():
        model.x.copy_(hx, non_blocking=True)
        model.pos.copy_(hpos, non_blocking=True)
        g.replay()
        hout.copy_(model.x, non_blocking=True)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    e2 = torch.cuda.Event(enable_timing=True)
    e3 = torch.cuda.Event(enable_timing=True)
    e2.record(st)
    for _ in range(args.steps):
        e2e_step()
    e3.record(st)
    e3.synchronize()
    e2e_ms = e2.elapsed_time(e3) / args.steps
    e2e_wall_ms = (time.perf_counter() - t0) * 1e3 / args.steps

    # per-kernel roofline: each op of the layer timed alone over the data of every layer that
    # has the first layer's shape and cache capacity (a mixed stack's other layers differ)
    shape0, cap0 = wl.layers[0], wl.cache_cap[0]
    same = [i for i in range(nL) if wl.layers[i] == shape0 and wl.cache_cap[i] == cap0]
    nS = len(same)
    kern = {}
    q = torch.randn((wl.B, shape0.n_q * shape0.d), device="cuda")
    out = torch.empty_like(q)
    aws = torch.empty(max(1, gem.gqa_decode_attn_workspace(wl.B, shape0.n_q, shape0.n_kv, shape0.d, cap0,
                                                           shape0.window)), dtype=torch.uint8, device="cuda")

    def attn_all():
        for i in same:
            k, v = model.kc[i], model.vc[i]
            gem.gqa_decode_attn(q, k, v, shape0.n_q, shape0.n_kv, shape0.d, model.pos, shape0.window,
                                float(shape0.scale), out, aws)
    ga = capture(torch, attn_all)
    ms_a = time_graph(torch, ga, max(5, args.steps)) / nS
    Ta = min(T, shape0.window) if shape0.window else T
    kern["gqa_decode_attn"] = {"us": ms_a * 1e3, "bytes": attn_bytes(shape0, wl.B, Ta)}

    xin = torch.randn((wl.B, max(shape0.H, shape0.F, shape0.n_q * shape0.d)), device="cuda")
    layers0 = [model.layers[i] for i in same]
    gate_up = [torch.cat([dl.w_gate, dl.w_up]) for dl in layers0]
    yb = torch.empty((wl.B, 2 * shape0.F), device="cuda")
    for name, mats, N, K in [("q4_0_gemv_gate_up", gate_up, 2 * shape0.F, shape0.H),
                             ("q4_0_gemv_qkv", [dl.w_qkv for dl in layers0], shape0.n_qkv, shape0.H),
                             ("q4_0_gemv_down", [dl.w_down for dl in layers0], shape0.H, shape0.F),
                             ("q4_0_gemv_o", [dl.w_o for dl in layers0], shape0.H, shape0.n_q * shape0.d)]:
        xk = xin[:, :K].contiguous()
        yk = torch.empty((wl.B, N), device="cuda")

        def gemv_all(mats=mats, N=N, K=K, xk=xk, yk=yk):
            for W in mats:
                gem.q4_0_gemv(W, N, K, xk, yk)
        gg = capture(torch, gemv_all)
        ms_g = time_graph(torch, gg, max(5, args.steps)) / nS
        kern[name] = {"us": ms_g * 1e3, "bytes": gemv_bytes(N, K, wl.B)}
    del gate_up, yb

    # the 31B FFN projection (5376 -> 21504), 8 distinct matrices (520 MB) rotated
    gemv31 = {}
    W31 = [torch.from_numpy(gem_synth.q4_0_matrix(0, 5000 + i, 21504, 5376)).cuda() for i in range(8)]
    for B in (1, 8):
        x31 = torch.from_numpy(gem_synth.normal_f32(0, 6000, (B, 5376))).cuda()
        y31 = torch.empty((B, 21504), device="cuda")

        def g31(x31=x31, y31=y31):
            for W in W31:
                gem.q4_0_gemv(W, 21504, 5376, x31, y31)
        gg = capture(torch, g31)
        us = time_graph(torch, gg, max(5, args.steps)) / len(W31) * 1e3
        b = gemv_bytes(21504, 5376, B)
        gemv31["b%d" % B] = {"us": us, "gbs": b / us / 1e3}
    del W31

    # the same step as one persistent launch (gem_decode_step), where the layers allow it
    persistent = None
    try:
        plan = gem.StepPlan(model.layers, wl.B, model.kc, model.vc)
        gp = capture(torch, lambda: plan.step(model.x, model.pos))
        ms_p = time_graph(torch, gp, max(5, args.steps))
        persistent = {"ms_per_step": round(ms_p, 4), "us_per_layer": round(ms_p * 1e3 / nL, 3)}
        plan.close()
    except gem.GemError as e:
        persistent = {"unsupported": str(e)}

    peak, peak_kind = measured_peaks()
    for k in kern.values():
        k["gbs"] = k["bytes"] / k["us"] / 1e3
        k["frac"] = k["gbs"] / peak
    for v in gemv31.values():
        v["frac"] = v["gbs"] / peak
    # dominant kernel: largest time per step inside the layer chain
    per_step_us = {"gqa_decode_attn": kern["gqa_decode_attn"]["us"],
                   "q4_0_gemv_gate_up": kern["q4_0_gemv_gate_up"]["us"],
                   "q4_0_gemv_qkv": kern["q4_0_gemv_qkv"]["us"],
                   "q4_0_gemv_down": kern["q4_0_gemv_down"]["us"],
                   "q4_0_gemv_o": kern["q4_0_gemv_o"]["us"]}
    dom = max(per_step_us, key=per_step_us.get)
    dk = kern[dom]

    tokens = wl.B * world
    value = whole_job_gbs(step_bytes, world, ms)
    if rank == 0:
        cpu = cpu_baseline(wl, args) if world == 1 else None
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded Q4_0 weights, N(0,1) fp16 KV cache and fp32 activations)",
            "config": {"workload": wl.name, "layers": nL, "B": wl.B, "n_kv": wl.pos,
                       "hidden": wl.layers[0].H, "heads": [wl.layers[0].n_q, wl.layers[0].n_kv],
                       "head_dim": wl.layers[0].d, "ffn": wl.layers[0].F,
                       "bytes_per_step": step_bytes,
                       "l2": "inputs larger than L2 (%.2f GB streamed per step vs 129 MB L2)" % (step_bytes / 1e9),
                       "parallelism": "replicas" if world > 1 else "single GPU"},
            "tok_s": round(tokens / (ms * 1e-3), 1),
            "us_per_layer": round(ms * 1e3 / nL, 3),
            "frac_of_peak": round(value / world / peak, 4),
            "roofline": {"bound": "hbm", "kernel": dom, "achieved": round(dk["gbs"], 1), "peak": peak,
                         "peak_kind": peak_kind, "unit": "GB/s", "frac": round(dk["frac"], 4),
                         "traffic": traffic_record(dom), "algorithmic_bytes": dk["bytes"],
                         "us_per_launch": round(dk["us"], 3)},
            "kernels": {k: {"us": round(v["us"], 3), "gbs": round(v["gbs"], 1), "frac": round(v["frac"], 4)}
                        for k, v in kern.items()},
            "kernels_layers": "the %d of %d layers shaped like the first" % (nS, nL),
            "persistent_step_kernel": persistent,
            "gemv_k5376_n21504": {k: {"us": round(v["us"], 3), "gbs": round(v["gbs"], 1),
                                      "frac": round(v["frac"], 4)} for k, v in gemv31.items()},
            "e2e": {"value": round(step_bytes / (e2e_ms * 1e-3) / 1e9, 1), "unit": UNIT,
                    "ms_per_step": round(e2e_ms, 4), "wall_ms_per_step": round(e2e_wall_ms, 4),
                    "h2d_bytes_per_step": int(hx.numel() * 4 + hpos.numel() * 4),
                    "d2h_bytes_per_step": int(hout.numel() * 4)},
            "gpu_launches": model.launches_per_step() * args.steps,
            "clocks": clk.summary(),
            "device": device_record(torch, local),
            "device_flags": flags,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()


_ORACLE_TENSORS = {}


def _oracle_sample(wl, budget_s, max_cached=4):
    """Oracle layer steps on the workload's layers, in order and cycling over the first
    `max_cached` of them (tensors built once), until ~budget_s of CPU work (at least one step)."""
    import oracle
    T = wl.pos + 1
    pos = np.full(wl.B, wl.pos, np.int32)
    done, bytes_done, t_spent = 0, 0, 0.0
    x = configs.layer_input(wl.layers[0].H, wl.B, 0).astype(np.float64)
    ncyc = min(max_cached, len(wl.layers))
    while done == 0 or t_spent < budget_s:
        li = done % ncyc
        key = (wl.name, li, wl.B)
        if key not in _ORACLE_TENSORS:
            _ORACLE_TENSORS[key] = configs.layer_tensors(wl.layers[li], wl.B, wl.cache_cap[li], 0, li)
        tens = _ORACLE_TENSORS[key]
        t0 = time.perf_counter()   # (a repeated step rewrites the same appended slot: same work)
        x = oracle.decode_layer(wl.layers[li], tens, x, pos, tens.k_cache, tens.v_cache)
        t_spent += time.perf_counter() - t0
        s = wl.layers[li]
        bytes_done += layer_bytes(s, wl.B, min(T, s.window) if s.window else T)["total"]
        done += 1
    return done, bytes_done, t_spent, oracle.num_threads()


def cpu_baseline(wl, args):
    done, b, t, cores = _oracle_sample(wl, args.cpu_budget)
    return {"value": round(b / t / 1e9, 3), "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": "%d layer steps of %s (its first %d layers in turn; fp64 scalar C, OpenMP over "
                      "rows/heads), %.1f s" % (done, wl.name, min(4, len(wl.layers)), t),
            "ms_per_layer": round(t * 1e3 / done, 1)}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    wl = configs.workload(args.workload)
    if args.layers:
        wl = configs.with_layers(wl, args.layers)
    per_step = args.cpu_budget / max(1, args.steps + args.warmup)   # at least one layer step each
    for _ in range(args.warmup):
        _oracle_sample(configs.with_layers(wl, 1), 0.0)
    tot_b, tot_t, cores, done = 0, 0.0, 1, 0
    for _ in range(args.steps):
        d, b, t, cores = _oracle_sample(wl, per_step)
        tot_b += b
        tot_t += t
        done += d
    v = tot_b / tot_t / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": round(v, 3), "unit": UNIT, "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(tot_t * 1e3 / args.steps, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (same seeded inputs as the GPU arm)",
            "config": {"workload": wl.name, "layers": len(wl.layers), "B": wl.B, "n_kv": wl.pos},
            "cpu_baseline": {"value": round(v, 3), "unit": UNIT, "kind": "oracle", "cores": cores,
                             "sample": "%d layer steps of %s per %d steps" % (done, wl.name, args.steps)},
            "e2e": {"value": round(v, 3), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["gem", "reference"], default="gem")
    ap.add_argument("--workload", default="qwen3-1.7b",
                    choices=["tiny", "qwen3-1.7b", "qwen3-4b-b8", "gemma4-31b-group"])
    ap.add_argument("--layers", type=int, default=0, help="use only the first n layers")
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle work")
    ap.add_argument("--kernel", choices=["step", "gemv", "attn"], default="step",
                    help="time one op alone (for profiler captures) instead of the step")
    ap.add_argument("--batch", type=int, default=1, help="--kernel gemv: activation rows")
    ap.add_argument("--mats", type=int, default=8, help="--kernel gemv: rotated matrices")
    ap.add_argument("--gemv-shape", choices=["up", "down"], default="up",
                    help="--kernel gemv: 31B FFN up (5376 -> 21504) or down (21504 -> 5376) projection")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    elif args.kernel != "step":
        run_kernel_only(args)
    else:
        run_gem(args)


if __name__ == "__main__":
    main()
