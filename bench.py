"""Decode-step benchmark of the GB300 Q4_0 decoder-layer library.

One step = one new token through every layer of the workload (all steps of the hot path:
norm, Q4_0 QKV, QK-norm, RoPE, KV append, split-K GQA attention, O + residual, norm,
gate/up + gated activation, down + residual).  Default workload (the headline line): the
Qwen3-1.7B-shape decode step at batch 1 (28 layers, hidden 2048, 16/8 heads of 128, FFN
6144, 4096 cached positions), whose 1.27 GB of weights and KV per step exceed the 129 MB
L2, so nothing is flushed between steps.  The same run adds sub-records for the other
workloads: the Qwen3-4B-shape step at B = 8 (36 layers, 2048 cached positions per
sequence), one Gemma-4-31B-shape group (5 sliding-window layers + 1 full-attention layer,
32768 cached positions), the tiny layer, and the 31B FFN-shape GEMV at B = 1 and 8.

Prints one JSON line.  `value` is achieved HBM GB/s over the step's algorithmic bytes
(Q4_0 weights + KV cache read + appended rows + activations), with inputs resident; `e2e`
is the same metric through the C ABI with the step's input copied from pinned host memory
and the output read back inside the timed region.  --impl reference times the fp64 oracle
on the host cores on a bounded sample of the same workload.

Synthetic inputs: seeded Q4_0 weights (codes uniform 0..15, binary16 scales uniform
[0.002, 0.02]), N(0,1) binary16 KV caches, N(0,1) fp32 activations, norm weights
1 + N(0, 0.1).  Every layer has its own weight and cache buffers; the timing-only stacks
fill them from a few distinct seeded draws per layer shape (`distinct` in each record),
since generating every layer's draws on the host would dominate the run.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import gem_synth  # noqa: E402
from gem_synth import configs  # noqa: E402

METRIC = "Q4_0 decode GEMV+attn HBM GB/s (% of ~8 TB/s); decode layer-step tok/s at B=1/8"
UNIT = "GB/s"


# ---- algorithmic bytes ------------------------------------------------------------------------

def q4_bytes(n, k):
    return n * (k // 32) * 18


def layer_bytes(shape, B: int, T: int) -> dict:
    """Algorithmic bytes of one layer step: every byte the method must move once."""
    w = (q4_bytes(shape.n_qkv, shape.H) + q4_bytes(shape.H, shape.n_q * shape.d) + 2 * q4_bytes(shape.F, shape.H)
         + q4_bytes(shape.H, shape.F))
    rows = 1 if getattr(shape, "compact_kv", False) else 2   # a compact cache keeps V rows only
    kv = B * shape.n_kv * T * shape.d * 2 * rows
    kv_write = B * shape.n_kv * shape.d * 2 * rows
    act = 4 * B * (2 * shape.H + shape.n_qkv * 2 + 2 * shape.n_q * shape.d + 3 * shape.F + 4 * shape.H)
    return {"weights": w, "kv": kv + kv_write, "act": act, "total": w + kv + kv_write + act}


def attn_bytes(shape, B, T):
    rows = 1 if getattr(shape, "compact_kv", False) else 2
    return B * shape.n_kv * T * shape.d * 2 * rows + 4 * B * 2 * shape.n_q * shape.d


def gemv_bytes(N, K, B, nmat=1):
    return nmat * q4_bytes(N, K) + 4 * B * (K + N)


def attended(shape, pos):
    T = pos + 1
    return min(T, shape.window) if shape.window else T


def step_bytes(wl):
    return sum(layer_bytes(s, wl.B, attended(s, wl.pos))["total"] for s in wl.layers)


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


# ---- clocks during the timed region -----------------------------------------------------------

class Clocks:
    """SM clock, its maximum and the clock-event (throttle) reasons, read through NVML
    (libnvidia-ml, part of the driver) as often as every millisecond while a timed region
    runs, so even a short region carries samples.  Read-only: no setting is changed.  Falls
    back to one nvidia-smi query at each end of the region when NVML cannot be opened."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, index: int, pci_bus_id: str | None = None):
        self.nvml = None
        self.handle = ctypes.c_void_p()
        self.samples = []   # (sm_mhz, max_mhz, reasons mask)
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() == 0:
                ok = pci_bus_id is not None and lib.nvmlDeviceGetHandleByPciBusId_v2(
                    pci_bus_id.encode(), ctypes.byref(self.handle)) == 0
                if not ok:
                    ok = lib.nvmlDeviceGetHandleByIndex_v2(index, ctypes.byref(self.handle)) == 0
                if ok:
                    self.nvml = lib
                    self.reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                        getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
        except Exception:
            self.nvml = None
        self.index = index

    def sample(self):
        if self.nvml is not None:
            sm, mx, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
            if (self.nvml.nvmlDeviceGetClockInfo(self.handle, 1, ctypes.byref(sm)) == 0 and
                    self.nvml.nvmlDeviceGetMaxClockInfo(self.handle, 1, ctypes.byref(mx)) == 0 and
                    self.reasons_fn(self.handle, ctypes.byref(rs)) == 0):
                self.samples.append((float(sm.value), float(mx.value), int(rs.value)))
            return
        try:
            out = subprocess.run(["nvidia-smi", "-i", str(self.index), "--query-gpu=clocks.sm,clocks.max.sm,"
                                  "clocks_event_reasons.active", "--format=csv,noheader,nounits"],
                                 capture_output=True, text=True, timeout=20).stdout.strip().split(",")
            self.samples.append((float(out[0]), float(out[1]), int(out[2].strip(), 16)))
        except Exception:
            pass

    def run_timed(self, torch, enqueue, steps, stream):
        """Record an event, enqueue `steps` units of work, record an event, and sample the clocks
        while the queued work runs, until the second event has completed.  Returns the elapsed
        milliseconds.  Nothing is sampled between the launches: a sample takes the host long
        enough to leave the GPU idle between steps."""
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            enqueue()
        e1.record(stream)
        self.sample()   # the region's start (the queued steps are running)
        while not e1.query():
            self.sample()
            time.sleep(0.0005)
        self.sample()   # the region's end
        return e0.elapsed_time(e1)

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        reasons = set()
        for _, _, m in self.samples:
            for bit, name in self.REASONS.items():
                if m & bit:
                    reasons.add(name)
        return {"sm_mhz": statistics.median(s[0] for s in self.samples),
                "sm_max_mhz": max(s[1] for s in self.samples), "reasons": sorted(reasons),
                "samples": len(self.samples), "source": "nvml" if self.nvml is not None else "nvidia-smi"}


def pci_bus_id(torch, index: int):
    """The device's PCI bus id in NVML's form, when torch reports it."""
    pr = torch.cuda.get_device_properties(index)
    try:
        return "%08X:%02X:%02X.0" % (pr.pci_domain_id, pr.pci_bus_id, pr.pci_device_id)
    except AttributeError:
        return None


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
    """Every layer of a workload on the device, with its own weight, cache and workspace
    buffers.  The first `distinct` layers of each shape get their own seeded draws; later
    layers of that shape are device copies of them (distinct buffers, same values)."""

    def __init__(self, gem, torch, wl, seed=0, distinct=None):
        self.gem, self.t, self.wl = gem, torch, wl
        self.B = wl.B
        self.layers, self.kc, self.vc, self.ws = [], [], [], []
        seen = {}   # (shape, cap) -> list of (DeviceLayer, k, v)
        for li, (shape, cap) in enumerate(zip(wl.layers, wl.cache_cap)):
            key = (shape, cap)
            made = seen.setdefault(key, [])
            if distinct is None or len(made) < distinct:
                tens = configs.layer_weights(shape, seed, li)
                dl = gem.DeviceLayer(shape, tens)
                k, v = configs.kv_cache(shape, wl.B, cap, seed, li)
                kc = None if shape.compact_kv else torch.from_numpy(k.view(np.int16)).cuda()
                vc = torch.from_numpy(v.view(np.int16)).cuda()
                made.append((dl, kc, vc))
                del tens, k, v
            else:
                src, ks, vs = made[li % len(made)]
                dl = gem.DeviceLayer.clone(src)
                kc, vc = (None if ks is None else ks.clone()), vs.clone()
            self.layers.append(dl)
            self.kc.append(kc)
            self.vc.append(vc)
            self.ws.append(torch.empty(max(1, gem.decode_layer_workspace(dl, wl.B, cap)),
                                       dtype=torch.uint8, device="cuda"))
        H = wl.layers[0].H
        self.x0 = configs.layer_input(H, wl.B, seed)
        self.x = torch.from_numpy(self.x0.copy()).cuda()
        self.pos = torch.full((wl.B,), wl.pos, dtype=torch.int32, device="cuda")
        self.distinct = distinct

    def step(self):
        for dl, k, v, w in zip(self.layers, self.kc, self.vc, self.ws):
            self.gem.decode_layer(dl, self.x, k, v, self.pos, w)

    def launches_per_step(self):
        n = 0
        for s, cap in zip(self.wl.layers, self.wl.cache_cap):
            # QK-norm/RoPE/append inside attention (never for a compact cache)
            fused = s.d <= 256 and s.n_q // s.n_kv <= 4 and not s.compact_kv
            n += (5 if fused else 6) + (2 if s.post_norms else 0)
            if self.B >= 2:
                # an activation prep launch for each 2..8-row GEMV above 64M weights (the
                # records kernel); smaller ones build their operands in one launch
                mats = ((s.n_qkv, s.H, 1), (s.H, s.n_q * s.d, 1), (s.F, s.H, 2), (s.H, s.F, 1))
                n += sum(1 for N, K, m in mats if m * N * K > (64 << 20))
            if s.compact_kv:
                split = self.gem.gqa_decode_attn_compact_workspace(self.B, s.n_q, s.n_kv, s.d, cap, s.rope_dim) > 0
            elif fused:
                split = False   # the last-arriving split merges inside the attention kernel
            else:
                split = self.gem.gqa_decode_attn_workspace(self.B, s.n_q, s.n_kv, s.d, cap, s.window) > 0
            n += 1 if split else 0
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


# ---- the layer's ops, each as the chain launches it -------------------------------------------

def op_callers(gem, torch, model, idx):
    """One closure per op of the layer step over the layers `idx`, each calling the same fused
    kernel (same plan) the layer chain runs for it: QKV (pre-norm fused), attention (QK-norm,
    RoPE and the KV append fused where the shape allows), O (+ residual), gate/up (pre-norm,
    pair, gated activation), down (+ residual).  Returns {name: (fn, bytes per launch)}."""
    wl = model.wl
    s, cap, B = wl.layers[idx[0]], wl.cache_cap[idx[0]], wl.B
    nqd = s.n_q * s.d
    x = torch.randn((B, s.H), device="cuda")
    qkv = torch.randn((B, s.n_qkv), device="cuda")
    att = torch.randn((B, nqd), device="cuda")
    act = torch.randn((B, s.F), device="cuda")
    y = torch.empty((B, max(s.H, s.F, s.n_qkv)), device="cuda")
    aws_n = gem.gqa_decode_attn_workspace(B, s.n_q, s.n_kv, s.d, cap, s.window)
    aws = torch.empty(max(1, aws_n), dtype=torch.uint8, device="cuda")
    gws = torch.empty(max(1, gem.q4_0_gemv_workspace(B, max(s.H, s.F, nqd))), dtype=torch.uint8, device="cuda")
    L = [model.layers[i] for i in idx]
    T = attended(s, wl.pos)
    gq = None if not s.qk_norm else [dl.g_q for dl in L]
    gk = None if not s.qk_norm else [dl.g_k for dl in L]

    def qkv_fn():
        for dl in L:
            gem.q4_0_gemv_fused(dl.w_qkv, None, s.n_qkv, s.H, x, qkv, gamma=dl.g_attn, eps=s.eps, workspace=gws)

    def attn_fn():
        for j, i in enumerate(idx):
            gem.gqa_decode_attn_fused(qkv, s.n_q, s.n_kv, s.d, gq[j] if gq else None, gk[j] if gk else None,
                                      1 if s.v_from_k else 0, s.eps, model.pos, s.theta, s.rope_dim,
                                      model.kc[i], model.vc[i], s.window, float(s.scale), att,
                                      aws if aws_n else None)

    def o_fn():
        for dl in L:
            gem.q4_0_gemv_fused(dl.w_o, None, s.H, nqd, att, y, residual=x, workspace=gws)

    def gate_up_fn():
        for dl in L:
            gem.q4_0_gemv_fused(dl.w_gate, dl.w_up, s.F, s.H, x, act, gamma=dl.g_ffn, eps=s.eps, act=s.act,
                                workspace=gws)

    def down_fn():
        for dl in L:
            gem.q4_0_gemv_fused(dl.w_down, None, s.H, s.F, act, y, residual=x, workspace=gws)

    return {
        "q4_0_gemv_qkv": (qkv_fn, gemv_bytes(s.n_qkv, s.H, B)),
        "gqa_decode_attn": (attn_fn, attn_bytes(s, B, T) + B * s.n_kv * s.d * 4),
        "q4_0_gemv_o": (o_fn, gemv_bytes(s.H, nqd, B) + 4 * B * s.H),
        "q4_0_gemv_gate_up": (gate_up_fn, gemv_bytes(s.F, s.H, B, nmat=2)),
        "q4_0_gemv_down": (down_fn, gemv_bytes(s.H, s.F, B) + 4 * B * s.H),
    }


def same_shape_layers(wl):
    s0, c0 = wl.layers[0], wl.cache_cap[0]
    return [i for i in range(len(wl.layers)) if wl.layers[i] == s0 and wl.cache_cap[i] == c0]


# ---- arms -------------------------------------------------------------------------------------

def attn_full_runner(gem, torch, cache, B, ncopies=2):
    """The Gemma 4 31B full-attention layer's attention at 32,769 positions (B sequences) over
    `ncopies` cache copies: cache "standard" (K and V rows; QK-norm, RoPE and the append in the
    separate launch before it, as the layer chain runs it) or "compact" (V rows only, K rebuilt
    inside the attention).  Returns (run, algorithmic bytes per attention call, calls per run)."""
    s = configs.GEMMA31_FULL_COMPACT if cache == "compact" else configs.GEMMA31_FULL
    P = 32768
    cap = P + 1
    qkv = torch.randn((B, s.n_qkv), device="cuda")
    att = torch.empty((B, s.n_q * s.d), device="cuda")
    pos = torch.full((B,), P, dtype=torch.int32, device="cuda")
    gq = torch.ones(s.d, device="cuda")
    gk = torch.ones(s.d, device="cuda")
    caches = []
    for i in range(ncopies):
        v = torch.from_numpy(gem_synth.normal_f16_bits(0, 8000 + i, (B, s.n_kv, cap, s.d)).view(np.int16)).cuda()
        k = None if cache == "compact" else torch.from_numpy(
            gem_synth.normal_f16_bits(0, 8100 + i, (B, s.n_kv, cap, s.d)).view(np.int16)).cuda()
        caches.append((k, v))
    if cache == "compact":
        wsn = gem.gqa_decode_attn_compact_workspace(B, s.n_q, s.n_kv, s.d, cap, s.rope_dim)
    else:
        wsn = gem.gqa_decode_attn_workspace(B, s.n_q, s.n_kv, s.d, cap, 0)
    wsa = torch.empty(max(1, wsn), dtype=torch.uint8, device="cuda")

    def run():
        for k, v in caches:
            if cache == "compact":
                gem.rmsnorm_qknorm_rope(qkv, s.n_q, s.n_kv, s.d, gq, gk, 1, s.eps, pos, s.theta, s.rope_dim,
                                        None, v)
                gem.gqa_decode_attn_compact(qkv, v, s.n_q, s.n_kv, s.d, pos, float(s.scale), gk, s.rope_dim,
                                            s.theta, att, wsa if wsn else None)
            else:
                gem.gqa_decode_attn_fused(qkv, s.n_q, s.n_kv, s.d, gq, gk, 1, s.eps, pos, s.theta, s.rope_dim,
                                          k, v, 0, float(s.scale), att, wsa if wsn else None)
    return run, attn_bytes(s, B, cap), len(caches)


def run_kernel_only(args):
    """A single op on its own (for profiler captures): `gemv` = a 31B FFN projection over --mats
    rotated matrices at --batch (--gemv-shape up: K=5376 -> N=21504; down: K=21504 -> N=5376);
    `op` = one op of the workload's layer step (--op), as the chain launches it, over the
    workload's first --layers layers."""
    import torch
    import q4_gemv_gqa_gb300 as gem
    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    res = {"kernel": args.kernel}
    if args.kernel == "attn_full":
        res["shape"] = {"B": args.batch, "positions": 32769, "cache": args.cache}
        run, b, n = attn_full_runner(gem, torch, args.cache, args.batch)
    elif args.kernel == "persistent":
        # the persistent whole-step kernel over the workload's first --layers layers
        wl = configs.with_layers(configs.workload(args.workload), args.layers or 2)
        model = Model(gem, torch, wl, distinct=1)
        plan = gem.StepPlan(model.layers, wl.B, model.kc, model.vc)
        res["workload"] = wl.name

        def run():
            plan.step(model.x, model.pos)
        b = step_bytes(wl)
        n = 1
    elif args.kernel == "elementwise":
        # the stand-alone RMSNorm (B x 5376) and gated activation (B x 21504) calls
        B = args.batch
        xe = torch.randn((B, 5376), device="cuda")
        ge = torch.ones(5376, device="cuda")
        oe = torch.empty_like(xe)
        gate = torch.randn((B, 21504), device="cuda")
        up = torch.randn((B, 21504), device="cuda")
        act = torch.empty_like(gate)

        def run():
            gem.rmsnorm(xe, ge, 1e-6, oe)
            gem.swiglu(gate, up, 1, act)
        b = 4 * B * (2 * 5376 + 3 * 21504)
        n = 1
    elif args.kernel == "q8":
        # the tied Q8_0 logit projection (--vocab x 5376) and the device argmax of its logits
        B, V, Hl = args.batch, args.vocab, 5376
        res["shape"] = {"V": V, "H": Hl, "B": B}
        Wq = torch.from_numpy(gem_synth.q8_0_matrix(0, 7000, V, Hl)).cuda()
        xq = torch.from_numpy(gem_synth.normal_f32(0, 7001, (B, Hl))).cuda()
        yq = torch.empty((B, V), device="cuda")
        iq = torch.empty((B,), dtype=torch.int32, device="cuda")
        wsq = torch.empty(max(1, gem.argmax_workspace(B, V)), dtype=torch.uint8, device="cuda")

        def run():
            gem.q8_0_gemv(Wq, V, Hl, xq, yq)
            gem.argmax(yq, iq, wsq)
        b = V * (Hl // 32) * 34 + 4 * B * (Hl + V)
        n = 1
    elif args.kernel == "gemv":
        B = args.batch
        N, K = (21504, 5376) if args.gemv_shape == "up" else (5376, 21504)
        res["shape"] = {"N": N, "K": K, "B": B}
        mats = [torch.from_numpy(gem_synth.q4_0_matrix(0, 5000 + i, N, K)).cuda()
                for i in range(args.mats)]
        if args.cuda_core:
            # weights 2 bytes off a 16-byte boundary: the library's general CUDA-core kernel (one
            # warp per row, plain loads), the comparison point for the tensor-core path
            def shifted(W):
                buf = torch.empty(W.numel() + 16, dtype=torch.uint8, device="cuda")
                buf[2:2 + W.numel()].copy_(W.reshape(-1))
                return buf[2:2 + W.numel()]
            mats = [shifted(W) for W in mats]
            res["path"] = "cuda-core (general kernel)"
        x = torch.from_numpy(gem_synth.normal_f32(0, 6000, (B, K))).cuda()
        y = torch.empty((B, N), device="cuda")
        ws = torch.empty(max(1, gem.q4_0_gemv_workspace(B, K)), dtype=torch.uint8, device="cuda")

        if B > 8:   # the batched prefill GEMM
            ws = torch.empty(max(1, gem.q4_0_gemm_workspace(B, K)), dtype=torch.uint8, device="cuda")

        def run():
            for W in mats:
                if B > 8:
                    gem.q4_0_gemm(W, None, N, K, x, y, workspace=ws)
                else:
                    gem.q4_0_gemv(W, N, K, x, y, workspace=ws)
        b = gemv_bytes(N, K, B)
        n = len(mats)
    else:
        wl = configs.with_layers(configs.workload(args.workload), args.layers or 2)
        model = Model(gem, torch, wl, distinct=1)
        idx = same_shape_layers(wl)
        fn, b = op_callers(gem, torch, model, idx)[args.op]
        res["op"], res["workload"] = args.op, wl.name
        run = fn
        n = len(idx)
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


def config_of(wl):
    return {"workload": wl.name, "layers": len(wl.layers), "B": wl.B, "n_kv": wl.pos,
            "hidden": wl.layers[0].H, "heads": [wl.layers[0].n_q, wl.layers[0].n_kv],
            "head_dim": wl.layers[0].d, "ffn": wl.layers[0].F, "bytes_per_step": step_bytes(wl),
            "l2": "inputs larger than L2 (%.2f GB streamed per step vs 129 MB L2)" % (step_bytes(wl) / 1e9),
            "parallelism": "single GPU"}


def workload_record(gem, torch, name, reps, peak, distinct):
    """One step of another workload, captured as a CUDA graph and replayed: ms per step,
    us per layer, tokens/s and GB/s over its algorithmic bytes."""
    wl = configs.workload(name)
    model = Model(gem, torch, wl, distinct=distinct)
    g = capture(torch, model.step)
    ms = time_graph(torch, g, reps, warmup=3)
    flags = gem.device_status()
    sb = step_bytes(wl)
    gbs = sb / (ms * 1e-3) / 1e9
    rec = {"layers": len(wl.layers), "B": wl.B, "n_kv": wl.pos, "ms_per_step": round(ms, 4),
           "us_per_layer": round(ms * 1e3 / len(wl.layers), 3), "tok_s": round(wl.B / (ms * 1e-3), 1),
           "gbs": round(gbs, 1), "frac_of_peak": round(gbs / peak, 4), "bytes_per_step": sb,
           "replays": reps, "distinct_draws_per_shape": distinct, "device_flags": flags}
    if len(wl.layers) > 1:
        nL = len(wl.layers)
        rec["note"] = "%d-layer step" % nL
    del g, model
    torch.cuda.empty_cache()
    return rec


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

    peak, peak_kind = measured_peaks()
    wl = configs.workload(args.workload)
    if args.layers:
        wl = configs.with_layers(wl, args.layers)
    model = Model(gem, torch, wl)
    nL = len(wl.layers)
    sbytes = step_bytes(wl)

    g = capture(torch, model.step)
    for _ in range(args.warmup):
        g.replay()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    st = torch.cuda.current_stream()
    clk = Clocks(local, pci_bus_id(torch, local))
    ms = clk.run_timed(torch, g.replay, args.steps, st) / args.steps
    torch.cuda.synchronize()
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

    # per-op roofline: each op of the layer, launched as the chain launches it (same fused
    # kernel), timed alone over every layer shaped like the first (graph, CUDA events)
    idx = same_shape_layers(wl)
    kern = {}
    for name, (fn, b) in op_callers(gem, torch, model, idx).items():
        gg = capture(torch, fn)
        us = time_graph(torch, gg, max(5, min(args.steps, 200))) / len(idx) * 1e3
        kern[name] = {"us": us, "bytes": b, "gbs": b / us / 1e3, "frac": b / us / 1e3 / peak}
        del gg
    dom = max(kern, key=lambda k: kern[k]["us"])
    dk = kern[dom]
    persistent = None
    try:
        plan = gem.StepPlan(model.layers, wl.B, model.kc, model.vc)
        gp = capture(torch, lambda: plan.step(model.x, model.pos))
        ms_p = time_graph(torch, gp, max(5, min(args.steps, 200)))
        persistent = {"ms_per_step": round(ms_p, 4), "us_per_layer": round(ms_p * 1e3 / nL, 3)}
        del gp
        plan.close()
    except gem.GemError as e:
        persistent = {"unsupported": str(e)}
    launches = model.launches_per_step()
    del g, model
    torch.cuda.empty_cache()

    # the 31B FFN projection (5376 -> 21504), 8 distinct matrices (520 MB) rotated
    gemv31 = {}
    W31 = [torch.from_numpy(gem_synth.q4_0_matrix(0, 5000 + i, 21504, 5376)).cuda() for i in range(8)]
    for B in (1, 8):
        x31 = torch.from_numpy(gem_synth.normal_f32(0, 6000, (B, 5376))).cuda()
        y31 = torch.empty((B, 21504), device="cuda")
        ws31 = torch.empty(max(1, gem.q4_0_gemv_workspace(B, 5376)), dtype=torch.uint8, device="cuda")

        def g31(x31=x31, y31=y31, ws31=ws31):
            for W in W31:
                gem.q4_0_gemv(W, 21504, 5376, x31, y31, workspace=ws31)
        gg = capture(torch, g31)
        us = time_graph(torch, gg, max(5, min(args.steps, 200))) / len(W31) * 1e3
        b = gemv_bytes(21504, 5376, B)
        gemv31["b%d" % B] = {"us": round(us, 3), "gbs": round(b / us / 1e3, 1), "frac": round(b / us / 1e3 / peak, 4)}
        del gg
    # the batched prefill GEMM on the same matrices: 16 and 32 prompt rows per call
    prefill = {}
    for M in (16, 32):
        xm = torch.from_numpy(gem_synth.normal_f32(0, 6001, (M, 5376))).cuda()
        ym = torch.empty((M, 21504), device="cuda")
        wsm = torch.empty(max(1, gem.q4_0_gemm_workspace(M, 5376)), dtype=torch.uint8, device="cuda")

        def gm(xm=xm, ym=ym, wsm=wsm):
            for W in W31:
                gem.q4_0_gemm(W, None, 21504, 5376, xm, ym, workspace=wsm)
        gg = capture(torch, gm)
        us = time_graph(torch, gg, max(5, min(args.steps, 200))) / len(W31) * 1e3
        b = gemv_bytes(21504, 5376, M)
        prefill["m%d" % M] = {"us": round(us, 3), "rows_s": round(M / (us * 1e-6), 1),
                              "gbs": round(b / us / 1e3, 1), "frac": round(b / us / 1e3 / peak, 4),
                              "weight_gbs_equiv": round(M * q4_bytes(21504, 5376) / us / 1e3, 1)}
        del gg
    del W31
    torch.cuda.empty_cache()

    # the tied Q8_0 logit projection at the Gemma-4-31B embedding shape (262,144 x 5,376, 1.5 GB)
    # and the device argmax of its logits
    logits = {}
    V, Hl = 262144, 5376
    Wq8 = torch.from_numpy(gem_synth.q8_0_matrix(0, 7000, V, Hl)).cuda()
    for B in (1, 8):
        xl = torch.from_numpy(gem_synth.normal_f32(0, 7001, (B, Hl))).cuda()
        yl = torch.empty((B, V), device="cuda")
        il = torch.empty((B,), dtype=torch.int32, device="cuda")
        aws = torch.empty(max(1, gem.argmax_workspace(B, V)), dtype=torch.uint8, device="cuda")
        gl = capture(torch, lambda xl=xl, yl=yl: gem.q8_0_gemv(Wq8, V, Hl, xl, yl))
        us = time_graph(torch, gl, max(5, min(args.steps, 50))) * 1e3
        ga = capture(torch, lambda yl=yl, il=il, aws=aws: gem.argmax(yl, il, aws))
        us_a = time_graph(torch, ga, max(5, min(args.steps, 200))) * 1e3
        ti = torch.empty((B, 64), dtype=torch.int32, device="cuda")
        tv = torch.empty((B, 64), device="cuda")
        tws = torch.empty(max(1, gem.topk_workspace(B, V, 64)), dtype=torch.uint8, device="cuda")
        gt = capture(torch, lambda yl=yl, ti=ti, tv=tv, tws=tws: gem.topk(yl, 64, ti, tv, tws))
        us_t = time_graph(torch, gt, max(5, min(args.steps, 200))) * 1e3
        b = V * (Hl // 32) * 34 + 4 * B * (Hl + V)
        logits["b%d" % B] = {"us": round(us, 2), "gbs": round(b / us / 1e3, 1), "frac": round(b / us / 1e3 / peak, 4),
                             "argmax_us": round(us_a, 2), "top64_us": round(us_t, 2)}
        del gl, ga, gt
    del Wq8
    torch.cuda.empty_cache()

    # the Gemma 4 31B full-attention layer's attention (32,769 positions, B = 1): standard
    # K + V cache against the compact V-only cache (QK-norm / RoPE / append launch included)
    attn_full = {}
    for cache in ("standard", "compact"):
        run, b, n = attn_full_runner(gem, torch, cache, 1)
        ga = capture(torch, run)
        us = time_graph(torch, ga, max(5, min(args.steps, 100))) / n * 1e3
        attn_full[cache] = {"us": round(us, 2), "bytes": b, "gbs": round(b / us / 1e3, 1),
                            "frac": round(b / us / 1e3 / peak, 4)}
        del ga, run
        torch.cuda.empty_cache()

    # the other workloads' steps
    subs = {}
    if not args.no_workloads and rank == 0:
        reps = max(10, min(args.steps, 100))
        for name, distinct in (("qwen3-4b-b8", 4), ("gemma4-31b-group", 2), ("gemma4-31b-group-compact", 2),
                               ("tiny", 1)):
            if name == wl.name:
                continue
            subs[name] = workload_record(gem, torch, name, reps, peak, distinct)
        subs["tiny"]["note"] = "one 0.4 MB layer: launch-latency bound, reported in us (no roofline)"

    tokens = wl.B * world
    value = whole_job_gbs(sbytes, world, ms)
    if rank == 0:
        cpu = cpu_baseline(wl, args) if world == 1 else None
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded Q4_0 weights, N(0,1) fp16 KV cache and fp32 activations)",
            "config": config_of(wl),
            "tok_s": round(tokens / (ms * 1e-3), 1),
            "us_per_layer": round(ms * 1e3 / nL, 3),
            "frac_of_peak": round(value / world / peak, 4),
            "roofline": {"bound": "hbm", "kernel": dom, "achieved": round(dk["gbs"], 1), "peak": peak,
                         "peak_kind": peak_kind, "unit": "GB/s", "frac": round(dk["frac"], 4),
                         "traffic": traffic_record(dom), "algorithmic_bytes": dk["bytes"],
                         "us_per_launch": round(dk["us"], 3)},
            "kernels": {k: {"us": round(v["us"], 3), "gbs": round(v["gbs"], 1), "frac": round(v["frac"], 4)}
                        for k, v in kern.items()},
            "kernels_how": "each op as the layer chain launches it (same fused kernel), alone over the %d "
                           "layers shaped like the first, CUDA graph, CUDA events" % len(idx),
            "persistent_step_kernel": persistent,
            "gemv_k5376_n21504": gemv31,
            "prefill_gemm_k5376_n21504": prefill,
            "logits_q8_0_k5376_v262144": logits,
            "attn_gemma31_full_p32768": attn_full,
            "workloads": subs,
            "e2e": {"value": round(sbytes / (e2e_ms * 1e-3) / 1e9, 1), "unit": UNIT,
                    "ms_per_step": round(e2e_ms, 4), "wall_ms_per_step": round(e2e_wall_ms, 4),
                    "h2d_bytes_per_step": int(hx.numel() * 4 + hpos.numel() * 4),
                    "d2h_bytes_per_step": int(hout.numel() * 4)},
            "gpu_launches": launches * args.steps,
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
        bytes_done += layer_bytes(s, wl.B, attended(s, wl.pos))["total"]
        done += 1
    return done, bytes_done, t_spent, oracle.num_threads()


def cpu_baseline(wl, args):
    """The oracle as it stands on the host cores: OpenMP over output rows / heads on every
    core, then single-threaded (the same arithmetic; per-row sums are sequential either way)."""
    import oracle
    done, b, t, cores = _oracle_sample(wl, args.cpu_budget * 2 / 3)
    nthreads = oracle.num_threads()
    oracle.set_num_threads(1)
    try:
        d1, b1, t1, _ = _oracle_sample(wl, args.cpu_budget / 3)
    finally:
        oracle.set_num_threads(nthreads)
    return {"value": round(b / t / 1e9, 3), "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": "%d layer steps of %s (its first %d layers in turn; fp64 scalar C, OpenMP over "
                      "rows/heads), %.1f s" % (done, wl.name, min(4, len(wl.layers)), t),
            "ms_per_layer": round(t * 1e3 / done, 1),
            "single_thread": {"value": round(b1 / t1 / 1e9, 3), "unit": UNIT, "cores": 1,
                              "ms_per_layer": round(t1 * 1e3 / d1, 1),
                              "sample": "%d layer steps, %.1f s" % (d1, t1)}}


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
            "config": config_of(wl),
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
                    choices=["tiny", "qwen3-1.7b", "qwen3-4b-b8", "gemma4-31b-group", "gemma4-31b-group-compact"])
    ap.add_argument("--layers", type=int, default=0, help="use only the first n layers")
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle work")
    ap.add_argument("--no-workloads", action="store_true", help="skip the other workloads' sub-records")
    ap.add_argument("--vocab", type=int, default=262144, help="--kernel q8: vocabulary rows")
    ap.add_argument("--kernel", choices=["step", "gemv", "op", "q8", "attn_full", "persistent", "elementwise"], default="step",
                    help="time one op alone (for profiler captures) instead of the step")
    ap.add_argument("--op", default="gqa_decode_attn",
                    choices=["q4_0_gemv_qkv", "gqa_decode_attn", "q4_0_gemv_o", "q4_0_gemv_gate_up",
                             "q4_0_gemv_down"], help="--kernel op: which op of the layer step")
    ap.add_argument("--batch", type=int, default=1,
                    help="--kernel gemv: activation rows (9..32: the batched prefill GEMM)")
    ap.add_argument("--mats", type=int, default=8, help="--kernel gemv: rotated matrices")
    ap.add_argument("--cuda-core", action="store_true",
                    help="--kernel gemv: misaligned weights, so the general CUDA-core kernel runs")
    ap.add_argument("--cache", choices=["standard", "compact"], default="compact",
                    help="--kernel attn_full: the full-attention layer's cache layout")
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
