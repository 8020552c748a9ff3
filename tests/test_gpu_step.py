"""The persistent whole-step kernel (gem_step_plan / gem_decode_step) on the GPU.

A one-layer step is compared with the fp64 oracle exactly as the per-layer chain is (same
tolerances and binary16 rounding-band rule, tests/test_gpu_parity.py); a stack of layers is
compared with the oracle run layer by layer at the same tolerances, and with itself across
repeated calls."""
from dataclasses import replace

import numpy as np
import pytest

import gem_synth
from gem_synth import configs
from parity import assert_close, scale_q4_0
from test_gpu_parity import _bits, _cu, _half_cache, _layer_parity, _oracle_follow_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import q4_gemv_gqa_gb300 as g
    g.device_status(reset=True)
    return g, torch


STEP_CASES = [
    ("tiny", configs.TINY, 1, [128]),
    ("tiny-b2-ring", replace(configs.TINY, window=64), 2, [200, 30]),
    ("qwen3-1.7b", configs.QWEN3_1_7B, 1, [4096]),
    ("qwen3-4b-ragged", configs.QWEN3_4B, 3, [0, 1000, 2048]),
    ("qwen3-4b-b4", configs.QWEN3_4B, 4, [2048] * 4),
]


@pytest.mark.parametrize("name,shape,B,pos_l", STEP_CASES, ids=[c[0] for c in STEP_CASES])
def test_step_single_layer_matches_oracle(env, name, shape, B, pos_l):
    g, t = env
    pos = np.array(pos_l, np.int32)
    cap = shape.window if shape.window else int(pos.max()) + 1
    tens = configs.layer_tensors(shape, B, cap, 0, 0)
    x = gem_synth.normal_f32(0, gem_synth.tid(0, gem_synth.ROLE_X), (B, shape.H))
    dl = g.DeviceLayer(shape, tens)
    dk, dv = _half_cache(t, tens.k_cache), _half_cache(t, tens.v_cache)
    plan = g.StepPlan([dl], B, [dk], [dv])
    dx = _cu(t, x.astype(np.float32))
    status = t.zeros(1, dtype=t.int32, device="cuda")
    plan.step(dx, _cu(t, pos), status=status)
    t.cuda.synchronize()
    assert int(status.item()) == 0
    _layer_parity(shape, tens, x, pos, dx.cpu().numpy(), _bits(dk), _bits(dv), "step %s" % name)
    plan.close()


def _stack(g, t, wl, seed):
    layers, kcs, vcs, tens_l = [], [], [], []
    for li, (shape, cap) in enumerate(zip(wl.layers, wl.cache_cap)):
        tens = configs.layer_tensors(shape, wl.B, cap, seed, li)
        layers.append(g.DeviceLayer(shape, tens))
        kcs.append(tens.k_cache)
        vcs.append(tens.v_cache)
    return layers, kcs, vcs


def test_step_stack_matches_oracle(env):
    """Four layers in one persistent launch against the oracle run layer by layer (following
    the GPU's binary16 rounding of each appended row where it is ambiguous), at the stated
    tolerance.  The O and down projections' block scales are divided by 8 (exactly), which
    keeps this stack's residual stream near the scale of one layer's output; with the
    unscaled synthetic weights it grows to ~1e4 after four layers, where fp32 rounding of the
    residual alone approaches the absolute bound."""
    g, t = env
    wl = configs.with_layers(configs.workload("qwen3-1.7b"), 4)
    wl = replace(wl, pos=1024, cache_cap=(1025,) * 4)
    pos = np.full(wl.B, wl.pos, np.int32)
    tens_l, layers = [], []
    for li, (shape, cap) in enumerate(zip(wl.layers, wl.cache_cap)):
        tn = configs.layer_tensors(shape, wl.B, cap, 5, li)
        tn.w_o = scale_q4_0(tn.w_o, 3)
        tn.w_down = scale_q4_0(tn.w_down, 3)
        tens_l.append(tn)
        layers.append(g.DeviceLayer(shape, tn))
    x0 = gem_synth.normal_f32(0, gem_synth.tid(0, gem_synth.ROLE_X), (wl.B, wl.layers[0].H))
    kc = [_half_cache(t, tn.k_cache) for tn in tens_l]
    vc = [_half_cache(t, tn.v_cache) for tn in tens_l]
    plan = g.StepPlan(layers, wl.B, kc, vc)
    xs = _cu(t, x0)
    status = t.zeros(1, dtype=t.int32, device="cuda")
    plan.step(xs, _cu(t, pos), status=status)
    t.cuda.synchronize()
    assert int(status.item()) == 0
    x = x0.astype(np.float64)
    for li, (shape, tn) in enumerate(zip(wl.layers, tens_l)):
        x = _oracle_follow_gpu(shape, tn, x, pos, tn.k_cache.copy(), tn.v_cache.copy(), _bits(kc[li]),
                               _bits(vc[li]), "step layer %d" % li)
    assert float(np.abs(x).max()) < 2048, "the scaled stack's residual stream is larger than intended"
    assert_close(xs.cpu().numpy(), x, "persistent step, 4 layers, vs oracle")
    plan.close()


def test_step_repeat_is_deterministic(env):
    g, t = env
    wl = configs.with_layers(configs.workload("qwen3-1.7b"), 2)
    layers, kcs, vcs = _stack(g, t, wl, 6)
    pos = _cu(t, np.full(wl.B, wl.pos, np.int32))
    x0 = gem_synth.normal_f32(0, gem_synth.tid(0, gem_synth.ROLE_X), (wl.B, wl.layers[0].H))
    kc = [_half_cache(t, k) for k in kcs]
    vc = [_half_cache(t, v) for v in vcs]
    plan = g.StepPlan(layers, wl.B, kc, vc)
    outs = []
    for _ in range(3):
        xs = _cu(t, x0)
        plan.step(xs, pos)
        outs.append(xs)
    t.cuda.synchronize()
    assert t.equal(outs[0], outs[1]) and t.equal(outs[1], outs[2])
    assert g.device_status() == 0
    plan.close()


def test_step_rejects_unsupported_layers(env):
    g, t = env
    shape = configs.GEMMA31_SWA   # post-attention / post-FFN norms: per-layer chain only
    small = replace(shape, H=512, n_q=8, n_kv=4, d=64, F=1024, rope_dim=64, window=64)
    tens = configs.layer_tensors(small, 1, 64, 0, 0)
    dl = g.DeviceLayer(small, tens)
    dk, dv = _half_cache(t, tens.k_cache), _half_cache(t, tens.v_cache)
    with pytest.raises(g.GemError) as ei:
        g.StepPlan([dl], 1, [dk], [dv])
    assert ei.value.status == 3   # GEM_ERR_UNSUPPORTED_SHAPE
