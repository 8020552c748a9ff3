"""The persistent whole-step kernel (gem_step_plan / gem_decode_step) on the GPU.

A one-layer step is compared with the fp64 oracle exactly as the per-layer chain is (same
tolerances and binary16 rounding-band rule, tests/test_gpu_parity.py); a stack of layers is
compared with the per-layer chain (gem_decode_layer, itself checked against the oracle)
within the same tolerance, and with itself across repeated calls."""
from dataclasses import replace

import numpy as np
import pytest

import gem_synth
from gem_synth import configs
from parity import assert_close
from test_gpu_parity import _bits, _cu, _half_cache, _layer_parity

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


def test_step_stack_matches_layer_chain(env):
    g, t = env
    wl = configs.with_layers(configs.workload("qwen3-1.7b"), 4)
    wl = replace(wl, pos=1024, cache_cap=(1025,) * 4)
    layers, kcs, vcs = _stack(g, t, wl, 5)
    pos = _cu(t, np.full(wl.B, wl.pos, np.int32))
    x0 = gem_synth.normal_f32(0, gem_synth.tid(0, gem_synth.ROLE_X), (wl.B, wl.layers[0].H))
    # per-layer chain
    xc = _cu(t, x0)
    kc_c = [_half_cache(t, k) for k in kcs]
    vc_c = [_half_cache(t, v) for v in vcs]
    for dl, k, v, cap in zip(layers, kc_c, vc_c, wl.cache_cap):
        ws = t.empty(g.decode_layer_workspace(dl, wl.B, cap), dtype=t.uint8, device="cuda")
        g.decode_layer(dl, xc, k, v, pos, ws)
    # one persistent launch
    xs = _cu(t, x0)
    kc_s = [_half_cache(t, k) for k in kcs]
    vc_s = [_half_cache(t, v) for v in vcs]
    plan = g.StepPlan(layers, wl.B, kc_s, vc_s)
    status = t.zeros(1, dtype=t.int32, device="cuda")
    plan.step(xs, pos, status=status)
    t.cuda.synchronize()
    assert int(status.item()) == 0
    # Both sides are fp32 with different summation orders; after four random-weight layers
    # the residual stream reaches ~1e4, where one fp32 unit is ~1e-3, so the absolute bound
    # grows with the output scale (8 units at the largest magnitude).
    ref = xc.cpu().numpy()
    assert_close(xs.cpu().numpy(), ref, "step vs chain, 4 layers",
                 max_abs=2e-3 + 8 * 2.0 ** -23 * float(np.abs(ref).max()))
    slot = wl.pos
    for li in range(4):
        a, b = _bits(kc_s[li]), _bits(kc_c[li])
        mask = np.ones(a.shape[2], bool)
        mask[slot] = False
        assert np.array_equal(a[:, :, mask], b[:, :, mask]), "layer %d: K rows other than the new one" % li
        assert np.array_equal(_bits(vc_s[li])[:, :, mask], _bits(vc_c[li])[:, :, mask])
        # the new rows: binary16 of (nearly) the same fp32 values; at most one unit apart
        for new_a, new_b in ((a[:, :, slot], b[:, :, slot]), (_bits(vc_s[li])[:, :, slot], _bits(vc_c[li])[:, :, slot])):
            d = np.abs(new_a.astype(np.int32) - new_b.astype(np.int32))
            assert int(d.max()) <= 1 and int((d > 0).sum()) <= max(2, new_a.size // 100), "layer %d new row" % li
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
