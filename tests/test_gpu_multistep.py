"""Consecutive decode steps through the C ABI, checked step by step against the oracle (GPU only).

GELO LLM generation, section 05: each decode step attends n_cache + 1 positions, so the row a
step appends to the KV cache is read by every later step.  Inside one stream the layer chain's
kernels are linked by programmatic dependent launch and request cached K/V tiles before they
wait for their predecessor; these tests run S steps back to back in one stream (eagerly, and
as one CUDA graph replayed once), with nothing but the library's own kernels between the
steps, so step s + 1's attention follows step s's append at the shortest launch distance the
chain has.  A stale read of a row appended one step earlier would bring back the cache's
random initial contents there and fail the comparison.

Each step s takes its own input row block X[s] and position vector P[s] = P[0] + s.  After
the run, step s is recomputed by the oracle from X[s] on the cache as it stood before step s
(the initial cache plus the rows the GPU appended at steps < s, themselves checked against
the oracle's rounding of the same values), layer by layer, and compared with the GPU's X[s]
at the tolerances of tests/parity.py (max-abs 2e-3, relative L2 1e-5).  In the two-layer
stacks the O and down projections' block scales are divided by 8 (exactly), so the second
layer's input stays near one layer's output scale and the absolute tolerance keeps its
meaning through the two chained layers."""
from dataclasses import replace

import numpy as np
import pytest

import gem_synth
from gem_synth import configs
from parity import assert_close, scale_q4_0
from test_gpu_parity import _bits, _cu, _half_cache, _oracle_follow_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import q4_gemv_gqa_gb300 as g
    g.device_status(reset=True)
    return g, torch


def _small_swa():
    return replace(configs.GEMMA31_SWA, H=512, n_q=8, n_kv=4, d=64, F=1024, rope_dim=64, window=64)


def _small_full_fused():
    # Gemma-style full-attention layer with V from K, G = 4, d = 128: attention fused with
    # QK-norm / RoPE / append (one launch)
    return replace(configs.GEMMA31_FULL, H=512, n_q=8, n_kv=2, d=128, F=1024, rope_dim=32)


def _small_unfused():
    # G = 8: the separate QK-norm / RoPE / append launch, split attention and merge launch
    return replace(configs.QWEN3_1_7B, H=512, n_q=8, n_kv=1, d=128, F=1024)


CASES = [
    # (name, layer shapes, B, first positions, steps, cache capacity)
    ("tiny-1layer", (configs.TINY,), 1, [128], 4, 136),
    ("qwen3-1.7b-2layers", (configs.QWEN3_1_7B,) * 2, 1, [1024], 4, 1032),
    ("qwen3-1.7b-2layers-b3-ragged", (configs.QWEN3_1_7B,) * 2, 3, [0, 517, 1020], 4, 1032),
    ("swa-ring-wraps", (_small_swa(),) * 2, 2, [62, 126], 4, 64),
    # one layer: with V from the K projection a second chained layer's inputs carry the first
    # layer's fp32 error, which moves more binary16 rounding decisions than the per-layer rule allows
    ("full-v-from-k-fused", (_small_full_fused(),), 1, [300], 4, 310),
    ("unfused-g8", (_small_unfused(),) * 2, 2, [300, 45], 4, 310),
]


def _setup(g, t, shapes, B, cap, seed):
    tens = [configs.layer_tensors(s, B, cap, seed, li) for li, s in enumerate(shapes)]
    if len(shapes) > 1:
        # O and down block scales / 8 (exact): the second layer's input then stays near the
        # first layer's output scale, as in the per-layer checks (see scale_q4_0)
        for tn in tens:
            tn.w_o = scale_q4_0(tn.w_o, 3)
            tn.w_down = scale_q4_0(tn.w_down, 3)
    layers = [g.DeviceLayer(s, tn) for s, tn in zip(shapes, tens)]
    kc = [_half_cache(t, tn.k_cache) for tn in tens]
    vc = [_half_cache(t, tn.v_cache) for tn in tens]
    return tens, layers, kc, vc


def _inputs(t, shapes, B, pos0, S, seed):
    H = shapes[0].H
    xs = np.stack([gem_synth.normal_f32(seed, gem_synth.tid(s, gem_synth.ROLE_X), (B, H)) for s in range(S)])
    ps = np.stack([np.array(pos0, np.int32) + s for s in range(S)]).astype(np.int32)
    return xs, ps, _cu(t, xs), _cu(t, ps)


def _check_steps(shapes, tens, xs, ps, got_x, kc_final, vc_final, what):
    """Recompute every step with the oracle from its own input on the GPU-consistent cache."""
    S = xs.shape[0]
    kstate = [tn.k_cache.copy() for tn in tens]
    vstate = [tn.v_cache.copy() for tn in tens]
    for s in range(S):
        x = xs[s].astype(np.float64)
        for li, (shape, tn) in enumerate(zip(shapes, tens)):
            x = _oracle_follow_gpu(shape, tn, x, ps[s], kstate[li], vstate[li], kc_final[li], vc_final[li],
                                   "%s step %d layer %d" % (what, s, li))
        assert_close(got_x[s], x, "%s step %d" % (what, s))
    # every slot that no step wrote still holds the initial cache
    for li, (shape, tn) in enumerate(zip(shapes, tens)):
        written = np.zeros(kc_final[li].shape[:3], bool)
        for s in range(S):
            for b in range(xs.shape[1]):
                p = int(ps[s][b])
                written[b, :, p % shape.window if shape.window else p] = True
        assert np.array_equal(kc_final[li][~written], tn.k_cache[~written]), "%s layer %d: K slots" % (what, li)
        assert np.array_equal(vc_final[li][~written], tn.v_cache[~written]), "%s layer %d: V slots" % (what, li)


@pytest.mark.parametrize("graph", [False, True], ids=["eager", "graph"])
@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_consecutive_steps_match_oracle(env, case, graph):
    g, t = env
    name, shapes, B, pos0, S, cap = case
    tens, layers, kc, vc = _setup(g, t, shapes, B, cap, 31)
    xs, ps, dX, dP = _inputs(t, shapes, B, pos0, S, 32)
    ws = [t.empty(g.decode_layer_workspace(dl, B, cap), dtype=t.uint8, device="cuda") for dl in layers]
    status = t.zeros(1, dtype=t.int32, device="cuda")

    def run():
        for s in range(S):
            for dl, k, v, w in zip(layers, kc, vc, ws):
                g.decode_layer(dl, dX[s], k, v, dP[s], w, status=status)

    if graph:
        # warm-up outside the capture on copies (kernel attributes are set on first use)
        kw = [k.clone() for k in kc]
        vw = [v.clone() for v in vc]
        xw = dX.clone()
        for dl, k, v, w in zip(layers, kw, vw, ws):
            g.decode_layer(dl, xw[0], k, v, dP[0], w)
        t.cuda.synchronize()
        gr = t.cuda.CUDAGraph()
        st = t.cuda.Stream()
        with t.cuda.stream(st):
            with t.cuda.graph(gr, stream=st):
                run()
        gr.replay()
    else:
        run()
    t.cuda.synchronize()
    assert int(status.item()) == 0
    _check_steps(shapes, tens, xs, ps, dX.cpu().numpy(), [_bits(k) for k in kc], [_bits(v) for v in vc],
                 "%s (%s)" % (name, "graph" if graph else "eager"))


STEP_PLAN_CASES = [c for c in CASES if c[0] in ("tiny-1layer", "qwen3-1.7b-2layers", "qwen3-1.7b-2layers-b3-ragged")]


@pytest.mark.parametrize("case", STEP_PLAN_CASES, ids=[c[0] for c in STEP_PLAN_CASES])
def test_consecutive_persistent_steps_match_oracle(env, case):
    """The same steps through gem_decode_step (one persistent launch per step)."""
    g, t = env
    name, shapes, B, pos0, S, cap = case
    tens, layers, kc, vc = _setup(g, t, shapes, B, cap, 41)
    xs, ps, dX, dP = _inputs(t, shapes, B, pos0, S, 42)
    plan = g.StepPlan(layers, B, kc, vc)
    status = t.zeros(1, dtype=t.int32, device="cuda")
    for s in range(S):
        plan.step(dX[s], dP[s], status=status)
    t.cuda.synchronize()
    assert int(status.item()) == 0
    _check_steps(shapes, tens, xs, ps, dX.cpu().numpy(), [_bits(k) for k in kc], [_bits(v) for v in vc],
                 "%s (persistent)" % name)
    plan.close()
