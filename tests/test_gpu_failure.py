"""Failure detection without a GPU fault (GPU only).

Every device-side wait of the library is bounded (gem_set_wait_limit).  These tests make one
wait run out on purpose through the library's test hooks (gem_set_test_injection), with a
1 ms limit: a ring stage of the one-row GEMV that expects 16 bytes more than it receives, and
a grid barrier of the persistent step kernel that one CTA never arrives at.  Nothing waits
forever and nothing traps: each kernel gives up after the limit, lets its copies land
(bounded), records GEM_DEVFLAG_TIMEOUT and leaves.  The tests check the flag, the status it
maps to (GEM_ERR_TIMEOUT), and that the same process then runs the same call correctly."""
import numpy as np
import pytest

import gem_synth
import oracle
from gem_synth import configs
from parity import assert_close
from test_gpu_parity import _bits, _cu, _half_cache, _layer_parity

pytestmark = pytest.mark.gpu

GEM_ERR_TIMEOUT = 6


@pytest.fixture(scope="module")
def env():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import q4_gemv_gqa_gb300 as g
    torch.cuda.synchronize()
    g.device_status(reset=True)
    return g, torch


def _injected(g, t, mask, fn):
    t.cuda.synchronize()
    g.set_wait_limit(1_000_000)   # 1 ms
    g.set_test_injection(mask)
    try:
        fn()
        t.cuda.synchronize()
    finally:
        g.set_test_injection(0)
        g.set_wait_limit(0)


def test_ring_wait_runs_out_and_reports_timeout(env):
    g, t = env
    N, K = 16, 256   # one CTA, one stage: the short stage is the ring's last
    W = gem_synth.q4_0_matrix(3, 300, N, K)
    x = gem_synth.normal_f32(3, 301, (1, K))
    dW, dx = _cu(t, W), _cu(t, x)
    y = t.full((1, N), float("nan"), device="cuda")
    g.device_status(reset=True)
    _injected(g, t, g.INJECT_RING_SHORTFALL, lambda: g.q4_0_gemv(dW, N, K, dx, y))
    flags = g.device_status(reset=True)
    assert flags & g.DEVFLAG_TIMEOUT, "the short stage's wait did not report"
    assert g.status_from_flags(flags) == GEM_ERR_TIMEOUT
    # the device answers normally afterwards: the same call, checked against the oracle
    y2 = t.full((1, N), float("nan"), device="cuda")
    g.q4_0_gemv(dW, N, K, dx, y2)
    t.cuda.synchronize()
    assert_close(y2.cpu().numpy(), oracle.q4_0_gemv(W, N, K, x), "GEMV after the timeout")
    assert g.device_status() == 0


def test_grid_barrier_runs_out_and_aborts_the_step(env):
    g, t = env
    shape, B, pos_l = configs.TINY, 1, [128]
    pos = np.array(pos_l, np.int32)
    cap = 136
    tens = configs.layer_tensors(shape, B, cap, 0, 0)
    x = gem_synth.normal_f32(0, gem_synth.tid(0, gem_synth.ROLE_X), (B, shape.H))
    dl = g.DeviceLayer(shape, tens)
    dk, dv = _half_cache(t, tens.k_cache), _half_cache(t, tens.v_cache)
    status = t.zeros(1, dtype=t.int32, device="cuda")
    plan = g.StepPlan([dl], B, [dk], [dv])
    dx = _cu(t, x)
    _injected(g, t, g.INJECT_GRID_ARRIVAL, lambda: plan.step(dx, _cu(t, pos), status=status))
    flags = int(status.item())
    assert flags & g.DEVFLAG_TIMEOUT, "the barrier wait did not report"
    assert g.status_from_flags(flags) == GEM_ERR_TIMEOUT
    plan.close()   # an aborted plan is not reused
    # a fresh plan on fresh caches runs the step correctly
    dk2, dv2 = _half_cache(t, tens.k_cache), _half_cache(t, tens.v_cache)
    plan2 = g.StepPlan([dl], B, [dk2], [dv2])
    dx2 = _cu(t, x)
    status.zero_()
    plan2.step(dx2, _cu(t, pos), status=status)
    t.cuda.synchronize()
    assert int(status.item()) == 0
    _layer_parity(shape, tens, x, pos, dx2.cpu().numpy(), _bits(dk2), _bits(dv2), "step after the timeout")
    plan2.close()
    assert g.device_status(reset=True) == 0


def test_gemv_workspace_calls_on_two_streams(env):
    """gem_q4_0_gemv_ws with a workspace per call: two 8-row GEMVs on two streams at once."""
    g, t = env
    N, K, B = 6144, 2048, 8
    Ws = [gem_synth.q4_0_matrix(4, 400 + i, N, K) for i in range(2)]
    xs = [gem_synth.normal_f32(4, 410 + i, (B, K)) for i in range(2)]
    dWs, dxs = [_cu(t, W) for W in Ws], [_cu(t, x) for x in xs]
    ys = [t.full((B, N), float("nan"), device="cuda") for _ in range(2)]
    need = g.q4_0_gemv_workspace(B, K)
    assert need > 0
    wss = [t.empty(need, dtype=t.uint8, device="cuda") for _ in range(2)]
    streams = [t.cuda.Stream() for _ in range(2)]
    t.cuda.synchronize()
    for _ in range(3):   # several rounds so the two streams' launches interleave
        for i in range(2):
            with t.cuda.stream(streams[i]):
                g.q4_0_gemv(dWs[i], N, K, dxs[i], ys[i], workspace=wss[i])
    t.cuda.synchronize()
    for i in range(2):
        assert_close(ys[i].cpu().numpy(), oracle.q4_0_gemv(Ws[i], N, K, xs[i]), "stream %d GEMV" % i)
    # a workspace smaller than the query is rejected before anything is launched
    with pytest.raises(g.GemError) as ei:
        g.q4_0_gemv(dWs[0], N, K, dxs[0], ys[0], workspace=wss[0][: need - 256])
    assert ei.value.status == 7   # GEM_ERR_WORKSPACE
