"""gem_gqa_decode_attn_noalloc (split partials in the library's own per-device array) against
gem_gqa_decode_attn with a caller-allocated workspace, through the C ABI (GPU only).

The file name sorts last so that the shared array is exercised after every other test has
run on the same device; the tests pass alone as well.  Tolerance is that of tests/parity.py;
both entry points run the same kernels with the same split plan, so the outputs are also
expected to be bit-identical."""
import numpy as np
import pytest

import gem_synth
from parity import assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import q4_gemv_gqa_gb300 as g
    g.device_status(reset=True)
    return g, torch


def _inputs(t, seed, n_q, n_kv, d, pos_l, cap):
    B = len(pos_l)
    q = t.from_numpy(gem_synth.normal_f32(seed, 1, (B, n_q * d))).cuda()
    kc = t.from_numpy(gem_synth.normal_f16_bits(seed, 2, (B, n_kv, cap, d)).view(np.int16)).cuda()
    vc = t.from_numpy(gem_synth.normal_f16_bits(seed, 3, (B, n_kv, cap, d)).view(np.int16)).cuda()
    pos = t.from_numpy(np.array(pos_l, np.int32)).cuda()
    return q, kc, vc, pos


def _with_workspace(g, t, q, kc, vc, pos, n_q, n_kv, d, window, scale):
    B, cap = q.shape[0], kc.shape[2]
    need = g.gqa_decode_attn_workspace(B, n_q, n_kv, d, cap, window)
    ws = t.empty(max(need, 1), dtype=t.uint8, device="cuda")
    out = t.full((B, n_q * d), float("nan"), device="cuda")
    g.gqa_decode_attn(q, kc, vc, n_q, n_kv, d, pos, window, scale, out, ws if need else None)
    return out


CASES = [
    # (n_q, n_kv, d, window, positions, cap, scale)
    (16, 8, 128, 0, [4096], 4097, 128 ** -0.5),                          # Qwen3-1.7B shape
    (32, 8, 128, 0, [0, 1, 63, 64, 65, 700, 1500, 2048], 2049, 128 ** -0.5),  # B = 8, ragged
    (32, 16, 256, 1024, [32768], 1024, 1.0),                             # Gemma SWA ring
    (32, 4, 512, 0, [32768], 32769, 1.0),                                # Gemma full attention
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "G%d_d%d_w%d_B%d" % (c[0] // c[1], c[2], c[3], len(c[4])))
def test_noalloc_matches_workspace_entry_two_calls_in_a_row(env, case):
    g, t = env
    n_q, n_kv, d, window, pos_l, cap, scale = case
    B = len(pos_l)
    assert g.gqa_decode_attn_workspace(B, n_q, n_kv, d, cap, window) <= g.NOALLOC_SCRATCH_BYTES
    q1, kc, vc, pos1 = _inputs(t, 21, n_q, n_kv, d, pos_l, cap)
    q2 = t.from_numpy(gem_synth.normal_f32(22, 1, (B, n_q * d))).cuda()
    pos2 = t.from_numpy(np.array([max(0, p - 37) for p in pos_l], np.int32)).cuda()
    ref1 = _with_workspace(g, t, q1, kc, vc, pos1, n_q, n_kv, d, window, scale)
    ref2 = _with_workspace(g, t, q2, kc, vc, pos2, n_q, n_kv, d, window, scale)
    # two calls back to back on one stream, different queries and positions, same array
    o1 = t.full((B, n_q * d), float("nan"), device="cuda")
    o2 = t.full((B, n_q * d), float("nan"), device="cuda")
    g.gqa_decode_attn_noalloc(q1, kc, vc, n_q, n_kv, d, pos1, window, scale, o1)
    g.gqa_decode_attn_noalloc(q2, kc, vc, n_q, n_kv, d, pos2, window, scale, o2)
    t.cuda.synchronize()
    assert_close(o1.cpu().numpy(), ref1.cpu().numpy(), "noalloc call 1 vs workspace entry")
    assert_close(o2.cpu().numpy(), ref2.cpu().numpy(), "noalloc call 2 vs workspace entry")
    assert t.equal(o1, ref1) and t.equal(o2, ref2)
    assert g.device_status() == 0


def test_noalloc_rejects_shape_beyond_scratch(env):
    g, t = env
    # the Gemma 4 31B full-attention layer at B = 8: each split covers at most 1024 positions, so
    # 32,769 positions take 33 splits, 8 x 32 x 33 x 514 floats = 17.4 MB of partials
    n_q, n_kv, d, cap, B = 32, 4, 512, 32769, 8
    need = g.gqa_decode_attn_workspace(B, n_q, n_kv, d, cap, 0)
    if need <= g.NOALLOC_SCRATCH_BYTES:
        pytest.skip("this device's split plan fits the shape into the scratch array")
    q = t.zeros((B, n_q * d), device="cuda")
    kc = t.zeros((B, n_kv, cap, d), dtype=t.int16, device="cuda")
    pos = t.full((B,), cap - 1, dtype=t.int32, device="cuda")
    out = t.full((B, n_q * d), float("nan"), device="cuda")
    with pytest.raises(g.GemError) as ei:
        g.gqa_decode_attn_noalloc(q, kc, kc, n_q, n_kv, d, pos, 0, 1.0, out)
    assert ei.value.status == 7  # GEM_ERR_WORKSPACE
    t.cuda.synchronize()
    assert bool(t.isnan(out).all()), "a rejected call must launch nothing"
