"""The compact full-attention cache (V rows only) against the oracle (GPU only).

"gem" research record, "Verified model facts": on a Gemma 4 full-attention layer V is the
unweighted RMSNorm of the K projection and K the same row times key_norm, then RoPE, so the
cache can keep V alone and rebuild K_j = RoPE_j(V_j * gamma_k) inside the attention (the
reading of the rotation is the oracle's: each rebuilt row is rotated at its own position).

  - gem_gqa_decode_attn_compact is compared element by element with
    oracle.gqa_attention_compact on the same seeded caches, over every head_dim, group sizes
    1..8, rope_dim from 0 to d, ragged batches, one cached position, and the Gemma 4 31B
    full-attention shape at 32,769 positions;
  - the V-only append of gem_rmsnorm_qknorm_rope (k_cache NULL) and its rejections;
  - gem_decode_layer with compact_kv against oracle.decode_layer on a compact layer: a small
    layer, the full-size Gemma 4 31B full-attention layer, and consecutive steps run back to
    back in one stream (each step's appended V row read by the next step's attention).
Tolerances are tests/parity.py's (max-abs 2e-3, relative L2 1e-5).  Appended binary16 codes
follow the rule of tests/test_gpu_parity.py: a code may differ from the oracle's only where
the value lies within the fp32 arithmetic's precision of a binary16 midpoint, and the layer
output is then compared with the oracle evaluated for that same rounding outcome."""
from dataclasses import replace

import numpy as np
import pytest

import gem_synth
import oracle
from gem_synth import configs
from parity import assert_close
from test_gpu_parity import _bits, _code_in_band, _cu, _half_cache

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import q4_gemv_gqa_gb300 as g
    g.device_status(reset=True)
    return g, torch


def _gamma(seed, d):
    return (1.0 + 0.25 * gem_synth.normal_f32(seed, 77, (d,))).astype(np.float32)


ATTN_CASES = [
    # (n_q, n_kv, d, rope_dim, positions, cap, scale, theta)
    (4, 2, 64, 64, [128], 129, 0.125, 10000.0),            # every dim rotated
    (4, 4, 64, 16, [0], 1, 0.125, 10000.0),                 # one cached position: output = V
    (8, 1, 64, 32, [15], 16, 0.125, 10000.0),               # G = 8
    (16, 8, 128, 128, [4096], 4097, 128 ** -0.5, 1e6),
    (32, 8, 128, 64, [0, 1, 63, 64, 65, 700, 1500, 2048], 2049, 128 ** -0.5, 1e6),  # ragged
    (6, 2, 256, 0, [5000], 5001, 0.0625, 10000.0),          # no rotation: K = V * gamma_k
    (16, 4, 256, 256, [3000], 3001, 0.0625, 1e6),
    (32, 4, 512, 128, [32768], 32769, 1.0, 1e6),            # Gemma 4 31B full-attention layer
    (32, 4, 512, 128, [5, 20000], 32769, 1.0, 1e6),         # a short and a long sequence
]


@pytest.mark.parametrize("case", ATTN_CASES,
                         ids=lambda c: "G%d_d%d_R%d_p%d_B%d" % (c[0] // c[1], c[2], c[3], max(c[4]), len(c[4])))
def test_compact_attention_matches_oracle(env, case):
    g, t = env
    n_q, n_kv, d, R, pos_l, cap, scale, theta = case
    B = len(pos_l)
    q = gem_synth.normal_f32(31, d, (B, n_q * d))
    vc = gem_synth.normal_f16_bits(31, 2, (B, n_kv, cap, d))
    gk = _gamma(31, d)
    pos = np.array(pos_l, np.int32)
    ws_bytes = g.gqa_decode_attn_compact_workspace(B, n_q, n_kv, d, cap, R)
    ws = t.empty(max(ws_bytes, 1), dtype=t.uint8, device="cuda")
    out = t.full((B, n_q * d), float("nan"), device="cuda")
    g.gqa_decode_attn_compact(_cu(t, q), _half_cache(t, vc), n_q, n_kv, d, _cu(t, pos), scale, _cu(t, gk), R,
                              theta, out, ws if ws_bytes else None)
    t.cuda.synchronize()
    got = out.cpu().numpy()
    for b in range(B):
        ref = oracle.gqa_attention_compact(q[b].reshape(n_q, d), vc[b], gk, int(pos[b]), R, theta, scale)
        assert_close(got[b], ref.reshape(-1), "compact attention b=%d p=%d" % (b, pos[b]))
    assert g.device_status() == 0


def test_compact_attention_deterministic(env):
    g, t = env
    n_q, n_kv, d, R, cap = 32, 4, 512, 128, 32769
    q = _cu(t, gem_synth.normal_f32(32, 1, (1, n_q * d)))
    vc = _half_cache(t, gem_synth.normal_f16_bits(32, 2, (1, n_kv, cap, d)))
    gk = _cu(t, _gamma(32, d))
    pos = _cu(t, np.array([32768], np.int32))
    ws = t.empty(max(g.gqa_decode_attn_compact_workspace(1, n_q, n_kv, d, cap, R), 1), dtype=t.uint8, device="cuda")
    outs = []
    for _ in range(5):
        out = t.empty((1, n_q * d), device="cuda")
        g.gqa_decode_attn_compact(q, vc, n_q, n_kv, d, pos, 1.0, gk, R, 1e6, out, ws)
        outs.append(out)
    t.cuda.synchronize()
    for o in outs[1:]:
        assert t.equal(o, outs[0])


def test_compact_attention_rejections(env):
    g, t = env
    n_q, n_kv, d, cap = 8, 2, 128, 64
    q = t.zeros((1, n_q * d), device="cuda")
    vc = t.zeros((1, n_kv, cap, d), dtype=t.int16, device="cuda")
    gk = t.ones(d, device="cuda")
    pos = t.tensor([10], dtype=t.int32, device="cuda")
    out = t.zeros((1, n_q * d), device="cuda")
    with pytest.raises(g.GemError) as ei:   # rope_dim not a multiple of 16
        g.gqa_decode_attn_compact(q, vc, n_q, n_kv, d, pos, 1.0, gk, 24, 1e4, out)
    assert ei.value.status == 3
    with pytest.raises(g.GemError) as ei:   # head_dim 96
        g.gqa_decode_attn_compact(t.zeros((1, n_q * 96), device="cuda"),
                                  t.zeros((1, n_kv, cap, 96), dtype=t.int16, device="cuda"), n_q, n_kv, 96,
                                  pos, 1.0, t.ones(96, device="cuda"), 32, 1e4, t.zeros((1, n_q * 96), device="cuda"))
    assert ei.value.status == 3
    # a long cache is split: the call needs the workspace
    cap2 = 32769
    assert g.gqa_decode_attn_compact_workspace(1, 32, 4, 512, cap2, 128) > 0
    with pytest.raises(g.GemError) as ei:
        g.gqa_decode_attn_compact(t.zeros((1, 32 * 512), device="cuda"),
                                  t.zeros((1, 4, cap2, 512), dtype=t.int16, device="cuda"), 32, 4, 512,
                                  t.tensor([cap2 - 1], dtype=t.int32, device="cuda"), 1.0,
                                  t.ones(512, device="cuda"), 128, 1e6, t.zeros((1, 32 * 512), device="cuda"))
    assert ei.value.status == 7   # GEM_ERR_WORKSPACE
    # a position outside the cache is flagged on the device and nothing is written
    status = t.zeros(1, dtype=t.int32, device="cuda")
    out.fill_(7.0)
    g.gqa_decode_attn_compact(q, vc, n_q, n_kv, d, t.tensor([cap], dtype=t.int32, device="cuda"), 1.0, gk, 32,
                              1e4, out, status=status)
    t.cuda.synchronize()
    assert int(status.item()) & g.DEVFLAG_POS_RANGE
    assert bool((out == 7.0).all())


def test_v_only_append(env):
    """rmsnorm_qknorm_rope with k_cache None and v_mode 1 writes the V row alone."""
    g, t = env
    B, n_q, n_kv, d, R, cap = 2, 8, 2, 128, 32, 64
    qkv = gem_synth.normal_f32(33, 1, (B, (n_q + n_kv) * d))
    gq, gk = _gamma(33, d), _gamma(34, d)
    pos = np.array([5, 63], np.int32)
    vc0 = gem_synth.normal_f16_bits(33, 2, (B, n_kv, cap, d))
    dq = _cu(t, qkv)
    dv = _half_cache(t, vc0)
    g.rmsnorm_qknorm_rope(dq, n_q, n_kv, d, _cu(t, gq), _cu(t, gk), 1, 1e-6, _cu(t, pos), 1e6, R, None, dv)
    t.cuda.synchronize()
    got_v = _bits(dv)
    got_q = dq.cpu().numpy()
    for b in range(B):
        p = int(pos[b])
        for j in range(n_kv):
            raw = qkv[b, (n_q + j) * d:(n_q + j + 1) * d].astype(np.float64)
            v = oracle.rmsnorm(raw, None, 1e-6)
            want = np.array([oracle.double_to_half_via_f32(x) for x in v], np.uint16)
            rms = float(np.sqrt(np.mean(v ** 2)))
            diff = np.nonzero(got_v[b, j, p] != want)[0]
            for i in diff:
                assert _code_in_band(int(got_v[b, j, p, i]), v[i], rms)
            assert len(diff) <= 2
            k = oracle.rope_neox(oracle.rmsnorm(raw, gk, 1e-6), R, p, 1e6)
            assert_close(got_q[b, (n_q + j) * d:(n_q + j + 1) * d], k, "rotated K b=%d j=%d" % (b, j))
        mask = np.ones(cap, bool)
        mask[p] = False
        assert np.array_equal(got_v[b][:, mask], vc0[b][:, mask])
    with pytest.raises(g.GemError):   # v_mode 0 needs both caches
        g.rmsnorm_qknorm_rope(dq, n_q, n_kv, d, None, None, 0, 1e-6, _cu(t, pos), 1e6, R, None, dv)


# ---- the layer step --------------------------------------------------------------------------

def _small_compact():
    return replace(configs.GEMMA31_FULL_COMPACT, H=512, n_q=8, n_kv=2, d=128, F=1024, rope_dim=32)


def _weights(shape, B, cap, seed):
    tens = configs.layer_weights(shape, seed, 0)
    _, vc = configs.kv_cache(shape, B, cap, seed, 0)
    return tens, vc


def _oracle_following(shape, tens, x, pos, v_before, gv, what):
    """The oracle's step from x on v_before, following the GPU's binary16 rounding of the
    appended V rows (gv: the GPU's cache after the step) where they are ambiguous."""
    xin = np.ascontiguousarray(x, dtype=np.float64)
    vc = v_before.copy()
    ref, kvn = oracle.decode_layer(shape, tens, xin, pos, None, vc, kvnew=True)
    B, n_kv, d = len(pos), shape.n_kv, shape.d
    flip = np.zeros((B, 2, n_kv, d), np.int8)
    for b in range(B):
        p = int(pos[b])
        gg, o = gv[b, :, p], vc[b, :, p]
        for j, i in np.argwhere(gg != o):
            v = kvn[b, 1, j, i]
            rms = float(np.sqrt(np.mean(kvn[b, 1, j] ** 2)))
            assert _code_in_band(int(gg[j, i]), v, rms), "%s: appended code outside the precision band" % what
            if gg[j, i] == oracle.other_half_via_f32(v):
                flip[b, 1, j, i] = 1
    nflip = int(flip.sum())
    assert nflip <= max(2, 0.01 * flip.size), "%s: %d rounding decisions differ" % (what, nflip)
    if nflip:
        ref = oracle.decode_layer(shape, tens, xin, pos, None, v_before.copy(), flip=flip)
    return ref


@pytest.mark.parametrize("name,shape,B,pos_l", [
    ("small", _small_compact(), 2, [300, 17]),
    ("gemma4-31b-full-compact", configs.GEMMA31_FULL_COMPACT, 1, [32768]),
], ids=["small", "gemma4-31b-full-compact"])
def test_compact_layer_matches_oracle(env, name, shape, B, pos_l):
    g, t = env
    pos = np.array(pos_l, np.int32)
    cap = int(pos.max()) + 1
    tens, vc = _weights(shape, B, cap, 5)
    x = gem_synth.normal_f32(5, gem_synth.tid(0, gem_synth.ROLE_X), (B, shape.H))
    dl = g.DeviceLayer(shape, tens)
    dx = _cu(t, x)
    dv = _half_cache(t, vc)
    ws = t.empty(g.decode_layer_workspace(dl, B, cap), dtype=t.uint8, device="cuda")
    status = t.zeros(1, dtype=t.int32, device="cuda")
    g.decode_layer(dl, dx, None, dv, _cu(t, pos), ws, status=status)
    t.cuda.synchronize()
    assert int(status.item()) == 0
    gv = _bits(dv)
    for b in range(B):
        mask = np.ones(cap, bool)
        mask[int(pos[b])] = False
        assert np.array_equal(gv[b][:, mask], vc[b][:, mask]), "other V slots changed"
    ref = _oracle_following(shape, tens, x, pos, vc, gv, "compact layer %s" % name)
    assert_close(dx.cpu().numpy(), ref, "compact layer %s" % name)


def test_compact_layer_consecutive_steps(env):
    """Four steps back to back in one stream: each step's attention reads the V row the
    previous step appended (K rebuilt from it), with no host synchronisation in between."""
    g, t = env
    shape = _small_compact()
    B, S, cap = 2, 4, 320
    p0 = np.array([300, 40], np.int32)
    tens, vc = _weights(shape, B, cap, 6)
    dl = g.DeviceLayer(shape, tens)
    X = [gem_synth.normal_f32(6, 500 + s, (B, shape.H)) for s in range(S)]
    dX = [_cu(t, x) for x in X]
    dP = [_cu(t, p0 + s) for s in range(S)]
    dv = _half_cache(t, vc)
    ws = t.empty(g.decode_layer_workspace(dl, B, cap), dtype=t.uint8, device="cuda")
    status = t.zeros(1, dtype=t.int32, device="cuda")
    for s in range(S):
        g.decode_layer(dl, dX[s], None, dv, dP[s], ws, status=status)
    t.cuda.synchronize()
    assert int(status.item()) == 0
    gv = _bits(dv)
    for s in range(S):
        # slots beyond p0 + s are not attended at step s, and slot p0 + s is rewritten by the
        # oracle's own append, so the GPU's final cache is the state before every step
        ref = _oracle_following(shape, tens, X[s], p0 + s, gv, gv, "compact step %d" % s)
        assert_close(dX[s].cpu().numpy(), ref, "compact step %d" % s)


def test_compact_layer_rejections(env):
    """compact_kv needs V from K, QK-norm and full attention; only compact layers may omit k_cache."""
    g, t = env
    base = _small_compact()
    tens, vc = _weights(base, 1, 64, 7)
    for bad in (replace(base, window=64), replace(base, qk_norm=False)):
        assert g.decode_layer_workspace(g.DeviceLayer(bad, tens), 1, 64) == 0
    plain = replace(base, compact_kv=False)
    dl = g.DeviceLayer(plain, tens)
    ws = t.empty(g.decode_layer_workspace(dl, 1, 64), dtype=t.uint8, device="cuda")
    with pytest.raises(g.GemError) as ei:
        g.decode_layer(dl, t.zeros((1, plain.H), device="cuda"), None, _half_cache(t, vc),
                       t.zeros(1, dtype=t.int32, device="cuda"), ws)
    assert ei.value.status == 1
