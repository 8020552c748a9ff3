"""Pins of the fp64 oracle against facts fixed outside it: the block format's
hand-built examples, the page-printed matrix size, library routines for special cases,
closed forms, invariants and high-precision brute force.  CPU only."""
import json
import math
import os

import numpy as np
import pytest

import gem_synth
import oracle
from gem_synth import configs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _block(scale_bits: int, qs: bytes) -> np.ndarray:
    return np.frombuffer(bytes([scale_bits & 0xFF, scale_bits >> 8]) + qs, dtype=np.uint8).copy()


# ---- binary16 ---------------------------------------------------------------------------

def test_half_decode_all_patterns_match_numpy():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.half_to_double(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_half_encode_matches_numpy_rne():
    rng = np.random.default_rng(1)
    vals = np.concatenate([
        rng.standard_normal(4000) * np.exp2(rng.integers(-30, 18, 4000)),
        [0.0, -0.0, 65504.0, 65519.99, 65520.0, 1e9, -1e9, 2.0 ** -24, 2.0 ** -25,
         3 * 2.0 ** -26, 2.0 ** -14, 1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11, np.inf, -np.inf],
        # exact ties between adjacent halves, both parities
        (1024 + np.arange(0, 40) + 0.5) * 2.0 ** -10,
    ])
    with np.errstate(over="ignore"):
        ref = vals.astype(np.float32).astype(np.float16).view(np.uint16)
    got = np.array([oracle.double_to_half_via_f32(v) for v in vals], dtype=np.uint16)
    assert np.array_equal(got, ref)


# ---- Q4_0 block format ------------------------------------------------------------------

def test_q4_0_hand_built_blocks():
    g = json.load(open(os.path.join(GOLDEN, "q4_0_blocks.json")))
    for blk in g["blocks"]:
        W = _block(int(blk["scale_bits"], 16), bytes.fromhex(blk["qs"]))
        got = oracle.q4_0_dequant(W, 1, 32)[0]
        assert np.array_equal(got, np.array(blk["expect"])), blk["name"]


@pytest.mark.parametrize("j", range(32))
def test_q4_0_nibble_order_one_hot(j):
    # element j alone carries code 9 (weight +d); every other code is 8 (weight 0)
    qs = bytearray([0x88] * 16)
    if j < 16:
        qs[j] = 0x89
    else:
        qs[j - 16] = 0x98
    W = _block(0x4000, bytes(qs))  # d = 2.0
    expect = np.zeros(32)
    expect[j] = 2.0
    assert np.array_equal(oracle.q4_0_dequant(W, 1, 32)[0], expect)


def test_q4_0_ffn_matrix_bytes_match_page():
    # "gem" research record, "Native Metal diagnostic: buffer ownership": the 31B FFN
    # projection (5376 in, 21504 out) is 65,028,096 matrix bytes.
    assert 21504 * (5376 // 32) * 18 == 65_028_096
    W = gem_synth.q4_0_matrix(0, 99, 64, 5376)
    assert W.nbytes * (21504 // 64) == 65_028_096


def _encode_q4_0(codes: np.ndarray, scale_bits: np.ndarray) -> np.ndarray:
    """Pack integer codes [N, K] (0..15) and binary16 scales [N, K/32] into Q4_0 bytes."""
    N, K = codes.shape
    nb = K // 32
    c = codes.reshape(N, nb, 32).astype(np.uint8)
    out = np.empty((N, nb, 18), dtype=np.uint8)
    out[:, :, 0] = scale_bits & 0xFF
    out[:, :, 1] = scale_bits >> 8
    out[:, :, 2:] = c[:, :, :16] | (c[:, :, 16:] << 4)
    return out.reshape(N, nb * 18)


@pytest.mark.parametrize("B", [1, 3, 8])
def test_gemv_equals_dense_matmul_on_known_weights(B):
    N, K = 37, 256
    u = gem_synth.draws(7, 1, N * K)
    codes = (u & np.uint64(15)).astype(np.int64).reshape(N, K)
    scales = (0.002 + 0.018 * gem_synth.uniform(7, 2, N * K // 32)).astype(np.float16)
    Wdense = (codes - 8).astype(np.float64) * np.repeat(
        scales.astype(np.float64).reshape(N, K // 32), 32, axis=1)
    Wq = _encode_q4_0(codes, scales.view(np.uint16).reshape(N, K // 32))
    x = gem_synth.normal_f32(7, 3, (B, K))
    r = gem_synth.normal_f32(7, 4, (B, N))
    y = oracle.q4_0_gemv(Wq, N, K, x)
    ref = x.astype(np.float64) @ Wdense.T
    assert np.allclose(y, ref, rtol=1e-13, atol=1e-13)
    yr = oracle.q4_0_gemv(Wq, N, K, x, residual=r)
    assert np.allclose(yr, ref + r.astype(np.float64), rtol=1e-13, atol=1e-13)


def test_gemv_linear_and_rows_independent():
    N, K = 19, 512
    W = gem_synth.q4_0_matrix(3, 5, N, K)
    x = gem_synth.normal(3, 6, 2 * K).reshape(2, K)
    y = oracle.q4_0_gemv(W, N, K, x)
    y_sum = oracle.q4_0_gemv(W, N, K, (x[0] + x[1])[None, :])
    assert np.allclose(y_sum[0], y[0] + y[1], rtol=1e-12, atol=1e-12)
    y0 = oracle.q4_0_gemv(W, N, K, x[:1])
    assert np.array_equal(y0[0], y[0])
    y3 = oracle.q4_0_gemv(W, N, K, 3.0 * x[:1])
    assert np.allclose(y3[0], 3.0 * y[0], rtol=1e-13, atol=1e-13)


def test_gemv_rejects_k_not_multiple_of_32():
    with pytest.raises(ValueError):
        oracle.q4_0_gemv(np.zeros(18, np.uint8), 1, 33, np.zeros((1, 33), np.float32))


# ---- RMSNorm ------------------------------------------------------------------------------

def test_rmsnorm_unit_rms_closed_form():
    x = gem_synth.normal(11, 1, 1000) * 3.0
    eps = 1e-6
    y = oracle.rmsnorm(x, None, eps)
    ms = np.mean(x * x)
    assert math.isclose(np.mean(y * y), ms / (ms + eps), rel_tol=1e-13)
    y0 = oracle.rmsnorm(x, None, 0.0)
    assert math.isclose(np.sqrt(np.mean(y0 * y0)), 1.0, rel_tol=1e-14)


def test_rmsnorm_scale_invariant_and_gamma_per_channel():
    x = gem_synth.normal(11, 2, 128)
    g = gem_synth.norm_weight(11, 3, 128)
    a = oracle.rmsnorm(x, None, 0.0)
    b = oracle.rmsnorm(7.5 * x, None, 0.0)
    assert np.allclose(a, b, rtol=1e-14, atol=1e-15)
    c = oracle.rmsnorm(x, g, 0.0)
    assert np.allclose(c, a * g.astype(np.float64), rtol=1e-14, atol=1e-15)


# ---- RoPE -----------------------------------------------------------------------------------

def test_rope_single_pair_is_rotation_by_pos_radians():
    v = np.array([0.6, -1.7])
    for p in [0, 1, 5, 4096, 32768]:
        got = oracle.rope_neox(v, 2, p, 1e6)
        c, s = np.cos(p), np.sin(p)  # one pair, frequency theta^0 = 1
        assert np.allclose(got, [v[0] * c - v[1] * s, v[0] * s + v[1] * c], rtol=1e-15, atol=1e-15)


def test_rope_second_pair_frequency():
    theta, R = 1e4, 4
    v = np.array([1.0, 0.0, 0.0, 0.0])   # pairs (0,2) and (1,3)
    w = np.array([0.0, 1.0, 0.0, 0.0])
    p = 3.0
    a1 = p * theta ** (-2.0 / R)
    got = oracle.rope_neox(w, R, p, theta)
    assert np.allclose(got, [0.0, np.cos(a1), 0.0, np.sin(a1)], atol=1e-15)
    got0 = oracle.rope_neox(v, R, p, theta)
    assert np.allclose(got0, [np.cos(p), 0.0, np.sin(p), 0.0], atol=1e-15)


@pytest.mark.parametrize("d,R,theta", [(64, 64, 1e6), (128, 128, 1e6), (256, 256, 1e4), (512, 128, 1e6)])
def test_rope_invariants(d, R, theta):
    v = gem_synth.normal(13, d, d)
    half = R // 2
    r0 = oracle.rope_neox(v, R, 0, theta)
    assert np.array_equal(r0, v)
    r = oracle.rope_neox(v, R, 32768, theta)
    pair_in = v[:half] ** 2 + v[half:R] ** 2
    pair_out = r[:half] ** 2 + r[half:R] ** 2
    assert np.allclose(pair_in, pair_out, rtol=1e-12)
    assert np.array_equal(r[R:], v[R:])
    r12 = oracle.rope_neox(oracle.rope_neox(v, R, 1000, theta), R, 3096, theta)
    r4096 = oracle.rope_neox(v, R, 4096, theta)
    assert np.allclose(r12, r4096, rtol=1e-10, atol=1e-11)


# ---- attention --------------------------------------------------------------------------------

def _rand_cache(seed, n_kv, cap, d):
    return (gem_synth.normal_f16_bits(seed, 1, (n_kv, cap, d)),
            gem_synth.normal_f16_bits(seed, 2, (n_kv, cap, d)))


def _f16(bits):
    return bits.view(np.float16).astype(np.float64)


def test_attention_weights_sum_to_one_and_gqa_shares_kv():
    n_q, n_kv, d, cap = 8, 2, 32, 50
    kc, vc = _rand_cache(21, n_kv, cap, d)
    q = gem_synth.normal(21, 3, n_q * d).reshape(n_q, d)
    q[1] = q[0]  # heads 0 and 1 share KV head 0
    out, P = oracle.gqa_attention(q, kc, vc, 40, 0, 0.2, return_probs=True)
    assert np.allclose(P.sum(axis=1), 1.0, atol=1e-12)
    assert np.array_equal(out[0], out[1])
    assert not np.allclose(out[0], out[4])


def test_attention_single_position_returns_v():
    kc, vc = _rand_cache(22, 2, 8, 16)
    q = gem_synth.normal(22, 3, 4 * 16).reshape(4, 16)
    out = oracle.gqa_attention(q, kc, vc, 0, 0, 1.0)
    for h in range(4):
        assert np.array_equal(out[h], _f16(vc[h // 2, 0]))


def test_attention_equal_keys_give_mean_of_v():
    n_kv, cap, d = 1, 30, 16
    kc, vc = _rand_cache(23, n_kv, cap, d)
    kc[:] = kc[0, 0]
    q = gem_synth.normal(23, 4, 2 * d).reshape(2, d)
    out = oracle.gqa_attention(q, kc, vc, 24, 0, 0.5)
    mean_v = _f16(vc[0, :25]).mean(axis=0)
    assert np.allclose(out[0], mean_v, rtol=1e-13, atol=1e-14)


def test_attention_g1_equals_per_head_mha():
    n, d, cap = 4, 24, 12
    kc, vc = _rand_cache(24, n, cap, d)
    q = gem_synth.normal(24, 5, n * d).reshape(n, d)
    out = oracle.gqa_attention(q, kc, vc, 9, 0, 0.3)
    for h in range(n):
        oh = oracle.gqa_attention(q[h:h + 1], kc[h:h + 1], vc[h:h + 1], 9, 0, 0.3)
        assert np.array_equal(out[h], oh[0])


def test_attention_order_invariant_under_slot_permutation():
    n_kv, cap, d = 2, 20, 16
    kc, vc = _rand_cache(25, n_kv, cap, d)
    q = gem_synth.normal(25, 6, 4 * d).reshape(4, d)
    perm = np.random.default_rng(0).permutation(cap)
    out = oracle.gqa_attention(q, kc, vc, cap - 1, 0, 0.4)
    outp = oracle.gqa_attention(q, kc[:, perm], vc[:, perm], cap - 1, 0, 0.4)
    assert np.allclose(out, outp, rtol=1e-12, atol=1e-13)


def test_attention_ring_window_equals_full_over_last_w():
    n_kv, W, d, pos = 1, 8, 16, 21           # window holds positions 14..21
    kc, vc = _rand_cache(26, n_kv, W, d)
    q = gem_synth.normal(26, 7, 2 * d).reshape(2, d)
    ring = oracle.gqa_attention(q, kc, vc, pos, W, 0.25)
    order = [(j % W) for j in range(pos - W + 1, pos + 1)]  # slots in position order
    lin = oracle.gqa_attention(q, kc[:, order], vc[:, order], W - 1, 0, 0.25)
    assert np.allclose(ring, lin, rtol=1e-13, atol=1e-14)
    # before the ring fills, the window is every position 0..pos
    few = oracle.gqa_attention(q, kc, vc, 5, W, 0.25)
    lin5 = oracle.gqa_attention(q, kc[:, :6], vc[:, :6], 5, 0, 0.25)
    assert np.allclose(few, lin5, rtol=1e-13, atol=1e-14)


def test_attention_brute_force_high_precision():
    mp = pytest.importorskip("mpmath")
    mp.mp.dps = 40
    n_q, n_kv, d, cap, pos, scale = 2, 1, 8, 6, 5, 1.0
    kc, vc = _rand_cache(27, n_kv, cap, d)
    q = gem_synth.normal(27, 8, n_q * d).reshape(n_q, d) * 4.0   # large, peaked scores
    out = oracle.gqa_attention(q, kc, vc, pos, 0, scale)
    K, V = _f16(kc[0]), _f16(vc[0])
    for h in range(n_q):
        s = [mp.mpf(scale) * mp.fsum(mp.mpf(q[h, i]) * mp.mpf(K[j, i]) for i in range(d))
             for j in range(pos + 1)]
        lse = mp.log(mp.fsum(mp.exp(t) for t in s))
        for i in range(d):
            ref = mp.fsum(mp.exp(s[j] - lse) * mp.mpf(V[j, i]) for j in range(pos + 1))
            assert abs(out[h, i] - float(ref)) <= 1e-13 * (1 + abs(float(ref)))


def test_attention_two_positions_logistic():
    d = 4
    kc = np.zeros((1, 2, d), np.float16)
    kc[0, 1, 0] = 1.0
    vc = np.zeros((1, 2, d), np.float16)
    vc[0, 0, :] = 1.0
    vc[0, 1, :] = -1.0
    q = np.array([[2.0, 0, 0, 0]])
    out = oracle.gqa_attention(q, kc.view(np.uint16), vc.view(np.uint16), 1, 0, 1.0)
    p1 = 1.0 / (1.0 + math.exp(-2.0))            # weight of position 1 (score 2 vs 0)
    assert np.allclose(out[0], (1 - p1) - p1, rtol=1e-15)


# ---- FFN activations ----------------------------------------------------------------------------

def test_activations_known_values_and_identities():
    assert oracle.silu(0.0) == 0.0
    assert math.isclose(oracle.silu(1.0), math.e / (1.0 + math.e), rel_tol=1e-15)
    assert math.isclose(oracle.gelu_tanh(1.0), 0.8411919906082768, rel_tol=1e-14)
    assert oracle.gelu_tanh(0.0) == 0.0
    for x in [0.3, 1.7, 5.0, 12.0]:
        assert math.isclose(oracle.silu(x) - oracle.silu(-x), x, rel_tol=1e-14)
        assert math.isclose(oracle.gelu_tanh(x) - oracle.gelu_tanh(-x), x, rel_tol=1e-14)


# ---- the layer step --------------------------------------------------------------------------------

def _tiny():
    w = configs.workload("tiny")
    s = w.layers[0]
    t = configs.layer_tensors(s, w.B, w.cache_cap[0], 0, 0)
    x = configs.layer_input(s.H, w.B, 0)
    return w, s, t, x


def _zero_scales(Wq):
    Wz = Wq.copy().reshape(-1, 18)
    Wz[:, 0:2] = 0
    return Wz.reshape(Wq.shape)


def test_layer_with_zero_weights_is_identity_and_appends_zero_row():
    w, s, t, x = _tiny()
    for name in ("w_qkv", "w_o", "w_gate", "w_up", "w_down"):
        setattr(t, name, _zero_scales(getattr(t, name)))
    pos = np.array([w.pos], np.int32)
    kc, vc = t.k_cache.copy(), t.v_cache.copy()
    out = oracle.decode_layer(s, t, x, pos, kc, vc)
    assert np.array_equal(out, x.astype(np.float64))
    # RoPE of a zero vector can produce -0.0; compare values, not bit patterns
    assert np.all(_f16(kc[:, :, w.pos]) == 0) and np.all(_f16(vc[:, :, w.pos]) == 0)
    assert np.array_equal(kc[:, :, :w.pos], t.k_cache[:, :, :w.pos])


def test_layer_stages_compose():
    w, s, t, x = _tiny()
    pos = np.array([w.pos], np.int32)
    kc, vc = t.k_cache.copy(), t.v_cache.copy()
    out, qkv, att, h = oracle.decode_layer(s, t, x, pos, kc, vc, stages=True)
    qd = s.n_q * s.d
    kd = s.n_kv * s.d
    # the appended row is the fp16 rounding (via fp32) of the normed, rotated k and raw v
    k_new = qkv[0, qd:qd + kd].reshape(s.n_kv, s.d)
    v_new = qkv[0, qd + kd:].reshape(s.n_kv, s.d)
    assert np.array_equal(kc[0, :, w.pos], k_new.astype(np.float32).astype(np.float16).view(np.uint16))
    assert np.array_equal(vc[0, :, w.pos], v_new.astype(np.float32).astype(np.float16).view(np.uint16))
    # q heads are unit-RMS before RoPE times gamma: RoPE preserves pair norms, so the
    # per-head squared norm equals that of rmsnorm(raw q) * gamma
    a = oracle.gqa_attention(qkv[0, :qd].reshape(s.n_q, s.d), kc[0], vc[0], w.pos, 0, s.scale)
    assert np.array_equal(a.reshape(-1), att[0])
    # FFN residual: with zero down-projection the output equals h
    t.w_down = _zero_scales(t.w_down)
    kc2, vc2 = t.k_cache.copy(), t.v_cache.copy()
    out2 = oracle.decode_layer(s, t, x, pos, kc2, vc2)
    assert np.array_equal(out2, h)


def test_qk_norm_heads_independent_and_gamma_per_channel():
    # GELO section 05 names the two properties of apply_qk_norm: each head is
    # normalised on its own, and gamma applies per channel.
    d = 16
    heads = gem_synth.normal(31, 1, 3 * d).reshape(3, d) * np.array([[0.1], [1.0], [30.0]])
    g = gem_synth.norm_weight(31, 2, d)
    outs = [oracle.rmsnorm(h, g, 0.0) for h in heads]
    for o in outs:
        assert math.isclose(np.sqrt(np.mean((o / g.astype(np.float64)) ** 2)), 1.0, rel_tol=1e-13)


def test_argmax_ties_lowest_index():
    v = np.array([1.0, 3.0, -2.0, 3.0, 3.0])
    assert oracle.argmax(v) == 1
    assert oracle.argmax(np.array([5.0])) == 0


def test_oracle_thread_count_does_not_change_results():
    N, K = 64, 1024
    W = gem_synth.q4_0_matrix(5, 5, N, K)
    x = gem_synth.normal_f32(5, 6, (2, K))
    n0 = oracle.num_threads()
    try:
        oracle.set_num_threads(1)
        a = oracle.q4_0_gemv(W, N, K, x)
        oracle.set_num_threads(max(2, n0))
        b = oracle.q4_0_gemv(W, N, K, x)
    finally:
        oracle.set_num_threads(n0)
    assert np.array_equal(a, b)


@pytest.mark.parametrize("which", ["tiny", "gemma_full_small", "gemma_swa_small"])
def test_layer_equals_composition_of_pinned_steps(which):
    """The layer step equals its steps (each pinned above) chained in the order of the
    GELO section 06 block: norm, QKV, QK-norm, RoPE, append, attention, O + residual,
    norm, gate/up, activation, down + residual (Gemma: V from K, post norms)."""
    if which == "tiny":
        w, s, t, x = _tiny()
        pos_v, cap = w.pos, w.cache_cap[0]
    else:
        from dataclasses import replace
        base = configs.GEMMA31_FULL if which == "gemma_full_small" else configs.GEMMA31_SWA
        s = replace(base, H=256, n_q=4, n_kv=2 if which == "gemma_full_small" else 4, d=64,
                    F=512, rope_dim=16 if which == "gemma_full_small" else 64,
                    window=0 if which == "gemma_full_small" else 16)
        pos_v = 40
        cap = s.window if s.window else pos_v + 1
        t = configs.layer_tensors(s, 1, cap, 3, 0)
        x = configs.layer_input(s.H, 1, 3)
    pos = np.array([pos_v], np.int32)
    kc, vc = t.k_cache.copy(), t.v_cache.copy()
    out = oracle.decode_layer(s, t, x, pos, kc, vc)

    xd = x[0].astype(np.float64)
    xn = oracle.rmsnorm(xd, t.g_attn, s.eps)
    qkv = oracle.q4_0_gemv(t.w_qkv, s.n_qkv, s.H, xn[None])[0]
    qd, kd = s.n_q * s.d, s.n_kv * s.d
    q = qkv[:qd].reshape(s.n_q, s.d).copy()
    k = qkv[qd:qd + kd].reshape(s.n_kv, s.d).copy()
    if s.v_from_k:
        v = np.stack([oracle.rmsnorm(k[j], None, s.eps) for j in range(s.n_kv)])
    else:
        v = qkv[qd + kd:].reshape(s.n_kv, s.d)
    q = np.stack([oracle.rope_neox(oracle.rmsnorm(h, t.g_q, s.eps), s.rope_dim, pos_v, s.theta) for h in q])
    k = np.stack([oracle.rope_neox(oracle.rmsnorm(h, t.g_k, s.eps), s.rope_dim, pos_v, s.theta) for h in k])
    kc2, vc2 = t.k_cache.copy(), t.v_cache.copy()
    slot = pos_v % s.window if s.window else pos_v
    kc2[0, :, slot] = k.astype(np.float32).astype(np.float16).view(np.uint16)
    vc2[0, :, slot] = v.astype(np.float32).astype(np.float16).view(np.uint16)
    assert np.array_equal(kc2, kc) and np.array_equal(vc2, vc)
    att = oracle.gqa_attention(q, kc2[0], vc2[0], pos_v, s.window, s.scale).reshape(-1)
    o = oracle.q4_0_gemv(t.w_o, s.H, qd, att[None])[0]
    h = xd + (oracle.rmsnorm(o, t.g_post_attn, s.eps) if s.post_norms else o)
    hn = oracle.rmsnorm(h, t.g_ffn, s.eps)
    g = oracle.q4_0_gemv(t.w_gate, s.F, s.H, hn[None])[0]
    u = oracle.q4_0_gemv(t.w_up, s.F, s.H, hn[None])[0]
    act = oracle.gelu_tanh if s.act == configs.ACT_GELU_TANH else oracle.silu
    a = np.array([act(gi) for gi in g]) * u
    dn = oracle.q4_0_gemv(t.w_down, s.H, s.F, a[None])[0]
    ref = h + (oracle.rmsnorm(dn, t.g_post_ffn, s.eps) if s.post_norms else dn)
    assert np.array_equal(out[0], ref)


def test_other_half_neighbour():
    # 1 + 2^-11 lies exactly between 1.0 (0x3c00) and 1 + 2^-10 (0x3c01): RNE picks the
    # even code 0x3c00, the other neighbour is 0x3c01
    assert oracle.double_to_half_via_f32(1.0 + 2.0 ** -11) == 0x3C00
    assert oracle.other_half_via_f32(1.0 + 2.0 ** -11) == 0x3C01
    assert oracle.other_half_via_f32(1.0) == 0x3C00                  # exact: no other code
    assert oracle.other_half_via_f32(-(1.0 + 2.0 ** -12)) == 0xBC01   # RNE -> -1.0, other -> away
    rng = np.random.default_rng(3)
    for v in rng.standard_normal(2000) * 10:
        a = oracle.double_to_half_via_f32(v)
        o = oracle.other_half_via_f32(v)
        fa = np.float64(np.uint16(a).view(np.float16))
        fo = np.float64(np.uint16(o).view(np.float16))
        vf = float(np.float32(v))
        assert min(fa, fo) <= vf <= max(fa, fo)      # the two codes bracket the value
        assert abs(fa - vf) <= abs(fo - vf)          # RNE is the nearer one


def test_layer_flip_changes_only_the_flipped_code():
    w, s, t, x = _tiny()
    pos = np.array([w.pos], np.int32)
    kc, vc = t.k_cache.copy(), t.v_cache.copy()
    out0, kvn = oracle.decode_layer(s, t, x, pos, kc, vc, kvnew=True)
    flip = np.zeros((1, 2, s.n_kv, s.d), np.int8)
    flip[0, 1, 1, 5] = 1
    kc2, vc2 = t.k_cache.copy(), t.v_cache.copy()
    out1 = oracle.decode_layer(s, t, x, pos, kc2, vc2, flip=flip)
    assert np.array_equal(kc2, kc)
    diff = vc2 != vc
    assert diff.sum() == 1 and diff[0, 1, w.pos, 5]
    assert vc2[0, 1, w.pos, 5] == oracle.other_half_via_f32(kvn[0, 1, 1, 5])
    assert not np.array_equal(out0, out1)


# ---- Q8_0 block format (tied embedding / logit projection) ------------------------------

def _q8_block(scale_bits: int, qs: bytes) -> np.ndarray:
    assert len(qs) == 32
    return np.frombuffer(bytes([scale_bits & 0xFF, scale_bits >> 8]) + qs, dtype=np.uint8).reshape(1, 34)


def test_q8_0_hand_built_blocks():
    g = json.load(open(os.path.join(GOLDEN, "q8_0_blocks.json")))
    for blk in g["blocks"]:
        W = _q8_block(int(blk["scale_bits"], 16), bytes.fromhex(blk["qs"]))
        got = oracle.q8_0_dequant(W, 1, 32)[0]
        assert np.array_equal(got, np.array(blk["expect"], dtype=np.float64)), blk["name"]


@pytest.mark.parametrize("j", [0, 1, 15, 16, 30, 31])
def test_q8_0_element_order_one_hot(j):
    qs = bytearray(32)
    qs[j] = 0xFD   # -3
    W = _q8_block(0x3400, bytes(qs))   # d = 0.25
    expect = np.zeros(32)
    expect[j] = -0.75
    assert np.array_equal(oracle.q8_0_dequant(W, 1, 32)[0], expect)


def test_q8_0_gemv_equals_dense_matmul_on_independently_decoded_weights():
    # the test decodes the blocks itself from the format definition (numpy binary16 and int8
    # views), then compares the oracle GEMV with a plain fp64 matmul
    N, K, B = 7, 96, 3
    W = gem_synth.q8_0_matrix(5, 9, N, K)
    blocks = W.reshape(N, K // 32, 34)
    d = blocks[:, :, 0:2].copy().view(np.float16).astype(np.float64)[:, :, 0]
    q = blocks[:, :, 2:].view(np.int8).astype(np.float64)
    dense = (q * d[:, :, None]).reshape(N, K)
    x = gem_synth.normal(5, 10, B * K).reshape(B, K)
    got = oracle.q8_0_gemv(W, N, K, x)
    assert np.allclose(got, x @ dense.T, rtol=1e-12, atol=1e-12)
    assert np.array_equal(oracle.q8_0_dequant(W, N, K), dense)


def test_argmax_ignores_nan():
    nan = float("nan")
    assert oracle.argmax(np.array([nan, 1.0, 2.0, 2.0])) == 2
    assert oracle.argmax(np.array([nan, nan])) == 0
    assert oracle.argmax(np.array([-np.inf, -5.0])) == 1


# ---- compact full-attention cache: K rebuilt from V ----------------------------------------

def _np_rope(v, R, pos, theta):
    """NeoX rotation of the first R dims by pos * theta^(-2i/R), written out with numpy."""
    out = v.copy()
    half = R // 2
    i = np.arange(half)
    ang = pos * theta ** (-2.0 * i / R)
    c, s = np.cos(ang), np.sin(ang)
    out[:half] = v[:half] * c - v[half:R] * s
    out[half:R] = v[:half] * s + v[half:R] * c
    return out


def test_compact_attention_equals_brute_force_over_rebuilt_keys():
    n_q, n_kv, d, R, theta, pos, cap = 4, 2, 16, 8, 1e4, 9, 12
    G = n_q // n_kv
    v16 = gem_synth.normal_f16_bits(41, 1, (n_kv, cap, d))
    gamma = gem_synth.norm_weight(41, 2, d)
    q = gem_synth.normal(41, 3, n_q * d).reshape(n_q, d)
    scale = 0.25
    got = oracle.gqa_attention_compact(q, v16, gamma, pos, R, theta, scale)
    vals = v16.view(np.float16).astype(np.float64)
    ref = np.empty((n_q, d))
    for h in range(n_q):
        g = h // G
        K = np.stack([_np_rope(vals[g, j] * gamma.astype(np.float64), R, j, theta) for j in range(pos + 1)])
        sc = scale * (K @ q[h])
        w = np.exp(sc - sc.max())
        w /= w.sum()
        ref[h] = w @ vals[g, :pos + 1]
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-13)


def test_compact_attention_without_rotation_or_weight_is_attention_with_k_equal_v():
    n_q, n_kv, d, pos, cap = 6, 3, 32, 20, 24
    v16 = gem_synth.normal_f16_bits(42, 1, (n_kv, cap, d))
    q = gem_synth.normal(42, 2, n_q * d).reshape(n_q, d)
    got = oracle.gqa_attention_compact(q, v16, None, pos, 0, 1e6, 0.125)
    ref = oracle.gqa_attention(q, v16, v16, pos, 0, 0.125)
    assert np.array_equal(got, ref)


def test_compact_layer_appends_v_only_and_tracks_the_standard_layer():
    """A compact full-attention layer writes the same V row as the standard one, leaves no K
    cache, and differs from the standard layer only by the binary16 rounding of the cached K
    rows (which the compact layer rebuilds from V instead)."""
    from dataclasses import replace
    shape = replace(configs.GEMMA31_FULL, H=512, n_q=8, n_kv=2, d=64, F=1024, rope_dim=16)
    compact = replace(shape, compact_kv=True)
    B, cap, pos = 1, 40, np.array([37], np.int32)
    tens = configs.layer_tensors(shape, B, cap, 43, 0)
    x = configs.layer_input(shape.H, B, 43)
    # a cache consistent with the compact layout: K rows rounded from the rebuilt keys
    v = tens.v_cache
    k = np.empty_like(v)
    for g in range(shape.n_kv):
        for j in range(cap):
            kk = _np_rope(v[0, g, j].view(np.float16).astype(np.float64) * tens.g_k.astype(np.float64),
                          shape.rope_dim, j, shape.theta)
            k[0, g, j] = kk.astype(np.float32).astype(np.float16).view(np.uint16)
    vs, ks = v.copy(), k.copy()
    ref = oracle.decode_layer(shape, tens, x, pos, ks, vs)
    vc = v.copy()
    got = oracle.decode_layer(compact, tens, x, pos, None, vc)
    assert np.array_equal(vc, vs)                   # same appended V row, nothing else touched
    assert np.allclose(got, ref, rtol=1e-3, atol=1e-3)
    assert not np.array_equal(got, ref)             # the K rows really are rebuilt, not read


# ---- top-k (the sampler's selection; ties by lowest index, NaN after every number) -----------

def test_topk_hand_cases():
    nan, inf = float("nan"), float("inf")
    i, v = oracle.topk(np.array([1.0, 3.0, 3.0, 2.0, 3.0]), 3)
    assert list(i) == [1, 2, 4] and list(v) == [3.0, 3.0, 3.0]
    i, _ = oracle.topk(np.array([nan, 1.0, nan, 0.0]), 4)
    assert list(i) == [1, 3, 0, 2]
    i, _ = oracle.topk(np.array([-inf, -inf, 5.0]), 3)
    assert list(i) == [2, 0, 1]
    i, v = oracle.topk(np.array([7.0]), 1)
    assert list(i) == [0] and v[0] == 7.0
    with pytest.raises(ValueError):
        oracle.topk(np.array([1.0, 2.0]), 3)


def test_topk_equals_a_stable_sort_and_the_argmax():
    """Against numpy's lexicographic sort (value descending, then index), NaN rows last."""
    rng = np.random.default_rng(5)
    for n, k in [(1, 1), (10, 10), (1000, 64), (4097, 17)]:
        v = np.round(rng.normal(size=n), 1)   # rounding makes ties common
        v[rng.integers(0, n, size=max(1, n // 50))] = np.nan
        num = np.nonzero(~np.isnan(v))[0]
        order = num[np.lexsort((num, -v[num]))]
        order = np.concatenate([order, np.nonzero(np.isnan(v))[0]])
        i, vals = oracle.topk(v, k)
        assert list(i) == list(order[:k])
        assert np.array_equal(vals, v[order[:k]], equal_nan=True)
        assert i[0] == oracle.argmax(v) or np.all(np.isnan(v))
