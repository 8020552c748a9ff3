"""The fused entry points the layer step runs, against the oracle (GPU only).

gem_q4_0_gemv_fused: pre-norm + Q4_0 GEMV (+ residual), or the gate/up pair with the gated
activation.  gem_gqa_decode_attn_fused: QK-norm + RoPE + binary16 KV append + decode attention
from the raw QKV projection row.  Tolerances are those of tests/parity.py; the appended rows
follow the binary16 rounding-band rule of tests/test_gpu_parity.py, and the attention output
is compared with the oracle's attention over the cache holding the GPU's appended rows."""
import numpy as np
import pytest

import gem_synth
import oracle
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


GEMV_FUSED_CASES = [
    # (N, K, B, pair, norm, residual, act)
    (4096, 2048, 1, False, True, False, 0),     # Qwen3-1.7B QKV projection with its pre-norm
    (4096, 2048, 3, False, True, False, 0),
    (6144, 2048, 1, True, True, False, 0),      # gate/up pair, SiLU
    (520, 2560, 8, True, True, False, 1),       # gate/up pair, GELU-tanh, 8 rows, ragged N
    (2048, 6144, 1, False, False, True, 0),     # down projection with the residual
    (2048, 2048, 5, False, False, True, 0),
    (2600, 16384, 1, True, True, False, 0),     # long K: the one-row K split over CTA pairs
]


@pytest.mark.parametrize("case", GEMV_FUSED_CASES,
                         ids=lambda c: "N%d_K%d_B%d_%s%s%s" % (c[0], c[1], c[2], "pair" if c[3] else "one",
                                                                "_norm" if c[4] else "", "_res" if c[5] else ""))
def test_gemv_fused_matches_oracle(env, case):
    g, t = env
    N, K, B, pair, norm, res, act = case
    W0 = gem_synth.q4_0_matrix(12, 1, N, K)
    W1 = gem_synth.q4_0_matrix(12, 2, N, K) if pair else None
    x = gem_synth.normal_f32(12, 3, (B, K)) * 3
    gamma = gem_synth.norm_weight(12, 4, K) if norm else None
    r = gem_synth.normal_f32(12, 5, (B, N)) if res else None
    eps = 1e-6
    y = t.full((B, N), float("nan"), device="cuda")
    g.q4_0_gemv_fused(_cu(t, W0), None if W1 is None else _cu(t, W1), N, K, _cu(t, x), y,
                      gamma=None if gamma is None else _cu(t, gamma), eps=eps, act=act,
                      residual=None if r is None else _cu(t, r))
    t.cuda.synchronize()
    # (without a norm the fp32 input itself is the operand; the oracle adds the fp32 residual)
    xh = np.stack([oracle.rmsnorm(x[b].astype(np.float64), gamma, eps) for b in range(B)]) if norm else x
    y0 = oracle.q4_0_gemv(W0, N, K, xh) if norm else oracle.q4_0_gemv(W0, N, K, xh, r)
    if pair:
        y1 = oracle.q4_0_gemv(W1, N, K, xh)
        f = oracle.gelu_tanh if act else oracle.silu
        ref = np.array([[f(float(y0[b, n])) * float(y1[b, n]) for n in range(N)] for b in range(B)])
    else:
        ref = y0
    assert_close(y.cpu().numpy(), ref, "fused GEMV %s" % (case,))


def test_gemv_fused_rejects_pair_with_residual(env):
    g, t = env
    W = t.zeros(16 * 8 * 18, dtype=t.uint8, device="cuda")
    x = t.zeros((1, 256), device="cuda")
    y = t.zeros((1, 16), device="cuda")
    with pytest.raises(g.GemError) as ei:
        g.q4_0_gemv_fused(W, W, 16, 256, x, y, residual=y)
    assert ei.value.status == 1


ATTN_FUSED_CASES = [
    # (n_q, n_kv, d, rope_dim, theta, v_mode, window, positions, cap, scale)
    (4, 2, 64, 64, 1e6, 0, 0, [128], 129, 0.125),                        # one launch
    (16, 8, 128, 128, 1e6, 0, 0, [4096], 4097, 128 ** -0.5),             # one launch, splits merged by the last to finish
    (32, 8, 128, 128, 1e6, 0, 0, [2048, 0, 17, 700], 2049, 128 ** -0.5),  # ragged batch
    (8, 2, 128, 32, 1e6, 1, 0, [300], 301, 1.0),                         # V from K, partial RoPE
    (32, 16, 256, 256, 1e4, 0, 64, [200, 30], 64, 1.0),                  # ring
    (8, 1, 128, 128, 1e6, 0, 0, [300, 45], 301, 128 ** -0.5),            # G = 8: two launches
    (32, 4, 512, 128, 1e6, 1, 0, [5000], 5001, 1.0),                     # d = 512: two launches
]


@pytest.mark.parametrize("case", ATTN_FUSED_CASES,
                         ids=lambda c: "G%d_d%d_v%d_w%d_B%d" % (c[0] // c[1], c[2], c[5], c[6], len(c[7])))
def test_attention_fused_matches_oracle(env, case):
    g, t = env
    n_q, n_kv, d, R, theta, v_mode, window, pos_l, cap, scale = case
    B = len(pos_l)
    nqkv = (n_q + n_kv + (0 if v_mode else n_kv)) * d
    qkv = gem_synth.normal_f32(13, d, (B, nqkv)) * 2
    gq = gem_synth.norm_weight(13, 1, d)
    gk = gem_synth.norm_weight(13, 2, d)
    kc = gem_synth.normal_f16_bits(13, 3, (B, n_kv, cap, d))
    vc = gem_synth.normal_f16_bits(13, 4, (B, n_kv, cap, d))
    pos = np.array(pos_l, np.int32)
    dk, dv = _half_cache(t, kc), _half_cache(t, vc)
    need = g.gqa_decode_attn_workspace(B, n_q, n_kv, d, cap, window)
    ws = t.empty(need, dtype=t.uint8, device="cuda") if need else None
    out = t.full((B, n_q * d), float("nan"), device="cuda")
    status = t.zeros(1, dtype=t.int32, device="cuda")
    g.gqa_decode_attn_fused(_cu(t, qkv), n_q, n_kv, d, _cu(t, gq), _cu(t, gk), v_mode, 1e-6, _cu(t, pos), theta, R,
                            dk, dv, window, scale, out, ws, status=status)
    t.cuda.synchronize()
    assert int(status.item()) == 0
    gk_bits, gv_bits, got = _bits(dk), _bits(dv), out.cpu().numpy()
    for b in range(B):
        p = int(pos[b])
        slot = p % window if window else p
        q = qkv[b, :n_q * d].reshape(n_q, d).astype(np.float64)
        k = qkv[b, n_q * d:(n_q + n_kv) * d].reshape(n_kv, d).astype(np.float64)
        rq = np.stack([oracle.rope_neox(oracle.rmsnorm(h, gq, 1e-6), R, p, theta) for h in q])
        rk = np.stack([oracle.rope_neox(oracle.rmsnorm(h, gk, 1e-6), R, p, theta) for h in k])
        rv = (np.stack([oracle.rmsnorm(h, None, 1e-6) for h in k]) if v_mode
              else qkv[b, (n_q + n_kv) * d:].reshape(n_kv, d).astype(np.float64))
        for gbits, vals in ((gk_bits, rk), (gv_bits, rv)):
            gnew = gbits[b, :, slot]
            nd = 0
            for j in range(n_kv):
                rms = float(np.sqrt(np.mean(vals[j] ** 2)))
                for i in range(d):
                    v = float(vals[j, i])
                    if gnew[j, i] != oracle.double_to_half_via_f32(v):
                        assert _code_in_band(int(gnew[j, i]), v, rms)
                        nd += 1
            assert nd <= max(2, 0.005 * n_kv * d)
        mask = np.ones(cap, bool)
        mask[slot] = False
        assert np.array_equal(gk_bits[b][:, mask], kc[b][:, mask])
        assert np.array_equal(gv_bits[b][:, mask], vc[b][:, mask])
        # attention over the cache as the GPU left it (its own appended codes)
        ref = oracle.gqa_attention(rq, gk_bits[b], gv_bits[b], p, window, scale)
        assert_close(got[b], ref.reshape(-1), "fused attention b=%d p=%d" % (b, p))
