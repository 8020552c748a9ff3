"""CUDA library vs the fp64 oracle on identical seeded inputs (GPU only).

Every comparison goes through the C ABI (via the thin Python binding).  Tolerances are
those of tests/parity.py: max-abs <= 2e-3 and relative L2 <= 1e-5.  Binary16 KV rows
written by the kernels are compared to the oracle's rounding of the same value; a
rounding decision may differ by one unit where the fp32 (GPU) and fp64 (oracle) values
straddle a binary16 rounding boundary, and such differences must stay rare."""
from dataclasses import replace

import numpy as np
import pytest

import gem_synth
import oracle
from gem_synth import configs
from parity import assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gem():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import q4_gemv_gqa_gb300 as g
    g.device_status(reset=True)
    return g


@pytest.fixture(scope="module")
def torch_mod():
    import torch
    return torch


def _cu(t, a, dtype=None):
    x = t.from_numpy(np.ascontiguousarray(a)).cuda()
    return x if dtype is None else x.to(dtype)


def _half_cache(t, bits):
    return t.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda()


def _bits(tens):
    return tens.cpu().numpy().view(np.uint16)


# Relative slack of a kernel's fp32 new K/V value against the oracle's fp64 value (scaled
# by the head's RMS): a binary16 rounding decision inside this band may go either way.
EPS_KV = 2e-6


def _ambiguous(v, rms):
    d = EPS_KV * max(abs(v), rms)
    return oracle.double_to_half_via_f32(v - d) != oracle.double_to_half_via_f32(v + d)


def _code_line(c):
    """binary16 code on a monotone integer line"""
    return -(c & 0x7FFF) if c & 0x8000 else c


def _code_in_band(code, v, rms):
    """code is the rounding of some value within the fp32 band around v.  Codes that are
    not the other neighbour of v differ from the oracle's by at most 2 * band, far below
    the tolerance downstream, so they need no separate oracle evaluation."""
    d = EPS_KV * max(abs(v), rms)
    lo = _code_line(oracle.double_to_half_via_f32(v - d))
    hi = _code_line(oracle.double_to_half_via_f32(v + d))
    return lo <= _code_line(code) <= hi


# ---- Q4_0 GEMV ----------------------------------------------------------------------------

GEMV_CASES = [
    # (N, K, B): ragged row tails, several K stages, every batch size
    (67, 256, 1), (67, 256, 2), (67, 256, 3), (67, 256, 4), (67, 256, 5), (67, 256, 6),
    (67, 256, 7), (67, 256, 8), (33, 512, 3), (16, 2048, 1), (4096, 2048, 1), (2048, 6144, 1),
    (6144, 2048, 8), (2560, 9728, 8), (1, 256, 1),
    (40000, 512, 2), (40000, 512, 6),   # more 16-row units per CTA than one pass holds
    (300, 21504, 3),                    # long K: several activation phases
    (1000, 21504, 1), (2560, 9728, 1),  # one row: 12 phases; a ragged last phase (38 groups)
    (8, 8192, 1), (40000, 512, 1),      # one row: half a row-block pair; several passes
    (40, 65536, 1),                     # one row, operand records beyond shared memory: fallback kernel
    (5376, 21504, 1), (2600, 16384, 1), # one row, K split over CTA pairs (uneven units per CTA)
    (2600, 32768, 1),                   # the same, each CTA's half of the row read twice
    (24, 131328, 2),                    # two rows, very long K: the one-launch kernel, 257 stages per tile
    (520, 131328, 2),                   # two rows above 64M weights, records beyond the library array:
                                        # fallback kernel
]


@pytest.mark.parametrize("N,K,B", GEMV_CASES)
def test_gemv_matches_oracle(gem, torch_mod, N, K, B):
    t = torch_mod
    W = gem_synth.q4_0_matrix(1, N * 7 + K, N, K)
    x = gem_synth.normal_f32(1, 3, (B, K))
    ref = oracle.q4_0_gemv(W, N, K, x)
    y = t.full((B, N), float("nan"), device="cuda")
    gem.q4_0_gemv(_cu(t, W), N, K, _cu(t, x), y)
    t.cuda.synchronize()
    assert_close(y.cpu().numpy(), ref, "gemv N=%d K=%d B=%d" % (N, K, B))


@pytest.mark.parametrize("B", [1, 8])
def test_gemv_31b_ffn_shape_full(gem, torch_mod, B):
    """The 31B FFN projection (5376 -> 21504, 65,028,096 weight bytes), every output."""
    t = torch_mod
    N, K = 21504, 5376
    W = gem_synth.q4_0_matrix(0, 1000, N, K)
    assert W.nbytes == 65_028_096
    x = gem_synth.normal_f32(0, 1001, (B, K))
    ref = oracle.q4_0_gemv(W, N, K, x)
    y = t.empty((B, N), device="cuda")
    gem.q4_0_gemv(_cu(t, W), N, K, _cu(t, x), y)
    t.cuda.synchronize()
    assert_close(y.cpu().numpy(), ref, "gemv 31B FFN B=%d" % B)


def test_gemv_residual_in_place(gem, torch_mod):
    t = torch_mod
    N, K, B = 300, 768, 2
    W = gem_synth.q4_0_matrix(2, 5, N, K)
    x = gem_synth.normal_f32(2, 6, (B, K))
    r = gem_synth.normal_f32(2, 7, (B, N))
    ref = oracle.q4_0_gemv(W, N, K, x, residual=r)
    y = _cu(t, r)
    gem.q4_0_gemv(_cu(t, W), N, K, _cu(t, x), y, residual=y)
    t.cuda.synchronize()
    assert_close(y.cpu().numpy(), ref, "gemv residual in place")


@pytest.mark.parametrize("N,K,B", [(2600, 16384, 1), (2600, 16384, 2)])
def test_gemv_residual_in_place_k_split(gem, torch_mod, N, K, B):
    """Long K and more units than CTAs: the partial sums of a CTA pair (or cluster) are combined
    before the residual is added, in place."""
    t = torch_mod
    W = gem_synth.q4_0_matrix(2, 8, N, K)
    x = gem_synth.normal_f32(2, 9, (B, K))
    r = gem_synth.normal_f32(2, 10, (B, N))
    ref = oracle.q4_0_gemv(W, N, K, x, residual=r)
    y = _cu(t, r)
    gem.q4_0_gemv(_cu(t, W), N, K, _cu(t, x), y, residual=y)
    t.cuda.synchronize()
    assert_close(y.cpu().numpy(), ref, "gemv residual in place, K split B=%d" % B)


@pytest.mark.parametrize("N,K,B,offset", [(45, 96, 2, 0), (40, 512, 1, 2), (130, 3200, 3, 0)])
def test_gemv_general_path(gem, torch_mod, N, K, B, offset):
    """K % 256 != 0 or a matrix not 16-byte aligned runs the general kernel."""
    t = torch_mod
    W = gem_synth.q4_0_matrix(3, K, N, K)
    x = gem_synth.normal_f32(3, 8, (B, K))
    ref = oracle.q4_0_gemv(W, N, K, x)
    buf = t.zeros(W.nbytes + 16, dtype=t.uint8, device="cuda")
    buf[offset:offset + W.nbytes] = _cu(t, W.reshape(-1))
    y = t.empty((B, N), device="cuda")
    gem.q4_0_gemv(buf[offset:offset + W.nbytes], N, K, _cu(t, x), y)
    t.cuda.synchronize()
    assert_close(y.cpu().numpy(), ref, "gemv general N=%d K=%d off=%d" % (N, K, offset))


def test_gemv_empty_and_rejected(gem, torch_mod):
    t = torch_mod
    W = t.zeros(18 * 8, dtype=t.uint8, device="cuda")
    x = t.zeros((1, 256), device="cuda")
    y = t.zeros((1, 1), device="cuda")
    gem.q4_0_gemv(W, 0, 256, x, y)          # N = 0: nothing to do
    with pytest.raises(gem.GemError):
        gem.q4_0_gemv(W, 1, 33, x, y)       # K % 32 != 0
    with pytest.raises(gem.GemError):
        gem.q4_0_gemv(W, 1, 256, t.zeros((9, 256), device="cuda"), t.zeros((9, 1), device="cuda"))


def test_gemv_deterministic(gem, torch_mod):
    t = torch_mod
    N, K, B = 5000, 4096, 4
    W = _cu(t, gem_synth.q4_0_matrix(4, 1, N, K))
    x = _cu(t, gem_synth.normal_f32(4, 2, (B, K)))
    y1 = t.empty((B, N), device="cuda")
    y2 = t.empty((B, N), device="cuda")
    gem.q4_0_gemv(W, N, K, x, y1)
    gem.q4_0_gemv(W, N, K, x, y2)
    t.cuda.synchronize()
    assert t.equal(y1, y2)


# ---- RMSNorm / activation -------------------------------------------------------------------

def test_rmsnorm(gem, torch_mod):
    t = torch_mod
    B, H = 3, 2560
    x = gem_synth.normal_f32(5, 1, (B, H)) * 4
    g = gem_synth.norm_weight(5, 2, H)
    out = t.empty((B, H), device="cuda")
    gem.rmsnorm(_cu(t, x), _cu(t, g), 1e-6, out)
    t.cuda.synchronize()
    ref = np.stack([oracle.rmsnorm(x[b].astype(np.float64), g, 1e-6) for b in range(B)])
    assert_close(out.cpu().numpy(), ref, "rmsnorm")


@pytest.mark.parametrize("act", [0, 1])
def test_gated_activation(gem, torch_mod, act):
    t = torch_mod
    B, F = 2, 9728
    g = gem_synth.normal_f32(6, 1, (B, F)) * 3
    u = gem_synth.normal_f32(6, 2, (B, F))
    out = t.empty((B, F), device="cuda")
    gem.swiglu(_cu(t, g), _cu(t, u), act, out)
    t.cuda.synchronize()
    f = oracle.gelu_tanh if act else oracle.silu
    ref = np.array([[f(float(g[b, i])) * float(u[b, i]) for i in range(F)] for b in range(B)])
    assert_close(out.cpu().numpy(), ref, "activation %d" % act)


# ---- QK-norm + RoPE + append ----------------------------------------------------------------

ROPE_CASES = [
    # (n_q, n_kv, d, rope_dim, theta, v_mode, window, pos list, cap)
    (4, 2, 64, 64, 1e6, 0, 0, [128], 129),
    (16, 8, 128, 128, 1e6, 0, 0, [4096], 4097),
    (32, 8, 128, 128, 1e6, 0, 0, [2048, 0, 17, 2047, 1, 5, 100, 2000], 2049),
    (32, 16, 256, 256, 1e4, 0, 1024, [32768], 1024),
    (32, 4, 512, 128, 1e6, 1, 0, [32768], 32769),
]


@pytest.mark.parametrize("case", ROPE_CASES, ids=lambda c: "d%d_R%d_v%d_w%d_B%d" % (c[2], c[3], c[5], c[6], len(c[7])))
def test_qknorm_rope_append(gem, torch_mod, case):
    t = torch_mod
    n_q, n_kv, d, R, theta, v_mode, window, pos_l, cap = case
    B = len(pos_l)
    nqkv = (n_q + n_kv + (0 if v_mode else n_kv)) * d
    qkv = gem_synth.normal_f32(7, d, (B, nqkv)) * 2
    gq = gem_synth.norm_weight(7, 1, d)
    gk = gem_synth.norm_weight(7, 2, d)
    kc = gem_synth.normal_f16_bits(7, 3, (B, n_kv, cap, d))
    vc = gem_synth.normal_f16_bits(7, 4, (B, n_kv, cap, d))
    pos = np.array(pos_l, np.int32)
    dq, dk, dv = _cu(t, qkv), _half_cache(t, kc), _half_cache(t, vc)
    gem.rmsnorm_qknorm_rope(dq, n_q, n_kv, d, _cu(t, gq), _cu(t, gk), v_mode, 1e-6, _cu(t, pos), theta,
                            R, dk, dv, window)
    t.cuda.synchronize()
    got = dq.cpu().numpy()
    gk_bits, gv_bits = _bits(dk), _bits(dv)
    for b in range(B):
        p = int(pos[b])
        slot = p % window if window else p
        q = qkv[b, :n_q * d].reshape(n_q, d).astype(np.float64)
        k = qkv[b, n_q * d:(n_q + n_kv) * d].reshape(n_kv, d).astype(np.float64)
        rq = np.stack([oracle.rope_neox(oracle.rmsnorm(h, gq, 1e-6), R, p, theta) for h in q])
        rk = np.stack([oracle.rope_neox(oracle.rmsnorm(h, gk, 1e-6), R, p, theta) for h in k])
        if v_mode:
            rv = np.stack([oracle.rmsnorm(h, None, 1e-6) for h in k])
        else:
            rv = qkv[b, (n_q + n_kv) * d:].reshape(n_kv, d).astype(np.float64)
        assert_close(got[b, :n_q * d], rq.reshape(-1), "rope q b=%d" % b)
        assert_close(got[b, n_q * d:(n_q + n_kv) * d], rk.reshape(-1), "rope k b=%d" % b)
        for which, gbits, vals in ((0, gk_bits, rk), (1, gv_bits, rv)):
            g = gbits[b, :, slot]
            nd = 0
            for j in range(n_kv):
                rms = float(np.sqrt(np.mean(vals[j] ** 2)))
                for i in range(d):
                    v = float(vals[j, i])
                    if g[j, i] != oracle.double_to_half_via_f32(v):
                        assert _code_in_band(int(g[j, i]), v, rms)
                        nd += 1
            assert nd <= max(2, 0.005 * n_kv * d)
        # all other slots untouched
        mask = np.ones(cap, bool)
        mask[slot] = False
        assert np.array_equal(gk_bits[b][:, mask], kc[b][:, mask])
        assert np.array_equal(gv_bits[b][:, mask], vc[b][:, mask])


def test_rope_bad_position_flags_and_skips(gem, torch_mod):
    t = torch_mod
    n_q, n_kv, d, cap = 2, 1, 64, 8
    qkv = _cu(t, gem_synth.normal_f32(8, 1, (1, (n_q + 2 * n_kv) * d)))
    before = qkv.clone()
    kc = t.zeros((1, n_kv, cap, d), dtype=t.int16, device="cuda")
    vc = t.zeros_like(kc)
    status = t.zeros(1, dtype=t.int32, device="cuda")
    gem.rmsnorm_qknorm_rope(qkv, n_q, n_kv, d, None, None, 0, 1e-6, _cu(t, np.array([8], np.int32)), 1e6, d,
                            kc, vc, 0, status=status)
    t.cuda.synchronize()
    assert int(status.item()) & gem.DEVFLAG_POS_RANGE
    assert t.equal(qkv, before) and int(kc.abs().sum()) == 0


# ---- attention ----------------------------------------------------------------------------------

ATTN_CASES = [
    # (n_q, n_kv, d, window, positions, cap, scale)
    (4, 2, 64, 0, [128], 129, 0.125),
    (4, 4, 64, 0, [0], 1, 0.125),                       # one cached position: output = V
    (8, 1, 64, 0, [15], 16, 0.125),                     # G = 8
    (16, 8, 128, 0, [4096], 4097, 128 ** -0.5),         # Qwen3-1.7B shape
    (32, 8, 128, 0, [2048] * 8, 2049, 128 ** -0.5),     # Qwen3-4B shape, B = 8
    (32, 8, 128, 0, [0, 1, 63, 64, 65, 700, 1500, 2048], 2049, 128 ** -0.5),  # ragged lengths
    (32, 16, 256, 1024, [32768], 1024, 1.0),            # Gemma SWA ring, full ring
    (32, 16, 256, 1024, [700], 1024, 1.0),              # ring not yet full
    (32, 4, 512, 0, [32768], 32769, 1.0),               # Gemma full-attention shape
    (6, 2, 256, 0, [5000], 5001, 0.0625),
    (16, 8, 128, 0, [0], 4097, 128 ** -0.5),            # a long cache with one position: one split
    (16, 8, 128, 0, [20], 4097, 128 ** -0.5),           #   and two of the planned splits busy
]


@pytest.mark.parametrize("case", ATTN_CASES, ids=lambda c: "G%d_d%d_w%d_p%d_B%d" % (c[0] // c[1], c[2], c[3], max(c[4]), len(c[4])))
def test_attention_matches_oracle(gem, torch_mod, case):
    t = torch_mod
    n_q, n_kv, d, window, pos_l, cap, scale = case
    B = len(pos_l)
    q = gem_synth.normal_f32(9, d, (B, n_q * d))
    kc = gem_synth.normal_f16_bits(9, 1, (B, n_kv, cap, d))
    vc = gem_synth.normal_f16_bits(9, 2, (B, n_kv, cap, d))
    pos = np.array(pos_l, np.int32)
    ws_bytes = gem.gqa_decode_attn_workspace(B, n_q, n_kv, d, cap, window)
    ws = t.empty(max(ws_bytes, 1), dtype=t.uint8, device="cuda")
    out = t.full((B, n_q * d), float("nan"), device="cuda")
    gem.gqa_decode_attn(_cu(t, q), _half_cache(t, kc), _half_cache(t, vc), n_q, n_kv, d, _cu(t, pos), window,
                        scale, out, ws if ws_bytes else None)
    t.cuda.synchronize()
    got = out.cpu().numpy()
    for b in range(B):
        ref = oracle.gqa_attention(q[b].reshape(n_q, d), kc[b], vc[b], int(pos[b]), window, scale)
        assert_close(got[b], ref.reshape(-1), "attention b=%d p=%d" % (b, pos[b]))
    assert gem.device_status() == 0


def test_attention_deterministic_repeat(gem, torch_mod):
    t = torch_mod
    n_q, n_kv, d, cap = 32, 4, 512, 9000
    q = _cu(t, gem_synth.normal_f32(10, 1, (1, n_q * d)))
    kc = _half_cache(t, gem_synth.normal_f16_bits(10, 2, (1, n_kv, cap, d)))
    vc = _half_cache(t, gem_synth.normal_f16_bits(10, 3, (1, n_kv, cap, d)))
    pos = _cu(t, np.array([cap - 1], np.int32))
    ws = t.empty(gem.gqa_decode_attn_workspace(1, n_q, n_kv, d, cap, 0), dtype=t.uint8, device="cuda")
    o1 = t.empty((1, n_q * d), device="cuda")
    o2 = t.empty((1, n_q * d), device="cuda")
    gem.gqa_decode_attn(q, kc, vc, n_q, n_kv, d, pos, 0, 1.0, o1, ws)
    gem.gqa_decode_attn(q, kc, vc, n_q, n_kv, d, pos, 0, 1.0, o2, ws)
    t.cuda.synchronize()
    assert t.equal(o1, o2)


def test_attention_deterministic_repeat_flash(gem, torch_mod):
    t = torch_mod
    n_q, n_kv, d, cap = 16, 8, 128, 4097
    q = _cu(t, gem_synth.normal_f32(11, 1, (1, n_q * d)))
    kc = _half_cache(t, gem_synth.normal_f16_bits(11, 2, (1, n_kv, cap, d)))
    vc = _half_cache(t, gem_synth.normal_f16_bits(11, 3, (1, n_kv, cap, d)))
    pos = _cu(t, np.array([cap - 1], np.int32))
    need = gem.gqa_decode_attn_workspace(1, n_q, n_kv, d, cap, 0)
    # the workspace starts as garbage: a stand-alone call writes every split partial it reads
    ws = t.full((max(need, 1),), 0xFF, dtype=t.uint8, device="cuda")
    outs = [t.empty((1, n_q * d), device="cuda") for _ in range(10)]
    for o in outs:   # which split merges varies from call to call; the result must not
        gem.gqa_decode_attn(q, kc, vc, n_q, n_kv, d, pos, 0, 1.0, o, ws if need else None)
    t.cuda.synchronize()
    for o in outs[1:]:
        assert t.equal(outs[0], o)
    ref = oracle.gqa_attention(q.cpu().numpy().reshape(n_q, d), _bits(kc)[0], _bits(vc)[0], cap - 1, 0, 1.0)
    assert_close(outs[0].cpu().numpy()[0], ref.reshape(-1), "attention after a garbage workspace")


def test_decode_layer_workspace_may_start_as_garbage(gem, torch_mod):
    """The layer chain's QKV projection clears the attention's arrival counters, so a layer
    workspace that starts as arbitrary bytes gives the same result as a zeroed one."""
    t = torch_mod
    shape, B, pos_l = configs.QWEN3_1_7B, 1, [1024]
    pos = np.array(pos_l, np.int32)
    cap = 1025
    tens = configs.layer_tensors(shape, B, cap, 3, 0)
    x = gem_synth.normal_f32(3, gem_synth.tid(0, gem_synth.ROLE_X), (B, shape.H))
    dl = gem.DeviceLayer(shape, tens)
    outs = []
    for fill in (0, 0xFF, 0x01):
        dx = _cu(t, x)
        dk, dv = _half_cache(t, tens.k_cache), _half_cache(t, tens.v_cache)
        ws = t.full((gem.decode_layer_workspace(dl, B, cap),), fill, dtype=t.uint8, device="cuda")
        gem.decode_layer(dl, dx, dk, dv, _cu(t, pos), ws)
        outs.append(dx)
    t.cuda.synchronize()
    assert t.equal(outs[0], outs[1]) and t.equal(outs[0], outs[2])


def test_attention_needs_workspace(gem, torch_mod):
    """The d = 512 kernel merges its splits through a caller workspace."""
    t = torch_mod
    n_q, n_kv, d, cap = 8, 4, 512, 4097
    need = gem.gqa_decode_attn_workspace(1, n_q, n_kv, d, cap, 0)
    assert need > 0
    q = t.zeros((1, n_q * d), device="cuda")
    kc = t.zeros((1, n_kv, cap, d), dtype=t.int16, device="cuda")
    with pytest.raises(gem.GemError):
        gem.gqa_decode_attn(q, kc, kc, n_q, n_kv, d, _cu(t, np.array([4096], np.int32)), 0, 1.0,
                            t.empty((1, n_q * d), device="cuda"), t.empty(need - 256, dtype=t.uint8, device="cuda"))


# ---- one decoder layer step ----------------------------------------------------------------------
#
# The new token's K and V rows are rounded to binary16 from fp32 (GPU) or from fp64 via
# fp32 (oracle).  Where the value lies within the fp32 arithmetic's precision of a binary16
# midpoint, both codes are valid outcomes.  The test accepts a differing code only if it
# is the other neighbour of the oracle's value and the oracle marks that value ambiguous
# (within EPS_KV of the midpoint, relative to the head's RMS); downstream outputs are then
# compared with the oracle evaluated for that same outcome.

def _small_gemma(full: bool):
    base = configs.GEMMA31_FULL if full else configs.GEMMA31_SWA
    return replace(base, H=512, n_q=8, n_kv=2 if full else 4, d=64 if not full else 128, F=1024,
                   rope_dim=32 if full else 64, window=0 if full else 64)


def _gpu_layer(gem, t, shape, tens, x, pos, cap):
    B = x.shape[0]
    dl = gem.DeviceLayer(shape, tens)
    dx = _cu(t, np.ascontiguousarray(x, dtype=np.float32))
    dk, dv = _half_cache(t, tens.k_cache), _half_cache(t, tens.v_cache)
    ws = t.empty(gem.decode_layer_workspace(dl, B, cap), dtype=t.uint8, device="cuda")
    status = t.zeros(1, dtype=t.int32, device="cuda")
    gem.decode_layer(dl, dx, dk, dv, _cu(t, pos), ws, status=status)
    t.cuda.synchronize()
    return dx.cpu().numpy(), _bits(dk), _bits(dv), int(status.item())


def _layer_parity(shape, tens, x, pos, got, gk, gv, what):
    """Compare one GPU layer step with the oracle; returns the number of appended codes
    on the other side of an ambiguous rounding decision."""
    xin = np.ascontiguousarray(x, dtype=np.float32)
    kc, vc = tens.k_cache.copy(), tens.v_cache.copy()
    ref, kvn = oracle.decode_layer(shape, tens, xin, pos, kc, vc, kvnew=True)
    B, n_kv, d = len(pos), shape.n_kv, shape.d
    flip = np.zeros((B, 2, n_kv, d), np.int8)
    for b in range(B):
        p = int(pos[b])
        slot = p % shape.window if shape.window else p
        for which, gbits, obits in ((0, gk, kc), (1, gv, vc)):
            g, o = gbits[b, :, slot], obits[b, :, slot]
            for j, i in np.argwhere(g != o):
                v = kvn[b, which, j, i]
                rms = float(np.sqrt(np.mean(kvn[b, which, j] ** 2)))
                assert _code_in_band(int(g[j, i]), v, rms), \
                    "%s: appended code outside the fp32 precision band of the value" % what
                if g[j, i] == oracle.other_half_via_f32(v):
                    flip[b, which, j, i] = 1
        mask = np.ones(gk.shape[2], bool)
        mask[slot] = False
        assert np.array_equal(gk[b][:, mask], tens.k_cache[b][:, mask]), "%s: other K slots changed" % what
        assert np.array_equal(gv[b][:, mask], tens.v_cache[b][:, mask]), "%s: other V slots changed" % what
    nflip = int(flip.sum())
    assert nflip <= max(2, 0.01 * flip.size), "%s: %d rounding decisions differ" % (what, nflip)
    if nflip:
        ref = oracle.decode_layer(shape, tens, xin, pos, tens.k_cache.copy(), tens.v_cache.copy(),
                                  flip=flip)
    assert_close(got, ref, what)
    return nflip, ref


def _oracle_follow_gpu(shape, tens, x, pos, k_cache, v_cache, gk, gv, what):
    """One oracle layer step from x on caches (k_cache, v_cache: the state before the step;
    updated in place with the GPU's appended rows), following the GPU's binary16 rounding
    decisions of the new rows where they are ambiguous (gk, gv: the GPU's caches after the
    step).  Returns the oracle's output (fp64)."""
    xin = np.ascontiguousarray(x, dtype=np.float64)
    kc, vc = k_cache.copy(), v_cache.copy()
    ref, kvn = oracle.decode_layer(shape, tens, xin, pos, kc, vc, kvnew=True)
    B, n_kv, d = len(pos), shape.n_kv, shape.d
    flip = np.zeros((B, 2, n_kv, d), np.int8)
    for b in range(B):
        p = int(pos[b])
        slot = p % shape.window if shape.window else p
        for which, gbits, obits in ((0, gk, kc), (1, gv, vc)):
            g, o = gbits[b, :, slot], obits[b, :, slot]
            for j, i in np.argwhere(g != o):
                v = kvn[b, which, j, i]
                rms = float(np.sqrt(np.mean(kvn[b, which, j] ** 2)))
                assert _code_in_band(int(g[j, i]), v, rms), \
                    "%s: appended code outside the fp32 precision band of the value" % what
                if g[j, i] == oracle.other_half_via_f32(v):
                    flip[b, which, j, i] = 1
        k_cache[b, :, slot] = gk[b, :, slot]
        v_cache[b, :, slot] = gv[b, :, slot]
    nflip = int(flip.sum())
    assert nflip <= max(2, 0.01 * flip.size), "%s: %d rounding decisions differ" % (what, nflip)
    if nflip:
        kc, vc = k_cache.copy(), v_cache.copy()
        # (the GPU's rows are already in place; the oracle rewrites them with the same codes)
        ref = oracle.decode_layer(shape, tens, xin, pos, kc, vc, flip=flip)
    return ref


LAYER_CASES = [
    ("tiny", configs.TINY, 1, [128]),
    ("qwen3-1.7b", configs.QWEN3_1_7B, 1, [4096]),
    ("qwen3-4b-b8", configs.QWEN3_4B, 8, [2048] * 8),
    ("qwen3-4b-ragged", configs.QWEN3_4B, 3, [0, 1000, 2048]),
    ("gemma-small-swa", _small_gemma(False), 2, [200, 30]),
    ("gemma-small-full", _small_gemma(True), 1, [300]),
    ("gemma4-31b-swa", configs.GEMMA31_SWA, 1, [32768]),
    ("gemma4-31b-full", configs.GEMMA31_FULL, 1, [32768]),
    # hidden 16384: the QKV and fused gate/up projections split K over CTA pairs
    ("wide-hidden", replace(configs.QWEN3_1_7B, H=16384, F=2816), 1, [700]),
]


@pytest.mark.parametrize("name,shape,B,pos_l", LAYER_CASES, ids=[c[0] for c in LAYER_CASES])
def test_decode_layer_matches_oracle(gem, torch_mod, name, shape, B, pos_l):
    pos = np.array(pos_l, np.int32)
    cap = shape.window if shape.window else int(pos.max()) + 1
    tens = configs.layer_tensors(shape, B, cap, 0, 0)
    x = gem_synth.normal_f32(0, gem_synth.tid(0, gem_synth.ROLE_X), (B, shape.H))
    got, gk, gv, status = _gpu_layer(gem, torch_mod, shape, tens, x, pos, cap)
    assert status == 0
    _layer_parity(shape, tens, x, pos, got, gk, gv, "layer %s" % name)


@pytest.mark.parametrize("name,nlayers", [("qwen3-1.7b", 4), ("gemma4-31b-group", 6)])
def test_decode_layer_stack_each_layer_from_oracle_input(gem, torch_mod, name, nlayers):
    """Stacked layers, each with its own weights and cache.  Layer l runs on both sides
    from the oracle's output of layer l - 1 (rounded to fp32), so error does not compound
    through the comparison; the oracle chain itself is carried in fp64."""
    t = torch_mod
    wl = configs.with_layers(configs.workload(name), nlayers)
    if name == "qwen3-1.7b":
        wl = replace(wl, pos=1024, cache_cap=(1025,) * nlayers)
    pos = np.full(wl.B, wl.pos, np.int32)
    x = gem_synth.normal_f32(0, gem_synth.tid(0, gem_synth.ROLE_X), (wl.B, wl.layers[0].H)).astype(np.float64)
    for layer, (shape, cap) in enumerate(zip(wl.layers, wl.cache_cap)):
        tens = configs.layer_tensors(shape, wl.B, cap, 11, layer)
        got, gk, gv, status = _gpu_layer(gem, t, shape, tens, x, pos, cap)
        assert status == 0
        _, ref = _layer_parity(shape, tens, x, pos, got, gk, gv, "%s layer %d" % (name, layer))
        x = ref


# ---- logit projection + argmax (test only) ---------------------------------------------------
#
# A Q4_0 GEMV from the final hidden state to a Qwen3-size vocabulary, then the token choice:
# the GPU logits must match the oracle's within the parity tolerance and pick the same argmax
# (lowest index on ties).  Rows whose oracle top-2 gap is within twice the max-abs tolerance are
# ambiguous by construction and are counted, not asserted.

@pytest.mark.parametrize("B", [1, 8])
def test_logit_projection_argmax(gem, torch_mod, B):
    from parity import MAX_ABS
    t = torch_mod
    V, H = 151936, 2048
    W = gem_synth.q4_0_matrix(7, 77, V, H)
    x = gem_synth.normal_f32(7, 78, (B, H))
    ref = oracle.q4_0_gemv(W, V, H, x)
    y = t.full((B, V), float("nan"), device="cuda")
    gem.q4_0_gemv(_cu(t, W), V, H, _cu(t, x), y)
    got_idx = t.argmax(y, dim=1).cpu().numpy()   # first maximal index
    t.cuda.synchronize()
    assert_close(y.cpu().numpy(), ref, "logits B=%d" % B)
    decided = 0
    for b in range(B):
        top2 = np.sort(ref[b])[-2:]
        if top2[1] - top2[0] < 2 * MAX_ABS:
            continue
        assert int(got_idx[b]) == oracle.argmax(ref[b]), "row %d: GPU argmax %d, oracle %d" % (
            b, int(got_idx[b]), oracle.argmax(ref[b]))
        decided += 1
    assert decided >= 1
