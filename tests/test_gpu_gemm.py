"""The batched prefill Q4_0 GEMM (9..32 activation rows) against the oracle (GPU only).

"gem" research record, "Native Metal diagnostic: buffer ownership": the batched-Q4 prefill
operator reuses each dequantised weight tile across up to 32 prompt rows with fp32
accumulation.  gem_q4_0_gemm must give, for every row, the oracle's fp64 GEMV of that row
(exact weights (q - 8) * d), with the optional pre-norm, gate/up pair with its activation and
residual of the fused decode GEMV, at the tolerances of tests/parity.py.  Cases cover one,
two and four column tiles of 8 rows with ragged last tiles, ragged N, several phases, several
passes over a CTA's units, and the Gemma 4 31B FFN shape (K 5376, N 21504) at 32 rows."""
import numpy as np
import pytest

import gem_synth
import oracle
from parity import assert_close
from test_gpu_parity import _cu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import q4_gemv_gqa_gb300 as g
    g.device_status(reset=True)
    return g, torch


def _ref(W0, W1, N, K, x, gamma, eps, act, r):
    M = x.shape[0]
    xh = np.stack([oracle.rmsnorm(x[b].astype(np.float64), gamma, eps) for b in range(M)]) if gamma is not None else x
    y0 = oracle.q4_0_gemv(W0, N, K, xh) if gamma is not None else oracle.q4_0_gemv(W0, N, K, xh, r)
    if W1 is None:
        return y0
    y1 = oracle.q4_0_gemv(W1, N, K, xh)
    f = oracle.gelu_tanh if act else oracle.silu
    return np.array([[f(float(y0[b, n])) * float(y1[b, n]) for n in range(N)] for b in range(M)])


GEMM_CASES = [
    # (N, K, M, pair, norm, residual, act)
    (37, 256, 9, False, False, False, 0),        # two column tiles, the second one row wide
    (100, 1280, 16, False, False, True, 0),      # two full tiles, residual
    (333, 2048, 17, False, True, False, 0),      # four tiles (17..32 rows), pre-norm
    (520, 2560, 24, True, True, False, 1),       # gate/up pair, GELU-tanh
    (2048, 6144, 32, False, False, True, 0),     # Qwen3-1.7B down projection shape, 32 rows
    (6144, 2048, 32, True, True, False, 0),      # Qwen3-1.7B gate/up pair, 32 rows
    (4096, 2048, 12, False, True, False, 0),     # Qwen3-1.7B QKV projection
    (40, 224, 20, False, False, False, 0),       # K % 256 != 0: chunks of 8 rows on the general path
]


@pytest.mark.parametrize("case", GEMM_CASES,
                         ids=lambda c: "N%d_K%d_M%d_%s%s%s" % (c[0], c[1], c[2], "pair" if c[3] else "one",
                                                                "_norm" if c[4] else "", "_res" if c[5] else ""))
def test_gemm_matches_oracle(env, case):
    g, t = env
    N, K, M, pair, norm, res, act = case
    W0 = gem_synth.q4_0_matrix(41, 1, N, K)
    W1 = gem_synth.q4_0_matrix(41, 2, N, K) if pair else None
    x = gem_synth.normal_f32(41, 3, (M, K)) * 3
    gamma = gem_synth.norm_weight(41, 4, K) if norm else None
    r = gem_synth.normal_f32(41, 5, (M, N)) if res else None
    eps = 1e-6
    y = t.full((M, N), float("nan"), device="cuda")
    g.q4_0_gemm(_cu(t, W0), None if W1 is None else _cu(t, W1), N, K, _cu(t, x), y,
                gamma=None if gamma is None else _cu(t, gamma), eps=eps, act=act,
                residual=None if r is None else _cu(t, r))
    t.cuda.synchronize()
    assert_close(y.cpu().numpy(), _ref(W0, W1, N, K, x, gamma, eps, act, r), "prefill GEMM %s" % (case,))
    assert g.device_status() == 0


def test_gemm_31b_ffn_shape_32_rows(env):
    """K 5376 -> N 21504 at 32 rows: every row against the oracle."""
    g, t = env
    N, K, M = 21504, 5376, 32
    W = gem_synth.q4_0_matrix(42, 1, N, K)
    x = gem_synth.normal_f32(42, 2, (M, K))
    y = t.full((M, N), float("nan"), device="cuda")
    g.q4_0_gemm(_cu(t, W), None, N, K, _cu(t, x), y)
    t.cuda.synchronize()
    assert_close(y.cpu().numpy(), oracle.q4_0_gemv(W, N, K, x), "prefill GEMM 31B FFN shape, 32 rows")


def test_gemm_rows_independent_and_deterministic(env):
    """Row b of a 32-row call equals the one-row decode GEMV of row b within the tolerance, and
    repeated calls are bit-identical."""
    g, t = env
    N, K, M = 1000, 3072, 32
    W = _cu(t, gem_synth.q4_0_matrix(43, 1, N, K))
    x = _cu(t, gem_synth.normal_f32(43, 2, (M, K)))
    ys = []
    for _ in range(3):
        y = t.empty((M, N), device="cuda")
        g.q4_0_gemm(W, None, N, K, x, y)
        ys.append(y)
    y1 = t.empty((M, N), device="cuda")
    for b in range(M):
        g.q4_0_gemv(W, N, K, x[b:b + 1], y1[b:b + 1])
    t.cuda.synchronize()
    for y in ys[1:]:
        assert t.equal(y, ys[0])
    assert_close(ys[0].cpu().numpy(), y1.cpu().numpy().astype(np.float64), "32-row GEMM vs one-row GEMVs")


def test_gemm_rejections(env):
    g, t = env
    W = t.zeros(16 * 8 * 18, dtype=t.uint8, device="cuda")
    x = t.zeros((33, 256), device="cuda")
    y = t.zeros((33, 16), device="cuda")
    with pytest.raises(g.GemError) as ei:   # more than 32 rows
        g.q4_0_gemm(W, None, 16, 256, x, y)
    assert ei.value.status == 3
    with pytest.raises(g.GemError) as ei:   # the decode entry points stay at 8 rows
        g.q4_0_gemv(W, 16, 256, x[:9], y[:9], shared_records=True)
    assert ei.value.status == 3
    assert g.q4_0_gemm_workspace(32, 5376) >= 4 * 32 * 5376
    assert g.q4_0_gemm_workspace(1, 5376) == 0
