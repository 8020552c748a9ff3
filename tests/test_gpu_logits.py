"""The tied Q8_0 logit projection and the device argmax against the oracle (GPU only).

gem_q8_0_gemv is compared element by element with the oracle's fp64 Q8_0 GEMV at the
tolerances of tests/parity.py, on ragged shapes and at the two vocabulary shapes of the
pages' models (Qwen3: 151,936 x 2,048; Gemma 4 31B tied embedding: 262,144 x 5,376) for one
token and for eight.  gem_argmax must return exactly the oracle's argmax of the same values
(lowest index on ties, NaN never chosen); on the logits themselves it must match the oracle's
token wherever the oracle's top two differ by more than twice the max-abs tolerance."""
import numpy as np
import pytest

import gem_synth
import oracle
from parity import MAX_ABS, assert_close
from test_gpu_parity import _cu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import q4_gemv_gqa_gb300 as g
    g.device_status(reset=True)
    return g, torch


Q8_CASES = [
    # (N, K, B): ragged tiles, one chunk, a chunk plus a tail chunk, several chunks
    (37, 256, 1), (37, 256, 8), (16, 1024, 2), (100, 1280, 3), (5000, 2048, 5), (333, 5376, 8),
]


@pytest.mark.parametrize("N,K,B", Q8_CASES)
def test_q8_0_gemv_matches_oracle(env, N, K, B):
    g, t = env
    W = gem_synth.q8_0_matrix(21, N, N, K)
    x = gem_synth.normal_f32(21, 1000 + K, (B, K))
    y = t.full((B, N), float("nan"), device="cuda")
    g.q8_0_gemv(_cu(t, W), N, K, _cu(t, x), y)
    t.cuda.synchronize()
    assert_close(y.cpu().numpy(), oracle.q8_0_gemv(W, N, K, x), "q8_0 gemv N=%d K=%d B=%d" % (N, K, B))
    assert g.device_status() == 0


def test_q8_0_gemv_rejects_bad_shapes(env):
    g, t = env
    W = t.zeros(64 * 8 * 34, dtype=t.uint8, device="cuda")
    x = t.zeros((1, 256), device="cuda")
    y = t.zeros((1, 64), device="cuda")
    with pytest.raises(g.GemError) as ei:
        g.q8_0_gemv(W, 64, 224, x, y)   # K % 256 != 0
    assert ei.value.status == 3
    with pytest.raises(g.GemError) as ei:
        g.q8_0_gemv(W[2:], 8, 256, x, y)   # not 16-byte aligned
    assert ei.value.status == 2


def _check_argmax(g, t, y_np, what):
    y = _cu(t, np.ascontiguousarray(y_np, dtype=np.float32))
    B = y.shape[0]
    idx = t.full((B,), -7, dtype=t.int32, device="cuda")
    g.argmax(y, idx)
    t.cuda.synchronize()
    got = idx.cpu().numpy()
    for b in range(B):
        assert int(got[b]) == oracle.argmax(y_np[b].astype(np.float64)), "%s row %d" % (what, b)


def test_argmax_semantics(env):
    g, t = env
    N = 70000   # several chunks, a ragged last one
    rows = []
    r = gem_synth.normal_f32(22, 1, (N,))
    rows.append(r)
    tie = r.copy()
    m = float(tie.max()) + 1.0
    tie[[12345, 54321, 69999]] = m            # equal maxima in three chunks: the first wins
    rows.append(tie)
    nan = r.copy()
    nan[::7] = np.nan                         # NaN never chosen
    nan[0] = np.nan
    rows.append(nan)
    allnan = np.full(N, np.nan, np.float32)   # nothing to choose: 0
    rows.append(allnan)
    neg = -np.abs(r) - 1.0
    neg[N - 1] = -0.5                         # the largest at the very end
    rows.append(neg)
    _check_argmax(g, t, np.stack(rows), "argmax semantics")
    _check_argmax(g, t, np.array([[3.0]], np.float32), "one column")
    _check_argmax(g, t, gem_synth.normal_f32(22, 2, (8, 151936)), "eight rows of a Qwen3 vocabulary")


@pytest.mark.parametrize("V,H", [(151936, 2048), (262144, 5376)])
@pytest.mark.parametrize("B", [1, 8])
def test_tied_q8_0_logits_and_argmax_full_size(env, V, H, B):
    """The logit projection at the pages' vocabulary shapes, then the next token on the device."""
    g, t = env
    W = gem_synth.q8_0_matrix(23, V + H, V, H)
    x = gem_synth.normal_f32(23, 7, (B, H))
    dW = _cu(t, W)
    del W
    y = t.full((B, V), float("nan"), device="cuda")
    g.q8_0_gemv(dW, V, H, _cu(t, x), y)
    idx = t.full((B,), -1, dtype=t.int32, device="cuda")
    g.argmax(y, idx)
    t.cuda.synchronize()
    W = gem_synth.q8_0_matrix(23, V + H, V, H)
    ref = oracle.q8_0_gemv(W, V, H, x)
    del W
    assert_close(y.cpu().numpy(), ref, "tied Q8_0 logits V=%d H=%d B=%d" % (V, H, B))
    got = idx.cpu().numpy()
    decided = 0
    for b in range(B):
        top2 = np.sort(ref[b])[-2:]
        if top2[1] - top2[0] < 2 * MAX_ABS:
            continue   # ambiguous by construction: counted, not judged
        assert int(got[b]) == oracle.argmax(ref[b]), "row %d: device argmax %d, oracle %d" % (
            b, int(got[b]), oracle.argmax(ref[b]))
        decided += 1
    assert decided >= 1
    assert g.device_status() == 0
