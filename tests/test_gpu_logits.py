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
    # (N, K, B): ragged tiles, one chunk, a chunk plus a tail chunk, several chunks; one row
    # takes the CUDA-core kernel, two to eight rows the tensor-core one (32-row tiles)
    (37, 256, 1), (37, 256, 8), (16, 1024, 2), (100, 1280, 3), (5000, 2048, 5), (333, 5376, 8),
    (31, 256, 4), (1025, 5376, 6), (96, 2560, 7), (3000, 768, 2),
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


def test_q8_0_gemv_rows_of_any_scale(env):
    """Each activation row is scaled by its own power of two before the binary16 split, so
    rows far outside the binary16 range (and a zero row) give the unscaled result times the
    same power of two, whatever the other rows of the call hold."""
    g, t = env
    N, K = 300, 2304
    W = gem_synth.q8_0_matrix(22, N, N, K)
    x = gem_synth.normal_f32(22, 5, (4, K))
    shifts = [-60, 0, 40, None]   # None: the row is zero
    xs = np.stack([x[i] * np.float32(2.0 ** s) if s is not None else np.zeros(K, np.float32)
                   for i, s in enumerate(shifts)]).astype(np.float32)
    y = t.full((4, N), float("nan"), device="cuda")
    g.q8_0_gemv(_cu(t, W), N, K, _cu(t, xs), y)
    t.cuda.synchronize()
    got = y.cpu().numpy().astype(np.float64)
    ref = oracle.q8_0_gemv(W, N, K, x)
    for i, s in enumerate(shifts):
        if s is None:
            assert np.all(got[i] == 0.0), "zero row"
        else:
            assert_close(got[i] * 2.0 ** -s, ref[i], "row scaled by 2^%d" % s)
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
            continue   # ambiguous by construction: counted, not asserted
        assert int(got[b]) == oracle.argmax(ref[b]), "row %d: device argmax %d, oracle %d" % (
            b, int(got[b]), oracle.argmax(ref[b]))
        decided += 1
    assert decided >= 1
    assert g.device_status() == 0


# ---- device top-k (the sampler's list) ---------------------------------------------------------

def _check_topk(g, t, y_np, k, what):
    y = _cu(t, np.ascontiguousarray(y_np, dtype=np.float32))
    B = y.shape[0]
    idx = t.full((B, k), -7, dtype=t.int32, device="cuda")
    val = t.full((B, k), -7.0, device="cuda")
    g.topk(y, k, idx, val)
    t.cuda.synchronize()
    gi, gv = idx.cpu().numpy(), val.cpu().numpy()
    for b in range(B):
        oi, ov = oracle.topk(y_np[b].astype(np.float32).astype(np.float64), k)
        assert list(gi[b]) == list(oi), "%s row %d: %s vs %s" % (what, b, gi[b][:8], oi[:8])
        assert np.array_equal(gv[b].astype(np.float64), ov, equal_nan=True), "%s row %d values" % (what, b)


@pytest.mark.parametrize("k", [1, 5, 40, 64])
def test_topk_semantics(env, k):
    g, t = env
    N = 70000   # several chunks and a ragged last one
    r = gem_synth.normal_f32(24, 1, (N,))
    rows = [r]
    tie = np.round(r, 1).astype(np.float32)   # many equal values: ties go to the lowest index
    rows.append(tie)
    nan = r.copy()
    nan[::7] = np.nan
    rows.append(nan)
    mostly_nan = np.full(N, np.nan, np.float32)
    mostly_nan[[5, 60000]] = [-np.inf, 1.0]   # fewer numbers than k: NaN rows fill by index
    rows.append(mostly_nan)
    _check_topk(g, t, np.stack(rows), k, "top-%d semantics" % k)


@pytest.mark.parametrize("N,k", [(1, 1), (7, 7), (300, 64), (2048, 3), (151936, 40), (262144, 64)])
def test_topk_shapes(env, N, k):
    g, t = env
    _check_topk(g, t, gem_synth.normal_f32(25, N, (3, N)), k, "top-%d of %d" % (k, N))


def test_topk_of_q8_0_logits_starts_with_the_argmax(env):
    g, t = env
    V, H = 65536, 5376
    W = gem_synth.q8_0_matrix(26, V + H, V, H)
    x = gem_synth.normal_f32(26, 7, (2, H))
    y = t.empty((2, V), device="cuda")
    g.q8_0_gemv(_cu(t, W), V, H, _cu(t, x), y)
    idx = t.empty((2, 50), dtype=t.int32, device="cuda")
    val = t.empty((2, 50), device="cuda")
    g.topk(y, 50, idx, val)
    am = t.empty((2,), dtype=t.int32, device="cuda")
    g.argmax(y, am)
    t.cuda.synchronize()
    assert t.equal(idx[:, 0], am)
    yc = y.cpu().numpy()
    for b in range(2):
        oi, _ = oracle.topk(yc[b].astype(np.float64), 50)
        assert list(idx[b].cpu().numpy()) == list(oi)


def test_topk_rejections(env):
    g, t = env
    y = t.zeros((1, 100), device="cuda")
    idx = t.empty((1, 65), dtype=t.int32, device="cuda")
    val = t.empty((1, 65), device="cuda")
    with pytest.raises(g.GemError) as ei:   # k > 64
        g.topk(y, 65, idx, val)
    assert ei.value.status == 3
    with pytest.raises(g.GemError) as ei:   # k > N
        g.topk(t.zeros((1, 10), device="cuda"), 11, idx, val)
    assert ei.value.status == 1
    with pytest.raises(g.GemError) as ei:   # a row too long for k = 64
        g.topk(t.zeros((1, 262145), device="cuda"), 64, idx, val)
    assert ei.value.status == 3
