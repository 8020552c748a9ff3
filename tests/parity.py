"""Shared comparison helpers for the GPU-vs-oracle parity tests.

Tolerance (stated for this library's fp32-accumulating kernels against the fp64 oracle):
max-abs error <= 2e-3 and relative L2 error <= 1e-5 on every compared output."""
import json
import os

import numpy as np

MAX_ABS = 2e-3
REL_L2 = 1e-5


def errors(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    diff = got - ref
    ma = float(np.max(np.abs(diff))) if diff.size else 0.0
    den = float(np.linalg.norm(ref))
    rl = float(np.linalg.norm(diff)) / den if den > 0 else float(np.linalg.norm(diff))
    return ma, rl


def assert_close(got, ref, what, max_abs=MAX_ABS, rel_l2=REL_L2):
    assert np.all(np.isfinite(np.asarray(got, dtype=np.float64))), "%s: non-finite output" % what
    ma, rl = errors(got, ref)
    log = os.environ.get("GEM_PARITY_LOG")
    if log:
        with open(log, "a") as f:
            f.write(json.dumps({"what": what, "max_abs": ma, "rel_l2": rl}) + "\n")
    assert ma <= max_abs and rl <= rel_l2, "%s: max_abs=%.3e rel_l2=%.3e" % (what, ma, rl)
    return ma, rl


def f16_ulp_diff(a_bits, b_bits):
    """Distance in binary16 units between two arrays of bit patterns (same sign assumed
    close to zero handled by integer ordering)."""
    a = np.asarray(a_bits).astype(np.uint16).astype(np.int32)
    b = np.asarray(b_bits).astype(np.uint16).astype(np.int32)
    # map sign-magnitude to a monotone integer line
    a = np.where(a & 0x8000, -(a & 0x7FFF), a)
    b = np.where(b & 0x8000, -(b & 0x7FFF), b)
    return np.abs(a - b)


def scale_q4_0(W, shift):
    """The same Q4_0 matrix (raw 18-byte blocks) with every block scale multiplied by
    2^-shift, exactly: the binary16 exponent field is lowered by `shift`, which every scale
    must survive as a normal number.  Used to keep a stack of random-weight layers' residual
    stream near one layer's output scale, so the absolute tolerance keeps its meaning."""
    blocks = np.asarray(W).reshape(-1, 18).copy()
    d = blocks[:, 0].astype(np.uint16) | (blocks[:, 1].astype(np.uint16) << 8)
    e = (d >> 10) & 0x1F
    assert np.all(e > shift) and np.all(e < 31), "a scale would leave the normal range"
    d = d - np.uint16(shift << 10)
    blocks[:, 0] = (d & 0xFF).astype(np.uint8)
    blocks[:, 1] = (d >> 8).astype(np.uint8)
    return blocks.reshape(np.asarray(W).shape)
