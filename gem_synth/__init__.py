"""Seeded synthetic inputs shared by the oracle tests, the CUDA parity tests and bench.py.

This module only draws random bytes and floats; it holds none of the decoder-step
arithmetic (no dequantisation, no norms, no RoPE, no attention).  Both sides of every
parity check receive exactly the bytes produced here.

Generator (counter-based, stateless):
  * splitmix64 finaliser  mix(z) = z ^ (z >> 31) after the two xor-shift-multiply rounds
    with constants 0xBF58476D1CE4E5B9 and 0x94D049BB133111EB (Steele, Lea, Flood,
    "Fast splittable pseudorandom number generators", OOPSLA 2014).
  * stream key  k(seed, tid) = mix(mix(seed + gamma) ^ (tid * 0xD1B54A32D192ED03))
    with gamma = 0x9E3779B97F4A7C15, and draw i of stream (seed, tid) is
    u64(i) = mix(k + (i + 1) * gamma)   (mod 2**64).
  * uniform in [0, 1): (u64 >> 11) * 2**-53.
  * normal: Box-Muller in double from draws 2i and 2i+1:
    sqrt(-2 ln(1 - u_{2i})) * cos(2 pi u_{2i+1}); then round-to-nearest-even to the
    target type (fp32 or fp16).

Workload value distributions follow the decode configurations the library is measured
on: Q4_0 nibbles uniform on 0..15, fp16 block scales uniform on [0.002, 0.02],
activations N(0,1) fp32, KV cache N(0,1) fp16, norm weights 1 + N(0, 0.1) fp32.
"""
from __future__ import annotations

import numpy as np

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_TID_MUL = np.uint64(0xD1B54A32D192ED03)

# Q4_0 block: 2-byte little-endian binary16 scale followed by 16 bytes of nibbles.
Q4_0_BLOCK_BYTES = 18
Q4_0_BLOCK_ELEMS = 32


def _mix(z: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        return z ^ (z >> np.uint64(31))


def stream_key(seed: int, tid: int) -> np.uint64:
    with np.errstate(over="ignore"):
        s = np.array([seed], dtype=np.uint64) + _GAMMA
        k = _mix(s) ^ (np.array([tid], dtype=np.uint64) * _TID_MUL)
        return _mix(k)[0]


def draws(seed: int, tid: int, count: int, start: int = 0) -> np.ndarray:
    """u64 draws start .. start+count-1 of stream (seed, tid)."""
    k = stream_key(seed, tid)
    idx = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix(k + idx * _GAMMA)


def uniform(seed: int, tid: int, count: int) -> np.ndarray:
    u = draws(seed, tid, count)
    return (u >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


_CHUNK = 1 << 22


def normal(seed: int, tid: int, count: int, out_dtype=np.float64) -> np.ndarray:
    """count N(0,1) values; value i uses draws 2i and 2i+1 (generated in chunks)."""
    out = np.empty(count, dtype=out_dtype)
    for s in range(0, count, _CHUNK):
        n = min(_CHUNK, count - s)
        out[s:s + n] = _normal_range(seed, tid, s, n)
    return out


def normal_f32(seed: int, tid: int, shape, mean: float = 0.0, std: float = 1.0) -> np.ndarray:
    n = int(np.prod(shape)) if len(shape) else 1
    return (mean + std * normal(seed, tid, n)).astype(np.float32).reshape(shape)


def normal_f16_bits(seed: int, tid: int, shape) -> np.ndarray:
    """N(0,1) rounded to binary16; returned as the uint16 bit patterns."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.float16)
    for s in range(0, n, _CHUNK):
        m = min(_CHUNK, n - s)
        out[s:s + m] = _normal_range(seed, tid, s, m).astype(np.float16)
    return out.view(np.uint16).reshape(shape)


def _normal_range(seed: int, tid: int, start: int, n: int) -> np.ndarray:
    k = stream_key(seed, tid)
    idx = np.arange(2 * start + 1, 2 * (start + n) + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        u = _mix(k + idx * _GAMMA)
    u1 = (u[0::2] >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
    u2 = (u[1::2] >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
    return np.sqrt(-2.0 * np.log1p(-u1)) * np.cos(2.0 * np.pi * u2)


def q4_0_matrix(seed: int, tid: int, n_rows: int, k: int,
                scale_lo: float = 0.002, scale_hi: float = 0.02) -> np.ndarray:
    """Random Q4_0 matrix bytes, shape (n_rows, k // 32 * 18), uint8.

    Each block's 16 nibble bytes come from two u64 draws (every nibble uniform on
    0..15); its scale is uniform on [scale_lo, scale_hi] rounded to binary16 and
    stored little-endian in the block's first two bytes.
    """
    if k % Q4_0_BLOCK_ELEMS:
        raise ValueError("k must be a multiple of 32")
    nb = n_rows * (k // Q4_0_BLOCK_ELEMS)
    out = np.empty((nb, Q4_0_BLOCK_BYTES), dtype=np.uint8)
    payload = draws(seed, tid, 2 * nb)                       # 16 bytes per block
    out[:, 2:] = payload.view(np.uint8).reshape(nb, 16)
    u = draws(seed, tid, nb, start=2 * nb)
    sc = scale_lo + (scale_hi - scale_lo) * ((u >> np.uint64(11)).astype(np.float64) * (2.0 ** -53))
    out[:, 0:2] = sc.astype(np.float16).view(np.uint8).reshape(nb, 2)
    return out.reshape(n_rows, (k // Q4_0_BLOCK_ELEMS) * Q4_0_BLOCK_BYTES)


Q8_0_BLOCK_BYTES = 34


def q8_0_matrix(seed: int, tid: int, n_rows: int, k: int,
                scale_lo: float = 0.0002, scale_hi: float = 0.002) -> np.ndarray:
    """Random Q8_0 matrix bytes, shape (n_rows, k // 32 * 34), uint8.

    Each block's 32 code bytes come from four u64 draws (every code uniform on the 256
    int8 values); its scale is uniform on [scale_lo, scale_hi] rounded to binary16 and
    stored little-endian in the block's first two bytes.
    """
    if k % Q4_0_BLOCK_ELEMS:
        raise ValueError("k must be a multiple of 32")
    nb = n_rows * (k // Q4_0_BLOCK_ELEMS)
    out = np.empty((nb, Q8_0_BLOCK_BYTES), dtype=np.uint8)
    payload = draws(seed, tid, 4 * nb)                       # 32 bytes per block
    out[:, 2:] = payload.view(np.uint8).reshape(nb, 32)
    u = draws(seed, tid, nb, start=4 * nb)
    sc = scale_lo + (scale_hi - scale_lo) * ((u >> np.uint64(11)).astype(np.float64) * (2.0 ** -53))
    out[:, 0:2] = sc.astype(np.float16).view(np.uint8).reshape(nb, 2)
    return out.reshape(n_rows, (k // Q4_0_BLOCK_ELEMS) * Q8_0_BLOCK_BYTES)


def norm_weight(seed: int, tid: int, n: int) -> np.ndarray:
    """RMSNorm weight ~ 1 + N(0, 0.1), fp32."""
    return normal_f32(seed, tid, (n,), mean=1.0, std=0.1)


# Tensor ids: a layer's tensors live at layer * 64 + role.
ROLE_X = 1
ROLE_W_QKV = 2
ROLE_W_O = 3
ROLE_W_GATE = 4
ROLE_W_UP = 5
ROLE_W_DOWN = 6
ROLE_G_ATTN = 7
ROLE_G_FFN = 8
ROLE_G_Q = 9
ROLE_G_K = 10
ROLE_K_CACHE = 11
ROLE_V_CACHE = 12
ROLE_G_POST_ATTN = 13
ROLE_G_POST_FFN = 14
ROLE_Q = 15
ROLE_GATE = 16
ROLE_UP = 17
ROLE_W_LOGIT = 18


def tid(layer: int, role: int) -> int:
    return layer * 64 + role
