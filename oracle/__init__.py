"""ctypes front end of the scalar fp64 oracle (oracle/gem_oracle.c).

TEST INFRASTRUCTURE ONLY.  Only tests/, the package smoke check and bench.py's
CPU-baseline / reference legs may import this module.  It shares no code with the
CUDA library and imports nothing from it.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gem_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, OpenMP) into oracle/liboracle.so."""
    if not force and os.path.exists(_LIB_PATH) and \
            os.path.getmtime(_LIB_PATH) >= max(os.path.getmtime(_SRC),
                                               os.path.getmtime(_SRC[:-2] + ".h")):
        return _LIB_PATH
    tmp = _LIB_PATH + ".tmp.%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-D_GNU_SOURCE", "-fPIC", "-shared", "-fopenmp",
           "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class Layer(C.Structure):
    _fields_ = [("H", C.c_int64), ("n_q", C.c_int64), ("n_kv", C.c_int64),
                ("d", C.c_int64), ("F", C.c_int64),
                ("eps", C.c_double), ("theta", C.c_double), ("scale", C.c_double),
                ("rope_dim", C.c_int), ("window", C.c_int), ("act", C.c_int),
                ("qk_norm", C.c_int), ("v_from_k", C.c_int), ("post_norms", C.c_int),
                ("w_qkv", C.c_void_p), ("w_o", C.c_void_p), ("w_gate", C.c_void_p),
                ("w_up", C.c_void_p), ("w_down", C.c_void_p),
                ("g_attn", C.c_void_p), ("g_ffn", C.c_void_p), ("g_q", C.c_void_p),
                ("g_k", C.c_void_p), ("g_post_attn", C.c_void_p),
                ("g_post_ffn", C.c_void_p), ("compact_kv", C.c_int)]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = C.CDLL(build())
            p = C.c_void_p
            L.gem_oracle_half_to_double.restype = C.c_double
            L.gem_oracle_half_to_double.argtypes = [C.c_uint16]
            L.gem_oracle_double_to_half_via_f32.restype = C.c_uint16
            L.gem_oracle_double_to_half_via_f32.argtypes = [C.c_double]
            L.gem_oracle_q4_0_dequant.argtypes = [p, C.c_int64, C.c_int64, p]
            L.gem_oracle_q4_0_gemv_f32.argtypes = [p, C.c_int64, C.c_int64, p, C.c_int64,
                                                   C.c_int, p, C.c_int64, p, C.c_int64]
            L.gem_oracle_q4_0_gemv_f64.argtypes = [p, C.c_int64, C.c_int64, p, C.c_int64,
                                                   C.c_int, p, C.c_int64]
            L.gem_oracle_rmsnorm.argtypes = [p, C.c_int64, p, C.c_double, p]
            L.gem_oracle_rope_neox.argtypes = [p, C.c_int, C.c_int, C.c_double, C.c_double]
            L.gem_oracle_gqa_attention.argtypes = [p, p, p, C.c_int, C.c_int, C.c_int,
                                                   C.c_int64, C.c_int64, C.c_int,
                                                   C.c_double, p, p]
            L.gem_oracle_silu.restype = C.c_double
            L.gem_oracle_silu.argtypes = [C.c_double]
            L.gem_oracle_gelu_tanh.restype = C.c_double
            L.gem_oracle_gelu_tanh.argtypes = [C.c_double]
            L.gem_oracle_decode_layer.argtypes = [C.POINTER(Layer), C.c_int, p, p, p,
                                                  C.c_int64, p, p, p, p, p]
            L.gem_oracle_decode_layer_f64.argtypes = [C.POINTER(Layer), C.c_int, p, p, p,
                                                      C.c_int64, p, p, p, p, p]
            L.gem_oracle_decode_layer_ex.argtypes = [C.POINTER(Layer), C.c_int, p, p, p,
                                                     C.c_int64, p, p, p, p, p, p, p]
            L.gem_oracle_other_half_via_f32.restype = C.c_uint16
            L.gem_oracle_other_half_via_f32.argtypes = [C.c_double]
            L.gem_oracle_argmax.restype = C.c_int64
            L.gem_oracle_argmax.argtypes = [p, C.c_int64]
            L.gem_oracle_q8_0_dequant.argtypes = [p, C.c_int64, C.c_int64, p]
            L.gem_oracle_topk.restype = C.c_int
            L.gem_oracle_topk.argtypes = [p, C.c_int64, C.c_int, p, p]
            L.gem_oracle_gqa_attention_compact.restype = C.c_int
            L.gem_oracle_gqa_attention_compact.argtypes = [p, p, p, C.c_int, C.c_int, C.c_int, C.c_int64,
                                                           C.c_int64, C.c_int, C.c_double, C.c_double, p]
            L.gem_oracle_q8_0_gemv_f64.restype = C.c_int
            L.gem_oracle_q8_0_gemv_f64.argtypes = [p, C.c_int64, C.c_int64, p, C.c_int64, C.c_int, p,
                                                   C.c_int64]
            L.gem_oracle_num_threads.restype = C.c_int
            L.gem_oracle_set_num_threads.argtypes = [C.c_int]
            _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def half_to_double(h: int) -> float:
    return lib().gem_oracle_half_to_double(int(h) & 0xFFFF)


def double_to_half_via_f32(v: float) -> int:
    return int(lib().gem_oracle_double_to_half_via_f32(float(v)))


def other_half_via_f32(v: float) -> int:
    return int(lib().gem_oracle_other_half_via_f32(float(v)))


def q4_0_dequant(W: np.ndarray, N: int, K: int) -> np.ndarray:
    W = _c(W, np.uint8)
    out = np.empty((N, K), dtype=np.float64)
    lib().gem_oracle_q4_0_dequant(_ptr(W), N, K, _ptr(out))
    return out


def q4_0_gemv(W: np.ndarray, N: int, K: int, x: np.ndarray,
              residual: np.ndarray | None = None) -> np.ndarray:
    """y[b] = deq(W) @ x[b] (+ residual[b]) in fp64.  x: [B, K] fp32 or fp64."""
    W = _c(W, np.uint8)
    x = np.atleast_2d(x)
    B = x.shape[0]
    y = np.empty((B, N), dtype=np.float64)
    if x.dtype == np.float64:
        assert residual is None
        x = _c(x, np.float64)
        rc = lib().gem_oracle_q4_0_gemv_f64(_ptr(W), N, K, _ptr(x), K, B, _ptr(y), N)
    else:
        x = _c(x, np.float32)
        r = _c(None if residual is None else np.atleast_2d(residual), np.float32)
        rc = lib().gem_oracle_q4_0_gemv_f32(_ptr(W), N, K, _ptr(x), K, B, _ptr(r), N,
                                            _ptr(y), N)
    if rc:
        raise ValueError("oracle gemv rejected arguments (rc=%d)" % rc)
    return y


def rmsnorm(x: np.ndarray, gamma: np.ndarray | None, eps: float) -> np.ndarray:
    x = _c(x, np.float64)
    g = _c(gamma, np.float32)
    out = np.empty_like(x)
    lib().gem_oracle_rmsnorm(_ptr(x), x.size, _ptr(g), eps, _ptr(out))
    return out


def rope_neox(v: np.ndarray, rope_dim: int, pos: float, theta: float) -> np.ndarray:
    v = np.array(v, dtype=np.float64, copy=True)
    lib().gem_oracle_rope_neox(_ptr(v), v.size, rope_dim, float(pos), float(theta))
    return v


def gqa_attention(q: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray, pos: int,
                  window: int, scale: float, return_probs: bool = False):
    """One sequence: q [n_q, d]; caches binary16 bits [n_kv, cap, d]."""
    q = _c(q, np.float64)
    kc = _c(k_cache, np.uint16)
    vc = _c(v_cache, np.uint16)
    n_q, d = q.shape
    n_kv, cap, _ = kc.shape
    j0 = max(0, pos - window + 1) if window else 0
    T = pos - j0 + 1
    out = np.empty((n_q, d), dtype=np.float64)
    probs = np.empty((n_q, T), dtype=np.float64) if return_probs else None
    rc = lib().gem_oracle_gqa_attention(_ptr(q), _ptr(kc), _ptr(vc), n_q, n_kv, d, cap,
                                        pos, window, scale, _ptr(out), _ptr(probs))
    if rc:
        raise ValueError("oracle attention rejected arguments (rc=%d)" % rc)
    return (out, probs) if return_probs else out


def gqa_attention_compact(q: np.ndarray, v_cache: np.ndarray, gamma_k: np.ndarray | None, pos: int,
                          rope_dim: int, theta: float, scale: float) -> np.ndarray:
    """One sequence over a compact full-attention cache (V rows only, binary16 bits
    [n_kv, cap, d]): K_j = RoPE_j(V_j * gamma_k) rebuilt in fp64.  q [n_q, d] rotated at pos."""
    q = _c(q, np.float64)
    vc = _c(v_cache, np.uint16)
    g = _c(gamma_k, np.float32)
    n_q, d = q.shape
    n_kv, cap, _ = vc.shape
    out = np.empty((n_q, d), dtype=np.float64)
    rc = lib().gem_oracle_gqa_attention_compact(_ptr(q), _ptr(vc), _ptr(g), n_q, n_kv, d, cap, pos,
                                                rope_dim, theta, scale, _ptr(out))
    if rc:
        raise ValueError("oracle compact attention rejected arguments (rc=%d)" % rc)
    return out


def silu(g: float) -> float:
    return lib().gem_oracle_silu(float(g))


def gelu_tanh(g: float) -> float:
    return lib().gem_oracle_gelu_tanh(float(g))


def q8_0_dequant(W: np.ndarray, N: int, K: int) -> np.ndarray:
    W = _c(W, np.uint8)
    out = np.empty((N, K), dtype=np.float64)
    lib().gem_oracle_q8_0_dequant(_ptr(W), N, K, _ptr(out))
    return out


def q8_0_gemv(W: np.ndarray, N: int, K: int, x: np.ndarray) -> np.ndarray:
    """y[b] = deq(W) @ x[b] in fp64 (Q8_0 rows).  x: [B, K]."""
    W = _c(W, np.uint8)
    x = _c(np.atleast_2d(x), np.float64)
    B = x.shape[0]
    y = np.empty((B, N), dtype=np.float64)
    rc = lib().gem_oracle_q8_0_gemv_f64(_ptr(W), N, K, _ptr(x), K, B, _ptr(y), N)
    if rc:
        raise ValueError("oracle Q8_0 gemv rejected arguments (rc=%d)" % rc)
    return y


def argmax(v: np.ndarray) -> int:
    v = _c(v, np.float64)
    return int(lib().gem_oracle_argmax(_ptr(v), v.size))


def topk(v: np.ndarray, k: int):
    """(indices, values) of the k largest entries, largest first; ties by lowest index, NaN
    after every number (by index)."""
    v = _c(v, np.float64)
    idx = np.empty(k, np.int64)
    val = np.empty(k, np.float64)
    rc = lib().gem_oracle_topk(_ptr(v), v.size, int(k), _ptr(idx), _ptr(val))
    if rc:
        raise ValueError("oracle top-k rejected arguments (rc=%d)" % rc)
    return idx, val


def num_threads() -> int:
    return int(lib().gem_oracle_num_threads())


def set_num_threads(n: int) -> None:
    lib().gem_oracle_set_num_threads(int(n))


def make_layer(shape, t) -> tuple:
    """Build the C layer struct from a LayerShape and LayerTensors (kept alive)."""
    keep = [np.ascontiguousarray(a) if a is not None else None for a in
            (t.w_qkv, t.w_o, t.w_gate, t.w_up, t.w_down, t.g_attn, t.g_ffn, t.g_q, t.g_k,
             t.g_post_attn, t.g_post_ffn)]
    L = Layer(H=shape.H, n_q=shape.n_q, n_kv=shape.n_kv, d=shape.d, F=shape.F,
              eps=shape.eps, theta=shape.theta, scale=float(shape.scale),
              rope_dim=shape.rope_dim, window=shape.window, act=shape.act,
              qk_norm=int(shape.qk_norm), v_from_k=int(shape.v_from_k),
              post_norms=int(shape.post_norms),
              w_qkv=keep[0].ctypes.data, w_o=keep[1].ctypes.data,
              w_gate=keep[2].ctypes.data, w_up=keep[3].ctypes.data,
              w_down=keep[4].ctypes.data, g_attn=keep[5].ctypes.data,
              g_ffn=keep[6].ctypes.data,
              g_q=keep[7].ctypes.data if keep[7] is not None else None,
              g_k=keep[8].ctypes.data if keep[8] is not None else None,
              g_post_attn=keep[9].ctypes.data if keep[9] is not None else None,
              g_post_ffn=keep[10].ctypes.data if keep[10] is not None else None,
              compact_kv=int(getattr(shape, "compact_kv", False)))
    return L, keep


def decode_layer(shape, tensors, x: np.ndarray, pos: np.ndarray, k_cache: np.ndarray,
                 v_cache: np.ndarray, stages: bool = False, flip: np.ndarray | None = None,
                 kvnew: bool = False):
    """One layer step.  k_cache / v_cache (uint16, [B, n_kv, cap, d]) are updated in
    place with the appended row.  Returns x_out (fp64), or with stages=True the tuple
    (x_out, qkv, attn, h); kvnew=True appends the unrounded new rows [B, 2, n_kv, d].
    flip (int8 [B, 2, n_kv, d]) selects the other binary16 neighbour for those elements."""
    L, keep = make_layer(shape, tensors)
    B = x.shape[0]
    assert (k_cache is None or k_cache.flags.c_contiguous) and v_cache.flags.c_contiguous
    cap = v_cache.shape[2]
    pos = _c(pos, np.int32)
    out = np.empty((B, shape.H), dtype=np.float64)
    qkv = np.empty((B, shape.n_qkv), dtype=np.float64) if stages else None
    att = np.empty((B, shape.n_q * shape.d), dtype=np.float64) if stages else None
    h = np.empty((B, shape.H), dtype=np.float64) if stages else None
    kvn = np.empty((B, 2, shape.n_kv, shape.d), dtype=np.float64) if kvnew else None
    fl = _c(flip, np.int8)
    xx = _c(x, np.float64)
    rc = lib().gem_oracle_decode_layer_ex(C.byref(L), B, _ptr(xx), _ptr(k_cache), _ptr(v_cache),
                                          cap, _ptr(pos), _ptr(out), _ptr(qkv), _ptr(att),
                                          _ptr(h), _ptr(kvn), _ptr(fl))
    del keep
    if rc:
        raise ValueError("oracle decode layer failed (rc=%d)" % rc)
    res = (out, qkv, att, h) if stages else (out,)
    if kvnew:
        res = res + (kvn,)
    return res if len(res) > 1 else res[0]
