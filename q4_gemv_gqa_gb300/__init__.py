"""Python binding of the GB300 decoder-step library (libgem.so, include/gem.h).

Each function marshals torch CUDA tensors into the C ABI call of the same name and
raises GemError on a non-zero status.  All computation runs in the CUDA library; torch
only provides device memory and the current stream.  Importing this package fails if
libgem.so is missing, and every call fails if the tensors are not on a CUDA device.
"""
from __future__ import annotations

import ctypes as C

import torch

from . import _lib
from ._lib import LayerDesc

lib = _lib.load()

GEM_OK = 0
ACT_SILU = 0
ACT_GELU_TANH = 1
DEVFLAG_POS_RANGE = 1
DEVFLAG_TIMEOUT = 2

__all__ = ["GemError", "q4_0_gemv", "q4_0_gemv_workspace", "q4_0_gemv_fused", "q8_0_gemv", "argmax", "argmax_workspace", "rmsnorm", "rmsnorm_qknorm_rope", "gqa_decode_attn",
           "gqa_decode_attn_workspace", "gqa_decode_attn_fused", "swiglu", "decode_layer", "decode_layer_workspace",
           "DeviceLayer", "device_status", "status_from_flags", "set_wait_limit",
           "set_test_injection", "LayerDesc"]


class GemError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        msg = lib.gem_status_string(status).decode()
        if status == 4:
            msg += " (cudaError %d)" % lib.gem_last_cuda_error()
        super().__init__("%s: %s [status %d]" % (what, msg, status))


def _check(st: int, what: str) -> None:
    if st != GEM_OK:
        raise GemError(st, what)


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


_HALF_BITS = (torch.int16, torch.uint16)   # binary16 bit patterns


def _dev(t: torch.Tensor | None, dtype, name: str):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    ok = t.dtype in dtype if isinstance(dtype, tuple) else t.dtype == dtype
    if not ok:
        raise ValueError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    return t.data_ptr()


def _cache_shape(k: torch.Tensor | None, v: torch.Tensor, B: int, n_kv: int, d: int) -> int:
    """Caches must be [B, n_kv, cap, d] (the kernels address them from these sizes); k may be
    None for a compact (V-only) cache."""
    for name, c in (("k_cache", k), ("v_cache", v)):
        if c is None and name == "k_cache":
            continue
        if c.dim() != 4 or c.shape[0] != B or c.shape[1] != n_kv or c.shape[3] != d:
            raise ValueError("%s must be [B=%d, n_kv=%d, cap, d=%d], got %s" % (name, B, n_kv, d, tuple(c.shape)))
    if k is not None and v.shape != k.shape:
        raise ValueError("k_cache and v_cache shapes differ")
    return int(v.shape[2])


def _q4_bytes(W: torch.Tensor, N: int, K: int) -> None:
    # K % 32 != 0 is left to the library, which rejects it with GEM_ERR_BAD_SHAPE
    if K % 32 == 0 and W.numel() < N * (K // 32) * 18:
        raise ValueError("W must hold N x K Q4_0 weights (%d bytes), has %d" % (N * (K // 32) * 18, W.numel()))


def version() -> int:
    return lib.gem_version()


def device_status(reset: bool = False) -> int:
    v = C.c_int32(0)
    _check(lib.gem_device_status(C.byref(v), int(reset)), "gem_device_status")
    return v.value


def status_from_flags(flags: int) -> int:
    """gem_status that a set of GEM_DEVFLAG_* bits stands for (host only)."""
    return int(lib.gem_status_from_flags(flags))


INJECT_RING_SHORTFALL = 1
INJECT_GRID_ARRIVAL = 2


def set_wait_limit(ns: int) -> None:
    """Wall-time limit of every device-side wait on the current device (0: default 1 s)."""
    _check(lib.gem_set_wait_limit(int(ns)), "gem_set_wait_limit")


def set_test_injection(mask: int) -> None:
    """GEM_INJECT_* bits: make one bounded wait run out (tests of the timeout path)."""
    _check(lib.gem_set_test_injection(int(mask)), "gem_set_test_injection")


def q4_0_gemv_workspace(B: int, K: int) -> int:
    return int(lib.gem_q4_0_gemv_workspace(B, K))


def q4_0_gemv(W: torch.Tensor, N: int, K: int, x: torch.Tensor, y: torch.Tensor,
              residual: torch.Tensor | None = None, stream=None,
              workspace: torch.Tensor | None = None, shared_records: bool = False) -> torch.Tensor:
    """y[b] = deq(W) @ x[b] (+ residual[b]).  x: [B, >=K] fp32, y: [B, >=N] fp32.

    With B >= 2 the call goes through gem_q4_0_gemv_ws with `workspace` (a uint8 device tensor
    of q4_0_gemv_workspace(B, K) bytes; allocated here when not given), so concurrent calls
    share no state.  shared_records=True calls gem_q4_0_gemv instead, whose records live in
    the library's own per-device array."""
    B = x.shape[0] if x.dim() == 2 else 1
    _q4_bytes(W, N, K)
    if x.shape[-1] < K or y.shape[-1] < N:
        raise ValueError("x must have >= K columns and y >= N")
    need = q4_0_gemv_workspace(B, K) if K % 32 == 0 else 0
    if shared_records or need == 0:
        st = lib.gem_q4_0_gemv(_dev(W, torch.uint8, "W"), N, K, _dev(x, torch.float32, "x"),
                               x.shape[-1], B, _dev(y, torch.float32, "y"), y.shape[-1],
                               _dev(residual, torch.float32, "residual"), _stream(stream))
        _check(st, "gem_q4_0_gemv")
        return y
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    st = lib.gem_q4_0_gemv_ws(_dev(W, torch.uint8, "W"), N, K, _dev(x, torch.float32, "x"),
                              x.shape[-1], B, _dev(y, torch.float32, "y"), y.shape[-1],
                              _dev(residual, torch.float32, "residual"),
                              _dev(workspace, torch.uint8, "workspace"), workspace.numel(),
                              _stream(stream))
    _check(st, "gem_q4_0_gemv_ws")
    return y


def q4_0_gemv_fused(W0: torch.Tensor, W1: torch.Tensor | None, N: int, K: int, x: torch.Tensor,
                    y: torch.Tensor, gamma: torch.Tensor | None = None, eps: float = 1e-6,
                    act: int = ACT_SILU, residual: torch.Tensor | None = None,
                    workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Pre-norm (gamma) + Q4_0 GEMV, or the gate/up pair (W1) with the gated activation.
    x: [B, >=K] fp32, y: [B, >=N] fp32; workspace as for q4_0_gemv (allocated when needed)."""
    B = x.shape[0] if x.dim() == 2 else 1
    _q4_bytes(W0, N, K)
    if W1 is not None:
        _q4_bytes(W1, N, K)
    if x.shape[-1] < K or y.shape[-1] < N:
        raise ValueError("x must have >= K columns and y >= N")
    need = q4_0_gemv_workspace(B, K) if K % 32 == 0 else 0
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    st = lib.gem_q4_0_gemv_fused(_dev(W0, torch.uint8, "W0"), _dev(W1, torch.uint8, "W1"), N, K,
                                 _dev(x, torch.float32, "x"), x.shape[-1], B,
                                 _dev(gamma, torch.float32, "gamma"), eps, act,
                                 _dev(y, torch.float32, "y"), y.shape[-1],
                                 _dev(residual, torch.float32, "residual"),
                                 _dev(workspace, torch.uint8, "workspace") if need else None,
                                 workspace.numel() if need else 0, _stream(stream))
    _check(st, "gem_q4_0_gemv_fused")
    return y


def q4_0_gemm_workspace(M: int, K: int) -> int:
    return int(lib.gem_q4_0_gemm_workspace(M, K))


def q4_0_gemm(W0: torch.Tensor, W1: torch.Tensor | None, N: int, K: int, x: torch.Tensor,
              y: torch.Tensor, gamma: torch.Tensor | None = None, eps: float = 1e-6,
              act: int = ACT_SILU, residual: torch.Tensor | None = None,
              workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Batched prefill GEMM: M = x.shape[0] (<= 32) prompt rows through W0 (or the W0/W1 pair),
    each weight read once.  Same options as q4_0_gemv_fused; workspace allocated when needed."""
    M = x.shape[0] if x.dim() == 2 else 1
    _q4_bytes(W0, N, K)
    if W1 is not None:
        _q4_bytes(W1, N, K)
    if x.shape[-1] < K or y.shape[-1] < N:
        raise ValueError("x must have >= K columns and y >= N")
    need = q4_0_gemm_workspace(M, K) if K % 32 == 0 else 0
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    st = lib.gem_q4_0_gemm(_dev(W0, torch.uint8, "W0"), _dev(W1, torch.uint8, "W1"), N, K,
                           _dev(x, torch.float32, "x"), x.shape[-1], M,
                           _dev(gamma, torch.float32, "gamma"), eps, act,
                           _dev(y, torch.float32, "y"), y.shape[-1],
                           _dev(residual, torch.float32, "residual"),
                           _dev(workspace, torch.uint8, "workspace") if need else None,
                           workspace.numel() if need else 0, _stream(stream))
    _check(st, "gem_q4_0_gemm")
    return y


def q8_0_gemv(W: torch.Tensor, N: int, K: int, x: torch.Tensor, y: torch.Tensor,
              stream=None) -> torch.Tensor:
    """Tied Q8_0 embedding / logit projection: y[b] = deq(W) @ x[b].  W: N x (K/32*34) bytes."""
    B = x.shape[0] if x.dim() == 2 else 1
    if K % 32 == 0 and W.numel() < N * (K // 32) * 34:
        raise ValueError("W must hold N x K Q8_0 weights (%d bytes), has %d" % (N * (K // 32) * 34, W.numel()))
    if x.shape[-1] < K or y.shape[-1] < N:
        raise ValueError("x must have >= K columns and y >= N")
    st = lib.gem_q8_0_gemv(_dev(W, torch.uint8, "W"), N, K, _dev(x, torch.float32, "x"), x.shape[-1], B,
                           _dev(y, torch.float32, "y"), y.shape[-1], _stream(stream))
    _check(st, "gem_q8_0_gemv")
    return y


def argmax_workspace(B: int, N: int) -> int:
    return int(lib.gem_argmax_workspace(B, N))


def argmax(y: torch.Tensor, idx: torch.Tensor, workspace: torch.Tensor | None = None,
           stream=None) -> torch.Tensor:
    """idx[b] = index of the largest y[b][n] (lowest index on ties; NaN never chosen)."""
    B = y.shape[0] if y.dim() == 2 else 1
    N = y.shape[-1]
    if idx.numel() < B:
        raise ValueError("idx must hold B indices")
    need = argmax_workspace(B, N)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=y.device)
    st = lib.gem_argmax(_dev(y, torch.float32, "y"), N, B, N, _dev(idx, torch.int32, "idx"),
                        _dev(workspace, torch.uint8, "workspace"), workspace.numel(), _stream(stream))
    _check(st, "gem_argmax")
    return idx


def topk_workspace(B: int, N: int, k: int) -> int:
    return int(lib.gem_topk_workspace(B, N, k))


def topk(y: torch.Tensor, k: int, idx: torch.Tensor, val: torch.Tensor,
         workspace: torch.Tensor | None = None, stream=None):
    """The k largest entries of each row of y [B, N] fp32, largest first (ties: lowest index;
    NaN after every number): idx int32 [B, k], val fp32 [B, k]."""
    B = y.shape[0] if y.dim() == 2 else 1
    N = y.shape[-1]
    need = topk_workspace(B, N, k)
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=y.device)
    st = lib.gem_topk(_dev(y, torch.float32, "y"), N, B, N, k, _dev(idx, torch.int32, "idx"),
                      _dev(val, torch.float32, "val"), _dev(workspace, torch.uint8, "workspace"),
                      workspace.numel() if workspace is not None else 0, _stream(stream))
    _check(st, "gem_topk")
    return idx, val


def rmsnorm(x: torch.Tensor, gamma: torch.Tensor | None, eps: float, out: torch.Tensor,
            stream=None) -> torch.Tensor:
    B = x.shape[0] if x.dim() == 2 else 1
    st = lib.gem_rmsnorm(_dev(x, torch.float32, "x"), B, x.shape[-1],
                         _dev(gamma, torch.float32, "gamma"), eps,
                         _dev(out, torch.float32, "out"), _stream(stream))
    _check(st, "gem_rmsnorm")
    return out


def rmsnorm_qknorm_rope(qkv: torch.Tensor, n_q: int, n_kv: int, d: int,
                        gamma_q: torch.Tensor | None, gamma_k: torch.Tensor | None, v_mode: int,
                        eps: float, pos: torch.Tensor, theta: float, rope_dim: int,
                        k_cache: torch.Tensor | None, v_cache: torch.Tensor, window: int = 0,
                        status: torch.Tensor | None = None, stream=None) -> None:
    """qkv [B, ldqkv] fp32 in place; caches binary16 bits (int16/uint16) [B, n_kv, cap, d]; pos int32 [B].

    k_cache None with v_mode 1 appends the V row only (a compact full-attention cache)."""
    B = qkv.shape[0]
    cap = _cache_shape(k_cache, v_cache, B, n_kv, d)
    st = lib.gem_rmsnorm_qknorm_rope(
        _dev(qkv, torch.float32, "qkv"), qkv.shape[-1], B, n_q, n_kv, d,
        _dev(gamma_q, torch.float32, "gamma_q"), _dev(gamma_k, torch.float32, "gamma_k"),
        v_mode, eps, _dev(pos, torch.int32, "pos"), theta, rope_dim,
        _dev(k_cache, _HALF_BITS, "k_cache"), _dev(v_cache, _HALF_BITS, "v_cache"), cap,
        window, _dev(status, torch.int32, "status"), _stream(stream))
    _check(st, "gem_rmsnorm_qknorm_rope")


def gqa_decode_attn_workspace(B: int, n_q: int, n_kv: int, d: int, cache_cap: int,
                              window: int = 0) -> int:
    return int(lib.gem_gqa_decode_attn_workspace(B, n_q, n_kv, d, cache_cap, window))


def gqa_decode_attn(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, n_q: int,
                    n_kv: int, d: int, pos: torch.Tensor, window: int, scale: float,
                    out: torch.Tensor, workspace: torch.Tensor | None = None,
                    status: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """q [B, ldq] fp32 (head h at column h*d); caches uint16 [B, n_kv, cap, d]."""
    B = q.shape[0]
    cap = _cache_shape(k_cache, v_cache, B, n_kv, d)
    ws_ptr = _dev(workspace, torch.uint8, "workspace")
    ws_bytes = workspace.numel() if workspace is not None else 0
    st = lib.gem_gqa_decode_attn(
        _dev(q, torch.float32, "q"), q.shape[-1], _dev(k_cache, _HALF_BITS, "k_cache"),
        _dev(v_cache, _HALF_BITS, "v_cache"), B, n_q, n_kv, d, cap,
        _dev(pos, torch.int32, "pos"), window, scale, _dev(out, torch.float32, "out"),
        out.shape[-1], ws_ptr, ws_bytes, _dev(status, torch.int32, "status"), _stream(stream))
    _check(st, "gem_gqa_decode_attn")
    return out


def gqa_decode_attn_fused(qkv: torch.Tensor, n_q: int, n_kv: int, d: int,
                          gamma_q: torch.Tensor | None, gamma_k: torch.Tensor | None, v_mode: int,
                          eps: float, pos: torch.Tensor, theta: float, rope_dim: int,
                          k_cache: torch.Tensor, v_cache: torch.Tensor, window: int, scale: float,
                          out: torch.Tensor, workspace: torch.Tensor | None = None,
                          status: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """QK-norm + RoPE + KV append + attention from the raw QKV projection row (qkv [B, ldqkv])."""
    B = qkv.shape[0]
    cap = _cache_shape(k_cache, v_cache, B, n_kv, d)
    st = lib.gem_gqa_decode_attn_fused(
        _dev(qkv, torch.float32, "qkv"), qkv.shape[-1], B, n_q, n_kv, d,
        _dev(gamma_q, torch.float32, "gamma_q"), _dev(gamma_k, torch.float32, "gamma_k"), v_mode, eps,
        _dev(pos, torch.int32, "pos"), theta, rope_dim, _dev(k_cache, _HALF_BITS, "k_cache"),
        _dev(v_cache, _HALF_BITS, "v_cache"), cap, window, scale, _dev(out, torch.float32, "out"),
        out.shape[-1], _dev(workspace, torch.uint8, "workspace"),
        workspace.numel() if workspace is not None else 0, _dev(status, torch.int32, "status"),
        _stream(stream))
    _check(st, "gem_gqa_decode_attn_fused")
    return out


def gqa_decode_attn_compact_workspace(B: int, n_q: int, n_kv: int, d: int, cache_cap: int,
                                      rope_dim: int) -> int:
    return int(lib.gem_gqa_decode_attn_compact_workspace(B, n_q, n_kv, d, cache_cap, rope_dim))


def gqa_decode_attn_compact(q: torch.Tensor, v_cache: torch.Tensor, n_q: int, n_kv: int, d: int,
                            pos: torch.Tensor, scale: float, gamma_k: torch.Tensor, rope_dim: int,
                            theta: float, out: torch.Tensor, workspace: torch.Tensor | None = None,
                            status: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Attention over a V-only cache; K_j = RoPE_j(V_j * gamma_k) is rebuilt inside the kernel."""
    B = q.shape[0]
    cap = _cache_shape(None, v_cache, B, n_kv, d)
    st = lib.gem_gqa_decode_attn_compact(
        _dev(q, torch.float32, "q"), q.shape[-1], _dev(v_cache, _HALF_BITS, "v_cache"), B, n_q, n_kv,
        d, cap, _dev(pos, torch.int32, "pos"), scale, _dev(gamma_k, torch.float32, "gamma_k"),
        rope_dim, theta, _dev(out, torch.float32, "out"), out.shape[-1],
        _dev(workspace, torch.uint8, "workspace"), workspace.numel() if workspace is not None else 0,
        _dev(status, torch.int32, "status"), _stream(stream))
    _check(st, "gem_gqa_decode_attn_compact")
    return out


NOALLOC_SCRATCH_BYTES = 8 << 20  # GEM_ATTN_NOALLOC_SCRATCH_BYTES


def gqa_decode_attn_noalloc(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                            n_q: int, n_kv: int, d: int, pos: torch.Tensor, window: int,
                            scale: float, out: torch.Tensor, status: torch.Tensor | None = None,
                            stream=None) -> torch.Tensor:
    """gqa_decode_attn with the split partials in the library's own per-device array.

    For callers that must not allocate device memory while decoding.  Allocates nothing;
    calls that may run concurrently on one device race on the shared array; shapes whose
    partials exceed NOALLOC_SCRATCH_BYTES raise GemError (GEM_ERR_WORKSPACE)."""
    B = q.shape[0]
    cap = _cache_shape(k_cache, v_cache, B, n_kv, d)
    st = lib.gem_gqa_decode_attn_noalloc(
        _dev(q, torch.float32, "q"), q.shape[-1], _dev(k_cache, _HALF_BITS, "k_cache"),
        _dev(v_cache, _HALF_BITS, "v_cache"), B, n_q, n_kv, d, cap,
        _dev(pos, torch.int32, "pos"), window, scale, _dev(out, torch.float32, "out"),
        out.shape[-1], _dev(status, torch.int32, "status"), _stream(stream))
    _check(st, "gem_gqa_decode_attn_noalloc")
    return out


def swiglu(gate: torch.Tensor, up: torch.Tensor, act: int, out: torch.Tensor,
           stream=None) -> torch.Tensor:
    B = gate.shape[0] if gate.dim() == 2 else 1
    st = lib.gem_swiglu(_dev(gate, torch.float32, "gate"), _dev(up, torch.float32, "up"), B,
                        gate.shape[-1], act, _dev(out, torch.float32, "out"), _stream(stream))
    _check(st, "gem_swiglu")
    return out


class DeviceLayer:
    """Device-resident weights of one decoder layer plus its gem_layer_desc."""

    def __init__(self, shape, tensors, device="cuda"):
        def up(a, dt):
            return None if a is None else torch.from_numpy(a).to(device=device, dtype=dt).contiguous()

        self.shape = shape
        self.w_qkv = up(tensors.w_qkv, torch.uint8)
        self.w_o = up(tensors.w_o, torch.uint8)
        self.w_gate = up(tensors.w_gate, torch.uint8)
        self.w_up = up(tensors.w_up, torch.uint8)
        self.w_down = up(tensors.w_down, torch.uint8)
        self.g_attn = up(tensors.g_attn, torch.float32)
        self.g_ffn = up(tensors.g_ffn, torch.float32)
        self.g_q = up(tensors.g_q, torch.float32)
        self.g_k = up(tensors.g_k, torch.float32)
        self.g_post_attn = up(tensors.g_post_attn, torch.float32)
        self.g_post_ffn = up(tensors.g_post_ffn, torch.float32)
        self._make_desc()

    _TENSORS = ("w_qkv", "w_o", "w_gate", "w_up", "w_down", "g_attn", "g_ffn", "g_q", "g_k",
                "g_post_attn", "g_post_ffn")

    @classmethod
    def clone(cls, src: "DeviceLayer") -> "DeviceLayer":
        """A layer with its own device copies of src's weights (same values, new buffers)."""
        obj = cls.__new__(cls)
        obj.shape = src.shape
        for name in cls._TENSORS:
            t = getattr(src, name)
            setattr(obj, name, None if t is None else t.clone())
        obj._make_desc()
        return obj

    def _make_desc(self):
        ptr = lambda t: None if t is None else t.data_ptr()
        s = self.shape
        self.desc = LayerDesc(
            H=s.H, n_q=s.n_q, n_kv=s.n_kv, d=s.d, F=s.F, eps=s.eps, theta=s.theta,
            scale=float(s.scale), rope_dim=s.rope_dim, window=s.window, act=s.act,
            qk_norm=int(s.qk_norm), v_from_k=int(s.v_from_k), post_norms=int(s.post_norms),
            w_qkv=ptr(self.w_qkv), w_o=ptr(self.w_o), w_gate=ptr(self.w_gate),
            w_up=ptr(self.w_up), w_down=ptr(self.w_down), g_attn=ptr(self.g_attn),
            g_ffn=ptr(self.g_ffn), g_q=ptr(self.g_q), g_k=ptr(self.g_k),
            g_post_attn=ptr(self.g_post_attn), g_post_ffn=ptr(self.g_post_ffn),
            compact_kv=int(getattr(s, "compact_kv", False)))

    def weight_bytes(self) -> int:
        return sum(t.numel() for t in (self.w_qkv, self.w_o, self.w_gate, self.w_up, self.w_down))


def decode_layer_workspace(layer: DeviceLayer, B: int, cache_cap: int) -> int:
    return int(lib.gem_decode_layer_workspace(C.byref(layer.desc), B, cache_cap))


def decode_layer(layer: DeviceLayer, x: torch.Tensor, k_cache: torch.Tensor | None,
                 v_cache: torch.Tensor, pos: torch.Tensor, workspace: torch.Tensor,
                 status: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """One layer step, in place on x [B, H] fp32; caches uint16 [B, n_kv, cap, d] (a compact_kv
    layer keeps the V cache alone: k_cache may be None)."""
    B = x.shape[0]
    s = layer.shape
    cap = _cache_shape(k_cache, v_cache, B, s.n_kv, s.d)
    if x.dim() != 2 or x.shape[1] != s.H:
        raise ValueError("x must be [B, H=%d], got %s" % (s.H, tuple(x.shape)))
    st = lib.gem_decode_layer(C.byref(layer.desc), B, _dev(x, torch.float32, "x"),
                              _dev(k_cache, _HALF_BITS, "k_cache"),
                              _dev(v_cache, _HALF_BITS, "v_cache"), cap,
                              _dev(pos, torch.int32, "pos"), _dev(workspace, torch.uint8, "workspace"),
                              workspace.numel(), _dev(status, torch.int32, "status"),
                              _stream(stream))
    _check(st, "gem_decode_layer")
    return x


class StepPlan:
    """Every layer of a decode step in one persistent launch (gem_step_plan).

    layers: DeviceLayer list; k_caches, v_caches: per-layer uint16 [B, n_kv, cap, d]
    tensors, kept referenced by the plan."""

    def __init__(self, layers, B: int, k_caches, v_caches):
        n = len(layers)
        if len(k_caches) != n or len(v_caches) != n:
            raise ValueError("one K and one V cache per layer")
        for dl, k, v in zip(layers, k_caches, v_caches):
            _cache_shape(k, v, B, dl.shape.n_kv, dl.shape.d)
        self._keep = (list(layers), list(k_caches), list(v_caches))
        descs = (LayerDesc * n)(*[dl.desc for dl in layers])
        kp = (C.c_void_p * n)(*[_dev(k, _HALF_BITS, "k_cache") for k in k_caches])
        vp = (C.c_void_p * n)(*[_dev(v, _HALF_BITS, "v_cache") for v in v_caches])
        caps = (C.c_int64 * n)(*[int(k.shape[2]) for k in k_caches])
        h = C.c_void_p()
        st = lib.gem_step_plan_create(descs, n, B, kp, vp, caps, C.byref(h))
        _check(st, "gem_step_plan_create")
        self._h = h
        self.B = B

    def step(self, x: torch.Tensor, pos: torch.Tensor, status: torch.Tensor | None = None,
             stream=None) -> torch.Tensor:
        H = self._keep[0][0].shape.H
        if x.dim() != 2 or x.shape[0] != self.B or x.shape[1] != H:
            raise ValueError("x must be [B=%d, H=%d], got %s" % (self.B, H, tuple(x.shape)))
        if pos.numel() < self.B:
            raise ValueError("pos must hold B positions")
        st = lib.gem_decode_step(self._h, _dev(x, torch.float32, "x"), _dev(pos, torch.int32, "pos"),
                                 _dev(status, torch.int32, "status"), _stream(stream))
        _check(st, "gem_decode_step")
        return x

    def close(self) -> None:
        if getattr(self, "_h", None):
            lib.gem_step_plan_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
