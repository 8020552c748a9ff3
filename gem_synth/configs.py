"""Decoder-layer shapes of the measured workloads and their seeded tensors.

Shapes only: the arithmetic lives in the oracle and in the CUDA library.
Shapes come from the model tables of the two source pages: "GELO LLM generation"
(section 04, Qwen3 family table: Qwen3-1.7B and Qwen3-4B) and the "gem" engine
research record (section "Verified model facts": Gemma 4 31B geometry).
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import numpy as np

from . import (ROLE_G_ATTN, ROLE_G_FFN, ROLE_G_K, ROLE_G_POST_ATTN, ROLE_G_POST_FFN,
               ROLE_G_Q, ROLE_K_CACHE, ROLE_V_CACHE, ROLE_W_DOWN, ROLE_W_GATE, ROLE_W_O,
               ROLE_W_QKV, ROLE_W_UP, ROLE_X, norm_weight, normal_f16_bits, normal_f32,
               q4_0_matrix, tid)

ACT_SILU = 0
ACT_GELU_TANH = 1


@dataclass(frozen=True)
class LayerShape:
    H: int            # hidden width
    n_q: int          # query heads
    n_kv: int         # key/value heads
    d: int            # head dim
    F: int            # FFN width
    theta: float      # RoPE base
    rope_dim: int     # rotated dims (R); == d for full rotation
    window: int       # 0 = full causal attention, else sliding window W
    scale: float      # attention score scale
    act: int          # ACT_SILU or ACT_GELU_TANH
    qk_norm: bool     # per-head RMSNorm of q and k before RoPE
    v_from_k: bool    # V = unweighted RMSNorm of the K projection (no V rows)
    post_norms: bool  # RMSNorm of attention / FFN outputs before the residual adds
    eps: float = 1e-6
    compact_kv: bool = False   # full-attention layer whose cache keeps the V rows only

    @property
    def n_qkv(self) -> int:
        n_v = 0 if self.v_from_k else self.n_kv
        return (self.n_q + self.n_kv + n_v) * self.d


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    pos: int                 # position of the new token = number of cached positions
    layers: tuple            # tuple[LayerShape, ...]
    cache_cap: tuple         # per layer cache capacity (slots)


def qwen3_shape(H, n_q, n_kv, d, F) -> LayerShape:
    return LayerShape(H=H, n_q=n_q, n_kv=n_kv, d=d, F=F, theta=1e6, rope_dim=d, window=0,
                      scale=1.0 / np.sqrt(d), act=ACT_SILU, qk_norm=True, v_from_k=False,
                      post_norms=False)


TINY = qwen3_shape(256, 4, 2, 64, 512)
QWEN3_1_7B = qwen3_shape(2048, 16, 8, 128, 6144)
QWEN3_4B = qwen3_shape(2560, 32, 8, 128, 9728)
GEMMA31_SWA = LayerShape(H=5376, n_q=32, n_kv=16, d=256, F=21504, theta=1e4, rope_dim=256,
                         window=1024, scale=1.0, act=ACT_GELU_TANH, qk_norm=True,
                         v_from_k=False, post_norms=True)
GEMMA31_FULL = LayerShape(H=5376, n_q=32, n_kv=4, d=512, F=21504, theta=1e6, rope_dim=128,
                          window=0, scale=1.0, act=ACT_GELU_TANH, qk_norm=True,
                          v_from_k=True, post_norms=True)


# The same full-attention layer with the compact cache (V rows only; K rebuilt from V).
GEMMA31_FULL_COMPACT = replace(GEMMA31_FULL, compact_kv=True)


def _cap(shape: LayerShape, pos: int) -> int:
    return shape.window if shape.window else pos + 1


def workload(name: str) -> Workload:
    if name == "tiny":
        layers = (TINY,)
        pos, B = 128, 1
    elif name == "qwen3-1.7b":
        layers = (QWEN3_1_7B,) * 28
        pos, B = 4096, 1
    elif name == "qwen3-4b-b8":
        layers = (QWEN3_4B,) * 36
        pos, B = 2048, 8
    elif name == "gemma4-31b-group":
        layers = (GEMMA31_SWA,) * 5 + (GEMMA31_FULL,)
        pos, B = 32768, 1
    elif name == "gemma4-31b-group-compact":
        layers = (GEMMA31_SWA,) * 5 + (GEMMA31_FULL_COMPACT,)
        pos, B = 32768, 1
    else:
        raise KeyError(name)
    return Workload(name=name, B=B, pos=pos, layers=layers,
                    cache_cap=tuple(_cap(s, pos) for s in layers))


def with_layers(w: Workload, n: int) -> Workload:
    return replace(w, layers=w.layers[:n], cache_cap=w.cache_cap[:n])


@dataclass
class LayerTensors:
    w_qkv: np.ndarray
    w_o: np.ndarray
    w_gate: np.ndarray
    w_up: np.ndarray
    w_down: np.ndarray
    g_attn: np.ndarray
    g_ffn: np.ndarray
    g_q: np.ndarray | None
    g_k: np.ndarray | None
    g_post_attn: np.ndarray | None
    g_post_ffn: np.ndarray | None
    k_cache: np.ndarray      # uint16 [B, n_kv, cap, d]
    v_cache: np.ndarray      # uint16 [B, n_kv, cap, d]


def layer_tensors(shape: LayerShape, B: int, cap: int, seed: int, layer: int) -> LayerTensors:
    s, L = shape, layer
    return LayerTensors(
        w_qkv=q4_0_matrix(seed, tid(L, ROLE_W_QKV), s.n_qkv, s.H),
        w_o=q4_0_matrix(seed, tid(L, ROLE_W_O), s.H, s.n_q * s.d),
        w_gate=q4_0_matrix(seed, tid(L, ROLE_W_GATE), s.F, s.H),
        w_up=q4_0_matrix(seed, tid(L, ROLE_W_UP), s.F, s.H),
        w_down=q4_0_matrix(seed, tid(L, ROLE_W_DOWN), s.H, s.F),
        g_attn=norm_weight(seed, tid(L, ROLE_G_ATTN), s.H),
        g_ffn=norm_weight(seed, tid(L, ROLE_G_FFN), s.H),
        g_q=norm_weight(seed, tid(L, ROLE_G_Q), s.d) if s.qk_norm else None,
        g_k=norm_weight(seed, tid(L, ROLE_G_K), s.d) if s.qk_norm else None,
        g_post_attn=norm_weight(seed, tid(L, ROLE_G_POST_ATTN), s.H) if s.post_norms else None,
        g_post_ffn=norm_weight(seed, tid(L, ROLE_G_POST_FFN), s.H) if s.post_norms else None,
        k_cache=normal_f16_bits(seed, tid(L, ROLE_K_CACHE), (B, s.n_kv, cap, s.d)),
        v_cache=normal_f16_bits(seed, tid(L, ROLE_V_CACHE), (B, s.n_kv, cap, s.d)),
    )


def layer_weights(shape: LayerShape, seed: int, layer: int) -> LayerTensors:
    """The weights and norm weights of layer_tensors() (same draws), without the caches."""
    s, L = shape, layer
    return LayerTensors(
        w_qkv=q4_0_matrix(seed, tid(L, ROLE_W_QKV), s.n_qkv, s.H),
        w_o=q4_0_matrix(seed, tid(L, ROLE_W_O), s.H, s.n_q * s.d),
        w_gate=q4_0_matrix(seed, tid(L, ROLE_W_GATE), s.F, s.H),
        w_up=q4_0_matrix(seed, tid(L, ROLE_W_UP), s.F, s.H),
        w_down=q4_0_matrix(seed, tid(L, ROLE_W_DOWN), s.H, s.F),
        g_attn=norm_weight(seed, tid(L, ROLE_G_ATTN), s.H),
        g_ffn=norm_weight(seed, tid(L, ROLE_G_FFN), s.H),
        g_q=norm_weight(seed, tid(L, ROLE_G_Q), s.d) if s.qk_norm else None,
        g_k=norm_weight(seed, tid(L, ROLE_G_K), s.d) if s.qk_norm else None,
        g_post_attn=norm_weight(seed, tid(L, ROLE_G_POST_ATTN), s.H) if s.post_norms else None,
        g_post_ffn=norm_weight(seed, tid(L, ROLE_G_POST_FFN), s.H) if s.post_norms else None,
        k_cache=None,
        v_cache=None,
    )


def kv_cache(shape: LayerShape, B: int, cap: int, seed: int, layer: int) -> tuple:
    """The (K, V) caches of layer_tensors() (same draws): uint16 [B, n_kv, cap, d] each."""
    s, L = shape, layer
    return (normal_f16_bits(seed, tid(L, ROLE_K_CACHE), (B, s.n_kv, cap, s.d)),
            normal_f16_bits(seed, tid(L, ROLE_V_CACHE), (B, s.n_kv, cap, s.d)))


def layer_input(H: int, B: int, seed: int) -> np.ndarray:
    return normal_f32(seed, tid(0, ROLE_X), (B, H))
