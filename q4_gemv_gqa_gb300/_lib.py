"""ctypes loader of libgem.so (the CUDA library) and the C-ABI prototypes.

There is no fallback: if the library is missing or fails to load, importing the package
raises, so nothing can silently run a different implementation."""
from __future__ import annotations

import ctypes as C
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libgem.so")

p = C.c_void_p
i64 = C.c_int64
i32 = C.c_int


class LayerDesc(C.Structure):
    """Mirror of gem_layer_desc (include/gem.h)."""
    _fields_ = [("H", i64), ("n_q", i64), ("n_kv", i64), ("d", i64), ("F", i64),
                ("eps", C.c_float), ("theta", C.c_float), ("scale", C.c_float),
                ("rope_dim", i32), ("window", i32), ("act", i32),
                ("qk_norm", i32), ("v_from_k", i32), ("post_norms", i32),
                ("w_qkv", p), ("w_o", p), ("w_gate", p), ("w_up", p), ("w_down", p),
                ("g_attn", p), ("g_ffn", p), ("g_q", p), ("g_k", p),
                ("g_post_attn", p), ("g_post_ffn", p), ("compact_kv", i32)]


# name -> (restype, argtypes); every symbol declared in include/gem.h
PROTOTYPES = {
    "gem_status_string": (C.c_char_p, [i32]),
    "gem_last_cuda_error": (i32, []),
    "gem_version": (i32, []),
    "gem_device_status": (i32, [p, i32]),
    "gem_status_from_flags": (i32, [i32]),
    "gem_set_wait_limit": (i32, [C.c_uint64]),
    "gem_set_test_injection": (i32, [i32]),
    "gem_q4_0_gemv": (i32, [p, i64, i64, p, i64, i32, p, i64, p, p]),
    "gem_q4_0_gemv_workspace": (C.c_size_t, [i32, i64]),
    "gem_q4_0_gemv_ws": (i32, [p, i64, i64, p, i64, i32, p, i64, p, p, C.c_size_t, p]),
    "gem_q4_0_gemv_fused": (i32, [p, p, i64, i64, p, i64, i32, p, C.c_float, i32, p, i64, p, p,
                                  C.c_size_t, p]),
    "gem_q4_0_gemm_workspace": (C.c_size_t, [i32, i64]),
    "gem_q4_0_gemm": (i32, [p, p, i64, i64, p, i64, i32, p, C.c_float, i32, p, i64, p, p, C.c_size_t, p]),
    "gem_topk_workspace": (C.c_size_t, [i32, i64, i32]),
    "gem_topk": (i32, [p, i64, i32, i64, i32, p, p, p, C.c_size_t, p]),
    "gem_q8_0_gemv": (i32, [p, i64, i64, p, i64, i32, p, i64, p]),
    "gem_argmax_workspace": (C.c_size_t, [i32, i64]),
    "gem_argmax": (i32, [p, i64, i32, i64, p, p, C.c_size_t, p]),
    "gem_rmsnorm": (i32, [p, i32, i64, p, C.c_float, p, p]),
    "gem_rmsnorm_qknorm_rope": (i32, [p, i64, i32, i32, i32, i32, p, p, i32, C.c_float, p,
                                      C.c_float, i32, p, p, i64, i32, p, p]),
    "gem_gqa_decode_attn_workspace": (C.c_size_t, [i32, i32, i32, i32, i64, i32]),
    "gem_gqa_decode_attn": (i32, [p, i64, p, p, i32, i32, i32, i32, i64, p, i32, C.c_float,
                                  p, i64, p, C.c_size_t, p, p]),
    "gem_gqa_decode_attn_fused": (i32, [p, i64, i32, i32, i32, i32, p, p, i32, C.c_float, p, C.c_float,
                                        i32, p, p, i64, i32, C.c_float, p, i64, p, C.c_size_t, p, p]),
    "gem_gqa_decode_attn_compact_workspace": (C.c_size_t, [i32, i32, i32, i32, i64, i32]),
    "gem_gqa_decode_attn_compact": (i32, [p, i64, p, i32, i32, i32, i32, i64, p, C.c_float, p, i32,
                                          C.c_float, p, i64, p, C.c_size_t, p, p]),
    "gem_gqa_decode_attn_noalloc": (i32, [p, i64, p, p, i32, i32, i32, i32, i64, p, i32,
                                          C.c_float, p, i64, p, p]),
    "gem_swiglu": (i32, [p, p, i32, i64, i32, p, p]),
    "gem_decode_layer_workspace": (C.c_size_t, [C.POINTER(LayerDesc), i32, i64]),
    "gem_decode_layer": (i32, [C.POINTER(LayerDesc), i32, p, p, p, i64, p, p, C.c_size_t, p, p]),
    "gem_step_plan_create": (i32, [C.POINTER(LayerDesc), i32, i32, C.POINTER(p), C.POINTER(p),
                                   C.POINTER(i64), C.POINTER(p)]),
    "gem_decode_step": (i32, [p, p, p, p, p]),
    "gem_step_plan_destroy": (None, [p]),
}

_lib = None


def load() -> C.CDLL:
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError("libgem.so is not built (expected at %s); run "
                          "`python -c 'import __graft_entry__ as g; g.build()'`" % LIB_PATH)
    lib = C.CDLL(LIB_PATH)
    for name, (res, args) in PROTOTYPES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib
