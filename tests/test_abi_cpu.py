"""The C-ABI library builds, loads and exports every symbol include/gem.h declares; host-side
argument checks reject bad calls before any CUDA work.  CPU only (no compute calls)."""
import ctypes as C
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    text = open(os.path.join(ROOT, "include", "gem.h")).read()
    return set(re.findall(r"GEM_API\s+[\w\s\*]*?\b(gem_\w+)\s*\(", text))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    path = __graft_entry__._build_module().build()
    return C.CDLL(path)


def test_header_declares_the_boundary_calls():
    names = _declared()
    for n in ["gem_q4_0_gemv", "gem_rmsnorm_qknorm_rope", "gem_gqa_decode_attn", "gem_swiglu",
              "gem_decode_layer"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for n in sorted(_declared()):
        assert hasattr(lib, n), n


def test_binding_prototypes_cover_the_header():
    import importlib.util
    spec = importlib.util.spec_from_file_location("gem_lib", os.path.join(ROOT, "q4_gemv_gqa_gb300", "_lib.py"))
    m = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(m)
    assert set(m.PROTOTYPES) == _declared()


def test_status_strings(lib):
    lib.gem_status_string.restype = C.c_char_p
    assert lib.gem_status_string(0) == b"ok"
    assert lib.gem_status_string(3) == b"unsupported shape"
    assert lib.gem_status_string(99) == b"unknown status"


def test_gemv_host_checks_reject_before_cuda(lib):
    f = lib.gem_q4_0_gemv
    f.restype = C.c_int
    f.argtypes = [C.c_void_p, C.c_int64, C.c_int64, C.c_void_p, C.c_int64, C.c_int, C.c_void_p,
                  C.c_int64, C.c_void_p, C.c_void_p]
    dummy = C.c_void_p(0x1000)
    assert f(dummy, 4, 33, dummy, 33, 1, dummy, 4, None, None) == 3      # K % 32 != 0
    assert f(dummy, 4, 64, dummy, 64, 9, dummy, 4, None, None) == 3      # B > 8
    assert f(None, 4, 64, dummy, 64, 1, dummy, 4, None, None) == 1       # null W
    assert f(dummy, 4, 64, dummy, 32, 1, dummy, 4, None, None) == 1      # ldx < K
    assert f(dummy, -1, 64, dummy, 64, 1, dummy, 4, None, None) == 1     # negative N
    assert f(dummy, 4, 64, dummy, 64, 0, dummy, 4, None, None) == 0      # B == 0: nothing to do
    assert f(dummy, 0, 64, dummy, 64, 2, dummy, 4, None, None) == 0      # N == 0: nothing to do


def test_rope_and_attention_host_checks(lib):
    r = lib.gem_rmsnorm_qknorm_rope
    r.restype = C.c_int
    i, p, f = C.c_int, C.c_void_p, C.c_float
    r.argtypes = [p, C.c_int64, i, i, i, i, p, p, i, f, p, f, i, p, p, C.c_int64, i, p, p]
    d = C.c_void_p(0x1000)
    assert r(d, 512, 1, 4, 2, 64, None, None, 0, 1e-6, d, 1e6, 63, d, d, 10, 0, None, None) == 1   # odd rope_dim
    assert r(d, 512, 1, 4, 2, 64, None, None, 2, 1e-6, d, 1e6, 64, d, d, 10, 0, None, None) == 1   # bad v_mode
    assert r(d, 512, 1, 4, 2, 64, None, None, 0, 1e-6, d, 1e6, 64, d, d, 10, 16, None, None) == 1  # window > cap
    assert r(d, 100, 1, 4, 2, 64, None, None, 0, 1e-6, d, 1e6, 64, d, d, 10, 0, None, None) == 1   # ldqkv too small
    a = lib.gem_gqa_decode_attn
    a.restype = C.c_int
    a.argtypes = [p, C.c_int64, p, p, i, i, i, i, C.c_int64, p, i, f, p, C.c_int64, p, C.c_size_t, p, p]
    assert a(d, 512, d, d, 1, 4, 2, 96, 10, d, 0, 1.0, d, 512, None, 0, None, None) == 3   # head dim
    assert a(d, 1024, d, d, 1, 18, 2, 64, 10, d, 0, 1.0, d, 1024, None, 0, None, None) == 3  # G = 9 > 8
    assert a(d, 512, d, d, 1, 5, 2, 64, 10, d, 0, 1.0, d, 512, None, 0, None, None) == 1   # n_q % n_kv


def test_python_binding_imports_and_wraps(lib):
    import q4_gemv_gqa_gb300 as gem
    assert gem.version() == 100
    with pytest.raises(gem.GemError) as e:
        gem._check(3, "x")
    assert "unsupported shape" in str(e.value)


def test_status_from_flags_and_control_range_checks(lib):
    """Host-only mappings and range checks of the failure-detection controls (no CUDA call)."""
    f = lib.gem_status_from_flags
    f.restype = C.c_int
    f.argtypes = [C.c_int32]
    assert f(0) == 0
    assert f(1) == 5          # GEM_DEVFLAG_POS_RANGE -> GEM_ERR_DEVICE_FLAG
    assert f(2) == 6          # GEM_DEVFLAG_TIMEOUT -> GEM_ERR_TIMEOUT
    assert f(3) == 6          # timeout wins over other bits
    w = lib.gem_set_wait_limit
    w.restype = C.c_int
    w.argtypes = [C.c_uint64]
    assert w(999) == 1        # below 1 us
    assert w(61_000_000_000) == 1
    inj = lib.gem_set_test_injection
    inj.restype = C.c_int
    inj.argtypes = [C.c_int]
    assert inj(4) == 1        # unknown bit


def test_gemv_workspace_query_and_checks(lib):
    q = lib.gem_q4_0_gemv_workspace
    q.restype = C.c_size_t
    q.argtypes = [C.c_int, C.c_int64]
    assert q(1, 2048) == 0                 # one row: no records
    n2 = q(2, 2048)
    assert n2 > 0 and n2 % 256 == 0
    assert q(8, 2048) == n2                # records hold 8 rows' operands whatever B
    assert q(8, 4096) > n2
    f = lib.gem_q4_0_gemv_ws
    f.restype = C.c_int
    f.argtypes = [C.c_void_p, C.c_int64, C.c_int64, C.c_void_p, C.c_int64, C.c_int, C.c_void_p, C.c_int64,
                  C.c_void_p, C.c_void_p, C.c_size_t, C.c_void_p]
    d = C.c_void_p(0x1000)
    assert f(d, 64, 2048, d, 2048, 2, d, 64, None, None, 0, None) == 7             # no workspace
    assert f(d, 64, 2048, d, 2048, 2, d, 64, None, d, n2 - 256, None) == 7         # too small
    assert f(d, 64, 2048, d, 2048, 2, d, 64, None, C.c_void_p(0x1010), n2, None) == 2   # misaligned
    assert f(d, 64, 33, d, 64, 2, d, 64, None, d, n2, None) == 3                  # K % 32 != 0
