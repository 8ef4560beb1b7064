"""The C-ABI library builds, loads and exports what include/luce_moe.h
declares; host-side argument validation rejects bad calls before any CUDA
work (CPU only: no call here reaches a kernel)."""
import ctypes
import os
import re

import pytest

from quantized_moe_decode_luce_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "luce_moe.h")


@pytest.fixture(scope="module")
def lib():
    path = B.build()
    L = ctypes.CDLL(path)
    return L


def declared_symbols():
    txt = open(HEADER).read()
    return sorted(set(re.findall(r"LUCE_API\s+[\w\s\*]+?\b(luce_\w+)\s*\(", txt)))


def test_header_declares_the_six_ops_and_helpers():
    names = declared_symbols()
    for want in ["luce_route_topk", "luce_quantize_q8_1", "luce_moe_group", "luce_moe_glu_pair",
                 "luce_moe_prep", "luce_set_pdl",
                 "luce_moe_down_combine", "luce_argmax", "luce_argmax_workspace_bytes", "luce_status_string",
                 "luce_get_fault", "luce_version"]:
        assert want in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name
    out = os.popen(f"nm -D --defined-only {B.LIB}").read()
    exported = set(re.findall(r" T (\w+)", out))
    assert set(declared_symbols()) == exported  # nothing else leaks out


def test_status_strings(lib):
    lib.luce_status_string.restype = ctypes.c_char_p
    assert lib.luce_status_string(0) == b"ok"
    assert lib.luce_status_string(1) == b"invalid argument"
    assert lib.luce_status_string(3) == b"CUDA error"
    assert lib.luce_version() >= 100


def _p(v):
    return ctypes.c_void_p(v)


# A 16-byte aligned fake device address.  Every call below either fails
# host validation or is an empty call (T == 0 / R == 0), so nothing is ever
# launched with it; no call here may pass validation with real work.
GOOD = 0x10000


def test_quantize_validation(lib):
    f = lib.luce_quantize_q8_1
    f.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
    assert f(_p(GOOD), 4, 33, _p(GOOD), None) == 1          # K % 32
    assert f(_p(GOOD), 4, 0, _p(GOOD), None) == 1
    assert f(_p(GOOD), -1, 32, _p(GOOD), None) == 1
    assert f(_p(GOOD + 2), 4, 32, _p(GOOD), None) == 1      # misaligned x
    assert f(None, 4, 32, _p(GOOD), None) == 1
    assert f(_p(GOOD), 0, 32, _p(GOOD), None) == 0          # empty call: nothing enqueued


def test_route_validation(lib):
    f = lib.luce_route_topk
    f.argtypes = [ctypes.c_void_p] * 2 + [ctypes.c_int] * 3 + [ctypes.c_void_p] * 3
    assert f(_p(GOOD), None, 1, 1025, 2, _p(GOOD), _p(GOOD), None) == 1   # E > 1024
    assert f(_p(GOOD), None, 1, 8, 9, _p(GOOD), _p(GOOD), None) == 1      # k > E
    assert f(_p(GOOD), None, 1, 128, 65, _p(GOOD), _p(GOOD), None) == 1   # k > 64
    assert f(_p(GOOD), None, 1, 8, 0, _p(GOOD), _p(GOOD), None) == 1
    assert f(_p(GOOD), _p(GOOD + 1), 1, 8, 2, _p(GOOD), _p(GOOD), None) == 1
    assert f(_p(GOOD), None, 0, 8, 2, _p(GOOD), _p(GOOD), None) == 0


def test_group_validation(lib):
    f = lib.luce_moe_group
    f.argtypes = [ctypes.c_void_p] + [ctypes.c_int] * 3 + [ctypes.c_void_p] * 4
    assert f(_p(GOOD), 1, 2, 0, _p(GOOD), _p(GOOD), _p(GOOD), None) == 1
    assert f(_p(GOOD), 1 << 20, 2, 8, _p(GOOD), _p(GOOD), _p(GOOD), None) == 1  # T*k > 2^20
    assert f(_p(GOOD), 1, 2, 8, None, _p(GOOD), _p(GOOD), None) == 1


def test_glu_and_down_validation(lib):
    g = lib.luce_moe_glu_pair
    g.argtypes = [ctypes.c_void_p] * 7 + [ctypes.c_int] * 5 + [ctypes.c_float] + [ctypes.c_void_p] * 2 + \
        [ctypes.c_int, ctypes.c_void_p]
    P = [_p(GOOD)] * 7
    assert g(*P, 1, 2, 8, 480, 256, 0.0, _p(GOOD), _p(GOOD), 0, None) == 1       # H % 256
    assert g(*P, 1, 2, 8, 512, 96, 0.0, _p(GOOD), _p(GOOD), 0, None) == 1        # I % 256
    assert g(*P, 1, 2, 8, 512, 256, 0.0, _p(GOOD), _p(GOOD), 7, None) == 1       # variant
    assert g(_p(GOOD + 8), *P[1:], 1, 2, 8, 512, 256, 0.0, _p(GOOD), _p(GOOD), 0, None) == 1  # 16-B alignment
    assert g(P[0], P[1], P[2], None, *P[4:], 1, 2, 8, 512, 256, 0.0, _p(GOOD), _p(GOOD), 0, None) == 1
    assert g(*P, 1, 2, 8, 512, 256, 0.0, _p(GOOD), None, 0, None) == 1           # hq missing
    assert g(*P, 0, 2, 8, 512, 256, 0.0, _p(GOOD), _p(GOOD), 0, None) == 0       # T = 0
    d = lib.luce_moe_down_combine
    d.argtypes = [ctypes.c_void_p] * 7 + [ctypes.c_int] * 5 + [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p]
    assert d(*P, 1, 2, 8, 512, 100, _p(GOOD), 0, None) == 1
    assert d(*P, 1, 2, 2000, 512, 256, _p(GOOD), 0, None) == 1                   # E > 1024
    assert d(*P, 0, 2, 8, 512, 256, _p(GOOD), 0, None) == 0


def test_prep_and_pdl_validation(lib):
    f = lib.luce_moe_prep
    f.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int] * 4 + [ctypes.c_void_p] * 7
    G = [_p(GOOD)] * 6
    assert f(_p(GOOD), None, _p(GOOD), 1, 64, 65, 2048, *G, None) == 1     # k > 64
    assert f(_p(GOOD), None, _p(GOOD), 1, 64, 6, 2047, *G, None) == 1      # H % 32
    assert f(_p(GOOD), None, None, 1, 64, 6, 2048, *G, None) == 1          # x missing
    assert f(_p(GOOD + 2), None, _p(GOOD), 1, 64, 6, 2048, *G, None) == 1  # misaligned logits
    lib.luce_set_pdl.argtypes = [ctypes.c_int]
    assert lib.luce_set_pdl(1) == 0 and lib.luce_set_pdl(0) == 0


def test_argmax_validation_and_workspace(lib):
    w = lib.luce_argmax_workspace_bytes
    w.argtypes = [ctypes.c_int, ctypes.c_int64]
    w.restype = ctypes.c_size_t
    assert w(0, 10) == 0
    assert w(1, 4096) >= 8 + 4
    n5 = w(5, 129280)
    assert n5 % 16 == 0 and n5 >= 5 * 8 + 5 * 4
    f = lib.luce_argmax
    f.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,
                  ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
    assert f(_p(GOOD), 5, 129280, _p(GOOD), None, _p(GOOD), n5 - 1, None) == 1   # workspace too small
    assert f(_p(GOOD), 1, 0, _p(GOOD), None, _p(GOOD), 64, None) == 1
    assert f(_p(GOOD), 1, 10, _p(GOOD), None, _p(GOOD + 4), 64, None) == 1       # workspace alignment
    assert f(_p(GOOD), 0, 10, _p(GOOD), None, _p(GOOD), 64, None) == 0


def test_edge_ops_validation(lib):
    f = lib.luce_rmsnorm_router
    f.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_float, ctypes.c_void_p] + [ctypes.c_int] * 3 + \
        [ctypes.c_void_p] * 3
    G = _p(GOOD)
    assert f(G, G, 1e-6, G, 1, 64, 2046, G, G, None) == 1          # H % 4
    assert f(G, G, 1e-6, G, 1, 64, 16384, G, G, None) == 1         # H > 12288
    assert f(G, G, -1.0, G, 1, 64, 2048, G, G, None) == 1          # eps < 0
    assert f(G, G, float("nan"), G, 1, 64, 2048, G, G, None) == 1  # eps NaN
    assert f(_p(GOOD + 4), G, 1e-6, G, 1, 64, 2048, G, G, None) == 1  # x not 16-byte aligned
    assert f(G, G, 1e-6, G, 1, 0, 2048, G, G, None) == 1           # E < 1
    assert f(G, G, 1e-6, G, 1, 64, 2048, G, None, None) == 1       # logits missing
    assert f(G, G, 1e-6, G, 0, 64, 2048, None, G, None) == 0       # T = 0
    r = lib.luce_add_rmsnorm_router
    r.argtypes = [ctypes.c_void_p] * 4 + [ctypes.c_float, ctypes.c_void_p] + [ctypes.c_int] * 3 + \
        [ctypes.c_void_p] * 3
    S = _p(GOOD + (1 << 20))
    assert r(G, None, S, G, 1e-6, G, 1, 64, 2048, G, G, None) == 1          # residual missing
    assert r(G, _p(GOOD + 4), S, G, 1e-6, G, 1, 64, 2048, G, G, None) == 1  # residual not 16-byte aligned
    assert r(G, _p(GOOD + 8192), _p(GOOD + 4096), G, 1e-6, G, 1, 64, 2048, G, G, None) == 1  # x_sum overlaps x
    assert r(G, _p(GOOD + 8192), _p(GOOD + 12288), G, 1e-6, G, 1, 64, 2048, G, G, None) == 1  # ... or residual
    assert r(G, G, S, G, 1e-6, G, 1, 64, 2046, G, G, None) == 1             # H % 4, as the plain norm
    assert r(G, None, None, G, 1e-6, G, 0, 64, 2048, None, G, None) == 0    # T = 0
    s = lib.luce_argmax_shard
    s.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,
                  ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
    assert s(G, 2, 1000, -1, G, None, G, 1 << 20, None) == 1       # v0 < 0
    assert s(G, 2, 1000, (1 << 31) - 10, G, None, G, 1 << 20, None) == 1  # v0 + Vs beyond int32
    assert s(G, 2, 1000, 0, G, None, G, 0, None) == 1              # workspace too small
    assert s(G, 0, 1000, 500, G, None, G, 0, None) == 0            # R = 0
    p = lib.luce_argmax_pick
    p.argtypes = [ctypes.c_void_p] * 2 + [ctypes.c_int] * 2 + [ctypes.c_void_p] * 3
    assert p(G, G, 0, 4, G, None, None) == 1                       # S < 1
    assert p(G, None, 2, 4, G, None, None) == 1
    assert p(G, G, 2, 0, G, None, None) == 0
    m = lib.luce_ep_mask
    m.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
    assert m(G, 8, 4, 2, G, None) == 1                             # e1 < e0
    assert m(G, -1, 0, 2, G, None) == 1
    assert m(G, 0, 0, 2, G, None) == 0
    a = lib.luce_add_f32
    a.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int64, ctypes.c_void_p]
    assert a(G, _p(GOOD + 2), G, 8, None) == 1                     # misaligned b
    assert a(G, G, G, 0, None) == 0


def test_q4k_validation(lib):
    G = _p(GOOD)
    g = lib.luce_moe_glu_q4k
    g.argtypes = [ctypes.c_void_p] * 6 + [ctypes.c_int] * 5 + [ctypes.c_float] + [ctypes.c_void_p] * 3
    assert g(G, G, G, G, G, G, 1, 2, 8, 2048 + 32, 1024, 0.0, G, None, None) == 1   # H % 256
    assert g(G, G, G, G, G, G, 1, 2, 8, 2048, 1000, 0.0, G, None, None) == 1        # I % 256
    assert g(G, G, G, None, G, G, 1, 2, 8, 2048, 1024, 0.0, G, None, None) == 1     # one shared matrix missing
    assert g(_p(GOOD + 4), G, G, G, G, G, 1, 2, 8, 2048, 1024, 0.0, G, None, None) == 1  # 16-byte alignment
    assert g(G, G, G, G, G, G, 1, 9, 8, 2048, 1024, 0.0, G, None, None) == 1        # k > E
    assert g(G, G, G, G, G, G, 1, 2, 8, 2048, 1024, 0.0, G, _p(GOOD + 2), None) == 1  # hq alignment
    assert g(G, G, G, G, G, G, 0, 2, 8, 2048, 1024, 0.0, G, None, None) == 0        # T = 0
    d = lib.luce_moe_down_combine_q4k
    d.argtypes = [ctypes.c_void_p] * 5 + [ctypes.c_int] * 5 + [ctypes.c_void_p] * 2
    assert d(G, G, G, G, G, 1, 2, 8, 2048, 1000, G, None) == 1                # I % 256
    assert d(G, None, G, G, None, 1, 2, 8, 2048, 1024, G, None) == 1          # weights missing
    assert d(G, None, G, G, G, 0, 2, 8, 2048, 1024, G, None) == 0
