"""Python wrapper of the CPU oracle (``luce_oracle.c``).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  It shares no code
with the CUDA library: it compiles its own C file with gcc and is called with
numpy arrays.

Every function here is a thin ctypes call into the C oracle, plus two pieces
of tolerance bookkeeping (``tol`` and ``hq_flip_allowance``) that turn the
oracle's error scales into the pass/fail bounds the tests use.  Pages are
cited by title: [PR826] is Lucebox PR #826 "feat(ds41): two-box
expert-parallel serving".
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "luce_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libluce_oracle.so")
_LIB = None

QK = 32
Q8_0_BYTES = 34
Q8_1_BYTES = 36

#: float tolerance of the graded outputs: |gpu - oracle| <= REL * terms + ABS
REL = 1e-4
ABS = 1e-6


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (ISO C, no FMA contraction, no fast-math)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
             "-Wall", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _lib():
    global _LIB
    if _LIB is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        P = ctypes.c_void_p
        i64 = ctypes.c_int64
        i32 = ctypes.c_int
        d = ctypes.c_double
        lib.lo_fp16_encode.restype = ctypes.c_uint16
        lib.lo_fp16_encode.argtypes = [ctypes.c_float]
        lib.lo_fp16_decode.restype = ctypes.c_float
        lib.lo_fp16_decode.argtypes = [ctypes.c_uint16]
        lib.lo_fp16_encode_n.argtypes = [P, i64, P]
        lib.lo_fp16_decode_n.argtypes = [P, i64, P]
        lib.lo_quantize_q8_1.argtypes = [P, i64, i64, P]
        lib.lo_dot_q8_0_q8_1.restype = d
        lib.lo_dot_q8_0_q8_1.argtypes = [P, P, i64, P]
        lib.lo_block_isums.argtypes = [P, P, i64, P]
        lib.lo_matvec_q8_0.argtypes = [P, i64, i64, P, P, P]
        lib.lo_silu.restype = d
        lib.lo_silu.argtypes = [d]
        lib.lo_swiglu.restype = d
        lib.lo_swiglu.argtypes = [d, d, d]
        lib.lo_route_topk.argtypes = [P, P, i32, i32, i32, P, P]
        lib.lo_moe_group.argtypes = [P, i32, i32, i32, P, P, P]
        lib.lo_glu_pair.argtypes = [P, P, P, P, P, P, i32, i32, i32, i32, i32, d, P, P]
        lib.lo_down_combine.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i32, P, P]
        lib.lo_argmax.argtypes = [P, i32, i64, P, P]
        lib.lo_argmax_pick.argtypes = [P, P, i32, i32, P, P]
        lib.lo_q4_k_scale_min.argtypes = [P, i32, P, P]
        lib.lo_dot_q4_k_q8_1.restype = d
        lib.lo_dot_q4_k_q8_1.argtypes = [P, P, i64, P]
        lib.lo_glu_q4k.argtypes = [P, P, P, P, P, P, i32, i32, i32, i32, i32, d, P, P]
        lib.lo_down_combine_q4k.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i32, P, P]
        lib.lo_rmsnorm_router.argtypes = [P, P, d, P, i32, i32, i32, P, P, P]
        _LIB = lib
    return _LIB


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ----------------------------------------------------------------------------- fp16
def fp16_encode(x) -> np.ndarray:
    """IEEE binary16 bits of fp32 values, round to nearest even."""
    x = _c(x, np.float32)
    out = np.empty(x.shape, np.uint16)
    _lib().lo_fp16_encode_n(_p(x), x.size, _p(out))
    return out


def fp16_decode(h) -> np.ndarray:
    h = _c(h, np.uint16)
    out = np.empty(h.shape, np.float32)
    _lib().lo_fp16_decode_n(_p(h), h.size, _p(out))
    return out


# ----------------------------------------------------------------------------- q8_1
def quantize_q8_1(x) -> np.ndarray:
    """x [..., K] fp32 -> q8_1 blocks uint8 [..., K/32, 36] ([PR826] q8_1 memo)."""
    x = _c(x, np.float32)
    K = x.shape[-1]
    assert K % QK == 0
    rows = x.size // K
    out = np.empty(x.shape[:-1] + (K // QK, Q8_1_BYTES), np.uint8)
    _lib().lo_quantize_q8_1(_p(x), rows, K, _p(out))
    return out


def dequant_q8_1(blocks) -> np.ndarray:
    """q8_1 blocks [..., nb, 36] -> fp32 values d*q, [..., nb*32] (test helper)."""
    b = _c(blocks, np.uint8)
    d = fp16_decode(b[..., 0:2].copy().view(np.uint16)[..., 0])
    q = b[..., 4:36].view(np.int8).astype(np.float32)
    return (q * d[..., None]).reshape(b.shape[:-2] + (-1,))


def dot_q8_0_q8_1(w_row, x_row):
    """(value, terms) of one Q8_0 row times one q8_1 row."""
    w_row = _c(w_row, np.uint8)
    x_row = _c(x_row, np.uint8)
    nb = w_row.size // Q8_0_BYTES
    assert x_row.size == nb * Q8_1_BYTES
    t = np.zeros(1, np.float64)
    v = _lib().lo_dot_q8_0_q8_1(_p(w_row), _p(x_row), nb * QK, _p(t))
    return v, float(t[0])


def block_isums(w_row, x_row) -> np.ndarray:
    w_row = _c(w_row, np.uint8)
    x_row = _c(x_row, np.uint8)
    nb = w_row.size // Q8_0_BYTES
    out = np.empty(nb, np.int32)
    _lib().lo_block_isums(_p(w_row), _p(x_row), nb * QK, _p(out))
    return out


def matvec_q8_0(W, xq):
    """W [rows, nb, 34] uint8, xq [nb, 36] -> (y f64 [rows], terms f64 [rows])."""
    W = _c(W, np.uint8)
    xq = _c(xq, np.uint8)
    rows = W.shape[0]
    nb = W.size // rows // Q8_0_BYTES
    y = np.empty(rows, np.float64)
    t = np.empty(rows, np.float64)
    _lib().lo_matvec_q8_0(_p(W), rows, nb * QK, _p(xq), _p(y), _p(t))
    return y, t


def silu(g: float) -> float:
    return _lib().lo_silu(float(g))


def swiglu(g: float, u: float, clamp: float = 0.0) -> float:
    return _lib().lo_swiglu(float(g), float(u), float(clamp))


# ----------------------------------------------------------------------------- router
def route_topk(logits, bias, k: int):
    """logits [T, E] f32, bias [E] f32 or None -> ids int32 [T, k], weights f64 [T, k]."""
    logits = _c(logits, np.float32)
    T, E = logits.shape
    b = None if bias is None else _c(bias, np.float32)
    ids = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    _lib().lo_route_topk(_p(logits), _p(b), T, E, k, _p(ids), _p(w))
    return ids, w


def moe_group(ids, E: int):
    """ids int32 [T, k] -> counts [E], offsets [E+1], routes [T*k] (int32)."""
    ids = _c(ids, np.int32)
    T, k = ids.shape
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    routes = np.empty(T * k, np.int32)
    _lib().lo_moe_group(_p(ids), T, k, E, _p(counts), _p(offsets), _p(routes))
    return counts, offsets, routes


# ----------------------------------------------------------------------------- experts
def glu_pair(wg, wu, wsg, wsu, xq, ids, E: int, H: int, I: int, clamp: float):
    """Gate/up pair + SwiGLU for every kept route and the shared expert.

    wg, wu: [E, I, H/32, 34] uint8; wsg, wsu: [I, H/32, 34] or None;
    xq: [T, H/32, 36]; ids [T, k].  Returns h f64 [T*k (+T), I] (rows of
    masked routes are NaN) and the per-element error scale h_terms.
    """
    ids = _c(ids, np.int32)
    T, k = ids.shape
    wg = _c(wg, np.uint8)
    wu = _c(wu, np.uint8)
    xq = _c(xq, np.uint8)
    wsg = None if wsg is None else _c(wsg, np.uint8)
    wsu = None if wsu is None else _c(wsu, np.uint8)
    rows = T * k + (T if wsg is not None else 0)
    h = np.full((rows, I), np.nan, np.float64)
    ht = np.full((rows, I), np.nan, np.float64)
    _lib().lo_glu_pair(_p(wg), _p(wu), _p(wsg), _p(wsu), _p(xq), _p(ids), T, k, E, H, I, float(clamp),
                       _p(h), _p(ht))
    return h, ht


def down_combine(wd, wsd, hq, ids, weights, E: int, H: int, I: int):
    """Down product + masked route-weighted combine + shared expert.

    wd [E, H, I/32, 34], wsd [H, I/32, 34] or None, hq [T*k (+T), I/32, 36],
    ids [T, k], weights [T, k] (rounded to fp32).  Returns out f32 [T, H] and
    its error scale out_terms f64 [T, H].
    """
    ids = _c(ids, np.int32)
    T, k = ids.shape
    wd = _c(wd, np.uint8)
    wsd = None if wsd is None else _c(wsd, np.uint8)
    hq = _c(hq, np.uint8)
    w = _c(weights, np.float32)
    out = np.empty((T, H), np.float32)
    ot = np.empty((T, H), np.float64)
    _lib().lo_down_combine(_p(wd), _p(wsd), _p(hq), _p(ids), _p(w), T, k, E, H, I, _p(out), _p(ot))
    return out, ot


def argmax(logits):
    """logits [R, V] f32 -> idx int32 [R], val f32 [R] (first maximum)."""
    logits = _c(logits, np.float32)
    R, V = logits.shape
    idx = np.empty(R, np.int32)
    val = np.empty(R, np.float32)
    _lib().lo_argmax(_p(logits), R, V, _p(idx), _p(val))
    return idx, val


Q4_K_BYTES = 144
QK_K = 256


def q4_k_scale_min(scales12, j: int):
    """(sc_j, m_j) of a Q4_K super-block's 12 packed scale bytes."""
    s = _c(scales12, np.uint8)
    sc = ctypes.c_int(0)
    m = ctypes.c_int(0)
    _lib().lo_q4_k_scale_min(_p(s), int(j), ctypes.byref(sc), ctypes.byref(m))
    return sc.value, m.value


def dot_q4_k_q8_1(w_row, x_row):
    """(value, terms) of one Q4_K row [K/256, 144] times one q8_1 row [K/32, 36]."""
    w_row = _c(w_row, np.uint8)
    x_row = _c(x_row, np.uint8)
    K = x_row.shape[-2] * QK
    t = ctypes.c_double(0.0)
    v = _lib().lo_dot_q4_k_q8_1(_p(w_row), _p(x_row), K, ctypes.byref(t))
    return v, t.value


def glu_q4k(wg, wu, wsg, wsu, xq, ids, E: int, H: int, I: int, clamp: float):
    """glu_pair with Q4_K gate/up weights [E, I, H/256, 144] (shared [I, H/256, 144])."""
    ids = _c(ids, np.int32)
    T, k = ids.shape
    wg, wu, xq = _c(wg, np.uint8), _c(wu, np.uint8), _c(xq, np.uint8)
    wsg = None if wsg is None else _c(wsg, np.uint8)
    wsu = None if wsu is None else _c(wsu, np.uint8)
    rows = T * k + (T if wsg is not None else 0)
    h = np.full((rows, I), np.nan, np.float64)
    ht = np.full((rows, I), np.nan, np.float64)
    _lib().lo_glu_q4k(_p(wg), _p(wu), _p(wsg), _p(wsu), _p(xq), _p(ids), T, k, E, H, I, float(clamp), _p(h), _p(ht))
    return h, ht


def down_combine_q4k(wd, wsd, hq, ids, weights, E: int, H: int, I: int):
    """down_combine with Q4_K down weights [E, H, I/256, 144] (shared [H, I/256, 144])."""
    ids = _c(ids, np.int32)
    T, k = ids.shape
    wd, hq = _c(wd, np.uint8), _c(hq, np.uint8)
    wsd = None if wsd is None else _c(wsd, np.uint8)
    w = _c(weights, np.float32)
    out = np.empty((T, H), np.float32)
    ot = np.empty((T, H), np.float64)
    _lib().lo_down_combine_q4k(_p(wd), _p(wsd), _p(hq), _p(ids), _p(w), T, k, E, H, I, _p(out), _p(ot))
    return out, ot


def moe_layer_q4k(wg, wu, wd, wsg, wsu, wsd, x, logits, bias, k: int, clamp: float):
    """moe_layer with Q4_K expert weights (the same steps and roundings)."""
    x = _c(x, np.float32)
    T, H = x.shape
    E, I = wg.shape[0], wg.shape[1]
    ids, w = route_topk(logits, bias, k)
    xq = quantize_q8_1(x)
    h, ht = glu_q4k(wg, wu, wsg, wsu, xq, ids, E, H, I, clamp)
    h32 = np.nan_to_num(h, nan=0.0).astype(np.float32)
    ht0 = np.nan_to_num(ht, nan=0.0)
    hq = quantize_q8_1(h32)
    out, ot = down_combine_q4k(wd, wsd, hq, ids, w.astype(np.float32), E, H, I)
    return dict(ids=ids, weights=w, xq=xq, h=h, h_terms=ht, hq=hq, out=out, out_terms=ot,
                h_allow=hq_flip_allowance(h32, tol(ht0)))


def argmax_pick(vals, idxs):
    """Pairs of S vocabulary shards, vals f32 [S, R] and global idxs int32 [S, R]
    -> idx int32 [R], val f32 [R] (largest value, ties to the lower index)."""
    vals = _c(vals, np.float32)
    idxs = _c(idxs, np.int32)
    S, R = vals.shape
    idx = np.empty(R, np.int32)
    val = np.empty(R, np.float32)
    _lib().lo_argmax_pick(_p(vals), _p(idxs), S, R, _p(idx), _p(val))
    return idx, val


def rmsnorm_router(x, gamma, eps: float, w_router):
    """x [T, H] f32, gamma [H] f32, w_router [E, H] f32 -> (xn f64 [T, H],
    logits f64 [T, E], logit error scale f64 [T, E])."""
    x = _c(x, np.float32)
    gamma = _c(gamma, np.float32)
    w_router = _c(w_router, np.float32)
    T, H = x.shape
    E = w_router.shape[0]
    xn = np.empty((T, H), np.float64)
    logits = np.empty((T, E), np.float64)
    terms = np.empty((T, E), np.float64)
    _lib().lo_rmsnorm_router(_p(x), _p(gamma), float(eps), _p(w_router), T, E, H, _p(xn), _p(logits), _p(terms))
    return xn, logits, terms


def ep_layer(wg, wu, wd, wsg, wsu, wsd, x, logits, bias, k: int, clamp: float, bounds):
    """The step split over len(bounds) - 1 expert-parallel ranks ([PR826]:
    each rank holds a share of the routed experts, routes it does not own
    reach it masked to id -1, and the ranks sum their partial outputs every
    layer).  Rank s owns the routed experts [bounds[s], bounds[s + 1]); rank
    0 also runs the shared expert.  Each rank's partial is moe_layer's
    arithmetic with the other ranks' routes masked; out is the sum of the
    partials in rank order, each addition rounded to fp32.

    Returns a dict with ids (unmasked), weights, partials, out, out_terms and
    the q8_1 flip allowance of h (every route's h is computed by one rank).
    """
    x = _c(x, np.float32)
    T, H = x.shape
    E = wg.shape[0]
    I = wg.shape[1]
    ids, w = route_topk(logits, bias, k)
    xq = quantize_q8_1(x)
    parts, terms, allow = [], np.zeros((T, H)), None
    for s in range(len(bounds) - 1):
        ids_s = np.where((ids >= bounds[s]) & (ids < bounds[s + 1]), ids, -1).astype(np.int32)
        sg, su, sd = (wsg, wsu, wsd) if s == 0 else (None, None, None)
        h, ht = glu_pair(wg, wu, sg, su, xq, ids_s, E, H, I, clamp)
        h32 = np.nan_to_num(h, nan=0.0).astype(np.float32)
        a = hq_flip_allowance(h32, tol(np.nan_to_num(ht, nan=0.0)))
        a[:T * k][ids_s.reshape(-1) < 0] = 0.0  # rows of routes this rank does not own
        if allow is None:
            allow = np.zeros((T * k + (T if wsg is not None else 0), I))
        allow[:a.shape[0]] += a
        out_s, ot = down_combine(wd, sd, quantize_q8_1(h32), ids_s, w.astype(np.float32), E, H, I)
        parts.append(out_s)
        terms += ot
    out = parts[0].copy()
    for p in parts[1:]:
        out = (out + p).astype(np.float32)
    return dict(ids=ids, weights=w, partials=parts, out=out, out_terms=terms, h_allow=allow)


# ----------------------------------------------------------------------------- tolerance
def tol(terms):
    """The float bound: REL * terms + ABS."""
    return REL * np.asarray(terms, np.float64) + ABS


def hq_flip_allowance(h32, h_tol):
    """Where may a q8_1 quantization of h differ from the oracle's, and by how much?

    The oracle quantizes its own h (rounded to fp32); the GPU quantizes its own
    h, which may differ from the oracle's by up to h_tol per element.  Both
    quantize in fp32 with the same rule, so their codes can differ only where
    the perturbation of h can move x/d across a rounding midpoint (one step
    of q), or move d = amax/127 across an fp16 midpoint (one fp16 step of the
    stored d16).  Returns, per element, a bound on |d16*q (GPU) - d16*q
    (oracle)|: zero for every element whose quantization is stable.
    """
    h32 = np.asarray(h32, np.float32)
    shp = h32.shape
    hb = h32.reshape(-1, QK).astype(np.float64)
    tb = np.asarray(h_tol, np.float64).reshape(-1, QK)
    amax32 = np.abs(h32.reshape(-1, QK)).max(axis=1)
    d = (amax32 / np.float32(127.0)).astype(np.float64)  # the fp32 d of the rule
    tmax = tb.max(axis=1)
    delta_d = tmax / 127.0 * 1.01 + 1e-30
    # the stored d16 of any amax within the bound lies between fp16(d - delta_d)
    # and fp16(d + delta_d) (rounding is monotonic): several fp16 steps when
    # delta_d spans more than one
    d16 = d.astype(np.float16).astype(np.float64)
    d16_hi = (d + delta_d).astype(np.float16).astype(np.float64)
    d16_lo = np.maximum(d - delta_d, 0.0).astype(np.float16).astype(np.float64)
    d16_change = np.maximum(d16_hi - d16, d16 - d16_lo)
    safe_d = np.where(d > 0, d, 1.0)
    ratio = np.abs(hb) / safe_d[:, None]
    eps = (tb + ratio * delta_d[:, None]) / safe_d[:, None] * 1.01 + 1e-6
    dist = np.abs(ratio - np.floor(ratio) - 0.5)
    q_unstable = dist <= eps
    qmag = np.floor(ratio + 0.5)
    allow = (np.where(q_unstable, d16[:, None] + d16_change[:, None], 0.0)
             + (qmag + 1.0) * d16_change[:, None])
    # a block the oracle quantizes to all zeros may be non-zero on the GPU
    zero = (d == 0)[:, None] & (tmax[:, None] > 0)
    allow = np.where(zero, 2.0 * tb.max(axis=1, keepdims=True) + 1e-30, allow)
    return allow.reshape(shp)


# ----------------------------------------------------------------------------- composition
def moe_layer(wg, wu, wd, wsg, wsu, wsd, x, logits, bias, k: int, clamp: float):
    """The whole decode MoE-FFN step in the pages' order ([PR826]):
    route (select + weights), quantize x once to q8_1, gate/up pair + SwiGLU
    for every route and the shared expert, quantize h to q8_1 (from h rounded
    to fp32, the precision the quantization decision is made in), down
    product, masked route-weighted combine + shared expert.

    Returns a dict with ids, weights (f64), xq, h (f64), h_terms, hq, out (f32),
    out_terms and the q8_1 flip allowance of h.
    """
    x = _c(x, np.float32)
    T, H = x.shape
    E = wg.shape[0]
    I = wg.shape[1]
    ids, w = route_topk(logits, bias, k)
    xq = quantize_q8_1(x)
    h, ht = glu_pair(wg, wu, wsg, wsu, xq, ids, E, H, I, clamp)
    h32 = np.nan_to_num(h, nan=0.0).astype(np.float32)
    ht0 = np.nan_to_num(ht, nan=0.0)
    hq = quantize_q8_1(h32)
    out, ot = down_combine(wd, wsd, hq, ids, w.astype(np.float32), E, H, I)
    return dict(ids=ids, weights=w, xq=xq, h=h, h_terms=ht, hq=hq, out=out, out_terms=ot,
                h_allow=hq_flip_allowance(h32, tol(ht0)))
