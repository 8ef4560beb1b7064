"""Pins of the CPU oracle against things other than itself (CPU only).

Each test checks one oracle function against a value or property the pages
or the mathematics fix: hand-worked blocks, an independent fp16 codec
(numpy's), exact rational arithmetic, brute force over subsets, closed forms
and invariants.  Pages are cited by title: [PR826] is Lucebox PR #826
"feat(ds41): two-box expert-parallel serving".
"""
import itertools
import math
import os
import struct
from fractions import Fraction

import numpy as np
import pytest

import oracle
from quantized_moe_decode_luce_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------------------- fp16 codec
def test_fp16_decode_all_codes_match_numpy():
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.fp16_decode(codes)
    ref = codes.view(np.float16).astype(np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_fp16_encode_roundtrip_and_midpoints_match_numpy():
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = codes.view(np.float16).astype(np.float32)
    finite = np.isfinite(vals)
    # every fp16 value round-trips
    assert np.array_equal(oracle.fp16_encode(vals[finite]), codes[finite])
    # every midpoint between neighbouring finite fp16 values, and points just
    # beside it: ties go to the even code (IEEE round to nearest even)
    pos = np.arange(0, 0x7c00, dtype=np.uint16).view(np.float16).astype(np.float64)
    mids = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)  # exact in fp32
    for m in (mids, np.nextafter(mids, np.float32(np.inf)), np.nextafter(mids, np.float32(0))):
        for s in (1, -1):
            x = (s * m).astype(np.float32)
            assert np.array_equal(oracle.fp16_encode(x), x.astype(np.float16).view(np.uint16))


def test_fp16_encode_random_and_special_match_numpy():
    g = np.random.default_rng(7)
    bits = g.integers(0, 2**32, size=400000, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    x = x[~np.isnan(x)]
    assert np.array_equal(oracle.fp16_encode(x), x.astype(np.float16).view(np.uint16))
    special = np.array([0.0, -0.0, np.inf, -np.inf, 65504, 65519.99, 65520, 1e-8, 2.0**-25,
                        2.0**-25 * 1.0000001, 2.0**-24, 3 * 2.0**-25, 6.1e-5], np.float32)
    assert np.array_equal(oracle.fp16_encode(special), special.astype(np.float16).view(np.uint16))
    # Python's struct 'e' codec agrees too (another independent encoder)
    for v in [0.1, 1 / 3, 1e-3, 2e-2, 12345.678, -7.77]:
        f = float(np.float32(v))
        assert oracle.fp16_encode(np.array([f], np.float32))[0] == struct.unpack("<H", struct.pack("<e", f))[0]


# ----------------------------------------------------------------------------- q8_1 blocks
def _parse_pairs(s):
    out = np.zeros(32, np.float64)
    for tok in s.split():
        i, v = tok.split(":")
        out[int(i)] = float(v)
    return out


def test_q8_1_hand_worked_blocks():
    n = 0
    with open(os.path.join(GOLDEN, "q8_1_blocks.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            name, xs, d16, s16, qs = [p.strip() for p in line.split(";")]
            x = _parse_pairs(xs).astype(np.float32)
            b = oracle.quantize_q8_1(x[None])[0, 0]
            assert b[0:2].view(np.uint16)[0] == int(d16, 16), name
            assert b[2:4].view(np.uint16)[0] == int(s16, 16), name
            assert np.array_equal(b[4:].view(np.int8).astype(np.int64), _parse_pairs(qs).astype(np.int64)), name
            n += 1
    assert n == 5


def test_q8_1_codes_are_nearest_by_brute_force():
    """q is the integer in [-127, 127] nearest to x/d (ties away from zero), by search."""
    g = np.random.default_rng(1)
    x = np.concatenate([g.standard_normal((40, 32)), g.uniform(-3, 3, (40, 32)) * 10.0 ** g.integers(-6, 4, (40, 1)),
                        np.round(g.standard_normal((20, 32)) * 4) / 2]).astype(np.float32)
    blocks = oracle.quantize_q8_1(x)[:, 0]
    cand = np.arange(-127, 128, dtype=np.float64)
    for xb, b in zip(x, blocks):
        amax = float(np.max(np.abs(xb)))
        d = float(np.float32(amax) / np.float32(127.0))
        q = b[4:].view(np.int8).astype(np.int64)
        for xi, qi in zip(xb, q):
            r = float(np.float32(xi) / np.float32(d))  # the fp32 quotient of the rule
            dist = np.abs(cand - r)
            best = cand[dist == dist.min()]
            want = best[np.argmax(np.abs(best))] if len(best) > 1 else best[0]  # tie: away from 0
            assert qi == want
        assert np.max(np.abs(q)) == 127
        d16 = b[0:2].view(np.float16)[0]
        s16 = b[2:4].view(np.float16)[0]
        assert d16 == np.float16(d)
        assert s16 == np.float16(np.float32(d) * np.float32(q.sum()))


def test_q8_1_zero_block():
    b = oracle.quantize_q8_1(np.zeros((1, 64), np.float32))
    assert not b.any()


# ----------------------------------------------------------------------------- dot products
def _frac16(u16):
    return Fraction(float(np.array([u16], np.uint16).view(np.float16)[0]))


@pytest.mark.parametrize("K", [32, 64, 256])
def test_dot_equals_exact_rational_dequantized_dot(K):
    g = np.random.default_rng(K)
    for _ in range(6):
        w = W.q8_0_blocks(g, 1, K)[0]
        xq = oracle.quantize_q8_1(g.standard_normal((1, K)).astype(np.float32))[0]
        # exact: sum_i (d_w qw_i)(d_x qx_i), fp16 scales decoded by numpy
        exact = Fraction(0)
        tabs = Fraction(0)
        for b in range(K // 32):
            dw = _frac16(w[b, 0:2].view(np.uint16)[0])
            dx = _frac16(xq[b, 0:2].view(np.uint16)[0])
            s = sum(int(a) * int(c) for a, c in zip(w[b, 2:].view(np.int8), xq[b, 4:].view(np.int8)))
            exact += dw * dx * s
            tabs += abs(dw * dx * s)
        v, t = oracle.dot_q8_0_q8_1(w, xq)
        nb = K // 32
        assert abs(Fraction(v) - exact) <= Fraction(nb + 2) * Fraction(2.0 ** -52) * tabs
        assert abs(Fraction(t) - tabs) <= Fraction(nb + 2) * Fraction(2.0 ** -52) * tabs
        isums = oracle.block_isums(w, xq)
        ref = (w[:, 2:].view(np.int8).astype(np.int64) * xq[:, 4:].view(np.int8).astype(np.int64)).sum(1)
        assert np.array_equal(isums, ref)


def test_column_slice_equals_zero_padded_full_row():
    """[PR826, commit "whole-row-lane slice"]: a K-range of a weight row gives
    the same sums as the full product with the rest zero-padded, bit for bit."""
    g = np.random.default_rng(3)
    K = 512
    nb = K // 32
    w = W.q8_0_blocks(g, 4, K)
    xq = oracle.quantize_q8_1(g.standard_normal((1, K)).astype(np.float32))[0]
    for b0, b1 in [(0, nb), (0, 1), (3, 9), (nb - 1, nb), (5, 6), (2, 14)]:
        for r in range(4):
            sl, _ = oracle.dot_q8_0_q8_1(w[r, b0:b1], xq[b0:b1])
            pad = np.zeros_like(w[r])
            pad[b0:b1] = w[r, b0:b1]
            full, _ = oracle.dot_q8_0_q8_1(pad, xq)
            assert struct.pack("<d", sl) == struct.pack("<d", full)


def test_row_slice_of_matvec_is_bitwise_identical():
    g = np.random.default_rng(4)
    Wm = W.q8_0_blocks(g, 40, 256)
    xq = oracle.quantize_q8_1(g.standard_normal((1, 256)).astype(np.float32))[0]
    y, t = oracle.matvec_q8_0(Wm, xq)
    y2, t2 = oracle.matvec_q8_0(Wm[7:23], xq)
    assert np.array_equal(y[7:23].view(np.uint64), y2.view(np.uint64))
    for r in range(40):
        v, _ = oracle.dot_q8_0_q8_1(Wm[r], xq)
        assert v == y[r]


# ----------------------------------------------------------------------------- SwiGLU
def test_silu_closed_forms():
    assert oracle.silu(0.0) == 0.0
    # sigmoid(ln 3) = 3/4, so silu(ln 3) = 0.75 ln 3
    assert abs(oracle.silu(math.log(3.0)) - 0.75 * math.log(3.0)) < 1e-15
    # sigmoid(-ln 3) = 1/4
    assert abs(oracle.silu(-math.log(3.0)) + 0.25 * math.log(3.0)) < 1e-15
    assert abs(oracle.silu(40.0) - 40.0) < 1e-12          # -> g for large g
    assert 0 > oracle.silu(-40.0) > -1e-15                 # -> 0- for large negative g


def test_swiglu_clamp_special_cases():
    L = 10.0
    # clamp inactive inside [-L, L] (and for g below L)
    assert oracle.swiglu(3.0, -4.0, L) == oracle.swiglu(3.0, -4.0, 0.0)
    assert oracle.swiglu(-30.0, 2.0, L) == oracle.swiglu(-30.0, 2.0, 0.0)
    # g = 12 is clamped to 10; u = +-15 to +-10; g has no lower clamp
    assert oracle.swiglu(12.0, 1.0, L) == oracle.swiglu(10.0, 1.0, 0.0)
    assert oracle.swiglu(2.0, 15.0, L) == oracle.swiglu(2.0, 10.0, 0.0)
    assert oracle.swiglu(2.0, -15.0, L) == oracle.swiglu(2.0, -10.0, 0.0)
    assert oracle.swiglu(math.log(3.0), 15.0, L) == pytest.approx(0.75 * math.log(3.0) * 10.0, rel=1e-15)
    # unclamped: h = silu(g) * u
    assert oracle.swiglu(12.0, 15.0, 0.0) == pytest.approx(12.0 / (1.0 + math.exp(-12.0)) * 15.0, rel=1e-15)


# ----------------------------------------------------------------------------- router
def _rule_holds(scores, sel):
    """Every selected expert beats every other: higher score, or equal and lower index."""
    others = [f for f in range(len(scores)) if f not in sel]
    return all(scores[e] > scores[f] or (scores[e] == scores[f] and e < f) for e in sel for f in others)


@pytest.mark.parametrize("E,k", [(5, 1), (6, 2), (8, 3), (10, 4), (9, 9)])
def test_router_selection_brute_force_over_subsets(E, k):
    g = np.random.default_rng(E * 10 + k)
    logits = g.standard_normal((6, E)).astype(np.float32)
    logits[0] = 0.5  # all tied
    logits[1, :3] = logits[1, 3]  # partial ties
    bias = (g.standard_normal(E) * 0.3).astype(np.float32)
    for b in (None, bias):
        ids, w = oracle.route_topk(logits, b, k)
        scores = logits if b is None else (logits + b).astype(np.float32)
        for t in range(6):
            winners = [set(S) for S in itertools.combinations(range(E), k) if _rule_holds(scores[t], set(S))]
            assert len(winners) == 1 and winners[0] == set(ids[t].tolist())
            # slot order: by score, ties to the lower index
            for j in range(k - 1):
                a, c = ids[t, j], ids[t, j + 1]
                assert scores[t, a] > scores[t, c] or (scores[t, a] == scores[t, c] and a < c)
            # weights: softmax of the selected unbiased logits
            sel = logits[t, ids[t]].astype(np.float64)
            assert abs(w[t].sum() - 1.0) < 1e-15 * k * 4
            for j in range(k):
                assert w[t, j] / w[t, 0] == pytest.approx(math.exp(sel[j] - sel[0]), rel=1e-14)
    # all-tied row selects 0..k-1 in order
    ids, w = oracle.route_topk(np.full((1, E), 0.25, np.float32), None, k)
    assert ids[0].tolist() == list(range(k))
    assert np.allclose(w, 1.0 / k, rtol=1e-15)


def test_router_k1_weight_is_exactly_one():
    g = np.random.default_rng(5)
    logits = g.standard_normal((7, 16)).astype(np.float32)
    ids, w = oracle.route_topk(logits, None, 1)
    assert np.all(w == 1.0)
    assert np.array_equal(ids[:, 0], np.argmax(logits, axis=1))


def test_router_nan_scores_rank_below_every_number():
    # a NaN score counts as -infinity: never ahead of a number, ties to the
    # lower index among NaN and -infinity scores, and k distinct experts always
    nan, inf = float("nan"), float("inf")
    logits = np.array([[nan, 1.0, nan, 0.5],
                       [-inf, nan, 2.0, nan]], np.float32)
    ids, _ = oracle.route_topk(logits, None, 3)
    assert ids[0].tolist() == [1, 3, 0]
    assert ids[1].tolist() == [2, 0, 1]
    # a NaN bias on a finite logit gives a NaN score too
    ids, _ = oracle.route_topk(np.array([[3.0, 1.0, 2.0]], np.float32), np.array([nan, 0.0, 0.0], np.float32), 2)
    assert ids[0].tolist() == [2, 1]


def test_router_bias_changes_selection_not_weights():
    logits = np.array([[1.0, 0.9, 0.0, -1.0]], np.float32)
    bias = np.array([0.0, 0.0, 2.0, 0.0], np.float32)
    ids, w = oracle.route_topk(logits, bias, 2)
    assert ids[0].tolist() == [2, 0]
    e = np.exp(np.array([0.0, 1.0]) - 1.0)
    assert np.allclose(w[0], e / e.sum(), rtol=1e-15)


# ----------------------------------------------------------------------------- grouping
@pytest.mark.parametrize("T,k,E", [(1, 1, 1), (3, 2, 4), (7, 3, 5), (16, 4, 9), (40, 8, 128)])
def test_grouping_brute_force(T, k, E):
    g = np.random.default_rng(T * 1000 + E)
    ids = np.stack([g.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    ids[g.random(ids.shape) < 0.2] = -1  # masked routes
    counts, offsets, routes = oracle.moe_group(ids, E)
    flat = ids.reshape(-1)
    assert np.array_equal(counts, np.bincount(flat[flat >= 0], minlength=E))
    assert offsets[0] == 0 and np.array_equal(np.diff(offsets), counts)
    n = int(offsets[-1])
    assert n == int((flat >= 0).sum())
    want = sorted([r for r in range(T * k) if flat[r] >= 0], key=lambda r: (flat[r], r))
    assert routes[:n].tolist() == want
    assert np.all(routes[n:] == -1)
    for e in range(E):
        seg = routes[offsets[e]:offsets[e + 1]]
        assert np.all(flat[seg] == e) and np.all(np.diff(seg) > 0)


# ----------------------------------------------------------------------------- experts
def _dequant_q8_0(w):
    d = w[..., 0:2].copy().view(np.float16)[..., 0].astype(np.float64)
    q = w[..., 2:].view(np.int8).astype(np.float64)
    return (q * d[..., None]).reshape(w.shape[:-2] + (-1,))


def _dense_layer(L, ids, weights32, clamp):
    """The layer with dequantized operands and numpy float64 matmuls (a
    library primitive), independent of the oracle's block loop."""
    wl = L.wl
    T, k = ids.shape
    xq = oracle.quantize_q8_1(L.x)
    xd = oracle.dequant_q8_1(xq).astype(np.float64)
    Gd, Ud, Dd = _dequant_q8_0(L.wg), _dequant_q8_0(L.wu), _dequant_q8_0(L.wd)
    rows = T * k + (T if L.wsg is not None else 0)
    h = np.full((rows, wl.I), np.nan)
    for r in range(rows):
        if r < T * k:
            e = ids.reshape(-1)[r]
            if e < 0:
                continue
            gm, um, t = Gd[e], Ud[e], r // k
        else:
            gm, um, t = _dequant_q8_0(L.wsg), _dequant_q8_0(L.wsu), r - T * k
        gv, uv = gm @ xd[t], um @ xd[t]
        if clamp > 0:
            gv, uv = np.minimum(gv, clamp), np.clip(uv, -clamp, clamp)
        h[r] = gv / (1 + np.exp(-gv)) * uv
    return h, xq, Dd


@pytest.mark.parametrize("clamp", [0.0, 10.0])
def test_glu_pair_matches_dequantized_dense_matmul(clamp):
    wl = W.Workload("pin", T=3, H=256, I=96, E=4, k=2, shared=True, clamp=clamp, seed=11)
    L = W.host_layer(wl)
    ids = np.array([[1, 3], [3, -1], [0, 1]], np.int32)
    hd, xq, _ = _dense_layer(L, ids, None, clamp)
    h, ht = oracle.glu_pair(L.wg, L.wu, L.wsg, L.wsu, xq, ids, wl.E, wl.H, wl.I, clamp)
    ok = ~np.isnan(hd)
    assert np.array_equal(ok, ~np.isnan(h))
    assert np.all(np.abs(h[ok] - hd[ok]) <= 1e-12 * (1 + np.abs(hd[ok]) + ht[ok]))
    assert np.isnan(h[3]).all()  # masked route (t=1, j=1) left untouched


def test_down_combine_matches_dequantized_dense_matmul():
    wl = W.Workload("pin", T=3, H=128, I=64, E=4, k=2, shared=True, clamp=0.0, seed=12)
    L = W.host_layer(wl)
    g = np.random.default_rng(9)
    ids = np.array([[1, 3], [3, -1], [0, 1]], np.int32)
    weights = g.uniform(0.05, 0.9, (3, 2)).astype(np.float32)
    hq = oracle.quantize_q8_1(g.standard_normal((3 * 2 + 3, wl.I)).astype(np.float32))
    out, ot = oracle.down_combine(L.wd, L.wsd, hq, ids, weights, wl.E, wl.H, wl.I)
    hd = oracle.dequant_q8_1(hq).astype(np.float64)
    Dd = _dequant_q8_0(L.wd)
    Sd = _dequant_q8_0(L.wsd)
    for t in range(3):
        acc = np.float32(0)
        for j in range(2):
            e = ids[t, j]
            if e < 0:
                continue
            y = np.float32(Dd[e] @ hd[t * 2 + j])
            acc = np.float32(acc + np.float32(weights[t, j] * y))
        acc = np.float32(acc + np.float32(Sd @ hd[6 + t]))
        assert np.all(np.abs(out[t] - acc) <= 4 * np.spacing(np.abs(acc).astype(np.float32)) + 1e-12 * ot[t])


def test_combine_rounds_products_and_sums_separately():
    """[PR826, commit "fused routed combine ..."]: products and sums are each
    rounded to fp32 (no fused multiply-add).  Down rows with one non-zero code
    make y exact, so the expected result is the exact rational value of each
    step rounded to fp32, computed here with fractions."""
    H, I, E, k = 4, 32, 2, 2
    wd = np.zeros((E, H, 1, 34), np.uint8)
    for e in range(E):
        for n in range(H):
            wd[e, n, 0, 0:2] = np.array([np.float16(1.0 + 0.0009765625 * (3 * e + n))]).view(np.uint8)
            wd[e, n, 0, 2] = np.uint8(np.int8(101 - 7 * n - 13 * e))
    hq = np.zeros((2, 1, 36), np.uint8)
    hq[:, 0, 0:2] = np.array([np.float16(1.0)]).view(np.uint8)
    hq[:, 0, 4] = 1
    ids = np.array([[0, 1]], np.int32)
    wts = np.array([[0.3333333432674408, 0.6666666865348816]], np.float32)
    out, _ = oracle.down_combine(wd, None, hq, ids, wts, E, H, I)
    f32 = lambda fr: Fraction(float(np.float32(float(fr))))  # noqa: E731 (exact -> fp32, RNE)
    for n in range(H):
        ys = [Fraction(float(np.float16(1.0 + 0.0009765625 * (3 * e + n)))) * (101 - 7 * n - 13 * e) for e in range(E)]
        acc = Fraction(0)
        for j in range(k):
            acc = f32(acc + f32(Fraction(float(wts[0, j])) * ys[j]))
        assert Fraction(float(out[0, n])) == acc


def test_combine_masks_and_shared_expert():
    wl = W.Workload("pin", T=2, H=64, I=64, E=3, k=2, shared=True, clamp=0.0, seed=13)
    L = W.host_layer(wl)
    g = np.random.default_rng(2)
    hq = oracle.quantize_q8_1(g.standard_normal((2 * 2 + 2, wl.I)).astype(np.float32))
    w = np.ones((2, 2), np.float32)
    # all routes masked: out is the shared expert alone
    ids = np.full((2, 2), -1, np.int32)
    out, _ = oracle.down_combine(L.wd, L.wsd, hq, ids, w, wl.E, wl.H, wl.I)
    ys, _ = oracle.matvec_q8_0(L.wsd, hq[4])
    assert np.array_equal(out[0], ys.astype(np.float32))
    # one-hot weight reproduces one expert's product (+ shared)
    ids = np.array([[2, 0], [1, -1]], np.int32)
    w = np.array([[1.0, 0.0], [1.0, 0.0]], np.float32)
    out, _ = oracle.down_combine(L.wd, None, hq, ids, w, wl.E, wl.H, wl.I)
    y2, _ = oracle.matvec_q8_0(L.wd[2], hq[0])
    assert np.array_equal(out[0], y2.astype(np.float32))
    y1, _ = oracle.matvec_q8_0(L.wd[1], hq[2])
    assert np.array_equal(out[1], y1.astype(np.float32))


# ----------------------------------------------------------------------------- argmax
def test_argmax_exhaustive_against_numpy():
    g = np.random.default_rng(6)
    x = g.standard_normal((50, 777)).astype(np.float32)
    x[1, :] = 3.0                       # all equal -> 0
    x[2, 0] = 100.0                     # max at 0
    x[3, -1] = 100.0                    # max at V-1
    x[4, 10] = x[4, 500] = 50.0         # duplicated maximum -> first
    x[5, :] = -0.0
    x[5, 7] = 0.0                       # -0 == +0: tie -> index 0
    x[6] = np.round(x[6])               # many ties
    idx, val = oracle.argmax(x)
    assert np.array_equal(idx, np.argmax(x, axis=1))
    assert np.array_equal(val, x[np.arange(50), idx])
    assert idx[1] == 0 and idx[2] == 0 and idx[3] == 776 and idx[4] == 10 and idx[5] == 0


def test_argmax_pick_over_shards_equals_the_whole_row():
    # any split of the vocabulary into shards, each reporting its first
    # maximum with its global index, picks the whole row's first maximum
    g = np.random.default_rng(16)
    x = g.standard_normal((9, 1000)).astype(np.float32)
    x[1, 499] = x[1, 500] = 9.0    # a tie across the 2-way boundary -> 499
    x[2, 0] = x[2, 999] = 9.0      # first and last column tie -> 0
    x[3, :] = 1.0                  # all equal -> 0
    x[4, 250] = x[4, 750] = 9.0    # tie across non-adjacent shards -> 250
    full, fval = oracle.argmax(x)
    for cuts in ([0, 500, 1000], [0, 1, 999, 1000], [0, 250, 251, 750, 1000], [0, 1000]):
        vals, idxs = [], []
        for a, b in zip(cuts[:-1], cuts[1:]):
            i, v = oracle.argmax(x[:, a:b])
            vals.append(v)
            idxs.append(i + a)
        idx, val = oracle.argmax_pick(np.stack(vals), np.stack(idxs))
        assert np.array_equal(idx, full) and np.array_equal(val, fval)
    assert full[1] == 499 and full[2] == 0 and full[3] == 0 and full[4] == 250


# ----------------------------------------------------------------------------- the steps either side
def test_rmsnorm_closed_forms():
    one = np.ones(2, np.float32)
    # (3, 4): mean square 12.5, so xn = (3, 4) / sqrt(12.5)
    xn, _, _ = oracle.rmsnorm_router(np.array([[3.0, 4.0]], np.float32), one, 0.0, np.eye(2, dtype=np.float32))
    assert np.allclose(xn[0], np.array([3.0, 4.0]) / math.sqrt(12.5), rtol=1e-15)
    # a constant row c: xn = c / sqrt(c^2 + eps); gamma scales each element
    H, c, eps = 64, 0.5, 1e-3
    gamma = np.linspace(0.5, 2.0, H).astype(np.float32)
    xn, _, _ = oracle.rmsnorm_router(np.full((1, H), c, np.float32), gamma, eps, np.zeros((1, H), np.float32))
    assert np.allclose(xn[0], c / math.sqrt(c * c + eps) * gamma.astype(np.float64), rtol=1e-14)
    # zero input stays zero; scaling x by 2 (eps = 0) leaves xn unchanged exactly
    xn, lg, _ = oracle.rmsnorm_router(np.zeros((1, H), np.float32), gamma, 1e-6, np.ones((3, H), np.float32))
    assert np.all(xn == 0.0) and np.all(lg == 0.0)
    g = np.random.default_rng(17)
    x = g.standard_normal((3, H)).astype(np.float32)
    a, _, _ = oracle.rmsnorm_router(x, gamma, 0.0, np.zeros((1, H), np.float32))
    b, _, _ = oracle.rmsnorm_router(2.0 * x, gamma, 0.0, np.zeros((1, H), np.float32))
    assert np.array_equal(a, b)
    # with gamma = 1 and eps = 0 the normed row has mean square 1
    a, _, _ = oracle.rmsnorm_router(x, np.ones(H, np.float32), 0.0, np.zeros((1, H), np.float32))
    assert np.allclose((a ** 2).mean(axis=1), 1.0, rtol=1e-14)


def test_router_logits_against_numpy_and_one_hot_rows():
    g = np.random.default_rng(18)
    T, E, H = 3, 12, 256
    x = g.standard_normal((T, H)).astype(np.float32)
    gamma = g.uniform(0.5, 1.5, H).astype(np.float32)
    w = (g.standard_normal((E, H)) * 0.05).astype(np.float32)
    w[0] = 0.0
    w[0, 7] = 1.0                  # one-hot row: logit = xn[7]
    xn, lg, terms = oracle.rmsnorm_router(x, gamma, 1e-6, w)
    ref = xn @ w.astype(np.float64).T
    assert np.allclose(lg, ref, rtol=1e-12, atol=1e-12)
    assert np.array_equal(lg[:, 0], xn[:, 7])
    assert np.allclose(terms, np.abs(xn) @ np.abs(w.astype(np.float64)).T, rtol=1e-12)


def test_ep_split_sums_to_the_single_device_step():
    # two expert-parallel ranks (routed experts [0, E/2) with the shared
    # expert, and [E/2, E)): each route is computed by one rank, so the sum of
    # the partials is the single-device output up to the order of the sums
    wl = W.Workload("ep_pin", T=3, H=256, I=256, E=8, k=3, shared=True, clamp=0.0, seed=41, bias_std=0.1)
    L = W.host_layer(wl)
    full = oracle.moe_layer(L.wg, L.wu, L.wd, L.wsg, L.wsu, L.wsd, L.x, L.logits, L.bias, wl.k, wl.clamp)
    ep = oracle.ep_layer(L.wg, L.wu, L.wd, L.wsg, L.wsu, L.wsd, L.x, L.logits, L.bias, wl.k, wl.clamp, [0, 4, 8])
    assert np.array_equal(ep["ids"], full["ids"])
    assert np.all(np.abs(ep["out"] - full["out"]) <= oracle.tol(full["out_terms"]))
    assert np.allclose(ep["out_terms"], full["out_terms"], rtol=1e-12)
    # one rank owning everything is the single-device step, bit for bit
    one = oracle.ep_layer(L.wg, L.wu, L.wd, L.wsg, L.wsu, L.wsd, L.x, L.logits, L.bias, wl.k, wl.clamp, [0, 8])
    assert np.array_equal(one["out"], full["out"])
    # a rank that owns none of the selected experts contributes zero (rank 1 here has no shared expert)
    none = oracle.ep_layer(L.wg, L.wu, L.wd, L.wsg, L.wsu, L.wsd, L.x, L.logits, L.bias, wl.k, wl.clamp, [0, 8, 8])
    assert np.all(none["partials"][1] == 0.0) and np.array_equal(none["out"], full["out"])


# ----------------------------------------------------------------------------- Q4_K weights
def _pack_q4k(d, dmin, sc, m, q):
    """One Q4_K super-block from its parts, written from the layout's
    description in the packing direction (the oracle unpacks)."""
    s = [0] * 12
    for j in range(4):
        s[j] = (sc[j] & 63) | ((sc[j + 4] >> 4) << 6)
        s[j + 4] = (m[j] & 63) | ((m[j + 4] >> 4) << 6)
    for j in range(4, 8):
        s[j + 4] = (sc[j] & 15) | ((m[j] & 15) << 4)
    qs = [0] * 128
    for j in range(8):
        for i in range(32):
            qs[32 * (j // 2) + i] |= (q[j][i] & 15) << (4 * (j % 2))
    return bytes(struct.pack("<e", d) + struct.pack("<e", dmin) + bytes(s) + bytes(qs))


def _q8_1_block(d8, s8, codes):
    return struct.pack("<e", d8) + struct.pack("<e", s8) + bytes((c & 255) for c in codes)


def test_q4k_scales_and_mins_unpack_what_was_packed():
    g = np.random.default_rng(30)
    for _ in range(50):
        sc = g.integers(0, 64, 8).tolist()
        m = g.integers(0, 64, 8).tolist()
        blk = _pack_q4k(0.5, 0.25, sc, m, [[0] * 32] * 8)
        scales = np.frombuffer(blk[4:16], np.uint8)
        assert [oracle.q4_k_scale_min(scales, j) for j in range(8)] == list(zip(sc, m))


def test_q4k_dot_equals_the_exact_dequantized_dot():
    # d, dmin, d8 powers of two and small code sums: the stored s8 = d8 sum(q8)
    # is exact in fp16, so the dot is the exact rational dot of the values
    g = np.random.default_rng(31)
    for trial in range(20):
        d, dmin = 2.0 ** -int(g.integers(6, 10)), 2.0 ** -int(g.integers(6, 10))
        sc = g.integers(0, 64, 8).tolist()
        m = g.integers(0, 64, 8).tolist()
        q = g.integers(0, 16, (8, 32)).tolist()
        w = np.frombuffer(_pack_q4k(d, dmin, sc, m, q), np.uint8).reshape(1, 144)
        xb, exact = [], Fraction(0)
        for j in range(8):
            d8 = 2.0 ** -int(g.integers(5, 9))
            codes = g.integers(-20, 21, 32).tolist()
            s8 = d8 * sum(codes)
            xb.append(_q8_1_block(d8, s8, codes))
            for i in range(32):
                val = Fraction(d) * sc[j] * q[j][i] - Fraction(dmin) * m[j]
                exact += val * Fraction(d8) * codes[i]
        x = np.frombuffer(b"".join(xb), np.uint8).reshape(8, 36)
        v, terms = oracle.dot_q4_k_q8_1(w, x)
        assert abs(Fraction(v) - exact) <= Fraction(abs(terms)) * Fraction(1, 2 ** 50)
    # all codes zero: the value is -dmin m_j everywhere, the dot -sum_j dmin m_j s8_j
    w = np.frombuffer(_pack_q4k(0.5, 0.125, [1] * 8, list(range(8)), [[0] * 32] * 8), np.uint8).reshape(1, 144)
    x = np.frombuffer(b"".join(_q8_1_block(0.25, 0.25 * 3, [3] + [0] * 31) for _ in range(8)), np.uint8)
    v, _ = oracle.dot_q4_k_q8_1(w, x.reshape(8, 36))
    assert v == -sum(0.125 * mj * 0.75 for mj in range(8))


def test_q4k_row_slices_add_up():
    g = W.rng(32, 0)
    w = W.q4_k_blocks(g, 1, 1024)[0]
    x = oracle.quantize_q8_1(g.standard_normal(1024).astype(np.float32))
    full, t_full = oracle.dot_q4_k_q8_1(w, x)
    parts = [oracle.dot_q4_k_q8_1(w[s:s + 1], x[8 * s:8 * s + 8]) for s in range(4)]
    assert abs(full - sum(p[0] for p in parts)) <= 1e-13 * t_full
    assert abs(t_full - sum(p[1] for p in parts)) <= 1e-13 * t_full


def test_q4k_layer_routes_and_masks_like_the_q8_0_layer():
    wl = W.Workload("q4k_pin", T=2, H=256, I=256, E=4, k=2, shared=True, clamp=0.0, seed=33, bias_std=0.0)
    L = W.host_layer_q4k(wl)
    ref = oracle.moe_layer_q4k(L.wg, L.wu, L.wd, L.wsg, L.wsu, L.wsd, L.x, L.logits, L.bias, wl.k, wl.clamp)
    ids, _ = oracle.route_topk(L.logits, L.bias, wl.k)
    assert np.array_equal(ref["ids"], ids)
    # one masked route: its h row stays unwritten and the combine skips it
    m = ids.copy()
    m[0, 1] = -1
    xq = oracle.quantize_q8_1(L.x)
    h, _ = oracle.glu_q4k(L.wg, L.wu, L.wsg, L.wsu, xq, m, wl.E, wl.H, wl.I, 0.0)
    assert np.isnan(h[1]).all() and not np.isnan(h[0]).any()
    # h is silu(g) u of the two row dots
    g0, _ = oracle.dot_q4_k_q8_1(L.wg[m[0, 0], 5], xq[0])
    u0, _ = oracle.dot_q4_k_q8_1(L.wu[m[0, 0], 5], xq[0])
    assert h[0, 5] == oracle.swiglu(g0, u0)


def test_q4k_down_combine_matches_dequantized_dense_matmul():
    """The Q4_K down product + combine against numpy float64 matmuls of the
    values the packer was given (d sc_j q - dmin m_j per sub-block j; the dot
    reads the mins against the q8_1 block's stored sum s8), combined in slot
    order with each product and sum rounded to fp32, shared expert last."""
    g = np.random.default_rng(34)
    E, H, I, T, k = 3, 48, 512, 2, 2
    nsb = I // 256

    def expert_rows(nrows):
        blocks, vals, mins = [], np.zeros((nrows, I)), np.zeros((nrows, I // 32))
        for n in range(nrows):
            row = []
            for sb in range(nsb):
                d = float(np.float16(g.uniform(1e-4, 2e-3)))
                dmin = float(np.float16(g.uniform(1e-4, 2e-3)))
                sc = g.integers(0, 64, 8).tolist()
                m = g.integers(0, 64, 8).tolist()
                q = g.integers(0, 16, (8, 32)).tolist()
                row.append(_pack_q4k(d, dmin, sc, m, q))
                for j in range(8):
                    c0 = sb * 256 + 32 * j
                    vals[n, c0:c0 + 32] = d * sc[j] * np.array(q[j], np.float64)
                    mins[n, sb * 8 + j] = dmin * m[j]
            blocks.append(np.frombuffer(b"".join(row), np.uint8).reshape(nsb, 144))
        return np.stack(blocks), vals, mins

    wd, vd, md = zip(*[expert_rows(H) for _ in range(E)])
    wsd, vs, ms = expert_rows(H)
    wd = np.stack(wd)
    ids = np.array([[2, 0], [1, -1]], np.int32)
    weights = g.uniform(0.05, 0.9, (T, k)).astype(np.float32)
    hq = oracle.quantize_q8_1(g.standard_normal((T * k + T, I)).astype(np.float32))
    out, ot = oracle.down_combine_q4k(wd, wsd, hq, ids, weights, E, H, I)
    hd = oracle.dequant_q8_1(hq).astype(np.float64)
    s8 = oracle.fp16_decode(hq[..., 2:4].copy().view(np.uint16)[..., 0]).astype(np.float64)  # [rows, I/32]

    def y_of(vals, mins, r):
        return vals @ hd[r] - mins @ s8[r]

    for t in range(T):
        acc = np.float32(0)
        for j in range(k):
            e = ids[t, j]
            if e < 0:
                continue
            y = np.float32(y_of(vd[e], md[e], t * k + j))
            acc = np.float32(acc + np.float32(weights[t, j] * y))
        acc = np.float32(acc + np.float32(y_of(vs, ms, T * k + t)))
        assert np.all(np.abs(out[t] - acc) <= 4 * np.spacing(np.abs(acc).astype(np.float32)) + 1e-12 * ot[t])
    # a masked route and a missing shared expert: the combine of the remaining slots
    out2, _ = oracle.down_combine_q4k(wd, None, hq[:T * k], np.array([[-1, -1], [1, -1]], np.int32), weights,
                                      E, H, I)
    assert np.all(out2[0] == 0.0)
    y = np.float32(y_of(vd[1], md[1], 2))
    assert np.all(np.abs(out2[1] - np.float32(weights[1, 0] * y)) <= 4 * np.spacing(np.abs(y)) + 1e-30)


def _flip_setup():
    """h of the decode layer through the oracle, and its float bound."""
    wl = W.WORKLOADS["decode_layer"]
    L = W.host_layer(wl)
    ids, _ = oracle.route_topk(L.logits, L.bias, wl.k)
    xq = oracle.quantize_q8_1(L.x)
    h, ht = oracle.glu_pair(L.wg, L.wu, L.wsg, L.wsu, xq, ids, wl.E, wl.H, wl.I, wl.clamp)
    return h.astype(np.float32), oracle.tol(ht)


def test_hq_flip_allowance_covers_every_change_within_the_float_bound():
    """Perturb h by anything the float rule admits and re-quantize: every
    dequantized q8_1 value that changes does so where the allowance is
    positive, and by no more than it."""
    h32, htol = _flip_setup()
    allow = oracle.hq_flip_allowance(h32, htol)
    ref = oracle.dequant_q8_1(oracle.quantize_q8_1(h32)).astype(np.float64)
    g = np.random.default_rng(40)
    changed = 0
    for trial in range(60):
        if trial < 20:
            delta = g.uniform(-1.0, 1.0, h32.shape) * htol
        elif trial < 40:
            delta = g.choice([-1.0, 1.0], h32.shape) * htol  # the bound's corners
        else:
            delta = g.choice([-1.0, 0.0, 1.0], h32.shape) * htol * 0.999
        hp = (h32.astype(np.float64) + delta).astype(np.float32)
        got = oracle.dequant_q8_1(oracle.quantize_q8_1(hp)).astype(np.float64)
        diff = np.abs(got - ref)
        moved = diff > 0
        changed += int(moved.sum())
        assert np.all(allow[moved] > 0), "a q8_1 value changed where the allowance says it is stable"
        assert np.all(diff <= allow + 1e-30), "a q8_1 value moved by more than its allowance"
    assert changed > 0  # the perturbations do reach unstable elements


def test_hq_flip_allowance_is_sharp():
    """Sharpness.  With a perturbation of a few fp32 ulps of h (the size of a
    reordered fp32 sum) the allowance marks few elements at the decode shape;
    under the float bound itself (1e-4 of the terms, large against |h| where
    the gate and up sums cancel) d may cross an fp16 midpoint in nearly every
    block, and the allowance says so.  Hand-made blocks: an element on a
    rounding midpoint is marked, the block maximum and integers are not, and a
    block of exact integer codes far from every midpoint stays all zero."""
    h32, htol = _flip_setup()
    ulps = np.abs(h32).astype(np.float64) * 2.0 ** -23 * 16
    frac_ulps = float((oracle.hq_flip_allowance(h32, ulps) > 0).mean())
    assert frac_ulps < 0.01, frac_ulps
    frac_bound = float((oracle.hq_flip_allowance(h32, htol) > 0).mean())
    assert frac_bound > 0.5, frac_bound
    # zero perturbation: nothing can move
    assert np.all(oracle.hq_flip_allowance(h32, np.zeros_like(ulps)) == 0.0)
    # hand-made block: amax 127 gives d = 1 (exact); values k + 0.5 are on a
    # rounding midpoint, integers are far from one
    blk = np.zeros((1, 32), np.float32)
    blk[0, 0] = 127.0
    blk[0, 1] = 10.5
    blk[0, 2] = 11.0
    t = np.full((1, 32), 1e-4)
    a = oracle.hq_flip_allowance(blk, t)
    assert a[0, 1] > 0 and a[0, 2] == 0.0 and a[0, 0] == 0.0
    far = ((np.arange(32) - 16) * 4).astype(np.float32).reshape(1, 32)  # integers; amax 127 gives d = 1
    far[0, 0] = -127.0
    a2 = oracle.hq_flip_allowance(far, np.full((1, 32), 1e-9))
    assert np.all(a2 == 0.0)
    # the same block scaled by 127/16: x/d = 7.9375 (i - 16) lands on a
    # midpoint exactly for i - 16 = +-8 (63.5), and only there
    mid = far * np.float32(1.0)
    mid[0, :] = ((np.arange(32) - 16) * np.float32(127.0 / 16.0)).astype(np.float32)
    a3 = oracle.hq_flip_allowance(mid, np.full((1, 32), 1e-9))
    assert set(np.nonzero(a3[0])[0].tolist()) == {8, 24}
