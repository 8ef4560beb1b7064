"""GPU parity: every C-ABI entry point against the CPU oracle on the same
seeded inputs (GB300).  Integer outputs bit for bit; float outputs within
1e-4 * terms + 1e-6; q8_1 blocks of GPU-computed values identical wherever
the quantization is stable (see gpu_util)."""
import os

import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_close, assert_hq_is_rule_of_h, assert_hq_valid, chain_allowance, dev, host
from quantized_moe_decode_luce_gb300 import binding as B
from quantized_moe_decode_luce_gb300 import build as BLD
from quantized_moe_decode_luce_gb300 import workloads as W
from quantized_moe_decode_luce_gb300.layer import Argmax, MoEStep

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    BLD.build()
    B.lib()
    yield


@pytest.fixture(autouse=True)
def _no_device_faults(request):
    yield
    if "allow_fault" not in request.keywords:
        assert B.luce_get_fault() == 0


def _distinct_ids(g, T, k, E, mask_frac=0.0):
    ids = np.stack([g.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    if mask_frac > 0:
        ids[g.random(ids.shape) < mask_frac] = -1
    return ids


# ----------------------------------------------------------------------------- q8_1
@pytest.mark.parametrize("T,K,kind", [(1, 512, "normal"), (5, 4096, "normal"), (37, 96, "wide"),
                                      (3, 2048, "ties"), (2, 64, "zeros"), (512, 4096, "normal"),
                                      (1, 32, "single")])
def test_quantize_q8_1_bit_exact(T, K, kind):
    g = W.rng(100, T * K)
    x = g.standard_normal((T, K)).astype(np.float32)
    if kind == "wide":
        x *= (10.0 ** g.integers(-7, 5, (T, K // 32, 1))).repeat(32, axis=2).reshape(T, K).astype(np.float32)
    elif kind == "ties":
        x = (np.round(x * 8) / 2).astype(np.float32)   # many exact .5 quotients
        x[:, ::32] = 63.5
    elif kind == "zeros":
        x[:, 32:64] = 0.0
        x[0, :32] = -0.0
    elif kind == "single":
        x[:] = 0
        x[0, 7] = -254.0
    ref = oracle.quantize_q8_1(x)
    n = ref.size
    buf = torch.full((n + 64,), 0xA5, dtype=torch.uint8, device="cuda")
    xq = buf[:n].view(T, K // 32, 36)
    B.luce_quantize_q8_1(dev(x), xq)
    torch.cuda.synchronize()
    assert np.array_equal(host(xq), ref)
    assert torch.all(buf[n:] == 0xA5)  # nothing written past the output


# ----------------------------------------------------------------------------- router
@pytest.mark.parametrize("T,E,k,bias,kind", [(1, 64, 6, True, "normal"), (5, 128, 8, False, "shared_col"),
                                             (512, 128, 8, False, "normal"), (3, 1024, 64, True, "normal"),
                                             (4, 1, 1, False, "normal"), (6, 37, 5, True, "normal"),
                                             (2, 16, 4, False, "ties"), (9, 256, 33, True, "normal")])
def test_route_topk(T, E, k, bias, kind):
    g = W.rng(200, T * E + k)
    logits = g.standard_normal((T, E)).astype(np.float32)
    if kind == "shared_col":
        logits = (g.standard_normal(E) + 0.75 * logits).astype(np.float32)
    if kind == "ties":
        logits[0] = 0.5
        logits[1, ::2] = 0.25
    b = (g.standard_normal(E) * 0.1).astype(np.float32) if bias else None
    ids_ref, w_ref = oracle.route_topk(logits, b, k)
    ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    B.luce_route_topk(dev(logits), dev(b) if b is not None else None, k, ids, w)
    torch.cuda.synchronize()
    assert np.array_equal(host(ids), ids_ref)
    err = assert_close(host(w), w_ref, np.ones_like(w_ref), "route weights")
    assert np.abs(host(w) - w_ref).max() < 2e-6
    assert err < 0.1


# ----------------------------------------------------------------------------- grouping
@pytest.mark.parametrize("T,k,E,mask", [(1, 6, 64, 0.0), (5, 8, 128, 0.2), (512, 8, 128, 0.1),
                                        (100, 64, 1024, 0.5), (7, 3, 5, 0.0), (2048, 4, 4, 0.0),
                                        (3, 2, 2, 1.0), (1, 1, 1, 0.0)])
def test_moe_group_bit_exact(T, k, E, mask):
    g = W.rng(300, T * k + E)
    ids = _distinct_ids(g, T, k, E, mask)
    c_ref, o_ref, r_ref = oracle.moe_group(ids, E)
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    routes = torch.empty(T * k, dtype=torch.int32, device="cuda")
    B.luce_moe_group(dev(ids), E, counts, offsets, routes)
    torch.cuda.synchronize()
    assert np.array_equal(host(counts), c_ref)
    assert np.array_equal(host(offsets), o_ref)
    assert np.array_equal(host(routes), r_ref)


def test_moe_group_empty():
    counts = torch.full((8,), 7, dtype=torch.int32, device="cuda")
    offsets = torch.full((9,), 7, dtype=torch.int32, device="cuda")
    ids = torch.empty((0, 2), dtype=torch.int32, device="cuda")
    routes = torch.empty(0, dtype=torch.int32, device="cuda")
    B.lib().luce_moe_group(None, 0, 2, 8, counts.data_ptr(), offsets.data_ptr(), None, None)
    torch.cuda.synchronize()
    assert host(counts).tolist() == [0] * 8 and host(offsets).tolist() == [0] * 9
    del ids, routes


@pytest.mark.allow_fault
def test_moe_group_out_of_range_id_is_skipped_and_flagged():
    assert B.luce_get_fault() == 0
    ids = np.array([[0, 9], [3, 1]], np.int32)  # 9 >= E
    E = 4
    c_ref, o_ref, r_ref = oracle.moe_group(ids, E)
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    routes = torch.empty(4, dtype=torch.int32, device="cuda")
    B.luce_moe_group(dev(ids), E, counts, offsets, routes)
    assert B.luce_get_fault() == B.LUCE_FAULT_BAD_ID
    assert np.array_equal(host(counts), c_ref) and np.array_equal(host(routes), r_ref)
    assert B.luce_get_fault() == 0  # reading clears


# ----------------------------------------------------------------------------- gate/up pair
GLU_CASES = [
    # name, T, k, E, H, I, shared, clamp, mask
    ("tiny", 1, 1, 1, 512, 256, False, 0.0, 0.0),
    ("multi_col", 9, 4, 16, 512, 512, True, 10.0, 0.0),
    ("wide_split", 40, 2, 4, 256, 256, True, 0.0, 0.0),
    ("masked", 4, 3, 8, 256, 256, True, 10.0, 0.3),
    ("shared_only", 3, 2, 8, 256, 512, True, 0.0, 1.0),
    ("decode_shape", 1, 6, 64, 2048, 1024, True, 0.0, 0.0),
    ("verify_shape_small_E", 5, 8, 12, 4096, 512, True, 10.0, 0.0),
    ("h1024_many_groups", 3, 4, 40, 1024, 2048, False, 0.0, 0.1),
    ("x_through_l1", 40, 1, 2, 4096, 256, True, 0.0, 0.0),
]


def _glu_inputs(name, T, k, E, H, I, shared, clamp, mask):
    wl = W.Workload(name, T=T, H=H, I=I, E=E, k=k, shared=shared, clamp=clamp, seed=400 + len(name))
    L = W.host_layer(wl)
    ids = _distinct_ids(W.rng(wl.seed, 9), T, k, E, mask)
    if name == "masked":
        ids[1, :] = -1
    return wl, L, ids


@pytest.mark.parametrize("case", GLU_CASES, ids=[c[0] for c in GLU_CASES])
def test_glu_pair(case):
    name, T, k, E, H, I, shared, clamp, mask = case
    wl, L, ids = _glu_inputs(*case)
    xq = oracle.quantize_q8_1(L.x)
    _, offsets, routes = oracle.moe_group(ids, E)
    h_ref, h_terms = oracle.glu_pair(L.wg, L.wu, L.wsg, L.wsu, xq, ids, E, H, I, clamp)
    rows = T * k + (T if shared else 0)
    h = torch.full((rows, I), float("nan"), dtype=torch.float32, device="cuda")
    hq = torch.zeros((rows, I // 32, 36), dtype=torch.uint8, device="cuda")
    B.luce_moe_glu_pair(dev(L.wg), dev(L.wu), dev(L.wsg) if shared else None, dev(L.wsu) if shared else None,
                        dev(xq), dev(offsets), dev(routes), T, k, E, H, I, clamp, h, hq)
    torch.cuda.synchronize()
    hg = host(h)
    valid = ~np.isnan(h_ref[:, 0])
    assert np.isnan(hg[~valid]).all(), "rows of masked routes must not be written"
    assert_close(hg[valid], h_ref[valid], h_terms[valid], f"h ({name})")
    h32 = h_ref[valid].astype(np.float32)
    allow = oracle.hq_flip_allowance(h32, oracle.tol(h_terms[valid]))
    flips = assert_hq_valid(host(hq)[valid], oracle.quantize_q8_1(h32), allow, f"hq ({name})", h_gpu=hg[valid])
    assert flips <= max(2, h32.size // 1000)
    # hq is exactly the q8_1 rule applied to the h the kernel stored
    hq2 = torch.empty_like(hq)
    B.luce_quantize_q8_1(h.nan_to_num(0.0), hq2)
    assert torch.equal(hq2[torch.from_numpy(valid).cuda()], hq[torch.from_numpy(valid).cuda()])


# ----------------------------------------------------------------------------- down + combine
DOWN_CASES = [
    ("tiny", 1, 1, 1, 512, 256, False, 0.0),
    ("decode_shape", 1, 6, 64, 2048, 1024, True, 0.0),
    ("verify_like", 5, 8, 32, 1024, 512, True, 0.1),
    ("wide_tiles", 130, 3, 6, 256, 256, True, 0.1),
    ("all_masked", 3, 2, 4, 256, 256, True, 1.0),
    ("no_shared_masked", 4, 4, 8, 512, 256, False, 0.4),
    # large I: 69.6 KB stages, a ring of two, seven stages through it
    ("large_i_two_stage_ring", 1, 6, 8, 256, 8192, True, 0.0),
    ("large_i_tokens", 9, 4, 8, 256, 4096, True, 0.1),
]


@pytest.mark.parametrize("case", DOWN_CASES, ids=[c[0] for c in DOWN_CASES])
def test_down_combine(case):
    name, T, k, E, H, I, shared, mask = case
    wl = W.Workload(name, T=T, H=H, I=I, E=E, k=k, shared=shared, clamp=0.0, seed=500 + len(name))
    L = W.host_layer(wl)
    g = W.rng(wl.seed, 7)
    ids = _distinct_ids(g, T, k, E, mask)
    w = g.uniform(0.01, 1.0, (T, k)).astype(np.float32)
    w /= w.sum(axis=1, keepdims=True)
    w = w.astype(np.float32)
    rows = T * k + (T if shared else 0)
    hq = oracle.quantize_q8_1((g.standard_normal((rows, I)) * 300).astype(np.float32))
    _, offsets, routes = oracle.moe_group(ids, E)
    out_ref, out_terms = oracle.down_combine(L.wd, L.wsd, hq, ids, w, E, H, I)
    buf = torch.full((T * H + 16,), 12345.0, dtype=torch.float32, device="cuda")
    out = buf[:T * H].view(T, H)
    B.luce_moe_down_combine(dev(L.wd), dev(L.wsd) if shared else None, dev(hq), dev(ids), dev(w), dev(offsets),
                            dev(routes), T, k, E, H, I, out)
    torch.cuda.synchronize()
    assert_close(host(out), out_ref, out_terms, f"out ({name})")
    assert torch.all(buf[T * H:] == 12345.0)


# ----------------------------------------------------------------------------- whole step
def _run_chain(wl, L, layer=None, path="layer"):
    step = MoEStep(wl.T, wl.H, wl.I, wl.E, wl.k, wl.shared, wl.clamp)
    step.path = path
    if layer is None:
        layer = W.DeviceLayer(dev(L.wg), dev(L.wu), dev(L.wd), dev(L.wsg) if wl.shared else None,
                              dev(L.wsu) if wl.shared else None, dev(L.wsd) if wl.shared else None)
    out = step.run(layer, dev(L.x), dev(L.logits), dev(L.bias) if L.bias is not None else None)
    torch.cuda.synchronize()
    assert step.path == path  # the one-launch path did not decline the shape
    return step, out


def _check_chain(wl, L, step):
    ref = oracle.moe_layer(L.wg, L.wu, L.wd, L.wsg, L.wsu, L.wsd, L.x, L.logits, L.bias, wl.k, wl.clamp)
    assert np.array_equal(host(step.ids), ref["ids"])
    assert np.array_equal(host(step.xq), ref["xq"])
    valid = ~np.isnan(ref["h"][:, 0])
    assert_close(host(step.h)[valid], ref["h"][valid], ref["h_terms"][valid], "h")
    flips = assert_hq_valid(host(step.hq)[valid], ref["hq"][valid], ref["h_allow"][valid], "hq",
                            h_gpu=host(step.h)[valid])
    allow = chain_allowance(L.wd, L.wsd, ref["ids"], ref["weights"], ref["h_allow"])
    gout = host(step.out)
    bound = oracle.tol(ref["out_terms"]) + allow
    assert np.all(np.abs(gout - ref["out"]) <= bound), "out outside tolerance"
    return flips


@pytest.mark.parametrize("path", ["layer", "split"])
@pytest.mark.parametrize("name", ["tiny", "decode_layer"])
def test_layer_chain_workloads(name, path):
    wl = W.WORKLOADS[name]
    L = W.host_layer(wl)
    step, _ = _run_chain(wl, L, path=path)
    _check_chain(wl, L, step)


@pytest.mark.parametrize("path", ["layer", "split"])
def test_layer_chain_verify_like_small(path):
    wl = W.Workload("verify_small", T=5, H=1024, I=512, E=32, k=8, shared=True, clamp=10.0, seed=21,
                    logits="shared_col")
    L = W.host_layer(wl)
    step, _ = _run_chain(wl, L, path=path)
    _check_chain(wl, L, step)


@pytest.mark.parametrize("path", ["layer", "split"])
def test_layer_is_deterministic(path):
    wl = W.WORKLOADS["decode_layer"]
    L = W.host_layer(wl)
    step, out1 = _run_chain(wl, L, path=path)
    a = (out1.clone(), step.h.clone(), step.hq.clone())
    layer = W.DeviceLayer(dev(L.wg), dev(L.wu), dev(L.wd), dev(L.wsg), dev(L.wsu), dev(L.wsd))
    for _ in range(3):
        step.run(layer, dev(L.x), dev(L.logits), dev(L.bias))
        torch.cuda.synchronize()
        assert torch.equal(step.out, a[0]) and torch.equal(step.h, a[1]) and torch.equal(step.hq, a[2])


def _compact(wl, dl, used):
    """Host copies of the experts in `used` (device -> host), in that order."""
    idx = torch.tensor(used, dtype=torch.long, device=dl.wg.device)
    return (host(dl.wg.index_select(0, idx)), host(dl.wu.index_select(0, idx)),
            host(dl.wd.index_select(0, idx)))


@pytest.mark.parametrize("path", ["layer", "split"])
def test_verify_layer_full_size(path):
    wl = W.WORKLOADS["verify_layer"]
    dl = W.device_layer(wl, wl.seed, "cuda")
    gx = W.rng(wl.seed, 2)
    x = W.activations(gx, wl.T, wl.H)
    logits, bias = W.router_logits(W.rng(wl.seed, 3), wl)
    step = MoEStep(wl.T, wl.H, wl.I, wl.E, wl.k, wl.shared, wl.clamp)
    step.path = path
    step.run(dl, dev(x), dev(logits), None)
    torch.cuda.synchronize()
    assert step.path == path
    ids_ref, w_ref = oracle.route_topk(logits, bias, wl.k)
    assert np.array_equal(host(step.ids), ids_ref)
    c_ref, o_ref, r_ref = oracle.moe_group(ids_ref, wl.E)
    assert np.array_equal(host(step.offsets), o_ref) and np.array_equal(host(step.routes), r_ref)
    used = sorted(set(ids_ref.reshape(-1).tolist()))
    remap = {e: i for i, e in enumerate(used)}
    cids = np.vectorize(remap.get)(ids_ref).astype(np.int32)
    wg, wu, wd = _compact(wl, dl, used)
    wsg, wsu, wsd = host(dl.wsg), host(dl.wsu), host(dl.wsd)
    ref = oracle.moe_layer(wg, wu, wd, wsg, wsu, wsd, x, logits, None, wl.k, wl.clamp) \
        if False else None
    # the oracle step on the compacted experts with the router's ids
    xq = oracle.quantize_q8_1(x)
    assert np.array_equal(host(step.xq), xq)
    h_ref, h_terms = oracle.glu_pair(wg, wu, wsg, wsu, xq, cids, len(used), wl.H, wl.I, wl.clamp)
    assert_close(host(step.h), h_ref, h_terms, "h (verify)")
    h32 = h_ref.astype(np.float32)
    h_allow = oracle.hq_flip_allowance(h32, oracle.tol(h_terms))
    hq_ref = oracle.quantize_q8_1(h32)
    assert_hq_valid(host(step.hq), hq_ref, h_allow, "hq (verify)", h_gpu=host(step.h))
    out_ref, out_terms = oracle.down_combine(wd, wsd, hq_ref, cids, w_ref.astype(np.float32), len(used),
                                             wl.H, wl.I)
    allow = chain_allowance(wd, wsd, cids, w_ref, h_allow)
    assert np.all(np.abs(host(step.out) - out_ref) <= oracle.tol(out_terms) + allow)
    assert 8 <= len(used) <= 40
    del ref


def test_prefill_layer_full_size_every_token():
    """The 512-token prefill layer against the oracle on every token: the
    oracle's steps run on host threads over chunks of tokens (its C calls
    release the interpreter lock), on host copies of all the experts."""
    from concurrent.futures import ThreadPoolExecutor
    wl = W.WORKLOADS["prefill_layer"]
    T, k, E, H, I = wl.T, wl.k, wl.E, wl.H, wl.I
    dl = W.device_layer(wl, wl.seed, "cuda")
    x = W.activations(W.rng(wl.seed, 2), T, H)
    logits, bias = W.router_logits(W.rng(wl.seed, 3), wl)
    step = MoEStep(T, H, I, E, k, wl.shared, wl.clamp)
    step.run(dl, dev(x), dev(logits), None)
    torch.cuda.synchronize()
    ids_ref, w_ref = oracle.route_topk(logits, bias, k)
    assert np.array_equal(host(step.ids), ids_ref)
    c_ref, o_ref, r_ref = oracle.moe_group(ids_ref, E)
    assert np.array_equal(host(step.counts), c_ref)
    assert np.array_equal(host(step.offsets), o_ref) and np.array_equal(host(step.routes), r_ref)
    xq = oracle.quantize_q8_1(x)
    assert np.array_equal(host(step.xq), xq)
    hg, hqg, og = host(step.h), host(step.hq), host(step.out)
    assert_hq_is_rule_of_h(hqg, hg, "hq (prefill)")
    wg, wu, wd = host(dl.wg), host(dl.wu), host(dl.wd)
    wsg, wsu, wsd = host(dl.wsg), host(dl.wsu), host(dl.wsd)
    w32 = w_ref.astype(np.float32)

    def check(a, b):
        rows = list(range(a * k, b * k)) + [T * k + t for t in range(a, b)]
        h_ref, h_terms = oracle.glu_pair(wg, wu, wsg, wsu, xq[a:b], ids_ref[a:b], E, H, I, wl.clamp)
        assert_close(hg[rows], h_ref, h_terms, f"h (prefill tokens {a}..{b})")
        h32 = h_ref.astype(np.float32)
        h_allow = oracle.hq_flip_allowance(h32, oracle.tol(h_terms))
        hq_ref = oracle.quantize_q8_1(h32)
        assert_hq_valid(hqg[rows], hq_ref, h_allow, f"hq (prefill tokens {a}..{b})")
        out_ref, out_terms = oracle.down_combine(wd, wsd, hq_ref, ids_ref[a:b], w32[a:b], E, H, I)
        allow = chain_allowance(wd, wsd, ids_ref[a:b], w_ref[a:b], h_allow)
        assert np.all(np.abs(og[a:b] - out_ref) <= oracle.tol(out_terms) + allow), \
            f"out (prefill tokens {a}..{b}) outside tolerance"
        return b - a

    chunk = 16
    with ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 1)) as ex:
        done = sum(ex.map(lambda a: check(a, min(T, a + chunk)), range(0, T, chunk)))
    assert done == T


# ----------------------------------------------------------------------------- argmax
@pytest.mark.parametrize("R,V,kind", [(1, 4096, "normal"), (5, 129280, "normal"), (3, 1, "normal"),
                                      (2, 3, "normal"), (4, 2049, "normal"), (300, 1000, "normal"),
                                      (1, 129280, "ties_across_chunks"), (2, 5000, "equal"),
                                      (3, 7777, "unaligned"), (2, 4099, "zeros")])
def test_argmax_bit_exact(R, V, kind):
    g = W.rng(600, R * V)
    x = g.standard_normal((R, V)).astype(np.float32)
    if kind == "ties_across_chunks":
        x[0, 5000] = x[0, 100000] = x[0, V - 1] = 9.0
    elif kind == "equal":
        x[:] = 1.25
    elif kind == "zeros":
        x[:] = -1.0
        x[0, 3] = -0.0
        x[0, 4000] = 0.0
        x[1, V - 1] = 0.0
    ref_i, ref_v = oracle.argmax(x)
    am = Argmax(R, V)
    if kind == "unaligned":
        big = torch.zeros(R * V + 1, dtype=torch.float32, device="cuda")
        big[1:] = dev(x).reshape(-1)
        logits = big[1:].view(R, V)
    else:
        logits = dev(x)
    for _ in range(2):  # the workspace counters reset themselves
        idx, val = am.run(logits)
        torch.cuda.synchronize()
        assert np.array_equal(host(idx), ref_i)
        assert np.array_equal(host(val).view(np.uint32), ref_v.view(np.uint32))


# ----------------------------------------------------------------------------- fused prep
@pytest.mark.parametrize("T,E,k,H,bias", [(1, 64, 6, 2048, True), (5, 128, 8, 4096, False), (32, 256, 8, 512, True),
                                          (3, 16, 16, 256, False), (1, 1, 1, 512, False), (33, 64, 6, 256, True),
                                          (4, 300, 7, 256, True)])
def test_moe_prep_matches_the_three_calls(T, E, k, H, bias):
    g = W.rng(700, T * E + k)
    logits = g.standard_normal((T, E)).astype(np.float32)
    x = g.standard_normal((T, H)).astype(np.float32)
    b = (g.standard_normal(E) * 0.1).astype(np.float32) if bias else None
    ids_ref, w_ref = oracle.route_topk(logits, b, k)
    c_ref, o_ref, r_ref = oracle.moe_group(ids_ref, E)
    ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    xq = torch.empty((T, H // 32, 36), dtype=torch.uint8, device="cuda")
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    routes = torch.empty(T * k, dtype=torch.int32, device="cuda")
    B.luce_moe_prep(dev(logits), dev(b) if b is not None else None, dev(x), k, ids, w, xq, counts, offsets, routes)
    torch.cuda.synchronize()
    assert np.array_equal(host(ids), ids_ref)
    assert np.abs(host(w) - w_ref).max() < 2e-6
    assert np.array_equal(host(xq), oracle.quantize_q8_1(x))
    assert np.array_equal(host(counts), c_ref) and np.array_equal(host(offsets), o_ref)
    assert np.array_equal(host(routes), r_ref)


@pytest.mark.parametrize("path", ["layer", "split"])
@pytest.mark.parametrize("name", ["decode_layer", "tiny"])
def test_layer_chain_with_programmatic_launch(name, path):
    wl = W.WORKLOADS[name]
    L = W.host_layer(wl)
    B.luce_set_pdl(True)
    try:
        step, _ = _run_chain(wl, L, path=path)
        _check_chain(wl, L, step)
        # back-to-back steps on one stream: each one's early start must not
        # read the previous step's buffers before they are complete
        layer = W.DeviceLayer(dev(L.wg), dev(L.wu), dev(L.wd), dev(L.wsg) if wl.shared else None,
                              dev(L.wsu) if wl.shared else None, dev(L.wsd) if wl.shared else None)
        ref_out = step.out.clone()
        for _ in range(5):
            step.run(layer, dev(L.x), dev(L.logits), dev(L.bias) if L.bias is not None else None)
        torch.cuda.synchronize()
        assert torch.equal(step.out, ref_out)
    finally:
        B.luce_set_pdl(False)


def test_layer_chain_unfused_prep_path():
    wl = W.WORKLOADS["decode_layer"]
    L = W.host_layer(wl)
    step = MoEStep(wl.T, wl.H, wl.I, wl.E, wl.k, wl.shared, wl.clamp)
    step.path = "split"
    step.fused_prep = False
    layer = W.DeviceLayer(dev(L.wg), dev(L.wu), dev(L.wd), dev(L.wsg), dev(L.wsu), dev(L.wsd))
    step.run(layer, dev(L.x), dev(L.logits), dev(L.bias))
    torch.cuda.synchronize()
    _check_chain(wl, L, step)
