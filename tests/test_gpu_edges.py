"""GPU: the steps either side of the MoE FFN, against the oracle.

* RMS norm + router logits (luce_rmsnorm_router): xn and the logits within
  the float bound of the double-precision oracle, and the router's selection
  on the GPU's logits equal to the oracle's selection on the same logits.
* The argmax of a vocabulary split into shards (luce_argmax_shard on each,
  luce_argmax_pick across them): bit for bit the whole row's argmax.
* A two-way expert-parallel split (luce_ep_mask, the split path per rank,
  luce_add_f32): the masked ids exactly, the sum exactly the fp32 sum of the
  partials, the output within the bound of the oracle's split step.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_close, chain_allowance, dev, host
from quantized_moe_decode_luce_gb300 import binding as B
from quantized_moe_decode_luce_gb300 import build as BLD
from quantized_moe_decode_luce_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    BLD.build()
    B.lib()
    yield


@pytest.fixture(autouse=True)
def _no_device_faults():
    yield
    assert B.luce_get_fault() == 0


# ----------------------------------------------------------------------------- RMS norm + router
# T, E, H: decode and verify hidden sizes, several token tiles with a ragged
# last one, a ragged last expert chunk, the largest H (one token per tile)
NORM_CASES = [(1, 64, 2048), (5, 128, 4096), (13, 40, 512), (3, 9, 12288), (64, 256, 1024), (1, 9, 516),
              (1, 64, 4096)]


@pytest.mark.parametrize("T,E,H", NORM_CASES)
def test_rmsnorm_router_matches_oracle(T, E, H):
    g = W.rng(700, T * 1000 + E)
    x = g.standard_normal((T, H)).astype(np.float32)
    x[0, :7] *= 40.0  # a few large entries
    gamma = g.uniform(0.5, 1.5, H).astype(np.float32)
    w = (g.standard_normal((E, H)) * 0.02).astype(np.float32)
    eps = 1e-6
    xn_ref, lg_ref, terms = oracle.rmsnorm_router(x, gamma, eps, w)
    xn = torch.full((T, H), float("nan"), dtype=torch.float32, device="cuda")
    logits = torch.full((T, E), float("nan"), dtype=torch.float32, device="cuda")
    B.luce_rmsnorm_router(dev(x), dev(gamma), eps, dev(w), xn, logits)
    torch.cuda.synchronize()
    assert_close(host(xn), xn_ref, np.abs(xn_ref), "xn")
    assert_close(host(logits), lg_ref, terms, "logits")
    # without xn the logits are the same bits
    logits2 = torch.empty_like(logits)
    B.luce_rmsnorm_router(dev(x), dev(gamma), eps, dev(w), None, logits2)
    torch.cuda.synchronize()
    assert torch.equal(logits, logits2)
    # the router's selection from the GPU's logits is the oracle's from the same logits
    k = min(6, E)
    ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
    wts = torch.empty((T, k), dtype=torch.float32, device="cuda")
    B.luce_route_topk(logits, None, k, ids, wts)
    torch.cuda.synchronize()
    ids_ref, _ = oracle.route_topk(host(logits), None, k)
    assert np.array_equal(host(ids), ids_ref)


def test_rmsnorm_of_zero_rows_is_zero():
    T, E, H = 2, 8, 256
    x = np.zeros((T, H), np.float32)
    gamma = np.ones(H, np.float32)
    w = np.ones((E, H), np.float32)
    xn = torch.full((T, H), 7.0, dtype=torch.float32, device="cuda")
    logits = torch.full((T, E), 7.0, dtype=torch.float32, device="cuda")
    B.luce_rmsnorm_router(dev(x), dev(gamma), 1e-6, dev(w), xn, logits)
    torch.cuda.synchronize()
    assert torch.all(xn == 0.0) and torch.all(logits == 0.0)


@pytest.mark.parametrize("H", [2048, 516])
def test_rmsnorm_router_one_token_path_is_the_tiled_path(H):
    # one token takes the register path, a batch (or an unaligned gamma) the
    # tiled path: the same lane slices and sum orders give the same bits
    E = 40
    g = W.rng(720, H)
    x = g.standard_normal((3, H)).astype(np.float32)
    gamma = g.uniform(0.5, 1.5, H + 1).astype(np.float32)
    w = (g.standard_normal((E, H)) * 0.02).astype(np.float32)
    gam_d = dev(gamma)
    wd = dev(w)
    x1, lg1 = torch.empty((1, H), device="cuda"), torch.empty((1, E), device="cuda")
    x3, lg3 = torch.empty((3, H), device="cuda"), torch.empty((3, E), device="cuda")
    xu, lgu = torch.empty((1, H), device="cuda"), torch.empty((1, E), device="cuda")
    B.luce_rmsnorm_router(dev(x[:1]), gam_d[:H], 1e-6, wd, x1, lg1)
    B.luce_rmsnorm_router(dev(x), gam_d[:H], 1e-6, wd, x3, lg3)
    gam_u = dev(np.concatenate([[0.0], gamma[:H]]).astype(np.float32))[1:]  # 4-byte aligned only
    B.luce_rmsnorm_router(dev(x[:1]), gam_u, 1e-6, wd, xu, lgu)
    torch.cuda.synchronize()
    assert torch.equal(x1[0], x3[0]) and torch.equal(lg1[0], lg3[0])
    assert torch.equal(x1, xu) and torch.equal(lg1, lgu)
    xn_ref, lg_ref, terms = oracle.rmsnorm_router(x[:1], gamma[:H], 1e-6, w)
    assert_close(host(lg1), lg_ref, terms, "logits")


@pytest.mark.parametrize("T,E,H", [(1, 64, 2048), (5, 128, 4096), (1, 9, 516), (3, 9, 12288)])
def test_add_rmsnorm_router_is_the_add_then_the_norm(T, E, H):
    # the residual sum is one fp32 add (numpy's float32 addition, exactly);
    # xn and the logits are the oracle's of that sum, and the same bits as
    # luce_add_f32 followed by luce_rmsnorm_router
    g = W.rng(730, T * 1000 + H)
    x = g.standard_normal((T, H)).astype(np.float32)
    r = (g.standard_normal((T, H)) * 3.0).astype(np.float32)
    gamma = g.uniform(0.5, 1.5, H).astype(np.float32)
    w = (g.standard_normal((E, H)) * 0.02).astype(np.float32)
    s_ref = x + r
    xn_ref, lg_ref, terms = oracle.rmsnorm_router(s_ref, gamma, 1e-6, w)
    xd, rd, gd, wd = dev(x), dev(r), dev(gamma), dev(w)
    s_out = torch.full((T, H), float("nan"), device="cuda")
    xn = torch.full((T, H), float("nan"), device="cuda")
    lg = torch.full((T, E), float("nan"), device="cuda")
    B.luce_add_rmsnorm_router(xd, rd, s_out, gd, 1e-6, wd, xn, lg)
    s2, xn2, lg2 = torch.empty_like(s_out), torch.empty_like(xn), torch.empty_like(lg)
    B.luce_add_f32(xd, rd, s2)
    B.luce_rmsnorm_router(s2, gd, 1e-6, wd, xn2, lg2)
    lg3 = torch.empty_like(lg)
    B.luce_add_rmsnorm_router(xd, rd, None, gd, 1e-6, wd, None, lg3)
    torch.cuda.synchronize()
    assert np.array_equal(host(s_out).view(np.uint32), s_ref.view(np.uint32))
    assert_close(host(xn), xn_ref, np.abs(xn_ref), "xn")
    assert_close(host(lg), lg_ref, terms, "logits")
    assert torch.equal(s_out, s2) and torch.equal(xn, xn2) and torch.equal(lg, lg2) and torch.equal(lg, lg3)


# ----------------------------------------------------------------------------- vocabulary split
@pytest.mark.parametrize("cuts", [[0, 64640, 129280], [0, 1, 70000, 129280], [0, 43093, 86186, 129280],
                                  [0, 129280]])
def test_argmax_over_vocabulary_shards_is_the_whole_row(cuts):
    R, V = 5, 129280
    g = W.rng(710, len(cuts))
    x = g.standard_normal((R, V)).astype(np.float32)
    x[1, 64639] = x[1, 64640] = 9.0      # a tie across the two-way boundary
    x[2, 0] = x[2, V - 1] = 9.0          # first and last columns tie
    x[3, :] = 0.5                        # all equal
    x[4, 43092] = x[4, 129279] = 9.0     # tie across non-adjacent shards
    ref_i, ref_v = oracle.argmax(x)
    S = len(cuts) - 1
    vals = torch.empty((S, R), dtype=torch.float32, device="cuda")
    idxs = torch.empty((S, R), dtype=torch.int32, device="cuda")
    for s, (a, b) in enumerate(zip(cuts[:-1], cuts[1:])):
        shard = dev(np.ascontiguousarray(x[:, a:b]))  # the shard a rank would hold
        ws = torch.zeros(B.luce_argmax_workspace_bytes(R, b - a), dtype=torch.uint8, device="cuda")
        B.luce_argmax_shard(shard, a, idxs[s], vals[s], ws)
    idx = torch.empty(R, dtype=torch.int32, device="cuda")
    val = torch.empty(R, dtype=torch.float32, device="cuda")
    B.luce_argmax_pick(vals, idxs, idx, val)
    torch.cuda.synchronize()
    assert np.array_equal(host(idx), ref_i)
    assert np.array_equal(host(val).view(np.uint32), ref_v.view(np.uint32))
    assert ref_i[1] == 64639 and ref_i[2] == 0 and ref_i[3] == 0 and ref_i[4] == 43092
    # and the pick of the GPU's shard results is the oracle's pick of them
    p_i, p_v = oracle.argmax_pick(host(vals), host(idxs))
    assert np.array_equal(p_i, ref_i)


# ----------------------------------------------------------------------------- expert-parallel split
def _rank_partial(wl, L, logits, bias, e0, e1, shared):
    T, k, E, H, I = wl.T, wl.k, wl.E, wl.H, wl.I
    ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    B.luce_route_topk(logits, bias, k, ids, w)
    ids_m = torch.empty_like(ids)
    B.luce_ep_mask(ids, e0, e1, ids_m)
    xq = torch.empty((T, H // 32, 36), dtype=torch.uint8, device="cuda")
    B.luce_quantize_q8_1(dev(L.x), xq)
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    routes = torch.empty(T * k, dtype=torch.int32, device="cuda")
    B.luce_moe_group(ids_m, E, counts, offsets, routes)
    rows = T * k + T
    h = torch.full((rows, I), float("nan"), dtype=torch.float32, device="cuda")
    hq = torch.zeros((rows, I // 32, 36), dtype=torch.uint8, device="cuda")
    B.luce_moe_glu_pair(dev(L.wg), dev(L.wu), dev(L.wsg) if shared else None, dev(L.wsu) if shared else None, xq,
                        offsets, routes, T, k, E, H, I, wl.clamp, h, hq)
    out = torch.full((T, H), float("nan"), dtype=torch.float32, device="cuda")
    B.luce_moe_down_combine(dev(L.wd), dev(L.wsd) if shared else None, hq, ids_m, w, offsets, routes, T, k, E, H, I,
                            out)
    return ids, ids_m, out


@pytest.mark.parametrize("T", [1, 3])
def test_two_way_expert_parallel_split(T):
    wl = W.Workload("ep2", T=T, H=512, I=256, E=8, k=3, shared=True, clamp=0.0, seed=720 + T, bias_std=0.1)
    L = W.host_layer(wl)
    logits = dev(L.logits)
    bias = dev(L.bias) if L.bias is not None else None
    ids, ma, pa = _rank_partial(wl, L, logits, bias, 0, 4, True)     # rank 0: experts 0..3 and the shared one
    _, mb, pb = _rank_partial(wl, L, logits, bias, 4, 8, False)      # rank 1: experts 4..7
    out = torch.empty_like(pa)
    B.luce_add_f32(pa, pb, out)
    torch.cuda.synchronize()
    idh = host(ids)
    assert np.array_equal(host(ma), np.where(idh < 4, idh, -1))
    assert np.array_equal(host(mb), np.where(idh >= 4, idh, -1))
    assert np.array_equal(host(out), (host(pa) + host(pb)).astype(np.float32))
    ref = oracle.ep_layer(L.wg, L.wu, L.wd, L.wsg, L.wsu, L.wsd, L.x, L.logits, L.bias, wl.k, wl.clamp, [0, 4, 8])
    assert np.array_equal(idh, ref["ids"])
    allow = chain_allowance(L.wd, L.wsd, ref["ids"], ref["weights"], ref["h_allow"])
    bound = oracle.tol(ref["out_terms"]) + allow
    assert np.all(np.abs(host(out) - ref["out"]) <= bound), "EP output outside tolerance"
    # in place: the sum into the first partial
    B.luce_add_f32(pa, pb, pa)
    torch.cuda.synchronize()
    assert torch.equal(pa, out)
