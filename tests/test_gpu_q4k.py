"""GPU: the Q4_K expert-weight path (luce_moe_glu_q4k, luce_quantize_q8_1 of
h, luce_moe_down_combine_q4k) against the oracle: h within the float bound,
hq exactly the q8_1 rule where the quantization is stable, out within the
bound plus the allowance for q8_1 flips of h; masked routes untouched and
skipped; the decode-layer shape and a verify-like shape."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_close, assert_hq_valid, chain_allowance, dev, host
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
def _no_device_faults(request):
    yield
    if "allow_fault" not in request.keywords:
        assert B.luce_get_fault() == 0


# name, T, H, I, E, k, shared, clamp, masked route
CASES = [
    ("decode_shape", 1, 2048, 1024, 16, 6, True, 0.0, False),
    ("verify_like", 5, 1024, 512, 12, 4, True, 10.0, False),
    ("masked_no_shared", 3, 512, 256, 6, 2, False, 0.0, True),
    ("wide_rows", 2, 4096, 256, 4, 2, True, 0.0, False),
    ("odd_k_shared", 2, 512, 256, 8, 3, True, 0.0, False),     # the shared slot in the upper half-warp
    ("two_passes", 2, 512, 512, 10, 8, True, 0.0, True),       # k + 1 slots over two passes
    ("long_down_rows", 1, 256, 2048, 4, 2, True, 0.0, False),  # 32 sub-block pairs: one slot per warp
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_q4k_layer_matches_oracle(case):
    name, T, H, I, E, k, shared, clamp, masked = case
    wl = W.Workload(name, T=T, H=H, I=I, E=E, k=k, shared=shared, clamp=clamp, seed=800 + T * 10 + k, bias_std=0.1)
    L = W.host_layer_q4k(wl)
    ids, w = oracle.route_topk(L.logits, L.bias, k)
    if masked:
        ids[1, 0] = -1
    w32 = w.astype(np.float32)
    xq = oracle.quantize_q8_1(L.x)
    rows = T * k + (T if shared else 0)
    h_ref, h_terms = oracle.glu_q4k(L.wg, L.wu, L.wsg, L.wsu, xq, ids, E, H, I, clamp)

    h = torch.full((rows, I), float("nan"), dtype=torch.float32, device="cuda")
    hq = torch.full((rows, I // 32, 36), 0xAB, dtype=torch.uint8, device="cuda")
    B.luce_moe_glu_q4k(dev(L.wg), dev(L.wu), dev(L.wsg) if shared else None, dev(L.wsu) if shared else None, dev(xq),
                       dev(ids), E, H, I, clamp, h, hq)
    # the q8_1 blocks written in the gate/up launch are luce_quantize_q8_1 of h, bit for bit
    hq_sep = torch.zeros_like(hq)
    B.luce_quantize_q8_1(h.nan_to_num(0.0), hq_sep)
    # and h without hq is the same h
    h_only = torch.full_like(h, float("nan"))
    B.luce_moe_glu_q4k(dev(L.wg), dev(L.wu), dev(L.wsg) if shared else None, dev(L.wsu) if shared else None, dev(xq),
                       dev(ids), E, H, I, clamp, h_only)
    torch.cuda.synchronize()
    hg = host(h)
    valid = ~np.isnan(h_ref[:, 0])
    assert np.isnan(hg[~valid]).all(), "rows of masked routes must not be written"
    assert np.array_equal(host(hq)[valid], host(hq_sep)[valid])
    assert (host(hq)[~valid] == 0xAB).all(), "q8_1 rows of masked routes must not be written"
    assert torch.equal(h.nan_to_num(0.0), h_only.nan_to_num(0.0))
    assert_close(hg[valid], h_ref[valid], h_terms[valid], f"h ({name})")
    h32 = np.nan_to_num(h_ref, nan=0.0).astype(np.float32)
    allow = oracle.hq_flip_allowance(h32, oracle.tol(np.nan_to_num(h_terms, nan=0.0)))
    hq_ref = oracle.quantize_q8_1(h32)
    assert_hq_valid(host(hq)[valid], hq_ref[valid], allow[valid], f"hq ({name})", h_gpu=hg[valid])

    # the down product and combine, fed the oracle's own hq (so the bound is the plain float rule)
    out_ref, out_terms = oracle.down_combine_q4k(L.wd, L.wsd, hq_ref, ids, w32, E, H, I)
    out = torch.full((T, H), float("nan"), dtype=torch.float32, device="cuda")
    B.luce_moe_down_combine_q4k(dev(L.wd), dev(L.wsd) if shared else None, dev(hq_ref), dev(ids), dev(w32), E, H, I,
                                out)
    torch.cuda.synchronize()
    assert_close(host(out), out_ref, out_terms, f"out ({name})")

    # and the whole chain on the GPU's own hq, with the allowance for flips of h
    out2 = torch.empty_like(out)
    B.luce_moe_down_combine_q4k(dev(L.wd), dev(L.wsd) if shared else None, hq, dev(ids), dev(w32), E, H, I, out2)
    torch.cuda.synchronize()
    allow_out = chain_allowance_q4k(L.wd, L.wsd, ids, w32, allow)
    assert np.all(np.abs(host(out2) - out_ref) <= oracle.tol(out_terms) + allow_out)


def chain_allowance_q4k(wd, wsd, ids, weights, h_allow):
    """|out| change bound from flips of q8_1(h): sum_j |w_j| sum_i |Wd value| allow (values dequantized loosely:
    |d sc q - dmin m| <= |d| 63 15 + |dmin| 63 per element)."""
    T, k = ids.shape
    H = wd.shape[1]

    def bound_rows(W_rows):  # [H, I/256, 144] -> per-element magnitude bound [H, I]
        d = np.abs(W_rows[..., 0:2].copy().view(np.float16).astype(np.float64))
        dm = np.abs(W_rows[..., 2:4].copy().view(np.float16).astype(np.float64))
        b = (d * 63 * 15 + dm * 63)[..., 0]
        return np.repeat(b, 256, axis=-1)

    out = np.zeros((T, H))
    for t in range(T):
        for j in range(k):
            e = ids[t, j]
            if e < 0:
                continue
            a = h_allow[t * k + j]
            if a.any():
                out[t] += abs(float(weights[t, j])) * (bound_rows(wd[e]) @ a)
        if wsd is not None:
            a = h_allow[T * k + t]
            if a.any():
                out[t] += bound_rows(wsd) @ a
    return out * 1.001


@pytest.mark.allow_fault
def test_q4k_out_of_range_id_is_skipped_and_flagged():
    """An id >= E in either Q4_K call: that route is skipped (its h row is not
    written, the combine leaves it out) and LUCE_FAULT_BAD_ID is raised; the
    results equal the oracle's with that route masked."""
    assert B.luce_get_fault() == 0
    T, H, I, E, k = 2, 512, 256, 4, 2
    wl = W.Workload("q4k_bad_id", T=T, H=H, I=I, E=E, k=k, shared=True, clamp=0.0, seed=871, bias_std=0.0)
    L = W.host_layer_q4k(wl)
    ids_bad = np.array([[1, E], [3, 0]], np.int32)
    ids_masked = np.array([[1, -1], [3, 0]], np.int32)
    w32 = np.array([[0.6, 0.4], [0.7, 0.3]], np.float32)
    xq = oracle.quantize_q8_1(L.x)
    rows = T * k + T
    h_ref, h_terms = oracle.glu_q4k(L.wg, L.wu, L.wsg, L.wsu, xq, ids_masked, E, H, I, 0.0)
    h = torch.full((rows, I), float("nan"), dtype=torch.float32, device="cuda")
    hq = torch.full((rows, I // 32, 36), 0xAB, dtype=torch.uint8, device="cuda")
    B.luce_moe_glu_q4k(dev(L.wg), dev(L.wu), dev(L.wsg), dev(L.wsu), dev(xq), dev(ids_bad), E, H, I, 0.0, h, hq)
    torch.cuda.synchronize()
    assert B.luce_get_fault() == B.LUCE_FAULT_BAD_ID
    hg = host(h)
    assert np.isnan(hg[1]).all(), "the row of the out-of-range route must not be written"
    assert (host(hq)[1] == 0xAB).all(), "nor its q8_1 row"
    valid = ~np.isnan(h_ref[:, 0])
    assert_close(hg[valid], h_ref[valid], h_terms[valid], "h (bad id)")
    # the down product on the oracle's hq: the bad route is left out of the combine
    hq_ref = oracle.quantize_q8_1(np.nan_to_num(h_ref, nan=0.0).astype(np.float32))
    out_ref, out_terms = oracle.down_combine_q4k(L.wd, L.wsd, hq_ref, ids_masked, w32, E, H, I)
    out = torch.full((T, H), float("nan"), dtype=torch.float32, device="cuda")
    B.luce_moe_down_combine_q4k(dev(L.wd), dev(L.wsd), dev(hq_ref), dev(ids_bad), dev(w32), E, H, I, out)
    torch.cuda.synchronize()
    assert B.luce_get_fault() == B.LUCE_FAULT_BAD_ID
    assert_close(host(out), out_ref, out_terms, "out (bad id)")
    assert B.luce_get_fault() == 0  # reading clears
