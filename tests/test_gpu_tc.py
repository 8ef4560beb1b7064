"""GPU: the grouped tensor-core path of luce_moe_layer (more than 8 tokens, or
more than 64 routes) against the oracle.

Routing, grouping and the q8_1 input are integer results, compared bit for
bit.  h is within the float bound of the oracle's h; hq is, byte for byte,
the q8_1 kernel applied to the h the GPU stored, and differs from the
oracle's quantization of the oracle's h only where the flip allowance says it
may; out is within the float bound plus the allowance those flips carry.
The shapes cover: experts with more than 64 tokens (several token slices of
one expert), experts with none, no shared expert, the clamped SwiGLU, T*k > 64
at T <= 8, and H, I at their smallest (256)."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_close, assert_hq_is_rule_of_h, assert_hq_valid, chain_allowance, dev, host
from quantized_moe_decode_luce_gb300 import binding as B
from quantized_moe_decode_luce_gb300 import build as BLD
from quantized_moe_decode_luce_gb300 import workloads as W
from quantized_moe_decode_luce_gb300.layer import MoEStep

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


# name, T, H, I, E, k, shared, clamp, logits, bias_std, concentrate
CASES = [
    ("t9_smallest", 9, 256, 256, 8, 2, True, 0.0, "normal", 0.0, 0.0),
    ("t8_k9_routes", 8, 256, 512, 12, 9, True, 0.0, "normal", 0.1, 0.0),
    ("t40_no_shared", 40, 512, 256, 16, 3, False, 0.0, "normal", 0.1, 0.0),
    ("t64_clamped", 64, 512, 768, 8, 4, True, 10.0, "normal", 0.0, 0.0),
    ("t130_zipf_empty_experts", 130, 768, 512, 48, 4, True, 10.0, "zipf", 0.1, 0.0),
    # every token prefers the same few experts: 150 tokens on one expert -> three token slices
    ("t150_concentrated", 150, 256, 256, 16, 3, True, 0.0, "normal", 0.0, 25.0),
]


def _layer(wl):
    L = W.host_layer(wl)
    return L, W.DeviceLayer(dev(L.wg), dev(L.wu), dev(L.wd), dev(L.wsg) if wl.shared else None,
                            dev(L.wsu) if wl.shared else None, dev(L.wsd) if wl.shared else None)


def _run(wl, L, dl):
    st = MoEStep(wl.T, wl.H, wl.I, wl.E, wl.k, wl.shared, wl.clamp)
    assert st.path == "layer"
    st.h.fill_(float("nan"))
    st.run(dl, dev(L.x), dev(L.logits), dev(L.bias) if L.bias is not None else None)
    torch.cuda.synchronize()
    assert st.path == "layer"
    return st


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_tc_layer_matches_oracle(case):
    name, T, H, I, E, k, shared, clamp, logits, bias_std, conc = case
    wl = W.Workload(name, T=T, H=H, I=I, E=E, k=k, shared=shared, clamp=clamp, seed=1200 + T + k,
                    logits=logits, bias_std=bias_std)
    L, dl = _layer(wl)
    if conc > 0:
        pref = np.zeros(E, np.float32)
        pref[:k] = np.float32(conc) * np.arange(k, 0, -1, dtype=np.float32)
        L.logits = (L.logits + pref[None, :]).astype(np.float32)
    st = _run(wl, L, dl)
    ref = oracle.moe_layer(L.wg, L.wu, L.wd, L.wsg, L.wsu, L.wsd, L.x, L.logits, L.bias, k, clamp)
    assert np.array_equal(host(st.ids), ref["ids"])
    assert np.array_equal(host(st.xq), ref["xq"])
    c_ref, o_ref, r_ref = oracle.moe_group(ref["ids"], E)
    assert np.array_equal(host(st.counts), c_ref) and np.array_equal(host(st.offsets), o_ref)
    assert np.array_equal(host(st.routes), r_ref)
    if conc > 0:
        assert c_ref.max() > 128  # an expert with more than two token slices
    hg = host(st.h)
    valid = ~np.isnan(ref["h"][:, 0])
    assert valid.all()  # the router masks nothing
    assert_close(hg, ref["h"], ref["h_terms"], f"h ({name})")
    flips = assert_hq_valid(host(st.hq), ref["hq"], ref["h_allow"], f"hq ({name})", h_gpu=hg)
    allow = chain_allowance(L.wd, L.wsd, ref["ids"], ref["weights"], ref["h_allow"])
    gout = host(st.out)
    bound = oracle.tol(ref["out_terms"]) + allow
    bad = ~(np.abs(gout - ref["out"]) <= bound)
    assert not bad.any(), f"out ({name}): {bad.sum()} of {bad.size} outside tolerance"
    assert flips <= max(4, hg.size // 500)


def test_tc_layer_is_deterministic_and_reuses_its_workspace():
    wl = W.Workload("t96_repeat", T=96, H=512, I=512, E=16, k=4, shared=True, clamp=10.0, seed=1300)
    L, dl = _layer(wl)
    st = _run(wl, L, dl)
    ref = {n: getattr(st, n).clone() for n in ("out", "h", "hq")}
    x, lg = dev(L.x), dev(L.logits)
    b = dev(L.bias) if L.bias is not None else None
    for _ in range(3):
        st.run(dl, x, lg, b)
    torch.cuda.synchronize()
    for n, v in ref.items():
        assert torch.equal(getattr(st, n), v), f"{n} changed between repeated calls"


def test_tc_layer_workspace_too_small_is_an_argument_error():
    wl = W.Workload("t16_ws", T=16, H=256, I=256, E=8, k=2, shared=False, clamp=0.0, seed=1301)
    L, dl = _layer(wl)
    st = MoEStep(wl.T, wl.H, wl.I, wl.E, wl.k, wl.shared, wl.clamp)
    small = torch.zeros(st.workspace.numel() - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(B.LuceError) as ei:
        B.luce_moe_layer(dev(L.logits), None, dev(L.x), wl.k, wl.I, dl.wg, dl.wu, dl.wd, None, None, None, 0.0,
                         st.ids, st.weights, st.xq, st.counts, st.offsets, st.routes, st.h, st.hq, st.out, small)
    assert ei.value.status == B.LUCE_ERR_INVALID_ARG
