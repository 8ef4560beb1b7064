"""GPU: the whole layer in one launch (luce_moe_layer).

Its results must equal those of the three split launches (luce_moe_prep,
luce_moe_glu_pair, luce_moe_down_combine) bit for bit, for every output,
since every fused step repeats the split step's arithmetic in the same
order; the split path itself is checked against the oracle in
test_gpu_parity.py, and so is this path on the named workloads.  Also: its
device barrier state stays consistent over repeated calls and graph replays,
and shapes beyond its limits are declined before anything is launched."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import dev, host
from quantized_moe_decode_luce_gb300 import binding as B
from quantized_moe_decode_luce_gb300 import build as BLD
from quantized_moe_decode_luce_gb300 import workloads as W
from quantized_moe_decode_luce_gb300.layer import MoEStep

pytestmark = pytest.mark.gpu

OUTPUTS = ("ids", "weights", "xq", "counts", "offsets", "routes", "hq", "out")


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


def _layer(wl, L):
    return W.DeviceLayer(dev(L.wg), dev(L.wu), dev(L.wd), dev(L.wsg) if wl.shared else None,
                         dev(L.wsu) if wl.shared else None, dev(L.wsd) if wl.shared else None)


def _both(wl, L, layer=None, h_rows_valid=True):
    layer = layer or _layer(wl, L)
    x, lg = dev(L.x), dev(L.logits)
    b = dev(L.bias) if L.bias is not None else None
    res = {}
    for path in ("split", "layer"):
        st = MoEStep(wl.T, wl.H, wl.I, wl.E, wl.k, wl.shared, wl.clamp)
        st.path = path
        st.h.fill_(float("nan"))
        st.hq.fill_(0xAB)
        st.run(layer, x, lg, b)
        torch.cuda.synchronize()
        assert st.path == path
        res[path] = st
    return res["split"], res["layer"]


def _assert_equal(a, b, R):
    for name in OUTPUTS:
        ta, tb = getattr(a, name), getattr(b, name)
        if name == "hq":
            ta, tb = ta[:R], tb[:R]
        assert torch.equal(ta, tb), f"{name} differs between the split launches and the one launch"
    # h rows of routes and of the shared expert (every row is live: no masked routes)
    assert torch.equal(a.h[:R], b.h[:R])


SHAPES = [
    # name, T, H, I, E, k, shared, clamp, logits, bias_std
    ("decode", 1, 2048, 1024, 64, 6, True, 0.0, "normal", 0.1),
    ("tiny", 1, 512, 256, 1, 1, False, 0.0, "single", 0.0),
    ("verify_small", 5, 1024, 512, 32, 8, True, 10.0, "shared_col", 0.0),
    ("t8_e256", 8, 512, 256, 256, 8, True, 0.0, "normal", 0.1),
    ("t3_noshared", 3, 256, 512, 16, 4, False, 10.0, "normal", 0.0),
    ("t2_k1", 2, 768, 256, 8, 1, True, 0.0, "normal", 0.0),
    ("t7_k9", 7, 256, 768, 12, 9, True, 0.0, "normal", 0.05),
    ("wide_h", 4, 8192, 256, 64, 8, True, 0.0, "shared_col", 0.0),
    ("wide_i", 1, 256, 8192, 64, 6, True, 10.0, "zipf", 0.1),
    ("all_experts", 2, 256, 256, 4, 4, True, 0.0, "normal", 0.0),
    # flat-split kernel (hq > 24 KB) with more than 32 routed virtual experts:
    # the plan's lane scans take several 32-expert chunks
    ("flat_t6_e64", 6, 512, 512, 64, 8, True, 10.0, "normal", 0.0),
    ("flat_t8_e128", 8, 512, 512, 128, 8, True, 0.0, "normal", 0.1),
]


@pytest.mark.parametrize("case", SHAPES, ids=[c[0] for c in SHAPES])
def test_one_launch_equals_split_launches(case):
    name, T, H, I, E, k, shared, clamp, logits, bias_std = case
    wl = W.Workload(name, T=T, H=H, I=I, E=E, k=k, shared=shared, clamp=clamp, seed=900 + T * 7 + k,
                    logits=logits, bias_std=bias_std)
    L = W.host_layer(wl)
    a, b = _both(wl, L)
    R = T * k + (T if shared else 0)
    _assert_equal(a, b, R)
    # and the selection is the oracle's
    ids_ref, _ = oracle.route_topk(L.logits, L.bias, k)
    assert np.array_equal(host(b.ids), ids_ref)


def test_decode_layer_matches_oracle_through_one_launch():
    wl = W.WORKLOADS["decode_layer"]
    L = W.host_layer(wl)
    _, b = _both(wl, L)
    ref = oracle.moe_layer(L.wg, L.wu, L.wd, L.wsg, L.wsu, L.wsd, L.x, L.logits, L.bias, wl.k, wl.clamp)
    assert np.array_equal(host(b.ids), ref["ids"]) and np.array_equal(host(b.xq), ref["xq"])
    c_ref, o_ref, r_ref = oracle.moe_group(ref["ids"], wl.E)
    assert np.array_equal(host(b.counts), c_ref) and np.array_equal(host(b.offsets), o_ref)
    assert np.array_equal(host(b.routes), r_ref)


def test_repeated_calls_and_barrier_state():
    wl = W.WORKLOADS["decode_layer"]
    L = W.host_layer(wl)
    layer = _layer(wl, L)
    st = MoEStep(wl.T, wl.H, wl.I, wl.E, wl.k, wl.shared, wl.clamp)
    st.path = "layer"
    x, lg, b = dev(L.x), dev(L.logits), dev(L.bias)
    st.run(layer, x, lg, b)
    torch.cuda.synchronize()
    ref = st.out.clone()
    for i in range(20):
        st.run(layer, x, lg, b)
    torch.cuda.synchronize()
    assert torch.equal(st.out, ref) and st.path == "layer"
    # the 64-bit arrival count grows by the grid size per barrier, one barrier per decode call
    count = int(st.workspace[:8].view(torch.int64)[0].item())
    grid = torch.cuda.get_device_properties(0).multi_processor_count
    assert count == 21 * grid


def test_graph_replay_with_programmatic_launch():
    wl = W.WORKLOADS["decode_layer"]
    Ls = [W.host_layer(wl, seed=40 + i) for i in range(3)]
    layers = [_layer(wl, L) for L in Ls]
    xs = [dev(L.x) for L in Ls]
    lgs = [dev(L.logits) for L in Ls]
    bs = [dev(L.bias) for L in Ls]
    st = MoEStep(wl.T, wl.H, wl.I, wl.E, wl.k, wl.shared, wl.clamp)
    st.path = "layer"
    outs = torch.empty((3, wl.T, wl.H), dtype=torch.float32, device="cuda")
    # references: one layer at a time, eager, no programmatic launch
    refs = []
    for i in range(3):
        st.run(layers[i], xs[i], lgs[i], bs[i])
        torch.cuda.synchronize()
        refs.append(st.out.clone())
    B.luce_set_pdl(True)
    try:
        stream = torch.cuda.Stream()
        with torch.cuda.stream(stream):
            for i in range(3):  # a chain of layers, eager
                st.run(layers[i], xs[i], lgs[i], bs[i], out=outs[i])
            torch.cuda.synchronize()
            for i in range(3):
                assert torch.equal(outs[i], refs[i])
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for i in range(3):
                    st.run(layers[i], xs[i], lgs[i], bs[i], out=outs[i])
            outs.zero_()
            for _ in range(10):
                g.replay()
            torch.cuda.synchronize()
    finally:
        B.luce_set_pdl(False)
    for i in range(3):
        assert torch.equal(outs[i], refs[i])
    assert st.path == "layer"
    count = int(st.workspace[:8].view(torch.int64)[0].item())
    assert count % torch.cuda.get_device_properties(0).multi_processor_count == 0


def test_shapes_beyond_the_limits_are_declined_without_a_launch():
    # few tokens but more than 256 experts: beyond the one-launch kernels, and
    # not a many-token shape for the grouped tensor-core path
    T, H, I, E, k = 2, 256, 256, 300, 2
    f = torch.zeros((T, E), dtype=torch.float32, device="cuda")
    x = torch.zeros((T, H), dtype=torch.float32, device="cuda")
    w = torch.zeros((E, I, H // 32, 34), dtype=torch.uint8, device="cuda")
    wd = torch.zeros((E, H, I // 32, 34), dtype=torch.uint8, device="cuda")
    ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
    wts = torch.empty((T, k), dtype=torch.float32, device="cuda")
    xq = torch.empty((T, H // 32, 36), dtype=torch.uint8, device="cuda")
    cnt = torch.empty(E, dtype=torch.int32, device="cuda")
    off = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    rt = torch.empty(T * k, dtype=torch.int32, device="cuda")
    hq = torch.empty((T * k, I // 32, 36), dtype=torch.uint8, device="cuda")
    h = torch.empty((T * k, I), dtype=torch.float32, device="cuda")
    out = torch.full((T, H), 7.0, dtype=torch.float32, device="cuda")
    ws = torch.zeros(B.luce_moe_layer_workspace_bytes(T, k, H, I), dtype=torch.uint8, device="cuda")
    with pytest.raises(B.LuceError) as ei:
        B.luce_moe_layer(f, None, x, k, I, w, w, wd, None, None, None, 0.0, ids, wts, xq, cnt, off, rt, h, hq,
                         out, ws)
    assert ei.value.status == B.LUCE_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert torch.all(out == 7.0) and torch.all(ws == 0)
    # MoEStep serves such a shape with the split launches, even when asked for one launch
    st = MoEStep(T, H, I, E, k, False, 0.0)
    st.path = "layer"
    layer = W.DeviceLayer(w, w, wd)
    st.run(layer, x, f, None)
    torch.cuda.synchronize()
    assert st.path == "split"


@pytest.mark.parametrize("T", [1, 3])
def test_nan_scores_select_like_the_oracle_on_every_path(T):
    # NaN logits (and a NaN bias entry): both paths and the separate router
    # rank them below every number, as the oracle does; no fault is raised
    wl = W.Workload("nan_scores", T=T, H=256, I=256, E=40, k=6, shared=True, clamp=0.0, seed=77 + T,
                    logits="normal", bias_std=0.1)
    L = W.host_layer(wl)
    L.logits[:, ::3] = np.float32("nan")
    L.bias[5] = np.float32("nan")
    a, b = _both(wl, L)
    ids_ref, _ = oracle.route_topk(L.logits, L.bias, wl.k)
    assert np.array_equal(host(a.ids), ids_ref)
    assert np.array_equal(host(b.ids), ids_ref)
    ids = torch.empty((T, wl.k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, wl.k), dtype=torch.float32, device="cuda")
    B.luce_route_topk(dev(L.logits), dev(L.bias), wl.k, ids, w)
    torch.cuda.synchronize()
    assert np.array_equal(host(ids), ids_ref)
    for name in ("counts", "offsets", "routes"):
        assert torch.equal(getattr(a, name), getattr(b, name))
