"""Helpers of the GPU parity tests: device upload, oracle comparison rules.

Comparison rules (the pages' grading, made concrete):
* integer outputs (ids, counts, offsets, routes, argmax index, q8_1 codes of
  identical inputs) are compared bit for bit;
* float outputs satisfy |gpu - oracle| <= 1e-4 * terms + 1e-6, with the
  error scale `terms` the oracle computes for each output;
* q8_1 blocks quantized from a value the GPU computed itself (h) may differ
  from the oracle's quantization of the oracle's h only where the oracle
  marks the element as unstable (``oracle.hq_flip_allowance``) and by no
  more than the allowance; every other byte is identical.  They are also,
  byte for byte, the library's q8_1 kernel applied to the h the GPU stored
  (that kernel is checked bit for bit against the oracle on oracle inputs),
  so the fused quantization is the rule itself and not a near copy of it.
"""
import numpy as np
import torch

import oracle


def dev(a, device="cuda"):
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def host(t):
    return t.detach().cpu().numpy()


def assert_close(gpu, ref, terms, what=""):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    bound = oracle.tol(terms)
    err = np.abs(gpu - ref)
    bad = ~(err <= bound)
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outside tolerance; first at {tuple(i)}: "
                             f"gpu={gpu[tuple(i)]!r} oracle={ref[tuple(i)]!r} bound={bound[tuple(i)]!r}")
    return float((err / np.maximum(bound, 1e-300)).max()) if err.size else 0.0


def assert_hq_valid(hq_gpu, hq_ref, allow, what="hq", h_gpu=None):
    """hq blocks [rows, nb, 36]: equal bytes wherever the quantization is stable,
    dequantized difference within the allowance elsewhere; with the GPU's own h
    rows [rows, I] given, also bit-equal to the q8_1 kernel's output for them.
    Returns the number of codes that differ from hq_ref."""
    hq_gpu = np.asarray(hq_gpu, np.uint8)
    hq_ref = np.asarray(hq_ref, np.uint8)
    if h_gpu is not None:
        assert_hq_is_rule_of_h(hq_gpu, h_gpu, what)
    dg = oracle.dequant_q8_1(hq_gpu).astype(np.float64)
    dr = oracle.dequant_q8_1(hq_ref).astype(np.float64)
    allow = np.asarray(allow, np.float64).reshape(dg.shape)
    diff = np.abs(dg - dr)
    assert np.all(diff <= allow + 1e-30), f"{what}: dequantized values differ beyond the flip allowance"
    blk_unstable = (allow.reshape(hq_gpu.shape[:-1] + (32,)) > 0).any(axis=-1)
    stable = ~blk_unstable
    assert np.array_equal(hq_gpu[stable], hq_ref[stable]), f"{what}: stable blocks differ"
    codes_g = hq_gpu[..., 4:].view(np.int8)
    codes_r = hq_ref[..., 4:].view(np.int8)
    return int((codes_g != codes_r).sum())


def assert_hq_is_rule_of_h(hq_gpu, h_gpu, what="hq"):
    """hq [rows, nb, 36] equals luce_quantize_q8_1 of the h rows [rows, I]."""
    from quantized_moe_decode_luce_gb300 import binding as B
    h = dev(np.asarray(h_gpu, np.float32).reshape(-1, np.shape(h_gpu)[-1]))
    q = torch.empty((h.shape[0], h.shape[1] // 32, 36), dtype=torch.uint8, device=h.device)
    B.luce_quantize_q8_1(h, q)
    own = host(q)
    assert np.array_equal(np.asarray(hq_gpu, np.uint8).reshape(own.shape), own), \
        f"{what}: not the q8_1 rule applied to the h the GPU stored"


def dequant_q8_0_abs(w):
    """|d * q| of Q8_0 blocks [..., nb, 34] as float64 [..., nb*32]."""
    d = w[..., 0:2].copy().view(np.float16)[..., 0].astype(np.float64)
    q = w[..., 2:].view(np.int8).astype(np.float64)
    return np.abs(q * d[..., None]).reshape(w.shape[:-2] + (-1,))


def chain_allowance(wd, wsd, ids, weights, h_allow):
    """Bound on |out_gpu - out_oracle| added by q8_1(h) flips: for each token t
    and row n, sum_j |w_j| * sum_i |Wd[e_j][n][i]| * allow[r_j][i] (+ shared).
    Grouped by expert, so each expert's |Wd| is expanded once."""
    T, k = ids.shape
    H = wd.shape[1]
    out = np.zeros((T, H))
    h_allow = np.asarray(h_allow, np.float64)
    for e in np.unique(ids[ids >= 0]):
        ts, js = np.nonzero(ids == e)
        a = h_allow[ts * k + js] * np.abs(np.asarray(weights, np.float64)[ts, js])[:, None]
        live = a.any(axis=1)
        if live.any():
            np.add.at(out, ts[live], a[live] @ dequant_q8_0_abs(wd[e]).T)
    if wsd is not None:
        a = h_allow[T * k:T * k + T]
        if a.any():
            out += a @ dequant_q8_0_abs(wsd).T
    return out * 1.001
