"""Helpers of the GPU parity tests: device upload, oracle comparison rules.

Comparison rules (the pages' grading, made concrete):
* integer outputs (ids, counts, offsets, routes, argmax index, q8_1 codes of
  identical inputs) are compared bit for bit;
* float outputs satisfy |gpu - oracle| <= 1e-4 * terms + 1e-6, with the
  error scale `terms` the oracle computes for each output;
* q8_1 blocks quantized from a value the GPU computed itself (h) may differ
  from the oracle's quantization only where the oracle marks the element as
  unstable (``oracle.hq_flip_allowance``); every other byte is identical.
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


def assert_hq_valid(hq_gpu, hq_ref, allow, what="hq"):
    """hq blocks [rows, nb, 36]: equal bytes wherever the quantization is stable,
    dequantized difference within the allowance elsewhere.  Returns the number
    of differing codes."""
    hq_gpu = np.asarray(hq_gpu, np.uint8)
    hq_ref = np.asarray(hq_ref, np.uint8)
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


def dequant_q8_0_abs(w):
    """|d * q| of Q8_0 blocks [..., nb, 34] as float64 [..., nb*32]."""
    d = w[..., 0:2].copy().view(np.float16)[..., 0].astype(np.float64)
    q = w[..., 2:].view(np.int8).astype(np.float64)
    return np.abs(q * d[..., None]).reshape(w.shape[:-2] + (-1,))


def chain_allowance(wd, wsd, ids, weights, h_allow):
    """Bound on |out_gpu - out_oracle| added by q8_1(h) flips: for each token t
    and row n, sum_j |w_j| * sum_i |Wd[e_j][n][i]| * allow[r_j][i] (+ shared)."""
    T, k = ids.shape
    H = wd.shape[1]
    out = np.zeros((T, H))
    for t in range(T):
        for j in range(k):
            e = ids[t, j]
            if e < 0:
                continue
            a = h_allow[t * k + j]
            if a.any():
                out[t] += abs(float(weights[t, j])) * (dequant_q8_0_abs(wd[e]) @ a)
        if wsd is not None:
            a = h_allow[T * k + t]
            if a.any():
                out[t] += dequant_q8_0_abs(wsd) @ a
    return out * 1.001
