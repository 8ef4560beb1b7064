"""Seeded synthetic inputs of the MoE decode workloads.

This module only draws random inputs and packs them into the block layouts;
it holds none of the method's arithmetic.  Both the CUDA path (tests, bench)
and the CPU oracle (tests) take their inputs from here.

Workloads (sizes of the Lucebox DS4.1 serving pages' decode/verify path; the
pages publish no dataset and none is used):

* ``tiny``           one expert, gate/up 256 x 512, down 512 x 256, 1 token;
                     argmax over 4096 logits.  Seed 0.
* ``decode_layer``   T=1, H=2048, I=1024, E=64 routed + 1 shared, top-6,
                     unclamped SwiGLU, router bias ~ N(0, 0.1).  Seed 1.
* ``verify_layer``   T=5 (1 + 4 draft tokens), H=4096, I=2048, E=128 + 1
                     shared, top-8, SwiGLU clamped at 10, argmax over
                     5 x 129280 logits; logits share a per-expert mean across
                     columns so that columns share experts.  Seed 2.
* ``decode_stack43`` 43 resident decode_layer layers, 1 token per step,
                     64 pre-drawn steps, logits skewed by a Zipf(1.1) offset
                     per expert.  Seed 3.
* ``prefill_layer``  T=512, H=4096, I=1536, E=128 + 1 shared, top-8, clamped
                     SwiGLU.  Seed 4.

Weights are drawn directly as Q8_0 blocks: int8 codes uniform in [-127, 127]
and an fp16 scale uniform in [1e-3, 2e-2].  Activations are N(0, 1) fp32.
Router logits are redrawn per token until the gap between the k-th and the
(k+1)-th selection score is at least 1e-5.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

QK = 32
Q8_0_BYTES = 34
Q8_1_BYTES = 36
TOPK_MARGIN = 1e-5


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    H: int
    I: int
    E: int
    k: int
    shared: bool
    clamp: float
    seed: int
    logits: str = "normal"          # normal | shared_col | zipf | single
    bias_std: float = 0.0
    V: int = 0                      # argmax vocabulary (0: none)
    R: int = 0                      # argmax rows
    layers: int = 1
    steps: int = 1

    @property
    def q8_0_row_bytes_gate(self) -> int:
        return self.H // QK * Q8_0_BYTES

    @property
    def q8_0_row_bytes_down(self) -> int:
        return self.I // QK * Q8_0_BYTES

    @property
    def expert_bytes(self) -> int:
        """Q8_0 bytes of one expert's gate + up + down."""
        return 2 * self.I * self.q8_0_row_bytes_gate + self.H * self.q8_0_row_bytes_down


WORKLOADS = {
    "tiny": Workload("tiny", T=1, H=512, I=256, E=1, k=1, shared=False, clamp=0.0, seed=0,
                     logits="single", V=4096, R=1),
    "decode_layer": Workload("decode_layer", T=1, H=2048, I=1024, E=64, k=6, shared=True, clamp=0.0,
                             seed=1, logits="normal", bias_std=0.1),
    "verify_layer": Workload("verify_layer", T=5, H=4096, I=2048, E=128, k=8, shared=True, clamp=10.0,
                             seed=2, logits="shared_col", V=129280, R=5),
    "decode_stack43": Workload("decode_stack43", T=1, H=2048, I=1024, E=64, k=6, shared=True, clamp=0.0,
                               seed=3, logits="zipf", bias_std=0.1, layers=43, steps=64),
    "prefill_layer": Workload("prefill_layer", T=512, H=4096, I=1536, E=128, k=8, shared=True, clamp=10.0,
                              seed=4, logits="normal"),
}


# ----------------------------------------------------------------------------- host (numpy)
def rng(seed: int, stream: int = 0) -> np.random.Generator:
    """Independent, reproducible numpy stream per (seed, stream)."""
    return np.random.default_rng(np.random.SeedSequence([seed, stream]))


def q8_0_blocks(g: np.random.Generator, rows: int, K: int) -> np.ndarray:
    """Random Q8_0 weight rows: uint8 [rows, K/32, 34] (fp16 d, then 32 int8)."""
    assert K % QK == 0
    nb = K // QK
    qs = g.integers(-127, 128, size=(rows, nb, QK), dtype=np.int8)
    d = g.uniform(1e-3, 2e-2, size=(rows, nb)).astype(np.float16)
    out = np.empty((rows, nb, Q8_0_BYTES), np.uint8)
    out[..., 0:2] = d.view(np.uint8).reshape(rows, nb, 2)
    out[..., 2:] = qs.view(np.uint8)
    return out


Q4_K_BYTES = 144
QK_K = 256


def q4_k_blocks(g: np.random.Generator, rows: int, K: int) -> np.ndarray:
    """Random Q4_K weight rows: uint8 [rows, K/256, 144] (fp16 d and dmin,
    12 bytes of packed 6-bit scales and mins, 128 bytes of 4-bit codes; every
    byte pattern of the scales and codes is a valid block)."""
    assert K % QK_K == 0
    nb = K // QK_K
    out = np.empty((rows, nb, Q4_K_BYTES), np.uint8)
    d = g.uniform(1e-4, 2e-3, size=(rows, nb)).astype(np.float16)
    dmin = g.uniform(1e-4, 2e-3, size=(rows, nb)).astype(np.float16)
    out[..., 0:2] = d.view(np.uint8).reshape(rows, nb, 2)
    out[..., 2:4] = dmin.view(np.uint8).reshape(rows, nb, 2)
    out[..., 4:] = g.integers(0, 256, size=(rows, nb, Q4_K_BYTES - 4), dtype=np.uint8)
    return out


def host_layer_q4k(wl: Workload) -> HostLayer:
    """A whole layer with Q4_K expert weights (H and I multiples of 256)."""
    assert wl.H % QK_K == 0 and wl.I % QK_K == 0
    gw = rng(wl.seed, 11)
    wg = q4_k_blocks(gw, wl.E * wl.I, wl.H).reshape(wl.E, wl.I, wl.H // QK_K, Q4_K_BYTES)
    wu = q4_k_blocks(gw, wl.E * wl.I, wl.H).reshape(wl.E, wl.I, wl.H // QK_K, Q4_K_BYTES)
    wd = q4_k_blocks(gw, wl.E * wl.H, wl.I).reshape(wl.E, wl.H, wl.I // QK_K, Q4_K_BYTES)
    wsg = wsu = wsd = None
    if wl.shared:
        wsg = q4_k_blocks(gw, wl.I, wl.H)
        wsu = q4_k_blocks(gw, wl.I, wl.H)
        wsd = q4_k_blocks(gw, wl.H, wl.I)
    x = activations(rng(wl.seed, 2), wl.T, wl.H)
    logits, bias = router_logits(rng(wl.seed, 3), wl)
    return HostLayer(wl, wg, wu, wd, wsg, wsu, wsd, x, logits, bias, None)


def activations(g: np.random.Generator, T: int, H: int) -> np.ndarray:
    return g.standard_normal((T, H), dtype=np.float32)


def _scores32(logits: np.ndarray, bias) -> np.ndarray:
    return logits if bias is None else (logits + bias[None, :]).astype(np.float32)


def _enforce_margin(draw, bias, k: int, E: int) -> np.ndarray:
    """Draw a token's logits until the k-th/(k+1)-th score gap is >= 1e-5."""
    for _ in range(1000):
        l = draw()
        if k >= E:
            return l
        s = np.sort(_scores32(l[None, :], bias)[0])[::-1]
        if float(s[k - 1]) - float(s[k]) >= TOPK_MARGIN:
            return l
    raise RuntimeError("could not draw router logits with the top-k margin")


def router_logits(g: np.random.Generator, wl: Workload, T: int | None = None, layer: int = 0):
    """(logits f32 [T, E], bias f32 [E] or None) for one layer of a workload."""
    T = wl.T if T is None else T
    E, k = wl.E, wl.k
    bias = None
    if wl.bias_std > 0:
        bias = (g.standard_normal(E) * wl.bias_std).astype(np.float32)
    if wl.logits == "single":
        return np.zeros((T, E), np.float32), bias
    base = np.zeros(E, np.float64)
    scale = 1.0
    if wl.logits == "shared_col":
        base = g.standard_normal(E)
        scale = 0.75
    elif wl.logits == "zipf":
        # per layer, a seeded ranking r_e = 1..E of the experts; offset -1.1 ln r
        # makes exp(offset) proportional to r^-1.1 (hot and cold experts)
        rank = g.permutation(E) + 1
        base = -1.1 * np.log(rank.astype(np.float64))
    rows = []
    for _ in range(T):
        rows.append(_enforce_margin(
            lambda: (base + scale * g.standard_normal(E)).astype(np.float32), bias, k, E))
    return np.stack(rows).astype(np.float32), bias


def vocab_logits(g: np.random.Generator, R: int, V: int) -> np.ndarray:
    return g.standard_normal((R, V), dtype=np.float32)


@dataclass
class HostLayer:
    """One MoE layer's weights and inputs on the host (numpy)."""
    wl: Workload
    wg: np.ndarray
    wu: np.ndarray
    wd: np.ndarray
    wsg: np.ndarray | None
    wsu: np.ndarray | None
    wsd: np.ndarray | None
    x: np.ndarray
    logits: np.ndarray
    bias: np.ndarray | None
    vocab: np.ndarray | None = None


def host_layer(wl: Workload, T: int | None = None, E: int | None = None, seed: int | None = None) -> HostLayer:
    """Draw a whole layer on the host (small workloads only)."""
    if E is not None or T is not None:
        wl = Workload(**{**wl.__dict__, "E": E if E is not None else wl.E, "T": T if T is not None else wl.T})
    seed = wl.seed if seed is None else seed
    gw = rng(seed, 1)
    wg = q8_0_blocks(gw, wl.E * wl.I, wl.H).reshape(wl.E, wl.I, wl.H // QK, Q8_0_BYTES)
    wu = q8_0_blocks(gw, wl.E * wl.I, wl.H).reshape(wl.E, wl.I, wl.H // QK, Q8_0_BYTES)
    wd = q8_0_blocks(gw, wl.E * wl.H, wl.I).reshape(wl.E, wl.H, wl.I // QK, Q8_0_BYTES)
    wsg = wsu = wsd = None
    if wl.shared:
        wsg = q8_0_blocks(gw, wl.I, wl.H)
        wsu = q8_0_blocks(gw, wl.I, wl.H)
        wsd = q8_0_blocks(gw, wl.H, wl.I)
    gx = rng(seed, 2)
    x = activations(gx, wl.T, wl.H)
    logits, bias = router_logits(rng(seed, 3), wl)
    vocab = vocab_logits(rng(seed, 4), wl.R, wl.V) if wl.V else None
    return HostLayer(wl, wg, wu, wd, wsg, wsu, wsd, x, logits, bias, vocab)


# ----------------------------------------------------------------------------- device (torch)
def q8_0_blocks_torch(gen, rows: int, K: int, device):
    """Random Q8_0 rows drawn on `device` with a seeded torch.Generator.

    Same distribution as :func:`q8_0_blocks` (a different random stream).
    Returns a uint8 tensor [rows, K/32, 34].
    """
    import torch
    nb = K // QK
    out = torch.empty((rows, nb, Q8_0_BYTES), dtype=torch.uint8, device=device)
    chunk = max(1, (1 << 26) // (nb * QK))
    for r0 in range(0, rows, chunk):
        r1 = min(rows, r0 + chunk)
        n = r1 - r0
        qs = torch.randint(-127, 128, (n, nb, QK), dtype=torch.int8, device=device, generator=gen)
        d = (torch.rand((n, nb), device=device, generator=gen) * (2e-2 - 1e-3) + 1e-3).to(torch.float16)
        out[r0:r1, :, 0:2] = d.view(torch.uint8).view(n, nb, 2)
        out[r0:r1, :, 2:] = qs.view(torch.uint8)
    return out


@dataclass
class DeviceLayer:
    """One layer's Q8_0 weights resident on the GPU (torch uint8 tensors)."""
    wg: object
    wu: object
    wd: object
    wsg: object = None
    wsu: object = None
    wsd: object = None
    extra: dict = field(default_factory=dict)


def device_layer(wl: Workload, seed: int, device) -> DeviceLayer:
    import torch
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    wg = q8_0_blocks_torch(gen, wl.E * wl.I, wl.H, device).view(wl.E, wl.I, wl.H // QK, Q8_0_BYTES)
    wu = q8_0_blocks_torch(gen, wl.E * wl.I, wl.H, device).view(wl.E, wl.I, wl.H // QK, Q8_0_BYTES)
    wd = q8_0_blocks_torch(gen, wl.E * wl.H, wl.I, device).view(wl.E, wl.H, wl.I // QK, Q8_0_BYTES)
    lay = DeviceLayer(wg, wu, wd)
    if wl.shared:
        lay.wsg = q8_0_blocks_torch(gen, wl.I, wl.H, device)
        lay.wsu = q8_0_blocks_torch(gen, wl.I, wl.H, device)
        lay.wsd = q8_0_blocks_torch(gen, wl.H, wl.I, device)
    return lay


def touched_weight_bytes(wl: Workload, n_active_routed: int) -> int:
    """Expert-weight bytes one layer reads: the active routed experts + shared."""
    n = n_active_routed + (1 if wl.shared else 0)
    return n * wl.expert_bytes


def floor_us(nbytes: int, gbs: float) -> float:
    return nbytes / (gbs * 1e9) * 1e6


__all__ = ["Workload", "WORKLOADS", "rng", "q8_0_blocks", "activations", "router_logits", "vocab_logits",
           "host_layer", "HostLayer", "q8_0_blocks_torch", "device_layer", "DeviceLayer",
           "touched_weight_bytes", "floor_us"]
