"""Seeded synthetic inputs for the routed NVFP4 SiTU MoE forward.

This module is the one place that draws random inputs.  It serves the CUDA
path (benchmark, smoke check) and the tests of the CPU oracle alike, and it
holds none of the method's arithmetic: no quantizer, no routing, no GEMM.
Inputs that the pages define in the quantized domain (packed E2M1 codes, E4M3
block-scale bytes) are drawn directly as bytes.  Tensors that must first be
quantized (the tiny case's fp32 weights) are returned as fp32 and quantized
by whoever consumes them.

Generator: numpy PCG64 through ``default_rng([seed, tag])``, one stream per
tensor so that no input depends on the order of draws.

Workloads (shapes and distributions of the pages' cases; all synthetic):

* ``tiny``     T=16, H=512, I=128, E=32, k=4; x ~ N(0,1) bf16; 4 distinct
               uniform experts per row; route weights bf16(softmax(N(0,1)^4));
               W13 [32,256,512], W2 [32,512,128] fp32 ~ N(0, 0.02).
* ``routing``  NUM_ROWS=4096, K=16, E=896, H=3584; x ~ N(0,1) bf16, uniform
               distinct ids (init-routing alone, dropless and drop/pad C=96).
* ``decode``   H=3584, I=384, E=896, k=16, T in {1, 8, 16}; uniform distinct ids.
* ``prefill``  T=4096, ids drawn without replacement from Zipf(s=1.1) over a
               seeded permutation of the experts (Gumbel-top-k).
* ``maxbatch`` T=16384, uniform distinct ids, 1% of rows of x scaled by 50.

Full-shape NVFP4 weights: codes are uniform random bytes (every E2M1 nibble
equally likely); W13 block scales are E4M3 bytes uniform over codes 0x08..0x27
(2^-6 .. 0.234) and W2 block scales uniform over 0x50..0x77 (8 .. 240), chosen
so that FC1 pre-activations span SiTU's interior and saturation and the
outputs are O(0.1-1).  Per-expert dX*dW13, qA and dA*dW2 are log-uniform in
[1e-4, 1e-2]; qX = 1/dX with dX = amax(x)/(6*448).
"""
from __future__ import annotations

import dataclasses

import numpy as np

FULL = dict(H=3584, I=384, E=896, k=16)
TINY = dict(H=512, I=128, E=32, k=4)

# tensor tags: each tensor gets its own stream default_rng([seed, tag])
_TAG = dict(x=1, ids=2, route=3, w13=4, w2=5, sf13=6, sf2=7, s13=8, sqa=9, s2=10,
            big_rows=11, zipf_perm=12, beta=13, lam=14)


def rng(seed: int, tag: str) -> np.random.Generator:
    return np.random.default_rng([seed, _TAG[tag]])


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest even) and return the raw 16-bit patterns."""
    u = np.ascontiguousarray(a, np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16).astype(np.uint16)
    return r


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32)


def draw_x(seed: int, T: int, H: int, big_rows_frac: float = 0.0, big_scale: float = 50.0) -> np.ndarray:
    """x ~ N(0,1) as bf16 bits [T, H]; optionally floor(T*frac) rows x big_scale."""
    x = rng(seed, "x").standard_normal((T, H), dtype=np.float32)
    nbig = int(T * big_rows_frac)
    if nbig > 0:
        rows = rng(seed, "big_rows").choice(T, size=nbig, replace=False)
        x[rows] *= np.float32(big_scale)
    return f32_to_bf16_bits(x)


def draw_ids_uniform(seed: int, T: int, E: int, k: int) -> np.ndarray:
    """k distinct experts per row, uniformly (first k of a random ordering)."""
    keys = rng(seed, "ids").random((T, E))
    return np.argsort(keys, axis=1, kind="stable")[:, :k].astype(np.int32)


def draw_ids_zipf(seed: int, T: int, E: int, k: int, s: float = 1.1) -> np.ndarray:
    """k distinct experts per row drawn without replacement with probability
    proportional to Zipf(s) over a seeded permutation of the experts
    (Gumbel-top-k)."""
    perm = rng(seed, "zipf_perm").permutation(E)
    logp = np.empty(E, np.float64)
    logp[perm] = -s * np.log(np.arange(1, E + 1, dtype=np.float64))
    g = rng(seed, "ids").gumbel(size=(T, E))
    keys = logp[None, :] + g
    return np.argsort(-keys, axis=1, kind="stable")[:, :k].astype(np.int32)


def draw_route_weights(seed: int, T: int, k: int) -> np.ndarray:
    """bf16(softmax over k N(0,1) logits) as bf16 bits [T, k]."""
    lg = rng(seed, "route").standard_normal((T, k))
    p = np.exp(lg - lg.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    return f32_to_bf16_bits(p.astype(np.float32))


def qx_for(x_bits: np.ndarray) -> np.float32:
    """qX = 1/dX with dX = amax(x)/(6*448), in fp32."""
    amax = np.float32(np.abs(bf16_bits_to_f32(x_bits)).max())
    dX = np.float32(amax / np.float32(6 * 448))
    return np.float32(np.float32(1.0) / dX)


def log_uniform(seed: int, tag: str, n: int, lo: float = 1e-4, hi: float = 1e-2) -> np.ndarray:
    u = rng(seed, tag).random(n)
    return np.exp(np.log(lo) + u * (np.log(hi) - np.log(lo))).astype(np.float32)


def draw_nvfp4_weights(seed: int, E: int, rows: int, K: int, which: str):
    """Packed codes [E, rows, K/2] (uniform bytes) and E4M3 block scales
    [E, rows, K/16] (uniform over a code range) in the canonical layout."""
    codes = rng(seed, which).integers(0, 256, size=(E, rows, K // 2), dtype=np.uint8)
    lo, hi = (0x08, 0x27) if which == "w13" else (0x50, 0x77)
    sf = rng(seed, "sf13" if which == "w13" else "sf2").integers(lo, hi + 1, size=(E, rows, K // 16),
                                                                 dtype=np.uint8)
    return codes, sf


@dataclasses.dataclass
class MoEInputs:
    H: int
    I: int
    E: int
    k: int
    T: int
    x: np.ndarray            # [T, H] bf16 bits
    expert_ids: np.ndarray   # [T, k] int32
    route_weights: np.ndarray  # [T, k] bf16 bits
    qX: np.float32
    w13: np.ndarray | None = None     # [E, 2I, H/2] u8 (canonical)
    sf13: np.ndarray | None = None    # [E, 2I, H/16] u8
    w2: np.ndarray | None = None      # [E, H, I/2] u8
    sf2: np.ndarray | None = None     # [E, H, I/16] u8
    dXdW13: np.ndarray | None = None  # [E] f32
    qA: np.ndarray | None = None      # [E] f32
    dAdW2: np.ndarray | None = None   # [E] f32
    w13_f32: np.ndarray | None = None  # tiny case only: [E, 2I, H] fp32 before quantization
    w2_f32: np.ndarray | None = None   # tiny case only: [E, H, I] fp32


def tiny(seed: int = 0, T: int = 16) -> MoEInputs:
    """The tiny case; weights come back as fp32 (the consumer quantizes)."""
    return small(seed, T, **TINY)


def small(seed: int, T: int, H: int, I: int, E: int, k: int) -> MoEInputs:
    """A small case of any shape, drawn like the tiny one (fp32 weights)."""
    x = draw_x(seed, T, H)
    ids = draw_ids_uniform(seed, T, E, k)
    rw = draw_route_weights(seed, T, k)
    w13 = (rng(seed, "w13").standard_normal((E, 2 * I, H), dtype=np.float32) * np.float32(0.02))
    w2 = (rng(seed, "w2").standard_normal((E, H, I), dtype=np.float32) * np.float32(0.02))
    return MoEInputs(H, I, E, k, T, x, ids, rw, qx_for(x), w13_f32=w13, w2_f32=w2)


def full(seed: int = 0, T: int = 16, routing: str = "uniform", big_rows_frac: float = 0.0,
         weights: bool = True, E: int | None = None) -> MoEInputs:
    """A full-shape case (H=3584, I=384, E=896, k=16) with weights drawn
    directly as NVFP4 codes and block scales."""
    H, I, k = FULL["H"], FULL["I"], FULL["k"]
    E = E or FULL["E"]
    x = draw_x(seed, T, H, big_rows_frac)
    if routing == "uniform":
        ids = draw_ids_uniform(seed, T, E, k)
    elif routing == "zipf":
        ids = draw_ids_zipf(seed, T, E, k)
    else:
        raise ValueError(routing)
    rw = draw_route_weights(seed, T, k)
    inp = MoEInputs(H, I, E, k, T, x, ids, rw, qx_for(x))
    if weights:
        inp.w13, inp.sf13 = draw_nvfp4_weights(seed, E, 2 * I, H, "w13")
        inp.w2, inp.sf2 = draw_nvfp4_weights(seed, E, H, I, "w2")
    inp.dXdW13 = log_uniform(seed, "s13", E)
    inp.qA = log_uniform(seed, "sqa", E)
    inp.dAdW2 = log_uniform(seed, "s2", E)
    return inp


WORKLOADS = {
    "decode1": dict(T=1, routing="uniform"),
    "decode8": dict(T=8, routing="uniform"),
    "decode16": dict(T=16, routing="uniform"),
    "prefill": dict(T=4096, routing="zipf"),
    "maxbatch": dict(T=16384, routing="uniform", big_rows_frac=0.01),
}
SWEEP_T = (32, 128, 512, 1024, 2048, 8192)
