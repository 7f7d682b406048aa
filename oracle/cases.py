"""Preparation of the tiny case through the oracle -- TEST INFRASTRUCTURE.

The tiny case draws fp32 weights (in ``nvfp4_routed_moe_gb300.inputs``); this
module quantizes them with the oracle's NVFP4 quantizer and calibrates the
per-expert scales, so that both the oracle and the CUDA path receive the same
quantized inputs.  Calibration follows the "Cake SiTU backend" page: qX = 1/dX,
qA = 1/dA, and a shared intermediate scale expanded to one entry per expert.
The amax-based choice dX = amax/(6*448) is the tiny case's own recipe; the same
rule is used for the weight global scales dW[e] and for dA (from the oracle's
own fp32 SiTU outputs, with a provisional qA that does not affect them).
"""
from __future__ import annotations

import numpy as np

import oracle
from nvfp4_routed_moe_gb300 import inputs as gen

_FP4_E4M3_MAX = np.float32(6 * 448)


def quantize_expert_weights(w_f32: np.ndarray):
    """Per-expert NVFP4 quantization of [E, rows, K] fp32: returns packed
    codes [E, rows, K/2], E4M3 scales [E, rows, K/16], dW [E] (fp32)."""
    E, rows, K = w_f32.shape
    amax = np.abs(w_f32).reshape(E, -1).max(axis=1).astype(np.float32)
    dW = (amax / _FP4_E4M3_MAX).astype(np.float32)
    qW = (np.float32(1.0) / dW).astype(np.float32)
    q_rows = np.repeat(qW, rows)
    packed, sf = oracle.nvfp4_quant_rows(w_f32.reshape(E * rows, K), q_per_row=q_rows)
    return packed.reshape(E, rows, K // 2), sf.reshape(E, rows, K // 16), dW


def prepare_tiny(seed: int = 0, T: int = 16) -> gen.MoEInputs:
    return prepare(gen.tiny(seed, T))


def prepare_small(seed: int, T: int, H: int, I: int, E: int, k: int) -> gen.MoEInputs:
    """A small case of another shape, prepared like the tiny one."""
    return prepare(gen.small(seed, T, H, I, E, k))


def prepare(inp: gen.MoEInputs) -> gen.MoEInputs:
    T = inp.T
    inp.w13, inp.sf13, dW13 = quantize_expert_weights(inp.w13_f32)
    inp.w2, inp.sf2, dW2 = quantize_expert_weights(inp.w2_f32)
    dX = np.float32(np.float32(1.0) / inp.qX)
    inp.dXdW13 = (dX * dW13).astype(np.float32)
    # provisional qA: SiTU outputs do not depend on it
    ones = np.ones(inp.E, np.float32)
    _, mid = oracle.moe_forward_tokens(H=inp.H, I=inp.I, E=inp.E, k=inp.k, x=inp.x, expert_ids=inp.expert_ids,
                                       route_weights=inp.route_weights, tokens=np.arange(T),
                                       w13=inp.w13, sf13=inp.sf13, w2=inp.w2, sf2=inp.sf2, qX=inp.qX,
                                       dXdW13=inp.dXdW13, qA=ones, dAdW2=ones, want_intermediates=True)
    amax_a = np.float32(np.abs(mid["a"]).max())
    dA = np.float32(amax_a / _FP4_E4M3_MAX)
    inp.qA = np.full(inp.E, np.float32(1.0) / dA, np.float32)
    inp.dAdW2 = (dA * dW2).astype(np.float32)
    return inp


def run_oracle(inp: gen.MoEInputs, tokens=None, beta=None, lam=None, want_intermediates=False):
    toks = np.arange(inp.T) if tokens is None else np.asarray(tokens)
    return oracle.moe_forward_tokens(H=inp.H, I=inp.I, E=inp.E, k=inp.k, x=inp.x, expert_ids=inp.expert_ids,
                                     route_weights=inp.route_weights, tokens=toks, w13=inp.w13, sf13=inp.sf13,
                                     w2=inp.w2, sf2=inp.sf2, qX=inp.qX, dXdW13=inp.dXdW13, qA=inp.qA,
                                     dAdW2=inp.dAdW2, beta=beta, lam=lam, want_intermediates=want_intermediates)
