"""Helpers for the GPU tests: move generator inputs to the device, prepare
weights and workspace, run moe_forward through the C ABI, compare with the
oracle.  All compute goes through nvfp4_routed_moe_gb300.api."""
from __future__ import annotations

import numpy as np
import torch

from nvfp4_routed_moe_gb300 import api
from nvfp4_routed_moe_gb300 import inputs as gen

TOL_MAX_ABS = 2e-2
TOL_REL_L2 = 1e-2


def dev(a: np.ndarray, dtype=None) -> torch.Tensor:
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    t = torch.from_numpy(a)
    if dtype is not None:
        t = t.view(dtype)
    return t.cuda()


class Model:
    """Prepared weights and per-expert scales of one MoEInputs on the GPU."""

    def __init__(self, inp: gen.MoEInputs):
        self.inp = inp
        self.shape = api.shape(inp.H, inp.I, inp.E, inp.k)
        sizes = api.moe_prepared_weight_bytes(self.shape)
        w13, sf13, w2, sf2 = (dev(inp.w13), dev(inp.sf13), dev(inp.w2), dev(inp.sf2))
        assert [t.numel() for t in (w13, sf13, w2, sf2)] == list(sizes)
        self.w13 = torch.empty(sizes[0], dtype=torch.uint8, device="cuda")
        self.sf13 = torch.empty(sizes[1], dtype=torch.uint8, device="cuda")
        self.w2 = torch.empty(sizes[2], dtype=torch.uint8, device="cuda")
        self.sf2 = torch.empty(sizes[3], dtype=torch.uint8, device="cuda")
        api.moe_prepare_weights(self.shape, w13, sf13, w2, sf2, self.w13, self.sf13, self.w2, self.sf2)
        torch.cuda.synchronize()
        del w13, sf13, w2, sf2
        self.qX = dev(np.array([inp.qX], np.float32))
        self.dXdW13 = dev(inp.dXdW13)
        self.qA = dev(inp.qA)
        self.dAdW2 = dev(inp.dAdW2)

    def workspace(self, max_tokens: int) -> torch.Tensor:
        n = api.moe_workspace_size(self.shape, max_tokens)
        return torch.empty(n, dtype=torch.uint8, device="cuda")

    def forward(self, x, ids, rw, ws=None, T=None, beta=None, lam=None, out=None, prepare=True, qX=None):
        T = T if T is not None else x.shape[0]
        qX = self.qX if qX is None else qX
        if ws is None:
            ws = self.workspace(T)
        if prepare:
            api.moe_prepare_workspace(self.shape, ws, T)
        if out is None:
            out = torch.empty((T, self.inp.H), dtype=torch.bfloat16, device="cuda")
        api.moe_forward(self.shape, T, x, ids, rw, self.w13, self.sf13, self.w2, self.sf2, qX, self.dXdW13,
                        self.qA, self.dAdW2, beta, lam, ws, out)
        return out, ws

    def forward_inputs(self, inp: gen.MoEInputs | None = None, **kw):
        """Forward of `inp`'s activations, routing and qX (weights and
        per-expert scales are the model's)."""
        inp = inp or self.inp
        x = dev(inp.x, torch.bfloat16)
        ids = dev(inp.expert_ids)
        rw = dev(inp.route_weights, torch.bfloat16)
        kw.setdefault("qX", dev(np.array([inp.qX], np.float32)))
        return self.forward(x, ids, rw, **kw)


def out_bits(out: torch.Tensor) -> np.ndarray:
    return out.view(torch.int16).cpu().numpy().view(np.uint16)


def bf16_ulp(v: np.ndarray) -> np.ndarray:
    """Spacing of BF16 values at |v| (8 significant bits; 2^-133 below the
    normal range)."""
    a = np.abs(v.astype(np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return 2.0 ** (e - 7)


def compare(got_bits: np.ndarray, ref_bits: np.ndarray):
    """(max_abs, rel_l2, excess) between two bf16 bit arrays; excess is the
    largest |got - ref| / max(TOL_MAX_ABS, one BF16 ulp of ref)."""
    g = gen.bf16_bits_to_f32(got_bits).astype(np.float64)
    r = gen.bf16_bits_to_f32(ref_bits).astype(np.float64)
    d = np.abs(g - r)
    max_abs = float(d.max()) if g.size else 0.0
    excess = float((d / np.maximum(TOL_MAX_ABS, bf16_ulp(r))).max()) if g.size else 0.0
    den = float(np.sqrt((r ** 2).sum()))
    rel = float(np.sqrt(((g - r) ** 2).sum()) / den) if den > 0 else float(np.sqrt((g ** 2).sum()))
    return max_abs, rel, excess


def assert_close(got_bits, ref_bits, what=""):
    """The forward's tolerance: relative L2 error <= 1e-2 and, per element,
    |got - ref| <= max(2e-2, one BF16 ulp of ref).  Above magnitude 4 the
    BF16 spacing itself exceeds 2e-2, and two fp32 sums that differ only in
    the order of their additions (hardware accumulation against the oracle's
    fp64 sum) can round to neighbouring BF16 values there; one ulp is the
    least any BF16 result can be held to."""
    max_abs, rel, excess = compare(got_bits, ref_bits)
    assert np.isfinite(gen.bf16_bits_to_f32(got_bits)).all(), f"{what}: non-finite output"
    assert excess <= 1.0 and rel <= TOL_REL_L2, f"{what}: max_abs={max_abs:.3g} ({excess:.3g} of the bound) rel_l2={rel:.3g}"
    return max_abs, rel


def ws_view(model: Model, ws: torch.Tensor):
    return api.moe_workspace_layout(model.shape, ws.numel())


def ws_i32(ws: torch.Tensor, offset: int, n: int) -> np.ndarray:
    return ws[offset:offset + 4 * n].cpu().numpy().view(np.int32).copy()


def ws_u8(ws: torch.Tensor, offset: int, n: int) -> np.ndarray:
    return ws[offset:offset + n].cpu().numpy().copy()
