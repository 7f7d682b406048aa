"""Pins of the oracle's routing and init-routing ("npu_moe_init_routing_v2",
formulas 1-5): brute force on small cases, numpy's stable argsort, invariants,
hand-worked int8 values."""
import os

import numpy as np
import pytest

import oracle
from nvfp4_routed_moe_gb300 import inputs as gen


def _read(path):
    with open(path) as f:
        return [l.split() for l in f if l.strip() and not l.startswith("#")]


def _brute_routing(ids, E):
    T, k = ids.shape
    flat = [(int(ids[t, j]), t * k + j) for t in range(T) for j in range(k) if 0 <= ids[t, j] < E]
    order = sorted(flat)  # (expert, rowIdx) lexicographic = stable by rowIdx
    return [r for _, r in order], [e for e, _ in order]


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_routing_brute_force_tiny(seed):
    inp = gen.tiny(seed)
    r = oracle.routing(inp.expert_ids, inp.E)
    sr, se = _brute_routing(inp.expert_ids, inp.E)
    assert list(r["sorted_row"]) == sr
    assert list(r["sorted_expert"]) == se
    for i, f in enumerate(sr):
        assert r["gather"][f] == i
    counts = np.bincount(inp.expert_ids.ravel(), minlength=inp.E)
    np.testing.assert_array_equal(r["count"], counts)
    np.testing.assert_array_equal(r["cumsum"], np.cumsum(counts))


def test_routing_matches_numpy_stable_argsort_and_invariants():
    ids = gen.draw_ids_zipf(5, 512, 896, 16)
    r = oracle.routing(ids, 896)
    flat = ids.ravel()
    order = np.argsort(flat, kind="stable")
    np.testing.assert_array_equal(r["sorted_row"], order)
    P = flat.size
    assert r["count"].sum() == P and r["cumsum"][-1] == P
    g = r["gather"]
    np.testing.assert_array_equal(g[r["sorted_row"]], np.arange(P))          # gather o scatter = id
    keys = flat[r["sorted_row"]]
    assert np.all(np.diff(keys) >= 0)
    same = np.diff(keys) == 0
    assert np.all(np.diff(r["sorted_row"])[same] > 0)                          # stable within expert


def test_routing_invalid_ids_not_routed():
    ids = np.array([[0, 5], [-1, 2], [7, 0]], np.int32)
    r = oracle.routing(ids, 6)
    assert r["nvalid"] == 4
    assert list(r["sorted_row"][:4]) == [0, 5, 3, 1]
    assert r["gather"][2] == -1 and r["gather"][4] == -1
    assert list(r["count"]) == [2, 0, 1, 0, 0, 1]


def test_routing_empty_experts_and_single_token():
    ids = np.array([[3, 1, 2, 0]], np.int32)
    r = oracle.routing(ids, 8)
    assert list(r["sorted_row"]) == [3, 1, 2, 0]
    assert list(r["cumsum"]) == [1, 2, 3, 4, 4, 4, 4, 4]


def test_int8_dynamic_golden(golden_dir):
    xs, qs, s = _read(os.path.join(golden_dir, "int8_dynamic_quant.txt"))
    x = gen.f32_to_bf16_bits(np.array([float(v) for v in xs], np.float32))
    q, scale = oracle.dynamic_int8_row(x)
    assert list(q) == [int(v) for v in qs]
    assert scale == float(s[0])


def test_int8_closed_form_properties():
    x = gen.draw_x(3, 64, 512)
    xf = gen.bf16_bits_to_f32(x)
    for t in range(64):
        q, s = oracle.dynamic_int8_row(x[t])
        amax = np.float32(np.abs(xf[t]).max())
        assert s == np.float32(amax / np.float32(127))
        assert np.abs(q).max() == 127
        # q is the nearest integer to x/s (fp32 quotient), ties to even
        quo = (xf[t] / np.float32(s)).astype(np.float32)
        np.testing.assert_array_equal(q, np.clip(np.rint(quo), -127, 127).astype(np.int8))
    q, s = oracle.dynamic_int8_row(np.zeros(16, np.uint16))
    assert s == 0.0 and not q.any()


def test_init_routing_dropless_gather_moves_rows():
    inp = gen.full(0, T=64, weights=False, E=64)
    ex, ridx, tok, scale, nvalid = oracle.init_routing(inp.x, inp.expert_ids, 64, quant_mode=1)
    r = oracle.routing(inp.expert_ids, 64)
    np.testing.assert_array_equal(ridx, r["gather"])
    np.testing.assert_array_equal(tok, r["cumsum"])
    for f in range(64 * 16):
        t = f // 16
        q, s = oracle.dynamic_int8_row(inp.x[t])
        np.testing.assert_array_equal(ex[ridx[f]], q)
        assert scale[ridx[f]] == s
    ex1, ridx1, tok1, _, _ = oracle.init_routing(inp.x, inp.expert_ids, 64, quant_mode=-1, row_idx_type=1,
                                                 tokens_num_type=1)
    np.testing.assert_array_equal(ridx1, r["sorted_row"])
    np.testing.assert_array_equal(tok1, r["count"])
    for i in range(64 * 16):
        np.testing.assert_array_equal(ex1[i], inp.x[ridx1[i] // 16])   # expandedX[i] = x[scatter[i]//K]


def test_init_routing_drop_pad():
    E, C = 32, 20
    inp = gen.full(1, T=64, weights=False, E=E)
    ex, ridx, tok, scale, nvalid = oracle.init_routing(inp.x, inp.expert_ids, E, drop_pad=1, expert_capacity=C)
    counts = np.bincount(inp.expert_ids.ravel(), minlength=E)
    assert ex.shape == (E * C, 3584)
    filled = (scale != 0)
    assert filled.sum() == np.minimum(counts, C).sum()
    for e in range(E):
        n = min(counts[e], C)
        assert filled[e * C:e * C + n].all() and not filled[e * C + n:(e + 1) * C].any()
        assert not ex[e * C + n:(e + 1) * C].any()
    assert (ridx == -1).sum() == np.maximum(counts - C, 0).sum()
    np.testing.assert_array_equal(tok, np.cumsum(counts))   # histogram is not clipped
