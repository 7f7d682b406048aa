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


# --------------------------------------------------------------- every option
# (active_expert_range, active_num, key_value histogram, static quant, smooth
# scale): "npu_moe_init_routing_v2", formulas 1-6 and its parameter list.

def test_init_routing_ex_defaults_reduce_to_the_plain_op():
    inp = gen.full(2, T=48, weights=False, E=64)
    for kw in (dict(quant_mode=1), dict(quant_mode=-1, row_idx_type=1, tokens_num_type=1),
               dict(quant_mode=1, drop_pad=1, expert_capacity=9)):
        a = oracle.init_routing(inp.x, inp.expert_ids, 64, **kw)
        b = oracle.init_routing_ex(inp.x, inp.expert_ids, 64, **kw)
        for u, v in zip(a, b):
            if isinstance(u, np.ndarray):
                np.testing.assert_array_equal(u, v)
            else:
                assert u == v


def test_active_expert_range_brute_force():
    T, E, k, lo, hi = 40, 32, 4, 5, 19
    inp = gen.full(3, T=T, weights=False, E=E)
    ids = gen.draw_ids_uniform(3, T, E, k)
    ex, ridx, tok, sc, avail = oracle.init_routing_ex(inp.x[:, :512], ids, E, expert_start=lo, expert_end=hi)
    flat = ids.ravel()
    inr = (flat >= lo) & (flat < hi)
    assert avail == int(inr.sum())
    order = [f for e in range(lo, hi) for f in range(flat.size) if flat[f] == e]     # stable by construction
    assert len(order) == avail
    gather = np.full(flat.size, -1)
    gather[order] = np.arange(avail)
    np.testing.assert_array_equal(ridx, gather)
    counts = np.array([(flat == e).sum() for e in range(lo, hi)])
    np.testing.assert_array_equal(tok, np.cumsum(counts))
    for i, f in enumerate(order):
        q, s = oracle.dynamic_int8_row(inp.x[f // k, :512])
        np.testing.assert_array_equal(ex[i], q)
        assert sc[i] == s
    assert not ex[avail:].any()
    _, ridx1, tok1, _, _ = oracle.init_routing_ex(inp.x[:, :512], ids, E, expert_start=lo, expert_end=hi,
                                                  row_idx_type=1, tokens_num_type=1, quant_mode=-1)
    np.testing.assert_array_equal(ridx1[:avail], order)
    assert (ridx1[avail:] == -1).all()
    np.testing.assert_array_equal(tok1, counts)


def test_key_value_histogram():
    ids = np.array([[3, 7], [7, 1], [3, 9], [12, 7]], np.int32)
    x = np.zeros((4, 16), np.uint16)
    _, _, kv, _, avail = oracle.init_routing_ex(x, ids, 16, expert_start=2, expert_end=10, tokens_num_type=2)
    assert avail == 6                                  # 3, 7, 7, 3, 9, 7 are in [2, 10)
    expect = np.zeros((16, 2), np.int32)
    expect[:3] = [[3, 2], [7, 3], [9, 1]]
    np.testing.assert_array_equal(kv, expect)


def test_active_num_keeps_the_first_sorted_rows():
    T, E, k = 24, 16, 4
    inp = gen.full(4, T=T, weights=False, E=E)
    ids = gen.draw_ids_uniform(4, T, E, k)
    full = oracle.init_routing_ex(inp.x[:, :256], ids, E, quant_mode=-1)
    part = oracle.init_routing_ex(inp.x[:, :256], ids, E, quant_mode=-1, active_num=37)
    np.testing.assert_array_equal(part[0][:37], full[0][:37])
    assert not part[0][37:].any()
    g_full, g_part = full[1], part[1]
    np.testing.assert_array_equal(g_part, np.where(g_full < 37, g_full, -1))
    np.testing.assert_array_equal(part[2], full[2])     # the histogram is over every available pair
    assert part[4] == full[4] == T * k


def test_static_int8_hand_worked():
    # x*scale + offset with scale 2, offset 0.5 (x as bf16: 0.3 -> 0.30078125,
    # -150.25 -> -150): 2.5 -> 2 (ties to even), -4.5 -> -4, 200.5 -> 127
    # (saturated), 1.1015625 -> 1, -299.5 -> -128 (saturated)
    xv = np.array([1.0, -2.5, 100.0, 0.3, -150.25] + [0.0] * 11, np.float32)
    x = gen.f32_to_bf16_bits(xv)[None, :]
    ex, ridx, _, sc, avail = oracle.init_routing_ex(x, np.array([[0]], np.int32), 1, quant_mode=0,
                                                    scale=[2.0], offset=[0.5])
    assert sc is None and avail == 1
    assert list(ex[0, :5]) == [2, -4, 127, 1, -128]
    assert not ex[0, 5:].any()


def test_dynamic_smooth_scale_power_of_two_rows():
    """A smooth row of 2^e scales x exactly: the codes equal the plain dynamic
    codes and the row scale is 2^e times the plain one."""
    T, E, k, lo, hi = 16, 8, 2, 2, 6
    inp = gen.full(5, T=T, weights=False, E=E)
    ids = gen.draw_ids_uniform(5, T, E, k)
    x = inp.x[:, :256]
    smooth = np.stack([np.full(256, 2.0 ** e, np.float32) for e in range(hi - lo)])
    a = oracle.init_routing_ex(x, ids, E, expert_start=lo, expert_end=hi)
    b = oracle.init_routing_ex(x, ids, E, expert_start=lo, expert_end=hi, scale=smooth)
    np.testing.assert_array_equal(a[0], b[0])
    flat = ids.ravel()
    order = [f for e in range(lo, hi) for f in range(flat.size) if flat[f] == e]
    for i, f in enumerate(order):
        assert b[3][i] == a[3][i] * np.float32(2.0 ** (flat[f] - lo))
    c = oracle.init_routing_ex(x, ids, E, expert_start=lo, expert_end=hi, scale=smooth[:1])   # one shared row
    np.testing.assert_array_equal(c[3], a[3])


def test_unquantized_rows_carry_the_token_scale():
    T, E, k = 12, 8, 2
    inp = gen.full(6, T=T, weights=False, E=E)
    ids = gen.draw_ids_uniform(6, T, E, k)
    s = np.arange(1, T + 1, dtype=np.float32) * 0.25
    ex, ridx, _, sc, avail = oracle.init_routing_ex(inp.x[:, :128], ids, E, quant_mode=-1, scale=s)
    for f in range(T * k):
        np.testing.assert_array_equal(ex[ridx[f]], inp.x[f // k, :128])
        assert sc[ridx[f]] == s[f // k]
