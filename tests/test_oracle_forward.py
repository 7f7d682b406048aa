"""Pins of the oracle's forward ("Cake SiTU backend": quantize X, FC1, SiTU,
requant, FC2, BF16 weighted finalize) and of its SiTU.

The dense restatement below decodes the codes with its own tables (torch's
float8_e4m3fn cast and the E2M1 grid) and does the contractions with numpy
matmuls; it reuses the oracle's quantized X and A codes only as inputs.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import cases
from nvfp4_routed_moe_gb300 import inputs as gen

E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0])
E4M3 = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()


def _dense(packed, sf):
    """Decode canonical packed codes [..., K/2] + scales [..., K/16] to fp64."""
    lo = E2M1[packed & 15]
    hi = E2M1[packed >> 4]
    v = np.stack([lo, hi], axis=-1).reshape(*packed.shape[:-1], packed.shape[-1] * 2)
    s = np.repeat(E4M3[sf], 16, axis=-1)
    return v * s


@pytest.fixture(scope="module")
def tiny():
    return cases.prepare_tiny(0)


def test_situ_special_cases():
    assert oracle.situ(0.0, 5.0) == 0.0
    assert oracle.situ(3.0, 0.0) == 0.0
    for g, u in [(0.3, -1.2), (2.0, 7.0), (-5.0, 30.0)]:
        assert oracle.situ(g, -u) == -oracle.situ(g, u)
    # saturation: gate -> beta, linear -> lambda
    assert abs(oracle.situ(200.0, 1e4) - 100.0) < 1e-9
    assert abs(oracle.situ(-200.0, 1e4)) < 1e-9
    for g in np.linspace(-50, 50, 101):
        for u in (-1e3, -3.0, 0.5, 80.0):
            gate = oracle.situ(g, 1e12, 4.0, 1.0) / 1.0   # linear part saturated at lambda = 1
            assert abs(gate) <= 4.0 + 1e-12
            lin = oracle.situ(60.0, u, 1.0, 25.0)          # gate saturated at beta = 1
            assert abs(lin) <= 25.0 + 1e-12


def _golden_rows(name):
    path = __file__.rsplit("/", 1)[0] + "/golden/" + name
    return [list(map(float, ln.split())) for ln in open(path) if ln.strip() and not ln.startswith("#")]


def test_situ_distinct_parameters_golden():
    """Gate and linear smoothing parameters in their own places ("Cake SiTU
    backend": situ_beta smooths the gate, situ_linear_beta the linear half):
    values worked by hand from the closed form, and the exchanged call, which
    a swap of the two parameters would give, differs from each of them."""
    rows = _golden_rows("situ_distinct_parameters.txt")
    assert len(rows) == 4
    for g, u, beta, lam, want, swapped in rows:
        got = oracle.situ(g, u, beta, lam)
        assert abs(got - want) <= 1e-13 * abs(want), (g, u, beta, lam, got, want)
        assert abs(oracle.situ(g, u, lam, beta) - swapped) <= 1e-13 * abs(swapped)
        assert abs(got - swapped) > 1e-3 * abs(want)


def test_dequant_rows_matches_independent_decode():
    """oracle.nvfp4_dequant_rows (the reference of the tile-product check)
    against this file's own decode (E2M1 grid table, torch's float8_e4m3fn
    cast): every code byte, every scale byte including zero and subnormal
    scales, low nibble first."""
    rs = np.random.default_rng(17)
    rows, cols = 256, 64
    packed = rs.integers(0, 256, size=(rows, cols // 2), dtype=np.uint8)
    packed[0] = np.arange(32, dtype=np.uint8)           # every byte value appears
    packed[1] = np.arange(32, 64, dtype=np.uint8)
    packed[2:8].reshape(-1)[:192] = np.arange(64, 256, dtype=np.uint8)
    sf = np.arange(rows * cols // 16, dtype=np.int64).reshape(rows, cols // 16) % 256
    sf = sf.astype(np.uint8)
    sf[sf == 0x7F] = 0x7E                                # E4M3 NaN codes are never produced
    sf[sf == 0xFF] = 0xFE
    got = oracle.nvfp4_dequant_rows(packed, sf)
    np.testing.assert_array_equal(got, _dense(packed, sf))
    # a hand-checked element: byte 0x9E holds code 0xE (-4) low, 0x9 (-0.5) high;
    # scale 0x38 is 1.0 and 0x01 is the smallest subnormal 2^-9
    one = oracle.nvfp4_dequant_rows(np.full((1, 8), 0x9E, np.uint8), np.array([[0x38]], np.uint8))
    assert one[0, 0] == -4.0 and one[0, 1] == -0.5
    tiny_sf = oracle.nvfp4_dequant_rows(np.full((1, 8), 0x07, np.uint8), np.array([[0x01]], np.uint8))
    assert tiny_sf[0, 0] == 6.0 * 2.0 ** -9 and tiny_sf[0, 1] == 0.0


def test_situ_limit_is_swiglu():
    """As beta, lambda -> infinity SiTU becomes SiLU(g) * u (textbook SwiGLU)."""
    g = torch.linspace(-8, 8, 41, dtype=torch.float64)
    u = torch.linspace(-3, 3, 41, dtype=torch.float64)
    ref = torch.nn.functional.silu(g) * u
    got = torch.tensor([oracle.situ(float(a), float(b), 1e7, 1e7) for a, b in zip(g, u)], dtype=torch.float64)
    torch.testing.assert_close(got, ref, rtol=1e-9, atol=1e-9)


def test_dense_restatement_tiny(tiny):
    """FC1 / FC2 / finalize against a numpy dense restatement (fp64 matmuls)."""
    inp = tiny
    out, mid = cases.run_oracle(inp, want_intermediates=True)
    H, I, k = inp.H, inp.I, inp.k
    xq, xsf = oracle.nvfp4_quant_rows(gen.bf16_bits_to_f32(inp.x), q=inp.qX)
    X = _dense(xq, xsf)                              # [T, H]
    W13 = _dense(inp.w13, inp.sf13)                  # [E, 2I, H]
    W2 = _dense(inp.w2, inp.sf2)                     # [E, H, I]
    rw = gen.bf16_bits_to_f32(inp.route_weights).astype(np.float64)
    for t in range(inp.T):
        acc_out = np.zeros(H)
        for j in range(k):
            e = inp.expert_ids[t, j]
            z = (W13[e] @ X[t]).astype(np.float32) * inp.dXdW13[e]
            np.testing.assert_array_equal(mid["z"][t, j], z)
            A = _dense(mid["aq"][t, j][None], mid["asf"][t, j][None])[0]
            y = (W2[e] @ A).astype(np.float32) * inp.dAdW2[e]
            np.testing.assert_array_equal(mid["y"][t, j], y)
            acc_out += rw[t, j] * y
        ref = gen.f32_to_bf16_bits(acc_out.astype(np.float32))
        np.testing.assert_array_equal(out[t], ref)


def test_gate_is_first_half(tiny):
    """w13 rows 0..I-1 feed g (the SiLU-like gate), rows I..2I-1 feed u."""
    inp = tiny
    _, mid = cases.run_oracle(inp, tokens=[0], want_intermediates=True)
    z = mid["z"][0, 0].astype(np.float64)
    a_ref = np.array([oracle.situ(z[i], z[inp.I + i]) for i in range(inp.I)], np.float32)
    np.testing.assert_array_equal(mid["a"][0, 0], a_ref)


def test_zero_input_gives_zero_output(tiny):
    inp = cases.prepare_tiny(0)
    inp.x = np.zeros_like(inp.x)
    out = cases.run_oracle(inp)
    assert not gen.bf16_bits_to_f32(out).any()


def test_one_hot_route_weight_is_single_expert_ffn(tiny):
    inp = cases.prepare_tiny(0)
    w = np.zeros((inp.T, inp.k), np.float32)
    w[:, 2] = 1.0
    inp.route_weights = gen.f32_to_bf16_bits(w)
    out, mid = cases.run_oracle(inp, want_intermediates=True)
    np.testing.assert_array_equal(out, gen.f32_to_bf16_bits(mid["y"][:, 2, :]))


def test_token_permutation_equivariance(tiny):
    inp = tiny
    out = cases.run_oracle(inp)
    perm = np.random.default_rng(4).permutation(inp.T)
    inp2 = cases.prepare_tiny(0)
    inp2.x, inp2.expert_ids, inp2.route_weights = inp.x[perm], inp.expert_ids[perm], inp.route_weights[perm]
    out2 = cases.run_oracle(inp2)
    np.testing.assert_array_equal(out2, out[perm])


def test_route_weights_enter_linearly(tiny):
    """The combine is linear in the route weights: doubling every weight
    doubles every output exactly (a power-of-two scale commutes with the fp64
    sum and the one BF16 rounding), and splitting the weights w = w1 + w2
    (both exact in BF16) gives out(w1) + out(w2) up to the BF16 roundings."""
    inp = cases.prepare_tiny(0)
    w = gen.bf16_bits_to_f32(inp.route_weights).astype(np.float64)
    out = gen.bf16_bits_to_f32(cases.run_oracle(inp)).astype(np.float64)
    inp.route_weights = gen.f32_to_bf16_bits((2.0 * w).astype(np.float32))
    out2 = gen.bf16_bits_to_f32(cases.run_oracle(inp)).astype(np.float64)
    np.testing.assert_array_equal(out2, 2.0 * out)
    w1 = gen.bf16_bits_to_f32(gen.f32_to_bf16_bits((0.75 * w).astype(np.float32))).astype(np.float64)
    w2 = w - w1
    assert np.array_equal(gen.bf16_bits_to_f32(gen.f32_to_bf16_bits(w2.astype(np.float32))), w2)
    parts = []
    for wp in (w1, w2):
        inp.route_weights = gen.f32_to_bf16_bits(wp.astype(np.float32))
        parts.append(gen.bf16_bits_to_f32(cases.run_oracle(inp)).astype(np.float64))
    # each output carries at most half a BF16 ulp of rounding (relative 2^-9)
    bound = 2.0 ** -8 * (np.abs(out) + np.abs(parts[0]) + np.abs(parts[1])) + 1e-30
    assert (np.abs(parts[0] + parts[1] - out) <= bound).all()


def test_exact_arithmetic_case():
    """Power-of-two scales and small codes: every sum is exact, so the whole
    forward is computable by hand (here: in fp64 with exact integers)."""
    H, I, E, k, T = 512, 128, 4, 2, 3
    rs = np.random.default_rng(11)
    # x: values in {0, +-1, +-2} -> with qX = 1 blocks containing a 2 get S = 2/6 ... keep it simple:
    # choose x so every block holds a 6 and other entries in the E2M1 grid, qX = 1 -> S = 1.
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], np.float32)
    x = rs.choice(np.concatenate([grid, -grid]), size=(T, H)).astype(np.float32)
    x[:, ::16] = 6.0
    xb = gen.f32_to_bf16_bits(x)
    codes13 = rs.integers(0, 256, size=(E, 2 * I, H // 2), dtype=np.uint8)
    sf13 = np.full((E, 2 * I, H // 16), 0x38, np.uint8)     # 1.0
    codes2 = rs.integers(0, 256, size=(E, H, I // 2), dtype=np.uint8)
    sf2 = np.full((E, H, I // 16), 0x30, np.uint8)          # 0.5
    ids = np.array([[0, 1], [2, 3], [1, 0]], np.int32)
    rw = gen.f32_to_bf16_bits(np.array([[0.5, 0.25], [1.0, 0.0], [0.125, 2.0]], np.float32))
    one = np.ones(E, np.float32)
    scale13 = np.full(E, 2.0 ** -12, np.float32)
    out, mid = oracle.moe_forward_tokens(H=H, I=I, E=E, k=k, x=xb, expert_ids=ids, route_weights=rw,
                                         tokens=np.arange(T), w13=codes13, sf13=sf13, w2=codes2, sf2=sf2,
                                         qX=np.float32(1.0), dXdW13=scale13, qA=one, dAdW2=one,
                                         want_intermediates=True)
    W13 = _dense(codes13, sf13)
    for t in range(T):
        for j in range(k):
            e = ids[t, j]
            acc = W13[e] @ x[t].astype(np.float64)          # integers and halves: exact
            assert np.all(np.abs(acc) < 2 ** 24)
            np.testing.assert_array_equal(mid["z"][t, j], (acc * 2.0 ** -12).astype(np.float32))
