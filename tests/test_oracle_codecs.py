"""Pins of the oracle's E2M1 / E4M3 codecs and its NVFP4 group quantizer.

Each check ties the oracle to something other than itself: hand-worked values
(tests/golden), brute-force nearest-value search over the format's grid, torch's
float8_e4m3fn cast, closed-form properties of the quantizer.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle

E2M1_GRID = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def _read(path):
    rows = []
    with open(path) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


def _brute_e2m1(v: float) -> float:
    """Nearest grid value by exhaustive search; ties go to the even code."""
    a = abs(v)
    if a >= 6.0:
        m = 6.0
    else:
        best = None
        for code, g in enumerate(E2M1_GRID):
            d = abs(a - g)
            if best is None or d < best[0] or (d == best[0] and code % 2 == 0):
                best = (d, code, g)
        m = best[2]
    return -m if math.copysign(1.0, v) < 0 else m


def test_e2m1_golden(golden_dir):
    for inp, want in _read(os.path.join(golden_dir, "e2m1_rounding.txt")):
        code = oracle.e2m1_encode(float(inp))
        assert oracle.e2m1_value(code) == float(want), (inp, code)


def test_e2m1_decode_table():
    vals = [oracle.e2m1_value(c) for c in range(16)]
    assert vals[:8] == E2M1_GRID
    assert vals[8:] == [-v for v in E2M1_GRID]


def test_e2m1_brute_force_random_and_midpoints():
    rs = np.random.default_rng(123)
    xs = list(rs.uniform(-8, 8, 20000).astype(np.float32))
    mids = [(a + b) / 2 for a, b in zip(E2M1_GRID, E2M1_GRID[1:])]
    for m in mids + E2M1_GRID:
        for s in (-1, 1):
            f = np.float32(s * m)
            xs += [f, np.nextafter(f, np.float32(np.inf)), np.nextafter(f, np.float32(-np.inf))]
    for v in xs:
        code = oracle.e2m1_encode(float(v))
        assert oracle.e2m1_value(code) == _brute_e2m1(float(v)), v


def test_e2m1_sign_of_zero():
    assert oracle.e2m1_encode(0.0) == 0
    assert oracle.e2m1_encode(-0.0) == 8
    assert oracle.e2m1_encode(-0.1) == 8


def test_e4m3_decode_against_torch():
    b = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    for c in range(256):
        v = oracle.e4m3_value(c)
        if math.isnan(b[c]):
            assert math.isnan(v)
        else:
            assert v == float(b[c]), c


def test_e4m3_encode_against_torch_in_range():
    rs = np.random.default_rng(7)
    mags = np.concatenate([np.exp(rs.uniform(np.log(1e-5), np.log(448.0), 200000)),
                           rs.uniform(0, 448.0, 50000)]).astype(np.float32)
    vals = np.concatenate([mags, -mags])
    ref = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_encode(float(v)) for v in vals[:20000]], np.uint8)
    np.testing.assert_array_equal(got, ref[:20000])
    # the rest via the range sweep (bit patterns between the smallest and largest input)
    bits = np.sort(np.abs(vals).view(np.uint32))
    lo, hi = int(bits[0]), int(bits[-1])
    sweep = oracle.e4m3_encode_range(lo, hi - lo + 1)
    idx = (np.abs(vals).view(np.uint32).astype(np.int64) - lo)
    sgn = np.where(np.signbit(vals), 0x80, 0).astype(np.uint8)
    np.testing.assert_array_equal(sweep[idx] | sgn, ref)


def test_e4m3_midpoints_round_to_even_and_saturate():
    codes = [c for c in range(0x7F)]
    vals = [oracle.e4m3_value(c) for c in codes]
    for c in range(len(vals) - 1):
        mid = (vals[c] + vals[c + 1]) / 2
        f = np.float32(mid)
        assert float(f) == mid  # midpoints are exact in fp32
        want = c if c % 2 == 0 else c + 1
        assert oracle.e4m3_encode(float(f)) == want, (c, mid)
        assert oracle.e4m3_encode(float(np.nextafter(f, np.float32(0)))) == c
        assert oracle.e4m3_encode(float(np.nextafter(f, np.float32(1e9)))) == c + 1
    for v in (448.0, 449.0, 464.0, 500.0, 1e30, float("inf")):
        assert oracle.e4m3_encode(v) == 0x7E
        assert oracle.e4m3_encode(-v) == 0xFE


def test_e4m3_ml_dtypes_if_present():
    ml = pytest.importorskip("ml_dtypes")
    rs = np.random.default_rng(9)
    vals = np.exp(rs.uniform(np.log(1e-4), np.log(440.0), 5000)).astype(np.float32)
    ref = vals.astype(ml.float8_e4m3fn).view(np.uint8)
    got = np.array([oracle.e4m3_encode(float(v)) for v in vals], np.uint8)
    np.testing.assert_array_equal(got, ref)


def test_e2m1_ml_dtypes_if_present():
    ml = pytest.importorskip("ml_dtypes")
    if not hasattr(ml, "float4_e2m1fn"):
        pytest.skip("no float4_e2m1fn")
    rs = np.random.default_rng(10)
    vals = rs.uniform(-6, 6, 5000).astype(np.float32)
    ref = vals.astype(ml.float4_e2m1fn).astype(np.float32)
    got = np.array([oracle.e2m1_value(oracle.e2m1_encode(float(v))) for v in vals])
    np.testing.assert_array_equal(got, ref)


# ------------------------------------------------------------- group quantizer

def test_global_amax_block_gets_scale_448():
    """qX = 1/dX with dX = amax/(6*448) ("Cake SiTU backend", qX=1/dX) puts the
    block holding the global amax at block scale 448."""
    rs = np.random.default_rng(1)
    for _ in range(200):
        x = rs.standard_normal(16 * 8).astype(np.float32) * np.float32(rs.uniform(0.01, 100))
        amax = np.float32(np.abs(x).max())
        dX = np.float32(amax / np.float32(2688))
        qX = np.float32(np.float32(1) / dX)
        g = int(np.abs(x).argmax()) // 16
        codes, sf = oracle.nvfp4_quant_group(x[g * 16:(g + 1) * 16], qX)
        assert oracle.e4m3_value(sf) == 448.0


def test_block_max_element_maps_to_six():
    """With a normal block scale, the E4M3 relative rounding error (<= 1/16)
    keeps the largest element's scaled value above 5, so it encodes to 6."""
    rs = np.random.default_rng(2)
    for _ in range(500):
        v = rs.standard_normal(16).astype(np.float32)
        q = np.float32(np.exp(rs.uniform(-2, 4)))
        codes, sf = oracle.nvfp4_quant_group(v, q)
        S = oracle.e4m3_value(sf)
        if S >= 2.0 ** -6:
            j = int(np.abs(v).argmax())
            assert abs(oracle.e2m1_value(codes[j])) == 6.0


def test_round_trip_of_representable_values():
    """x = code * S * d is re-encoded to the same codes when the block holds a 6."""
    rs = np.random.default_rng(3)
    for _ in range(300):
        sf_b = int(rs.integers(0x08, 0x7E))
        S = oracle.e4m3_value(sf_b)
        q = np.float32(2.0 ** int(rs.integers(-3, 4)))
        codes = rs.integers(0, 16, 16)
        codes[int(rs.integers(0, 16))] = 7 | (8 * int(rs.integers(0, 2)))
        x = np.array([oracle.e2m1_value(c) * S / float(q) for c in codes], np.float32)
        got, sf2 = oracle.nvfp4_quant_group(x, q)
        assert sf2 == sf_b
        np.testing.assert_array_equal([oracle.e2m1_value(c) for c in got], [oracle.e2m1_value(c) for c in codes])


def test_zero_block():
    codes, sf = oracle.nvfp4_quant_group(np.zeros(16, np.float32), np.float32(3.0))
    assert sf == 0 and all(c == 0 for c in codes)


def test_quant_rows_packing_low_nibble_even():
    x = np.zeros((1, 16), np.float32)
    x[0, 0] = 6.0   # code 7 in the low nibble of byte 0
    x[0, 1] = -1.0  # code 0xA in the high nibble of byte 0
    x[0, 3] = 3.0   # code 5 in the high nibble of byte 1
    packed, sf = oracle.nvfp4_quant_rows(x, q=np.float32(448.0))
    assert oracle.e4m3_value(sf[0, 0]) == 448.0
    assert packed[0, 0] == 0xA7 and packed[0, 1] == 0x50


def test_scale_atom_offsets_golden(golden_dir):
    for m, kc, ncols, off in _read(os.path.join(golden_dir, "scale_atom_offsets.txt")):
        assert oracle.scale_atom_offset(int(m), int(kc), int(ncols)) == int(off)


def test_scale_atom_layout_is_a_bijection():
    rows, cols = 256, 24
    seen = set()
    for r in range(rows):
        for c in range(cols):
            seen.add(oracle.scale_atom_offset(r, c, cols))
    assert len(seen) == rows * cols and max(seen) == rows * cols - 1
