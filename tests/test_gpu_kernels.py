"""GPU checks of the building blocks, through the C ABI, against the oracle:
hardware FP4/FP8 conversions (exhaustive), the device NVFP4 quantizer (both
forms, bit-exact), SiTU + requant of the FC1 epilogue, and one tcgen05
block-scaled tile product."""
import numpy as np
import pytest
import torch

import oracle
from nvfp4_routed_moe_gb300 import api

pytestmark = pytest.mark.gpu

E2M1_GRID = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], np.float64)


@pytest.mark.parametrize("n,k", [(16, 256), (48, 512), (128, 3584), (7, 256)])
def test_mma_tile_product(n, k):
    """One tcgen05 kind::mxf4nvf4 tile vs an fp64 dense restatement: with
    power-of-two scales every partial sum is exact in fp32."""
    rs = np.random.default_rng(n + k)
    a = rs.integers(0, 256, (128, k // 2), dtype=np.uint8)
    b = rs.integers(0, 256, (n, k // 2), dtype=np.uint8)
    sfa = rs.choice(np.array([0x30, 0x38, 0x40], np.uint8), (128, k // 16))   # 0.5, 1, 2
    sfb = rs.choice(np.array([0x38, 0x40, 0x30], np.uint8), (n, k // 16))
    sfb_pad = np.zeros((128, k // 16), np.uint8)
    sfb_pad[:n] = sfb
    A = oracle.nvfp4_dequant_rows(a, sfa)
    B = oracle.nvfp4_dequant_rows(b, sfb)
    ref = A @ B.T
    d = torch.empty((128, n), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.moe_test_mma_fp4(torch.from_numpy(a).cuda(), torch.from_numpy(oracle.to_atom_layout(sfa)).cuda(),
                         torch.from_numpy(b).cuda(), torch.from_numpy(oracle.to_atom_layout(sfb_pad)).cuda(), n, k,
                         d, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    got = d.cpu().numpy().astype(np.float64)
    if not np.array_equal(got, ref):
        diff = np.abs(got - ref)
        i, j = np.unravel_index(diff.argmax(), diff.shape)
        raise AssertionError(f"max diff {diff.max()} at {(i, j)}: got {got[i, j]} ref {ref[i, j]}; "
                             f"{(diff > 0).sum()} of {diff.size} differ; got[:2,:4]={got[:2, :4]} "
                             f"ref[:2,:4]={ref[:2, :4]}")


def _quant_case(rows, cols, seed):
    rs = np.random.default_rng(seed)
    x = rs.standard_normal((rows, cols)).astype(np.float32)
    x *= np.exp(rs.uniform(-6, 6, (rows, 1))).astype(np.float32)
    x[0] = 0.0                                     # zero row
    x[1, :16] = 1e-30                              # tiny group
    x[2, 16:32] = -3.0e4                           # huge group
    x[3, ::7] *= 40.0                              # outliers
    q = np.exp(rs.uniform(-4, 8, rows)).astype(np.float32)
    q[4] = np.float32(2688.0 / np.abs(x[4]).max())  # qX = 1/dX with dX = amax/(6*448)
    return x, q


@pytest.mark.parametrize("rows,cols", [(64, 512), (37, 3584), (5, 384)])
def test_quantize_rows_bit_exact(rows, cols):
    x, q = _quant_case(rows, cols, rows)
    packed = torch.empty((rows, cols // 2), dtype=torch.uint8, device="cuda")
    sf = torch.empty((rows, cols // 16), dtype=torch.uint8, device="cuda")
    api.moe_test_quantize_rows(torch.from_numpy(x).cuda(), torch.from_numpy(q).cuda(), packed, sf)
    rp, rsf = oracle.nvfp4_quant_rows(x, q_per_row=q)
    np.testing.assert_array_equal(sf.cpu().numpy(), rsf)
    np.testing.assert_array_equal(packed.cpu().numpy(), rp)


@pytest.mark.parametrize("I", [128, 384])
def test_requant_lanes_bit_exact(I):
    rows = 50
    x, q = _quant_case(rows, I, I)
    for qa in (float(q[7]), 1e-4, 3.0):
        packed = torch.empty((rows, I // 2), dtype=torch.uint8, device="cuda")
        sf = torch.empty((rows, I // 16), dtype=torch.uint8, device="cuda")
        api.moe_test_requant_lanes(torch.from_numpy(x).cuda(), qa, packed, sf)
        rp, rsf = oracle.nvfp4_quant_rows(x, q=np.float32(qa))
        np.testing.assert_array_equal(sf.cpu().numpy(), rsf)
        np.testing.assert_array_equal(packed.cpu().numpy(), rp)


def _near_boundary(a, qa, sf_bytes, rel=1e-6):
    """Where the oracle's scaled value a*r lies within rel of an E2M1 rounding
    midpoint, or the group's amax*qA/6 within rel of an E4M3 midpoint."""
    S = np.array([oracle.e4m3_value(int(b)) for b in sf_bytes.ravel()]).reshape(sf_bytes.shape)
    r = np.where(S == 0, 0.0, qa / np.where(S == 0, 1, S))
    y = np.abs(a.reshape(a.shape[0], -1, 16) * r[..., None])
    mids = (E2M1_GRID[1:] + E2M1_GRID[:-1]) / 2
    near_e2 = (np.abs(y[..., None] - mids) <= rel * np.maximum(y[..., None], 1e-30)).any(-1)
    amax = np.abs(a.reshape(a.shape[0], -1, 16)).max(-1) * qa / 6
    vals = np.array(sorted({oracle.e4m3_value(c) for c in range(0x7F)}))
    emids = (vals[1:] + vals[:-1]) / 2
    near_e4 = (np.abs(amax[..., None] - emids) <= rel * np.maximum(amax[..., None], 1e-30)).any(-1)
    return near_e2, near_e4


def test_situ_requant_matches_oracle():
    rows, I = 256, 384
    rs = np.random.default_rng(5)
    z = (rs.standard_normal((rows, 2 * I)) * np.exp(rs.uniform(-3, 3.5, (rows, 1)))).astype(np.float32)
    for qa, beta, lam in ((0.5, 4.0, 25.0), (11.0, 2.5, 10.0), (1e-3, 4.0, 25.0)):
        a = torch.empty((rows, I), dtype=torch.float32, device="cuda")
        packed = torch.empty((rows, I // 2), dtype=torch.uint8, device="cuda")
        sf = torch.empty((rows, I // 16), dtype=torch.uint8, device="cuda")
        api.moe_test_situ_requant(torch.from_numpy(z).cuda(), I, qa, beta, lam, a, packed, sf)
        ra, rp, rsf = oracle.situ_requant_rows(z, I, np.float32(qa), beta, lam)
        ga = a.cpu().numpy()
        np.testing.assert_allclose(ga, ra, rtol=4e-6, atol=1e-30)
        near_e2, near_e4 = _near_boundary(ra.astype(np.float64), np.float64(np.float32(qa)), rsf)
        gsf = sf.cpu().numpy()
        bad_sf = (gsf != rsf) & ~near_e4
        assert not bad_sf.any(), f"{bad_sf.sum()} scale mismatches away from a rounding boundary"
        gp = packed.cpu().numpy()
        gcodes = np.stack([gp & 15, gp >> 4], -1).reshape(rows, -1, 16)
        rcodes = np.stack([rp & 15, rp >> 4], -1).reshape(rows, -1, 16)
        same_sf = (gsf == rsf)[..., None]
        bad = (gcodes != rcodes) & same_sf & ~near_e2
        assert not bad.any(), f"{bad.sum()} code mismatches away from a rounding boundary"



def test_situ_gate_across_the_exponential_range():
    """Gate pre-activations from -95 to 95, so the sigmoid's e^{-g} runs from
    underflow to overflow, with ordinary up values: activations within the
    same rtol 4e-6 of the oracle's (fp64) as elsewhere."""
    rows, I = 64, 384
    g = np.linspace(-95.0, 95.0, rows * I).astype(np.float32).reshape(rows, I)
    u = np.resize(np.array([1.0, -3.7, 0.2, 40.0], np.float32), (rows, I))
    z = np.ascontiguousarray(np.concatenate([g, u], axis=1))
    a = torch.empty((rows, I), dtype=torch.float32, device="cuda")
    packed = torch.empty((rows, I // 2), dtype=torch.uint8, device="cuda")
    sf = torch.empty((rows, I // 16), dtype=torch.uint8, device="cuda")
    api.moe_test_situ_requant(torch.from_numpy(z).cuda(), I, 1.0, 4.0, 25.0, a, packed, sf)
    ra, _, _ = oracle.situ_requant_rows(z, I, np.float32(1.0), 4.0, 25.0)
    np.testing.assert_allclose(a.cpu().numpy(), ra, rtol=4e-6, atol=1e-30)

def _nan_inputs(start, n):
    bits = np.arange(start, start + n, dtype=np.uint64).astype(np.uint32)
    return (((bits >> 23) & 0xFF) == 0xFF) & ((bits & 0x7FFFFF) != 0)


def test_codec_sweep_exhaustive():
    """Every fp32 bit pattern: the oracle's E2M1 / E4M3 encoders agree with
    cvt.rn.satfinite.{e2m1x2,e4m3x2}.f32 (NaN inputs excluded: the pages give
    FP4 no NaN)."""
    chunk = 1 << 27
    lo = torch.empty(chunk, dtype=torch.uint8, device="cuda")
    hi = torch.empty_like(lo)
    e4 = torch.empty_like(lo)
    for start in range(0, 1 << 32, chunk):
        api.moe_test_codec_sweep(start, chunk, lo, hi, e4)
        g_lo, g_hi, g_e4 = lo.cpu().numpy(), hi.cpu().numpy(), e4.cpu().numpy()
        r2 = oracle.e2m1_encode_range(start, chunk)
        r4 = oracle.e4m3_encode_range(start, chunk)
        keep = ~_nan_inputs(start, chunk)
        bad = np.nonzero(keep & ((g_lo != r2) | (g_hi != r2) | (g_e4 != r4)))[0]
        assert bad.size == 0, (f"start={start:#x}: {bad.size} mismatches, first bits={start + int(bad[0]):#010x} "
                               f"lo={g_lo[bad[0]]} hi={g_hi[bad[0]]} e4={g_e4[bad[0]]} oracle e2m1={r2[bad[0]]} "
                               f"e4m3={r4[bad[0]]}")


@pytest.mark.parametrize("n,copies", [(256, 0), (128, 8), (256, 12)])
def test_mma_peak_microbenchmark_runs(n, copies):
    """The FP4 tensor-peak microbenchmark completes on every SM with a clean
    status, and a longer run takes proportionally more cycles: the MMAs are
    really issued (a plausible cost per MMA, neither skipped nor stalled)."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    cyc = torch.zeros(sms, dtype=torch.int64, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    per = []
    for mmas in (1024, 4096):
        api.moe_test_mma_peak(sms, n, mmas, copies, cyc, st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        c = cyc.cpu().numpy()
        assert (c > 0).all()
        per.append(float(np.median(c)) / mmas)
    assert per[1] <= per[0] * 1.2
    assert 16 <= per[1] <= 1024
    with pytest.raises(api.MoeError):
        api.moe_test_mma_peak(sms + 1, n, 1024, copies, cyc, st)
