"""GPU forward through the C ABI against the oracle.

Tiny case: every output, plus the intermediates in the workspace (routing
arrays and quantized X bit-exact, quantized A codes up to rounding-boundary
cases).  Full shape (H=3584, I=384, E=896, k=16): every output for decode
T in {1, 8, 16}; sampled tokens for prefill (T=4096, Zipf routing) and max
batch (T=16384, 1% of rows x50), with whole-output properties.  Edge cases:
ragged T, x = 0, exact-arithmetic inputs, invalid ids, per-expert SiTU
parameters, workspace reuse, CUDA-graph replay."""
import numpy as np
import pytest
import torch

import oracle
from oracle import cases
from nvfp4_routed_moe_gb300 import api
from nvfp4_routed_moe_gb300 import inputs as gen
from gpu_util import Model, assert_close, dev, out_bits, ws_i32, ws_u8, ws_view

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tiny():
    inp = cases.prepare_tiny(0)
    return inp, Model(inp)


def test_tiny_forward_matches_oracle(tiny):
    inp, m = tiny
    out, ws = m.forward_inputs()
    torch.cuda.synchronize()
    assert api.moe_read_status(ws) == (0, 0)
    ref = cases.run_oracle(inp)
    assert_close(out_bits(out), ref, "tiny")


@pytest.mark.parametrize("fc1", ["decode_kernel", "tcgen05"])
def test_tiny_intermediates(tiny, fc1, monkeypatch):
    """Routing arrays, quantized X (codes and block scales) bit-exact and the
    requantized A codes, with FC1 on the decode kernel (the default at this
    size: X's block scales token-major) and on the tcgen05 GEMM (block
    scales in the atoms of every routed row)."""
    inp, m = tiny
    if fc1 == "tcgen05":
        monkeypatch.setenv("NVFP4MOE_FC1_GEMV", "0")
    out, ws = m.forward_inputs()
    torch.cuda.synchronize()
    assert_close(out_bits(out), cases.run_oracle(inp), f"tiny, FC1 on the {fc1}")
    lay = ws_view(m, ws)
    T, k, E, H, I = inp.T, inp.k, inp.E, inp.H, inp.I
    P = T * k
    r = oracle.routing(inp.expert_ids, E)
    np.testing.assert_array_equal(ws_i32(ws, lay.count, E), r["count"])
    np.testing.assert_array_equal(ws_i32(ws, lay.cumsum, E), r["cumsum"])
    np.testing.assert_array_equal(ws_i32(ws, lay.sorted_row, P), r["sorted_row"])
    np.testing.assert_array_equal(ws_i32(ws, lay.gather, P), r["gather"])
    row_pos = ws_i32(ws, lay.row_pos, P)
    # padded row of pair f: expert segment start (rounded to 128) + rank within the expert
    pstart = np.concatenate([[0], np.cumsum((r["count"] + 127) // 128 * 128)])[:-1]
    rank = r["gather"] - (r["cumsum"] - r["count"])[inp.expert_ids.ravel()]
    np.testing.assert_array_equal(row_pos, pstart[inp.expert_ids.ravel()] + rank)
    # quantized X, bit-exact (oracle quantizes each token with qX): the codes
    # once per token, the block scales once per token (decode-kernel FC1) or
    # in the atoms of every routed row (tcgen05 FC1)
    xq_ref, xsf_ref = oracle.nvfp4_quant_rows(gen.bf16_bits_to_f32(inp.x), q=inp.qX)
    npad = int(row_pos.max()) + 1
    np.testing.assert_array_equal(ws_u8(ws, lay.xq, T * (H // 2)).reshape(T, H // 2), xq_ref)
    if fc1 == "decode_kernel":
        np.testing.assert_array_equal(ws_u8(ws, lay.sft, T * (H // 16)).reshape(T, H // 16), xsf_ref)
    else:
        sfx = ws_u8(ws, lay.sfx, ((npad + 127) // 128) * (H // 64) * 512)
        for f in range(P):
            t, p = f // k, row_pos[f]
            got_sf = [sfx[oracle.scale_atom_offset(p, c, H // 16)] for c in range(H // 16)]
            np.testing.assert_array_equal(got_sf, xsf_ref[t])
    # quantized A codes: equal except where FC1 sums round differently near a boundary
    _, mid = cases.run_oracle(inp, want_intermediates=True)
    aq = ws_u8(ws, lay.aq, npad * (I // 2)).reshape(npad, I // 2)
    table = np.array([oracle.e2m1_value(c) for c in range(16)])
    total = mism = 0
    for f in range(P):
        t, j, p = f // k, f % k, row_pos[f]
        g = np.stack([aq[p] & 15, aq[p] >> 4], -1).ravel()
        rr = np.stack([mid["aq"][t, j] & 15, mid["aq"][t, j] >> 4], -1).ravel()
        total += g.size
        mism += int((table[g] != table[rr]).sum())
    assert mism <= 0.01 * total, f"A code mismatch rate {mism}/{total}"


def test_two_pass_scale_layout_bit_exact():
    """Above 4096 routed pairs the X block scales are written per token and
    then laid out in atoms by a second pass.  On sampled tiles (and the last,
    partly filled one) the atoms equal the oracle's scales of each row's token
    scattered through the oracle's atom layout, zero on rows past the tile's
    fill, and the token-major packed codes equal the oracle's."""
    base = cases.prepare_tiny(3)
    inp = gen.tiny(3, 16400)          # weights and per-expert scales of the 16-token case
    for name in ("w13", "sf13", "w2", "sf2", "dXdW13", "qA", "dAdW2"):
        setattr(inp, name, getattr(base, name))
    m = Model(inp)
    out, ws = m.forward_inputs()
    torch.cuda.synchronize()
    assert api.moe_read_status(ws) == (0, 0)
    lay = ws_view(m, ws)
    T, k, H = inp.T, inp.k, inp.H
    ntiles = int(ws_i32(ws, lay.header, 8)[2])
    prow_pair = ws_i32(ws, lay.prow_pair, ntiles * 128)
    tl = ws_i32(ws, lay.tt_list, 4 * ntiles).reshape(ntiles, 4)
    xq_ref, xsf_ref = oracle.nvfp4_quant_rows(gen.bf16_bits_to_f32(inp.x), q=inp.qX)
    atom_bytes = (H // 64) * 512
    sample = set(np.random.default_rng(0).choice(ntiles, 6, replace=False).tolist()) | {ntiles - 1}
    for tile in sorted(sample):
        rows = int(tl[tile, 2])
        toks = prow_pair[tile * 128:tile * 128 + rows] // k
        exp_rows = np.zeros((128, H // 16), np.uint8)
        exp_rows[:rows] = xsf_ref[toks]
        got = ws_u8(ws, lay.sfx + tile * atom_bytes, atom_bytes)
        np.testing.assert_array_equal(got, oracle.to_atom_layout(exp_rows))
    np.testing.assert_array_equal(ws_u8(ws, lay.xq, T * (H // 2)).reshape(T, H // 2), xq_ref)
    toks = np.arange(0, T, 97)
    assert_close(out_bits(out)[toks], cases.run_oracle(inp, tokens=toks), "two-pass scales")


@pytest.mark.parametrize("T", [1, 2, 7, 33, 300])
def test_tiny_shape_ragged_token_counts(T):
    inp = cases.prepare_tiny(1, T=T)
    m = Model(inp)
    out, ws = m.forward_inputs()
    ref = cases.run_oracle(inp)
    assert_close(out_bits(out), ref, f"T={T}")
    assert api.moe_read_status(ws) == (0, 0)


@pytest.mark.parametrize("T", [33, 300])
def test_tiny_shape_decode_kernels_at_any_batch(T, monkeypatch):
    """FC1 and FC2 on the decode kernels forced above their default range:
    expert tiles of up to ~60 tokens (T = 300, 4 of 32 experts per token)
    take one job per 4 tokens over the same weight tiles, the last one
    ragged."""
    monkeypatch.setenv("NVFP4MOE_FC1_GEMV", "1")
    monkeypatch.setenv("NVFP4MOE_FC2_GEMV", "1")
    inp = cases.prepare_tiny(1, T=T)
    m = Model(inp)
    out, ws = m.forward_inputs()
    torch.cuda.synchronize()
    assert api.moe_read_status(ws) == (0, 0)
    assert_close(out_bits(out), cases.run_oracle(inp), f"T={T}, decode kernels")


def test_zero_input_gives_zero_output(tiny):
    inp, m = tiny
    x = torch.zeros((inp.T, inp.H), dtype=torch.bfloat16, device="cuda")
    out, _ = m.forward(x, dev(inp.expert_ids), dev(inp.route_weights, torch.bfloat16))
    assert not out.float().abs().sum().item()


def test_exact_inputs_match_to_the_last_bit():
    """Power-of-two block scales, grid-valued x and unit qX: X quantizes
    exactly and every FC1 sum is exact in fp32, so GPU and oracle see the same
    SiTU inputs; the outputs then agree bit for bit except where an fp32 sum
    lands on a bf16 rounding boundary (at most one bf16 ulp)."""
    H, I, E, k, T = 512, 128, 8, 2, 5
    rs = np.random.default_rng(11)
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], np.float32)
    x = rs.choice(np.concatenate([grid, -grid]), size=(T, H)).astype(np.float32)
    x[:, ::16] = 6.0
    ids = np.stack([rs.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    rw = gen.f32_to_bf16_bits(np.array([[0.5, 0.25]] * T, np.float32))
    inp = gen.MoEInputs(H, I, E, k, T, gen.f32_to_bf16_bits(x), ids, rw, np.float32(1.0))
    inp.w13 = rs.integers(0, 256, size=(E, 2 * I, H // 2), dtype=np.uint8)
    inp.sf13 = np.full((E, 2 * I, H // 16), 0x38, np.uint8)
    inp.w2 = rs.integers(0, 256, size=(E, H, I // 2), dtype=np.uint8)
    inp.sf2 = np.full((E, H, I // 16), 0x30, np.uint8)
    inp.dXdW13 = np.full(E, 2.0 ** -6, np.float32)
    inp.qA = np.full(E, 1.0, np.float32)
    inp.dAdW2 = np.full(E, 2.0 ** -6, np.float32)
    m = Model(inp)
    out, _ = m.forward_inputs()
    ref = cases.run_oracle(inp)
    got = out_bits(out)
    same = got == ref
    assert same.mean() >= 0.99, f"only {same.mean():.4f} of outputs identical"
    gv, rv = gen.bf16_bits_to_f32(got), gen.bf16_bits_to_f32(ref)
    assert np.all(np.abs(gv - rv) <= np.abs(rv) * 2.0 ** -7)


def test_invalid_ids_skipped_and_flagged(tiny):
    inp, m = tiny
    ids = inp.expert_ids.copy()
    ids[2, 1] = -5
    ids[9, 3] = inp.E + 3
    out, ws = m.forward(dev(inp.x, torch.bfloat16), dev(ids), dev(inp.route_weights, torch.bfloat16))
    st = api.moe_read_status(ws)
    assert st == (api.DEVSTAT_INVALID_EXPERT, 2)
    inp2 = cases.prepare_tiny(0)
    inp2.expert_ids = ids
    ref = cases.run_oracle(inp2)
    assert_close(out_bits(out), ref, "invalid ids")


def test_situ_parameters_per_expert(tiny):
    inp, m = tiny
    rs = np.random.default_rng(3)
    beta = rs.uniform(1.0, 6.0, inp.E).astype(np.float32)
    lam = rs.uniform(5.0, 40.0, inp.E).astype(np.float32)
    out, _ = m.forward_inputs(beta=dev(beta), lam=dev(lam))
    ref = cases.run_oracle(inp, beta=beta, lam=lam)
    assert_close(out_bits(out), ref, "situ beta/lambda")


def test_workspace_reuse_across_token_counts(tiny):
    """One maximum-size workspace serves every smaller prepared T."""
    inp, m = tiny
    ws = m.workspace(inp.T)
    for T in (inp.T, 3, 1):
        api.moe_prepare_workspace(m.shape, ws, T)
    x, ids, rw = dev(inp.x, torch.bfloat16), dev(inp.expert_ids), dev(inp.route_weights, torch.bfloat16)
    full = cases.run_oracle(inp)
    for T in (inp.T, 3, 1):
        out, _ = m.forward(x[:T], ids[:T], rw[:T], ws=ws, T=T, prepare=False)
        assert_close(out_bits(out), full[:T], f"reuse T={T}")


def test_not_prepared_is_rejected(tiny):
    """A workspace never passed to moe_prepare_workspace for this T is
    refused (its byte size is unique in this module, so no earlier prepared
    entry with a recycled address can match)."""
    inp, m = tiny
    ws = m.workspace(inp.T + 61)
    with pytest.raises(api.MoeError) as e:
        m.forward_inputs(ws=ws, prepare=False)
    assert e.value.status == 4


def test_cuda_graph_replay(tiny):
    inp, m = tiny
    x, ids, rw = dev(inp.x, torch.bfloat16), dev(inp.expert_ids), dev(inp.route_weights, torch.bfloat16)
    ws = m.workspace(inp.T)
    api.moe_prepare_workspace(m.shape, ws, inp.T)
    out = torch.empty((inp.T, inp.H), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        m.forward(x, ids, rw, ws=ws, out=out, prepare=False)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        m.forward(x, ids, rw, ws=ws, out=out, prepare=False)
    ref = cases.run_oracle(inp)
    for _ in range(3):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert_close(out_bits(out), ref, "graph replay")
    # new inputs in the same buffers
    inp2 = cases.prepare_tiny(0)
    inp2.x = gen.draw_x(9, inp.T, inp.H)
    inp2.expert_ids = gen.draw_ids_uniform(9, inp.T, inp.E, inp.k)
    inp2.qX = inp.qX          # the captured graph keeps reading the same qX buffer
    x.copy_(dev(inp2.x, torch.bfloat16))
    ids.copy_(dev(inp2.expert_ids))
    g.replay()
    torch.cuda.synchronize()
    assert_close(out_bits(out), cases.run_oracle(inp2), "graph replay new inputs")


# ------------------------------------------------------------------ full shape
@pytest.fixture(scope="module")
def full_model():
    inp = gen.full(0, T=16)
    return inp, Model(inp)


def _full_case(model_inp, T, routing, big=0.0, seed=0):
    inp = gen.full(seed, T=T, routing=routing, big_rows_frac=big, weights=False)
    inp.w13, inp.sf13, inp.w2, inp.sf2 = model_inp.w13, model_inp.sf13, model_inp.w2, model_inp.sf2
    inp.dXdW13, inp.qA, inp.dAdW2 = model_inp.dXdW13, model_inp.qA, model_inp.dAdW2
    return inp


@pytest.mark.parametrize("T", [1, 8, 16])
def test_full_shape_decode_all_tokens(full_model, T):
    minp, m = full_model
    inp = _full_case(minp, T, "uniform", seed=T)
    out, ws = m.forward_inputs(inp)
    torch.cuda.synchronize()
    assert api.moe_read_status(ws) == (0, 0)
    ref = cases.run_oracle(inp)
    assert_close(out_bits(out), ref, f"decode T={T}")


_GEMM_PATHS = [("1", "1"), ("0", "0"), ("1", "0"), ("0", "1")]


@pytest.mark.parametrize("T", [1, 8, 16, 32])
def test_full_shape_decode_kernels_and_tensor_core_gemms(full_model, T, monkeypatch):
    """FC1 and FC2 each on the decode kernels (warp-level MMAs over streamed
    weights; the default up to 16 tokens) or on the tcgen05 GEMMs, in all
    four combinations: each against the oracle on every token, and each
    within the tolerance of the tcgen05 pair."""
    minp, m = full_model
    inp = _full_case(minp, T, "uniform", seed=700 + T)
    ref = cases.run_oracle(inp)
    outs = {}
    for f1, f2 in _GEMM_PATHS:
        monkeypatch.setenv("NVFP4MOE_FC1_GEMV", f1)
        monkeypatch.setenv("NVFP4MOE_FC2_GEMV", f2)
        out, ws = m.forward_inputs(inp)
        torch.cuda.synchronize()
        assert api.moe_read_status(ws) == (0, 0)
        outs[f1, f2] = out_bits(out)
        assert_close(outs[f1, f2], ref, f"T={T}, NVFP4MOE_FC1_GEMV={f1} NVFP4MOE_FC2_GEMV={f2}")
    for key in _GEMM_PATHS[2:] + _GEMM_PATHS[:1]:
        assert_close(outs[key], outs["0", "0"], f"T={T}: {key} against the tcgen05 GEMMs")


@pytest.mark.parametrize("T", [7, 32])
@pytest.mark.parametrize("decode", ["default", "forced"])
def test_full_shape_crowded_expert_tiles_at_decode(full_model, T, decode, monkeypatch):
    """Every token routed to the same 16 experts (in its own order), so each
    expert tile holds all T tokens: the decode kernels take ceil(T/4) jobs
    per W13 tile and per group of W2 tiles, the last one ragged at T = 7
    (forced: the decode kernels at T = 32 too)."""
    minp, m = full_model
    if decode == "forced":
        monkeypatch.setenv("NVFP4MOE_FC1_GEMV", "1")
        monkeypatch.setenv("NVFP4MOE_FC2_GEMV", "1")
    inp = _full_case(minp, T, "uniform", seed=800 + T)
    rs = np.random.default_rng(800 + T)
    experts = rs.choice(inp.E, inp.k, replace=False).astype(np.int32)
    inp.expert_ids = np.stack([rs.permutation(experts) for _ in range(T)]).astype(np.int32)
    out, ws = m.forward_inputs(inp)
    torch.cuda.synchronize()
    assert api.moe_read_status(ws) == (0, 0)
    assert_close(out_bits(out), cases.run_oracle(inp), f"T={T}, crowded tiles, {decode}")


@pytest.mark.parametrize("T", [16, 2048])
def test_full_shape_per_expert_situ_parameters(full_model, T):
    """Non-default per-expert gate and linear smoothing ("Cake SiTU backend":
    situ_beta / situ_linear_beta, float32 [896]) at full shape: every token
    at decode size, sampled tokens at T=2048."""
    minp, m = full_model
    inp = _full_case(minp, T, "uniform", seed=40 + T)
    rs = np.random.default_rng(T)
    beta = rs.uniform(1.0, 8.0, inp.E).astype(np.float32)
    lam = rs.uniform(2.0, 60.0, inp.E).astype(np.float32)
    out, ws = m.forward_inputs(inp, beta=dev(beta), lam=dev(lam))
    torch.cuda.synchronize()
    assert api.moe_read_status(ws) == (0, 0)
    toks = np.arange(T) if T <= 16 else np.unique(np.concatenate([[0, T - 1], rs.choice(T, 14, replace=False)]))
    ref = cases.run_oracle(inp, tokens=toks, beta=beta, lam=lam)
    assert_close(out_bits(out)[toks], ref, f"situ params T={T}")
    default = cases.run_oracle(inp, tokens=toks[:4])
    assert not np.array_equal(ref[:4], default)      # the parameters do change the result


@pytest.mark.parametrize("T,routing,big", [(512, "uniform", 0.0)])
def test_full_shape_sampled_tokens(full_model, T, routing, big):
    minp, m = full_model
    inp = _full_case(minp, T, routing, big)
    out, ws = m.forward_inputs(inp)
    torch.cuda.synchronize()
    assert api.moe_read_status(ws) == (0, 0)
    rs = np.random.default_rng(T)
    sample = np.unique(np.concatenate([[0, T - 1], rs.choice(T, 14, replace=False)]))
    if big:
        xf = np.abs(gen.bf16_bits_to_f32(inp.x)).max(axis=1)
        sample = np.unique(np.concatenate([sample, np.argsort(-xf)[:2]]))
    ref = cases.run_oracle(inp, tokens=sample)
    assert_close(out_bits(out)[sample], ref, f"T={T} {routing}")
    assert torch.isfinite(out.float()).all()
    counts = np.bincount(inp.expert_ids.ravel(), minlength=inp.E)
    lay = ws_view(m, ws)
    np.testing.assert_array_equal(ws_i32(ws, lay.count, inp.E), counts)



def _tile_boundary_tokens(ids, E):
    """Tokens of the rows where the tiling changes: for every expert, the
    first row of its group, the first row of each further 128-row tile and
    the last row (the last, partly filled tile's end), in the stable expert
    order of the routing ("npu_moe_init_routing_v2", keyValueSort)."""
    r = oracle.routing(ids, E)
    k = ids.shape[1]
    start = r["cumsum"] - r["count"]
    rows = []
    for e in np.nonzero(r["count"])[0]:
        n = int(r["count"][e])
        rows += [int(start[e]) + j for j in range(0, n, 128)] + [int(start[e]) + n - 1]
    return np.unique(r["sorted_row"][np.array(rows)] // k)


@pytest.mark.parametrize("T,routing,big", [(4096, "zipf", 0.0), (16384, "uniform", 0.01)])
def test_full_shape_tile_boundary_tokens(full_model, T, routing, big):
    """Prefill (Zipf routing) and max batch (uniform, 1% of rows x50) at full
    shape: the tokens at every expert's first row, 128-row tile boundaries and
    last row -- the rows where tiles, padding and partly filled last tiles
    start and end -- plus the largest rows, against the oracle."""
    minp, m = full_model
    inp = _full_case(minp, T, routing, big)
    out, ws = m.forward_inputs(inp)
    torch.cuda.synchronize()
    assert api.moe_read_status(ws) == (0, 0)
    sample = _tile_boundary_tokens(inp.expert_ids, inp.E)
    if big:
        xf = np.abs(gen.bf16_bits_to_f32(inp.x)).max(axis=1)
        sample = np.unique(np.concatenate([sample, np.argsort(-xf)[:8]]))
    assert len(sample) >= (900 if T == 4096 else 1500)
    ref = cases.run_oracle(inp, tokens=sample)
    assert_close(out_bits(out)[sample], ref, f"T={T} {routing} tile boundaries")
    assert torch.isfinite(out.float()).all()
    counts = np.bincount(inp.expert_ids.ravel(), minlength=inp.E)
    lay = ws_view(m, ws)
    np.testing.assert_array_equal(ws_i32(ws, lay.count, inp.E), counts)


@pytest.mark.parametrize("T", [32, 128, 1024, 8192])
def test_full_shape_sweep_points(full_model, T):
    """The decode-to-prefill sweep's batch sizes (uniform ids): every token at
    T = 32 and 128 (FC1's two-tile units start above 16 tokens; FC2's
    accumulator slots widen at 32 and 64 rows), 256 sampled tokens plus the
    tile-boundary tokens of the first 64 experts above that."""
    minp, m = full_model
    inp = _full_case(minp, T, "uniform", seed=200 + T)
    out, ws = m.forward_inputs(inp)
    torch.cuda.synchronize()
    assert api.moe_read_status(ws) == (0, 0)
    if T <= 128:
        sample = np.arange(T)
    else:
        rs = np.random.default_rng(T)
        ids = inp.expert_ids
        bound = _tile_boundary_tokens(np.where(ids < 64, ids, 10 ** 6).astype(np.int32), 64)
        sample = np.unique(np.concatenate([rs.choice(T, 256, replace=False), bound, [0, T - 1]]))
    ref = cases.run_oracle(inp, tokens=sample)
    assert_close(out_bits(out)[sample], ref, f"sweep T={T}")


def _fc1_abs_sums(inp, toks):
    """sum_h |x^_h| |w^_{e,n,h}| for every listed token's pairs and FC1 row,
    from the oracle's quantized X and dequantized weights (fp64)."""
    xq, xsf = oracle.nvfp4_quant_rows(gen.bf16_bits_to_f32(inp.x[toks]), q=inp.qX)
    X = np.abs(oracle.nvfp4_dequant_rows(xq, xsf))
    out = np.zeros((len(toks), inp.k, 2 * inp.I))
    for ti, t in enumerate(toks):
        for j in range(inp.k):
            e = inp.expert_ids[t, j]
            W = np.abs(oracle.nvfp4_dequant_rows(inp.w13[e], inp.sf13[e]))
            out[ti, j] = W @ X[ti]
    return out


@pytest.mark.parametrize("fc1", ["decode_kernel", "tcgen05"])
def test_full_shape_decode_intermediate_codes(full_model, fc1, monkeypatch):
    """The requantized intermediate A of every routed pair at T = 16, read from
    the workspace, against the oracle's codes, with FC1 on the decode kernel
    (the default at this size) and on the tcgen05 GEMM.  FC1's fp32 sums
    round in the hardware's order, so a code may differ only where the
    oracle's SiTU value, moved by at most the fp32 summation error of its
    pre-activations (57 fp32 roundings of the sum of absolute products: one
    per K = 64 MMA step and one for the product; the decode kernel has fewer
    in any product's path: 16 MMA steps of a k-block in four chains, their
    3 sums, 14 k-block sums, the two k-block parities' sum and the product),
    crosses an E2M1 rounding midpoint -- or
    where the group's block scale itself differs because its amax crosses an
    E4M3 midpoint the same way.  The mismatch rate is reported."""
    minp, m = full_model
    T = 16
    inp = _full_case(minp, T, "uniform", seed=T)
    if fc1 == "tcgen05":
        monkeypatch.setenv("NVFP4MOE_FC1_GEMV", "0")
    out, ws = m.forward_inputs(inp)
    torch.cuda.synchronize()
    assert api.moe_read_status(ws) == (0, 0)
    lay = ws_view(m, ws)
    I, k = inp.I, inp.k
    toks = np.arange(T)
    _, mid = cases.run_oracle(inp, tokens=toks, want_intermediates=True)
    row_pos = ws_i32(ws, lay.row_pos, T * k)
    npad = int(row_pos.max()) + 1
    aq = ws_u8(ws, lay.aq, npad * (I // 2)).reshape(npad, I // 2)
    sfa = ws_u8(ws, lay.sfa, ((npad + 127) // 128) * (I // 64) * 512)
    dz = 57 * 2.0 ** -24 * _fc1_abs_sums(inp, toks) * inp.dXdW13[inp.expert_ids][..., None]
    table = np.array([oracle.e2m1_value(c) for c in range(16)])
    e4 = np.array(sorted({oracle.e4m3_value(c) for c in range(0x7F)}))
    e4_mids = (e4[1:] + e4[:-1]) / 2
    e2_mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
    n_codes = n_code_mis = n_sf_mis = 0
    for t in range(T):
        for j in range(k):
            e = inp.expert_ids[t, j]
            p = row_pos[t * k + j]
            z = mid["z"][t, j].astype(np.float64)
            g, u, dg, du = z[:I], z[I:], dz[t, j, :I], dz[t, j, I:]
            corners = np.stack([[oracle.situ(g[i] + sg * dg[i], u[i] + su * du[i]) for i in range(I)]
                                for sg in (-1, 1) for su in (-1, 1)] +
                               [[oracle.situ(g[i], u[i]) for i in range(I)]])
            a_lo, a_hi = corners.min(0), corners.max(0)
            got_codes = np.stack([aq[p] & 15, aq[p] >> 4], -1).ravel()
            ref_codes = np.stack([mid["aq"][t, j] & 15, mid["aq"][t, j] >> 4], -1).ravel()
            qa = np.float64(np.float32(inp.qA[e]))
            for grp in range(I // 16):
                sl = slice(16 * grp, 16 * grp + 16)
                got_sf = sfa[oracle.scale_atom_offset(p, grp, I // 16)]
                ref_sf = mid["asf"][t, j, grp]
                n_codes += 16
                if got_sf != ref_sf:
                    amax_lo = np.max(np.minimum(np.abs(a_lo[sl]), np.abs(a_hi[sl]))) * qa / 6
                    amax_hi = np.max(np.maximum(np.abs(a_lo[sl]), np.abs(a_hi[sl]))) * qa / 6
                    crossed = ((e4_mids >= amax_lo * (1 - 1e-7)) & (e4_mids <= amax_hi * (1 + 1e-7))).any()
                    assert crossed, f"scale of token {t} pair {j} group {grp} differs away from a boundary"
                    n_sf_mis += 1
                    continue
                S = oracle.e4m3_value(int(ref_sf))
                r = 0.0 if S == 0 else qa / S
                bad = table[got_codes[sl]] != table[ref_codes[sl]]
                for i in np.nonzero(bad)[0]:
                    y_lo, y_hi = sorted((abs(a_lo[sl][i]) * r, abs(a_hi[sl][i]) * r))
                    crossed = ((e2_mids >= y_lo * (1 - 1e-7)) & (e2_mids <= y_hi * (1 + 1e-7))).any()
                    assert crossed, f"code of token {t} pair {j} element {16 * grp + i} differs away from a boundary"
                    n_code_mis += 1
    print(f"A codes: {n_code_mis} of {n_codes} differ, {n_sf_mis} block scales differ (all at rounding boundaries)")
    assert n_code_mis <= 0.01 * n_codes

@pytest.mark.parametrize("T", [2048, 16384])
def test_back_to_back_forwards_share_a_workspace(full_model, T):
    """Two forwards with different inputs run back to back on one workspace,
    with no synchronization between them: the second one quantizes X and
    zeroes the accumulator rows ahead of its own routing, which must still
    come after the first one's finalize.  Both outputs match the oracle on
    sampled tokens (T=2048: block scales placed by the X quantizer; 16384:
    by the scale-atom kernel)."""
    minp, m = full_model
    cases_ab = (_full_case(minp, T, "uniform", seed=70 + T), _full_case(minp, T, "zipf", seed=71 + T))
    ws = m.workspace(T)
    api.moe_prepare_workspace(m.shape, ws, T)
    staged = [(dev(c.x, torch.bfloat16), dev(c.expert_ids), dev(c.route_weights, torch.bfloat16),
               dev(np.array([c.qX], np.float32))) for c in cases_ab]
    torch.cuda.synchronize()
    outs = [m.forward(x, ids, rw, ws=ws, T=T, prepare=False, qX=qx)[0] for x, ids, rw, qx in staged]
    torch.cuda.synchronize()
    assert api.moe_read_status(ws) == (0, 0)
    rs = np.random.default_rng(T)
    sample = np.unique(np.concatenate([[0, T - 1], rs.choice(T, 10, replace=False)]))
    for c, out, name in zip(cases_ab, outs, ("first", "second")):
        assert_close(out_bits(out)[sample], cases.run_oracle(c, tokens=sample), f"back to back, {name}, T={T}")


def test_concurrent_forwards_on_two_streams(full_model):
    """Two forwards with their own workspaces and outputs, enqueued on two
    streams without ordering between them (the library's contract for
    concurrent calls): both match the oracle on sampled tokens."""
    minp, m = full_model
    T = 2048
    cases_ab = (_full_case(minp, T, "uniform", seed=80), _full_case(minp, T, "zipf", seed=81))
    streams = (torch.cuda.Stream(), torch.cuda.Stream())
    staged, wss, outs = [], [], []
    for c in cases_ab:
        staged.append((dev(c.x, torch.bfloat16), dev(c.expert_ids), dev(c.route_weights, torch.bfloat16),
                       dev(np.array([c.qX], np.float32))))
        ws = m.workspace(T)
        api.moe_prepare_workspace(m.shape, ws, T)
        wss.append(ws)
        outs.append(torch.empty((T, c.H), dtype=torch.bfloat16, device="cuda"))
    torch.cuda.synchronize()
    for (x, ids, rw, qx), ws, out, st in zip(staged, wss, outs, streams):
        api.moe_forward(m.shape, T, x, ids, rw, m.w13, m.sf13, m.w2, m.sf2, qx, m.dXdW13, m.qA, m.dAdW2, None,
                        None, ws, out, st)
    torch.cuda.synchronize()
    rs = np.random.default_rng(5)
    sample = np.unique(np.concatenate([[0, T - 1], rs.choice(T, 10, replace=False)]))
    for c, ws, out, name in zip(cases_ab, wss, outs, ("first", "second")):
        assert api.moe_read_status(ws) == (0, 0)
        assert_close(out_bits(out)[sample], cases.run_oracle(c, tokens=sample), f"concurrent, {name}")

def test_full_shape_streamed_chunks(full_model):
    """The chunk-ready streaming front end at full shape: T = 4096 published
    as four 1024-token chunks through a two-slot ring, each routed on its own;
    sampled tokens match the oracle and the whole output matches the batch
    forward within the tolerance."""
    minp, m = full_model
    T, C = 4096, 1024
    inp = _full_case(minp, T, "uniform", seed=3)
    x, ids, rw = dev(inp.x, torch.bfloat16), dev(inp.expert_ids), dev(inp.route_weights, torch.bfloat16)
    qX = dev(np.array([inp.qX], np.float32))
    cfg = api.moe_stream_ring_t(2, C)
    ring = torch.empty(api.moe_stream_ring_size(m.shape, cfg), dtype=torch.uint8, device="cuda")
    api.moe_stream_ring_init(m.shape, cfg, ring)
    ws = m.workspace(C)
    api.moe_prepare_workspace(m.shape, ws, C)
    out = torch.empty((T, inp.H), dtype=torch.bfloat16, device="cuda")
    api.moe_stream_begin(m.shape, cfg, ring)
    for c in range(T // C):
        sl = slice(c * C, (c + 1) * C)
        api.moe_stream_publish(m.shape, cfg, ring, c, c * C, C, api.STREAM_ROUTE | api.STREAM_LAYOUT, x[sl], ids[sl],
                               rw[sl])
        api.moe_stream_forward(m.shape, cfg, ring, c, m.w13, m.sf13, m.w2, m.sf2, qX, m.dXdW13, m.qA, m.dAdW2,
                               None, None, ws, out)
    torch.cuda.synchronize()
    assert api.moe_read_status(ws) == (0, 0)
    assert api.moe_stream_read_status(ring) == 0
    sample = np.unique(np.concatenate([[0, C - 1, C, T - 1], np.random.default_rng(9).choice(T, 12, replace=False)]))
    assert_close(out_bits(out)[sample], cases.run_oracle(inp, tokens=sample), "streamed full shape")
    batch, _ = m.forward(x, ids, rw, qX=qX)
    assert_close(out_bits(out), out_bits(batch), "streamed vs batch, full shape")


# ------------------------------------------------------------- expert slices
# The forward of one expert-parallel rank ("npu_moe_init_routing_v2",
# active_expert_range): the rank holds experts [begin, begin + E_local) and
# returns the route-weighted sum over them only.  The oracle is the same
# forward with the ids shifted by -begin (ids outside [0, E_local) are not
# routed) and the slice's weights and scales.

def _slice(inp, begin, n):
    s = gen.MoEInputs(inp.H, inp.I, n, inp.k, inp.T, inp.x, inp.expert_ids - begin, inp.route_weights, inp.qX)
    s.w13, s.sf13, s.w2, s.sf2 = (a[begin:begin + n] for a in (inp.w13, inp.sf13, inp.w2, inp.sf2))
    s.dXdW13, s.qA, s.dAdW2 = (a[begin:begin + n] for a in (inp.dXdW13, inp.qA, inp.dAdW2))
    return s


def _local_forward(inp_slice, begin, global_ids):
    m = Model(inp_slice)
    T = inp_slice.T
    ws = m.workspace(T)
    api.moe_prepare_workspace(m.shape, ws, T)
    out = torch.empty((T, inp_slice.H), dtype=torch.bfloat16, device="cuda")
    api.moe_forward_local_experts(m.shape, begin, T, dev(inp_slice.x, torch.bfloat16), dev(global_ids),
                                  dev(inp_slice.route_weights, torch.bfloat16), m.w13, m.sf13, m.w2, m.sf2,
                                  dev(np.array([inp_slice.qX], np.float32)), m.dXdW13, m.qA, m.dAdW2, None, None,
                                  ws, out)
    torch.cuda.synchronize()
    return out, ws


@pytest.mark.parametrize("begin,n", [(0, 16), (16, 16), (5, 11)])
def test_local_expert_slice_tiny(begin, n):
    inp = cases.prepare_tiny(0, T=40)
    sl = _slice(inp, begin, n)
    out, ws = _local_forward(sl, begin, inp.expert_ids)
    assert api.moe_read_status(ws) == (0, 0)       # pairs of other ranks are not errors
    assert_close(out_bits(out), cases.run_oracle(sl), f"slice {begin}+{n}")


def test_local_expert_slices_sum_to_the_full_forward():
    inp = gen.full(21, T=16, routing="uniform", weights=True)
    full = cases.run_oracle(inp)
    total = np.zeros((inp.T, inp.H), np.float64)
    for begin in (0, 448):
        sl = _slice(inp, begin, 448)
        out, _ = _local_forward(sl, begin, inp.expert_ids)
        part = out_bits(out)
        assert_close(part, cases.run_oracle(sl), f"slice {begin}")
        total += gen.bf16_bits_to_f32(part)
    assert_close(gen.f32_to_bf16_bits(total.astype(np.float32)), full, "sum of slices")


def test_recycled_workspace_memory_is_refused_on_the_device(tiny):
    """A prepared workspace is freed and the caching allocator hands the
    same block back (same address, same size) holding other data: the host
    record still says "prepared", but the header's preparation stamp is gone,
    so the forward sets MOE_DEVSTAT_NOT_PREPARED and leaves the output zero
    instead of computing from foreign bytes.  Preparing it again restores
    the normal result."""
    inp, m = tiny
    nbytes = api.moe_workspace_size(m.shape, inp.T + 77)    # a size no other test uses
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    api.moe_prepare_workspace(m.shape, ws, inp.T)
    torch.cuda.synchronize()
    addr = ws.data_ptr()
    del ws
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    if ws.data_ptr() != addr:
        pytest.skip("the caching allocator returned another block")
    ws.fill_(0xA5)
    out, _ = m.forward_inputs(ws=ws, prepare=False)
    torch.cuda.synchronize()
    status, _ = api.moe_read_status(ws)
    assert status & api.DEVSTAT_NOT_PREPARED
    assert not out.float().abs().sum().item()
    api.moe_prepare_workspace(m.shape, ws, inp.T)
    out, _ = m.forward_inputs(ws=ws, prepare=False)
    torch.cuda.synchronize()
    assert api.moe_read_status(ws) == (0, 0)
    assert_close(out_bits(out), cases.run_oracle(inp), "re-prepared")


@pytest.mark.parametrize("env", [{"NVFP4MOE_FC1_DYNAMIC": "0", "NVFP4MOE_FC2_DYNAMIC": "0"},
                                 {"NVFP4MOE_FC2_TILE_STAGES": "0"}, {"NVFP4MOE_FC2_TAIL": "1"},
                                 {"NVFP4MOE_FC2_TAIL": "8", "NVFP4MOE_FC2_GROUP": "28"},
                                 {"NVFP4MOE_FC2_GROUP": "4", "NVFP4MOE_FC2_DYNAMIC": "0"}])
def test_full_shape_scheduling_options(full_model, env, monkeypatch):
    """The GEMMs' scheduling options give the same result: units by the
    routing-seeded work counters or by the static stride, FC2 ring stages of
    a whole output tile or of one k-block, FC2's last units split into
    parts or not, other unit widths.  T = 1024 (uniform ids), Zipf T = 4096
    (heavy tiles: the split applies by default) and T = 16384 with the
    options of the environment, sampled tile-boundary tokens against the
    oracle and the whole output against the default configuration within
    the tolerance."""
    minp, m = full_model
    for T, routing in ((1024, "uniform"), (4096, "zipf"), (16384, "uniform")):
        inp = _full_case(minp, T, routing, seed=300 + T)
        ref_out, _ = m.forward_inputs(inp)
        torch.cuda.synchronize()
        for k, v in env.items():
            monkeypatch.setenv(k, v)
        out, ws = m.forward_inputs(inp)
        torch.cuda.synchronize()
        for k in env:
            monkeypatch.delenv(k)
        assert api.moe_read_status(ws) == (0, 0)
        ids = inp.expert_ids
        sample = _tile_boundary_tokens(np.where(ids < 32, ids, 10 ** 6).astype(np.int32), 32)[:200]
        assert_close(out_bits(out)[sample], cases.run_oracle(inp, tokens=sample), f"T={T} {routing} {env}")
        assert_close(out_bits(out), out_bits(ref_out), f"T={T} {routing} {env} against the default")


def test_full_shape_zero_and_subnormal_weight_block_scales(full_model):
    """Full-shape decode (T = 16, every token) with a fifth of the W13 and W2
    block scales replaced by the zero scale (0x00) and E4M3 subnormals
    (0x01-0x07): zero blocks must contribute nothing and subnormal ones
    their exact 2^-9 multiples, in FC1 and FC2 alike."""
    minp, _ = full_model
    T = 16
    inp = _full_case(minp, T, "uniform", seed=500)
    rs = np.random.default_rng(500)
    used = np.unique(inp.expert_ids)
    sf13, sf2 = inp.sf13.copy(), inp.sf2.copy()
    for sf in (sf13, sf2):
        sub = sf[used]
        mask = rs.random(sub.shape) < 0.2
        sub[mask] = rs.integers(0, 8, size=int(mask.sum()), dtype=np.uint8)
        sf[used] = sub
    inp.sf13, inp.sf2 = sf13, sf2
    m = Model(inp)
    out, ws = m.forward_inputs(inp)
    torch.cuda.synchronize()
    assert api.moe_read_status(ws) == (0, 0)
    assert_close(out_bits(out), cases.run_oracle(inp), "zero and subnormal weight scales")
