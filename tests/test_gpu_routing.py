"""GPU init-routing ("npu_moe_init_routing_v2", formulas 1-5) through the C
ABI against the oracle, bit-exact: expanded_row_idx (gather and scatter),
histogram (cumsum and count), dynamic int8 rows and scales, drop/pad."""
import numpy as np
import pytest
import torch

import oracle
from nvfp4_routed_moe_gb300 import api
from nvfp4_routed_moe_gb300 import inputs as gen
from gpu_util import dev

pytestmark = pytest.mark.gpu


def _run(x, ids, E, opts: api.moe_routing_opts_t, inter=128):
    T, H = x.shape
    k = ids.shape[1]
    shp = api.shape(H, inter, E, k)
    ws = torch.empty(api.moe_workspace_size(shp, T), dtype=torch.uint8, device="cuda")
    api.moe_prepare_workspace(shp, ws, T)
    rows = E * opts.expert_capacity if opts.drop_pad else T * k
    if opts.quant_mode == 1:
        ex = torch.full((rows, H), 0x55, dtype=torch.int8, device="cuda")
    else:
        ex = torch.full((rows, H), 0x5555, dtype=torch.int16, device="cuda")
    ridx = torch.full((T * k,), -7, dtype=torch.int32, device="cuda")
    tok = torch.empty(E, dtype=torch.int32, device="cuda")
    scale = torch.full((rows,), -1.0, dtype=torch.float32, device="cuda") if opts.quant_mode == 1 else None
    api.moe_init_routing(shp, T, dev(x, torch.bfloat16), dev(ids), opts, ex, ridx, tok, scale, ws)
    st = api.moe_read_status(ws)
    return (ex.cpu().numpy(), ridx.cpu().numpy(), tok.cpu().numpy(),
            None if scale is None else scale.cpu().numpy(), st)


def _check(x, ids, E, drop_pad=0, C=0, row_idx_type=0, tokens_num_type=0, quant_mode=1):
    opts = api.moe_routing_opts_t(drop_pad, C, row_idx_type, tokens_num_type, quant_mode)
    ex, ridx, tok, scale, st = _run(x, ids, E, opts)
    rex, rridx, rtok, rscale, nvalid = oracle.init_routing(x, ids, E, drop_pad=drop_pad, expert_capacity=C,
                                                           row_idx_type=row_idx_type,
                                                           tokens_num_type=tokens_num_type, quant_mode=quant_mode)
    np.testing.assert_array_equal(tok, rtok)
    np.testing.assert_array_equal(ridx, rridx)
    if drop_pad:
        np.testing.assert_array_equal(ex.view(rex.dtype), rex)
    else:
        np.testing.assert_array_equal(ex[:nvalid].view(rex.dtype), rex[:nvalid])
    if quant_mode == 1:
        n = rscale.shape[0] if drop_pad else nvalid
        np.testing.assert_array_equal(scale[:n], rscale[:n])
    return st


def test_routing_config_dropless_gather_cumsum_int8():
    """NUM_ROWS=4096, K=16, E=896, H=3584, uniform distinct ids: dropless,
    gather index, cumsum, dynamic int8 (the init-routing workload)."""
    x = gen.draw_x(0, 4096, 3584)
    ids = gen.draw_ids_uniform(0, 4096, 896, 16)
    st = _check(x, ids, 896)
    assert st == (0, 0)


def test_routing_config_drop_pad_c96():
    x = gen.draw_x(0, 4096, 3584)
    ids = gen.draw_ids_uniform(0, 4096, 896, 16)
    _check(x, ids, 896, drop_pad=1, C=96)


@pytest.mark.parametrize("T,E,k", [(1, 32, 4), (16, 32, 4), (3, 896, 16), (300, 64, 8), (257, 896, 16),
                                   (1000, 128, 16)])
def test_routing_small_and_multiblock(T, E, k):
    x = gen.draw_x(T, T, 512)
    ids = gen.draw_ids_zipf(T, T, E, k)
    _check(x, ids, E)
    _check(x, ids, E, row_idx_type=1, tokens_num_type=1, quant_mode=-1)


def test_routing_invalid_ids_are_skipped_and_flagged():
    T, E, k = 40, 32, 4
    x = gen.draw_x(1, T, 512)
    ids = gen.draw_ids_uniform(1, T, E, k)
    ids[3, 1] = -1
    ids[17, 0] = E
    ids[39, 3] = 1 << 30
    st = _check(x, ids, E)
    assert st == (api.DEVSTAT_INVALID_EXPERT, 3)


def test_routing_zero_rows_and_duplicates():
    T, E, k = 24, 16, 4
    x = gen.draw_x(2, T, 512)
    x[5] = 0
    ids = gen.draw_ids_uniform(2, T, E, k)
    ids[7] = [3, 3, 3, 3]          # duplicates within a row: still a stable sort by flat index
    _check(x, ids, E)
    _check(x, ids, E, drop_pad=1, C=3)


# ------------------------------------------------- the op's remaining options
# active_expert_range, active_num, key_value histogram, static int8, smooth
# scale, carried token scale ("npu_moe_init_routing_v2", formulas 1-6).

def _run_ex(x, ids, E, kw, static=False):
    T, H = x.shape
    k = ids.shape[1]
    shp = api.shape(H, 128, E, k)
    qm = kw.get("quant_mode", 1)
    lo, hi = kw.get("expert_start", 0), kw.get("expert_end", 0) or E
    R = hi - lo
    rows = R * kw["expert_capacity"] if kw.get("drop_pad") else T * k
    ex = torch.full((rows, H), 0x55, dtype=torch.int8, device="cuda") if qm != -1 else \
        torch.full((rows, H), 0x5555, dtype=torch.int16, device="cuda")
    ridx = torch.full((T * k,), -7, dtype=torch.int32, device="cuda")
    ntok = 2 * E if kw.get("tokens_num_type") == 2 else R
    tok = torch.full((ntok,), -9, dtype=torch.int32, device="cuda")
    scale_out = torch.full((rows,), -1.0, dtype=torch.float32, device="cuda")
    avail = torch.full((1,), -3, dtype=torch.int32, device="cuda")
    sc = None if kw.get("scale") is None else dev(np.asarray(kw["scale"], np.float32))
    of = None if kw.get("offset") is None else dev(np.asarray(kw["offset"], np.float32))
    srows = sc.shape[0] if (sc is not None and qm == 1) else 0
    opts = api.routing_opts(drop_pad=kw.get("drop_pad", 0), expert_capacity=kw.get("expert_capacity", 0),
                            row_idx_type=kw.get("row_idx_type", 0), tokens_num_type=kw.get("tokens_num_type", 0),
                            quant_mode=qm, expert_start=lo, expert_end=kw.get("expert_end", 0),
                            active_num=kw.get("active_num", 0), scale=sc, scale_rows=srows, offset=of,
                            available_out=avail)
    xd, idd = dev(x, torch.bfloat16), dev(ids)
    if static:
        api.moe_init_routing_static(shp, T, xd, idd, opts, ex, ridx, tok, scale_out)
        torch.cuda.synchronize()
        st = None
    else:
        ws = torch.empty(api.moe_workspace_size(shp, T), dtype=torch.uint8, device="cuda")
        api.moe_prepare_workspace(shp, ws, T)
        api.moe_init_routing(shp, T, xd, idd, opts, ex, ridx, tok, scale_out, ws)
        st = api.moe_read_status(ws)
    return ex.cpu().numpy(), ridx.cpu().numpy(), tok.cpu().numpy(), scale_out.cpu().numpy(), int(avail.item()), st


def _check_ex(x, ids, E, static=False, **kw):
    ex, ridx, tok, sc, avail, st = _run_ex(x, ids, E, kw, static)
    okw = {k: v for k, v in kw.items() if k not in ("expert_end",)}
    if kw.get("expert_end"):
        okw["expert_end"] = kw["expert_end"]
    rex, rridx, rtok, rsc, ravail = oracle.init_routing_ex(x, ids, E, **okw)
    assert avail == ravail
    np.testing.assert_array_equal(ridx, rridx)
    np.testing.assert_array_equal(tok.reshape(rtok.shape), rtok)
    if kw.get("drop_pad"):
        moved = rex.shape[0]
    else:
        an = kw.get("active_num", 0)
        moved = min(an, ravail) if an > 0 else ravail
    np.testing.assert_array_equal(ex[:moved].view(rex.dtype), rex[:moved])
    if rsc is not None:
        np.testing.assert_array_equal(sc[:moved], rsc[:moved])
    return st


def test_expert_range_on_the_routing_workload():
    x = gen.draw_x(0, 4096, 3584)
    ids = gen.draw_ids_uniform(0, 4096, 896, 16)
    st = _check_ex(x, ids, 896, expert_start=100, expert_end=612)
    assert st == (0, 0)          # ids outside the range are not errors


@pytest.mark.parametrize("T,E,k,lo,hi", [(300, 64, 8, 5, 40), (1000, 128, 16, 0, 17), (3, 896, 16, 800, 896)])
def test_expert_range_scatter_count_unquantized(T, E, k, lo, hi):
    x = gen.draw_x(T, T, 512)
    ids = gen.draw_ids_zipf(T, T, E, k)
    _check_ex(x, ids, E, expert_start=lo, expert_end=hi, row_idx_type=1, tokens_num_type=1, quant_mode=-1)
    _check_ex(x, ids, E, expert_start=lo, expert_end=hi, quant_mode=1)


@pytest.mark.parametrize("lo,hi", [(0, 0), (300, 700)])
def test_key_value_histogram(lo, hi):
    x = gen.draw_x(7, 257, 512)
    ids = gen.draw_ids_zipf(7, 257, 896, 16)
    _check_ex(x, ids, 896, expert_start=lo, expert_end=hi, tokens_num_type=2)


@pytest.mark.parametrize("row_idx_type", [0, 1])
def test_active_num(row_idx_type):
    x = gen.draw_x(8, 1000, 512)
    ids = gen.draw_ids_uniform(8, 1000, 128, 16)
    _check_ex(x, ids, 128, active_num=5000, row_idx_type=row_idx_type)
    _check_ex(x, ids, 128, active_num=5000, expert_start=10, expert_end=90, quant_mode=-1)


def test_static_int8():
    x = gen.draw_x(9, 64, 512)
    ids = gen.draw_ids_uniform(9, 64, 32, 4)
    _check_ex(x, ids, 32, quant_mode=0, scale=[0.37], offset=[-1.5])
    _check_ex(x, ids, 32, quant_mode=0, scale=[40.0], offset=[3.0], drop_pad=1, expert_capacity=6)
    _check_ex(x, ids, 32, quant_mode=0, scale=[0.37], offset=[-1.5], row_idx_type=1)
    xb = gen.draw_x(10, 2048, 512)      # 8192 pairs: the multi-block routing path
    idsb = gen.draw_ids_uniform(10, 2048, 32, 4)
    _check_ex(xb, idsb, 32, quant_mode=0, scale=[3.0], offset=[0.5])


def test_dynamic_int8_with_smooth_scale():
    T, E, k, lo, hi = 200, 64, 8, 8, 40
    x = gen.draw_x(10, T, 512)
    ids = gen.draw_ids_zipf(10, T, E, k)
    rs = np.random.default_rng(10)
    shared = rs.uniform(0.2, 3.0, (1, 512)).astype(np.float32)
    per_expert = rs.uniform(0.2, 3.0, (hi - lo, 512)).astype(np.float32)
    _check_ex(x, ids, E, scale=shared)
    _check_ex(x, ids, E, expert_start=lo, expert_end=hi, scale=per_expert)


def test_unquantized_rows_carry_the_token_scale():
    x = gen.draw_x(11, 40, 512)
    ids = gen.draw_ids_uniform(11, 40, 32, 4)
    s = np.arange(1, 41, dtype=np.float32) * 0.5
    _check_ex(x, ids, 32, quant_mode=-1, scale=s)


def test_options_through_the_workspace_free_entry_point():
    x = gen.draw_x(12, 500, 512)
    ids = gen.draw_ids_zipf(12, 500, 128, 16)
    _check_ex(x, ids, 128, static=True, expert_start=20, expert_end=100, tokens_num_type=2)
    _check_ex(x, ids, 128, static=True, quant_mode=0, scale=[2.0], offset=[0.25], active_num=3000)
