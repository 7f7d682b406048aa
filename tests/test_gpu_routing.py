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
