"""moe_init_routing_static: init-routing for callers that cannot allocate
device memory (allocator callbacks, framework plug-ins without access to
device allocations).  Its routing scratch is a fixed static array inside the
library instead of a caller workspace.  Checked against moe_init_routing on
the same inputs, bit-exact like every routing test, on two calls in a row
(the second call reuses the array the first one left behind).

This file is collected last on purpose, so a failure here leaves every other
GPU test already run."""
import numpy as np
import pytest
import torch

from nvfp4_routed_moe_gb300 import api
from nvfp4_routed_moe_gb300 import inputs as gen
from gpu_util import dev

pytestmark = pytest.mark.gpu


def _outputs(T, H, E, k, opts):
    rows = E * opts.expert_capacity if opts.drop_pad else T * k
    xdt = torch.int8 if opts.quant_mode == 1 else torch.int16
    ex = torch.full((rows, H), 0x33, dtype=xdt, device="cuda")
    ridx = torch.full((T * k,), -9, dtype=torch.int32, device="cuda")
    tok = torch.full((E,), -9, dtype=torch.int32, device="cuda")
    sc = torch.full((rows,), -2.0, dtype=torch.float32, device="cuda") if opts.quant_mode == 1 else None
    return ex, ridx, tok, sc


def _run_both(x, ids, E, opts, calls=2):
    T, H = x.shape
    k = ids.shape[1]
    shp = api.shape(H, 128, E, k)
    xd, idd = dev(x, torch.bfloat16), dev(ids)
    ws = torch.empty(api.moe_workspace_size(shp, T), dtype=torch.uint8, device="cuda")
    api.moe_prepare_workspace(shp, ws, T)
    ref = _outputs(T, H, E, k, opts)
    api.moe_init_routing(shp, T, xd, idd, opts, *ref, ws)
    results = []
    for _ in range(calls):
        got = _outputs(T, H, E, k, opts)
        api.moe_init_routing_static(shp, T, xd, idd, opts, *got)
        torch.cuda.synchronize()
        results.append(got)
    return ref, results


def _compare(ref, got, nvalid_rows=None):
    ex_r, ridx_r, tok_r, sc_r = ref
    ex_g, ridx_g, tok_g, sc_g = got
    assert torch.equal(ridx_g, ridx_r)
    assert torch.equal(tok_g, tok_r)
    n = ex_r.shape[0] if nvalid_rows is None else nvalid_rows
    assert torch.equal(ex_g[:n], ex_r[:n])
    if sc_r is not None:
        assert torch.equal(sc_g[:n], sc_r[:n])


@pytest.mark.parametrize("T,E,k,drop_pad,C,quant", [
    (4096, 896, 16, 0, 0, 1),      # the init-routing workload, at the static limit of 65536 pairs
    (4096, 896, 16, 1, 96, 1),     # same, drop/pad to 96 rows per expert
    (37, 64, 8, 0, 0, -1),         # small, one-CTA routing path, bf16 rows
])
def test_static_scratch_matches_workspace_version_twice(T, E, k, drop_pad, C, quant):
    x = gen.draw_x(5, T, 3584 if T > 1000 else 512)
    ids = gen.draw_ids_uniform(5, T, E, k)
    opts = api.moe_routing_opts_t(drop_pad, C, 0, 0, quant)
    ref, results = _run_both(x, ids, E, opts)
    nvalid = None if drop_pad else T * k
    for got in results:
        _compare(ref, got, nvalid)


def test_static_scratch_second_call_with_other_inputs():
    """A second, different call on the same array gives that call's result,
    not a mix with the first call's leftovers."""
    E, k = 128, 16
    opts = api.moe_routing_opts_t(0, 0, 1, 1, 1)
    for T, seed in ((2000, 1), (300, 2)):
        x = gen.draw_x(seed, T, 512)
        ids = gen.draw_ids_zipf(seed, T, E, k)
        ref, results = _run_both(x, ids, E, opts, calls=1)
        _compare(ref, results[0], T * k)


def test_static_scratch_rejects_too_many_pairs():
    T, E, k = 4097, 896, 16          # 65552 pairs: one token over the limit
    shp = api.shape(3584, 128, E, k)
    opts = api.moe_routing_opts_t(0, 0, 0, 0, 1)
    buf = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(api.MoeError) as e:
        api.moe_init_routing_static(shp, T, buf, buf, opts, buf, buf, buf, buf)
    assert e.value.status == 3


@pytest.mark.parametrize("T,E,k", [(40, 32, 4), (2000, 128, 16)])
def test_static_scratch_skips_out_of_range_ids_like_the_workspace_version(T, E, k):
    """Ids outside [0, E) are skipped by both entry points alike: those pairs
    get expanded_row_idx -1, the histograms count only the valid ids, and
    the moved rows are the same (one-CTA and multi-CTA routing).  The static
    version has no status word to report; only the outputs are compared."""
    x = gen.draw_x(6, T, 512)
    ids = gen.draw_ids_uniform(6, T, E, k)
    ids[3, 1] = -1
    ids[17, 0] = E
    ids[T - 1, k - 1] = 1 << 30
    opts = api.moe_routing_opts_t(0, 0, 0, 1, 1)
    ref, results = _run_both(x, ids, E, opts)
    nvalid = T * k - 3
    ridx = ref[1].cpu().numpy()
    assert ridx[3 * k + 1] == -1 and ridx[17 * k] == -1 and ridx[T * k - 1] == -1
    assert int(ref[2].sum()) == nvalid
    for got in results:
        _compare(ref, got, nvalid)
