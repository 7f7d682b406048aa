"""The multi-rank paths on CPU with torch.distributed's gloo backend,
world_size 2 (no GPU): the replicated bench's whole-job timing, and the
expert-parallel combine, where each rank's forward over its own expert
slice is summed across ranks (the caller's all-reduce)."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _init(rank, world, port):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    return dist


def _timing_worker(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    dist = _init(rank, world, port)
    import bench
    ms_local = [12.5, 20.0][rank]
    out[rank] = bench.job_throughput(ms_local, 1000, 10, world, device="cpu")
    dist.destroy_process_group()


def test_replicated_timing_takes_the_slowest_rank():
    port = _free_port()
    out = mp.Manager().dict()
    mp.spawn(_timing_worker, args=(2, port, out), nprocs=2, join=True)
    for rank in (0, 1):
        ms, value = out[rank]
        assert ms == 20.0
        assert value == pytest.approx(2 * 1000 * 10 / 0.020)


def _ep_worker(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    dist = _init(rank, world, port)
    import torch
    from oracle import cases
    from nvfp4_routed_moe_gb300 import inputs as gen
    inp = cases.prepare_tiny(0, T=24)
    n = inp.E // world
    begin = rank * n
    sl = gen.MoEInputs(inp.H, inp.I, n, inp.k, inp.T, inp.x, inp.expert_ids - begin, inp.route_weights, inp.qX)
    sl.w13, sl.sf13, sl.w2, sl.sf2 = (a[begin:begin + n] for a in (inp.w13, inp.sf13, inp.w2, inp.sf2))
    sl.dXdW13, sl.qA, sl.dAdW2 = (a[begin:begin + n] for a in (inp.dXdW13, inp.qA, inp.dAdW2))
    _, mid = cases.run_oracle(sl, want_intermediates=True)
    # the rank's partial output in fp64: sum over its own experts of w * y
    part = np.zeros((inp.T, inp.H))
    rw = gen.bf16_bits_to_f32(inp.route_weights).astype(np.float64)
    for t in range(inp.T):
        for j in range(inp.k):
            if 0 <= inp.expert_ids[t, j] - begin < n:
                part[t] += rw[t, j] * mid["y"][t, j]
    buf = torch.from_numpy(part)
    dist.all_reduce(buf, op=dist.ReduceOp.SUM)
    if rank == 0:
        out["total"] = buf.numpy().copy()
        out["full"] = cases.run_oracle(inp)
    dist.destroy_process_group()


def test_expert_slices_all_reduce_to_the_full_forward():
    port = _free_port()
    out = mp.Manager().dict()
    mp.spawn(_ep_worker, args=(2, port, out), nprocs=2, join=True)
    from nvfp4_routed_moe_gb300 import inputs as gen
    total = gen.f32_to_bf16_bits(out["total"].astype(np.float32))
    np.testing.assert_array_equal(total, out["full"])
