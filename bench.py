#!/usr/bin/env python
"""Benchmark of the routed NVFP4 SiTU MoE forward on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload maxbatch] [--impl ours|reference]

One step is one moe_forward (routing, X quantization, FC1 + SiTU + requant,
FC2 + route-weighted combine, BF16 finalize) over one batch of seeded synthetic
input already resident in HBM.  Default workload: T=16384 tokens at
H=3584, I=384, E=896, k=16, uniform distinct expert ids, 1% of rows x50
(the max-batch case); its 2.08 GB of weights are larger than L2, so no flush
is needed between steps.  Under torchrun each rank runs its own batch on its
own GPU with replicated weights (weak scaling, no collective on the data
path); rank 0 prints one JSON line.

Also measured: per-stage times from timing events recorded between the
stages in a separate pass after the timed steps (events between kernels
serialize the chain; the dominant kernel's roofline uses these times), the
block-scaled FP4 tensor-core peak of this GPU from the library's own MMA
microbenchmark (the denominator of the tensor fraction),
an end-to-end pass through moe_forward with pinned host buffers (every
step's input copy and output read-back inside the timed region, pipelined on
copy-in / compute / copy-out streams with double buffers), SM clocks during
the timed region, a decode/prefill sweep (L2 flushed between steps; each
forward also replayed from a CUDA graph), init-routing alone in its modes
(dynamic and static int8, drop/pad, an expert range with the key_value
histogram), the widened paths beside the plain forward of the same batch
(streamed chunks, one expert-parallel rank's slice, per-expert SiTU
parameters), and the CPU oracle on a bounded sample of the same workload
(rank 0, one GPU only).

--impl reference times the CPU oracle alone (there is no other implementation
to run): each step evaluates a bounded sample of the same workload on the
host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from nvfp4_routed_moe_gb300 import inputs as gen  # noqa: E402

METRIC = "MoE tokens/s at H3584/I384/E896/k16 (T=1..16384); % HBM or FP4 roofline"
H, I, E, K = gen.FULL["H"], gen.FULL["I"], gen.FULL["E"], gen.FULL["k"]
FC1_BYTES_PER_EXPERT = 2 * I * H // 2 + 2 * I * H // 16          # 1,548,288
FC2_BYTES_PER_EXPERT = H * I // 2 + H * I // 16                  # 774,144
WORKLOADS = {
    "maxbatch": dict(T=16384, routing="uniform", big_rows_frac=0.01,
                     text="T=16384, H=3584, I=384, E=896, top-k=16, uniform distinct ids, 1% of rows x50"),
    "prefill": dict(T=4096, routing="zipf", big_rows_frac=0.0,
                    text="T=4096, H=3584, I=384, E=896, top-k=16, Zipf(1.1) ids without replacement"),
    "decode16": dict(T=16, routing="uniform", big_rows_frac=0.0,
                     text="T=16, H=3584, I=384, E=896, top-k=16, uniform distinct ids"),
    "T1024": dict(T=1024, routing="uniform", big_rows_frac=0.0,
                  text="T=1024, H=3584, I=384, E=896, top-k=16, uniform distinct ids"),
    # a small case of the same kernels for counter captures (weights 0.3 GB, still larger than L2)
    "small_e128": dict(T=1024, routing="uniform", big_rows_frac=0.0, E=128,
                       text="T=1024, H=3584, I=384, E=128, top-k=16, uniform distinct ids (profiling case)"),
}


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def init_routing_sweep(shp, flush, dev):
    """moe_init_routing alone on 4096 rows (k=16, E=896, H=3584, uniform distinct
    ids, dynamic int8): dropless with gather indices and cumsum, and drop/pad
    with capacity 96.  Achieved GB/s over the algorithmic bytes (x read, ids
    read, expanded rows, scales and indices written)."""
    import torch
    from nvfp4_routed_moe_gb300 import api
    rows, H, k, E = 4096, shp.hidden, shp.top_k, shp.num_experts
    b = gen.full(200, T=rows, routing="uniform", weights=False, E=E)
    x = dev(b.x, torch.bfloat16)
    ids = dev(b.expert_ids)
    ws = torch.empty(api.moe_workspace_size(shp, rows), dtype=torch.uint8, device="cuda")
    api.moe_prepare_workspace(shp, ws, rows)
    res = {}
    s_static = torch.tensor([0.5], dtype=torch.float32, device="cuda")
    o_static = torch.tensor([1.0], dtype=torch.float32, device="cuda")
    lo, hi = E // 8, 2 * E // 8   # one of eight expert-parallel ranks
    in_range = int(((b.expert_ids >= lo) & (b.expert_ids < hi)).sum())
    configs = (("dropless", 0, dict(quant_mode=1), rows * k),
               ("drop_pad_C96", 96, dict(drop_pad=1, expert_capacity=96, quant_mode=1), E * 96),
               ("static_int8", 0, dict(quant_mode=0, scale=s_static, offset=o_static), rows * k),
               ("range_key_value", 0, dict(quant_mode=1, expert_start=lo, expert_end=hi, tokens_num_type=2), in_range))
    for name, C, kw, n_out in configs:
        ex = torch.empty((max(n_out, 1) if C else rows * k, H), dtype=torch.int8, device="cuda")
        idx = torch.empty(rows * k, dtype=torch.int32, device="cuda")
        tok = torch.empty(2 * E, dtype=torch.int32, device="cuda")
        sc = torch.empty(ex.shape[0], dtype=torch.float32, device="cuda")
        opts = api.routing_opts(**kw)
        call = lambda: api.moe_init_routing(shp, rows, x, ids, opts, ex, idx, tok, sc, ws)
        for _ in range(3):
            call()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(20)]
        for a, c in evs:
            flush()
            a.record()
            call()
            c.record()
        torch.cuda.synchronize()
        t_ms = statistics.median([a.elapsed_time(c) for a, c in evs])
        byt = rows * H * 2 + rows * k * 4 + n_out * H + n_out * 4 + rows * k * 4 + E * 4
        res[name] = {"rows": rows, "rows_out": n_out, "ms": round(t_ms, 4), "bytes": byt,
                     "gb_per_s": byt / (t_ms * 1e-3) / 1e9}
    return res


class L2Flush:
    """Evicts this step's data from L2 between timed steps: writes a 512 MB
    buffer (larger than the 129 MB L2), then reads a second 256 MB one, so
    that the lines the write left dirty are written back here, outside the
    timed region, and not by the next step's kernels."""

    def __init__(self):
        import torch
        self.w = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
        self.r = torch.zeros(256 << 20, dtype=torch.uint8, device="cuda")

    def __call__(self):
        self.w.fill_(1)
        self.r.max()


def median_ms(call, flush, n=20):
    """Median CUDA-event time of `call` over n runs, L2 flushed before each."""
    import torch
    for _ in range(3):
        call()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    for a, c in evs:
        flush()
        a.record()
        call()
        c.record()
    torch.cuda.synchronize()
    return statistics.median([a.elapsed_time(c) for a, c in evs])


def next_rows_sweep(shp, flush, dev, w, scales, winp, peak):
    """The widened paths at T = 4096 (uniform ids), each beside the plain
    forward of the same batch: the chunk-ready streaming front end (four
    1024-token chunks through a two-slot ring, publish and forward on one
    stream, then on two streams with the forwards held to all but 16 SMs),
    one expert-parallel rank's slice (the first 112 of 896 experts,
    its own prepared weights), and per-expert SiTU parameters."""
    import torch
    from nvfp4_routed_moe_gb300 import api
    T, C, S = 4096, 1024, 2
    b = gen.full(300, T=T, routing="uniform", weights=False, E=shp.num_experts)
    x, ids, rw = dev(b.x, torch.bfloat16), dev(b.expert_ids), dev(b.route_weights, torch.bfloat16)
    qx = dev(np.array([b.qX], np.float32))
    out = torch.empty((T, shp.hidden), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(api.moe_workspace_size(shp, T), dtype=torch.uint8, device="cuda")
    api.moe_prepare_workspace(shp, ws, T)
    plain = lambda: api.moe_forward(shp, T, x, ids, rw, *w, qx, *scales, None, None, ws, out)
    t_plain = median_ms(plain, flush)
    res = {"T": T, "plain_ms": round(t_plain, 4)}

    cfg = api.moe_stream_ring_t(S, C)
    ring = torch.empty(api.moe_stream_ring_size(shp, cfg), dtype=torch.uint8, device="cuda")
    api.moe_stream_ring_init(shp, cfg, ring)
    ws_c = torch.empty(api.moe_workspace_size(shp, C), dtype=torch.uint8, device="cuda")
    api.moe_prepare_workspace(shp, ws_c, C)

    def streamed():
        api.moe_stream_begin(shp, cfg, ring)
        for c, base in enumerate(range(0, T, C)):
            api.moe_stream_publish(shp, cfg, ring, c, base, C, api.STREAM_ROUTE | api.STREAM_LAYOUT,
                                   x[base:base + C], ids[base:base + C], rw[base:base + C])
            api.moe_stream_forward(shp, cfg, ring, c, *w, qx, *scales, None, None, ws_c, out)
    t_st = median_ms(streamed, flush)
    assert api.moe_read_status(ws_c) == (0, 0) and api.moe_stream_read_status(ring) == 0
    res["stream"] = {"chunk": C, "slots": S, "ms": round(t_st, 4), "tokens_per_s": T / (t_st * 1e-3),
                     "vs_plain": t_plain / t_st}
    del ring

    # the same chunks with the producer on its own stream and the chunk
    # forwards held to all but 16 SMs (the ring's SM budget), so that each
    # publish overlaps the forward of the chunk before it; events order a
    # publish after the forward that frees its slot, so no device-side wait
    # ever depends on the other stream
    budget = max(1, torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count - 16)
    cfg2 = api.moe_stream_ring_t(S, C, budget)
    ring2 = torch.empty(api.moe_stream_ring_size(shp, cfg2), dtype=torch.uint8, device="cuda")
    api.moe_stream_ring_init(shp, cfg2, ring2)
    prod, cons = torch.cuda.Stream(), torch.cuda.Stream()
    n_chunks = T // C

    def streamed_two():
        cur = torch.cuda.current_stream()
        prod.wait_stream(cur)
        cons.wait_stream(cur)
        pub = [torch.cuda.Event() for _ in range(n_chunks)]
        con = [torch.cuda.Event() for _ in range(n_chunks)]
        api.moe_stream_begin(shp, cfg2, ring2, stream=prod)
        for c, base in enumerate(range(0, T, C)):
            if c >= S:
                prod.wait_event(con[c - S])
            api.moe_stream_publish(shp, cfg2, ring2, c, base, C, api.STREAM_ROUTE | api.STREAM_LAYOUT,
                                   x[base:base + C], ids[base:base + C], rw[base:base + C], stream=prod)
            pub[c].record(prod)
            cons.wait_event(pub[c])
            api.moe_stream_forward(shp, cfg2, ring2, c, *w, qx, *scales, None, None, ws_c, out, stream=cons)
            con[c].record(cons)
        cur.wait_stream(cons)
    t_two = median_ms(streamed_two, flush)
    assert api.moe_read_status(ws_c) == (0, 0) and api.moe_stream_read_status(ring2) == 0
    res["stream_two_streams"] = {"chunk": C, "slots": S, "max_sms": budget, "ms": round(t_two, 4),
                                 "tokens_per_s": T / (t_two * 1e-3), "vs_plain": t_plain / t_two}
    del ring2, ws_c

    EL, lo = shp.num_experts // 8, 0
    shp_l = api.shape(shp.hidden, shp.inter, EL, shp.top_k)
    w_l = [torch.empty(n, dtype=torch.uint8, device="cuda") for n in api.moe_prepared_weight_bytes(shp_l)]
    api.moe_prepare_weights(shp_l, dev(winp.w13[:EL]), dev(winp.sf13[:EL]), dev(winp.w2[:EL]), dev(winp.sf2[:EL]),
                            *w_l)
    sc_l = [dev(winp.dXdW13[:EL]), dev(winp.qA[:EL]), dev(winp.dAdW2[:EL])]
    ws_l = torch.empty(api.moe_workspace_size(shp_l, T), dtype=torch.uint8, device="cuda")
    api.moe_prepare_workspace(shp_l, ws_l, T)
    local = lambda: api.moe_forward_local_experts(shp_l, lo, T, x, ids, rw, *w_l, qx, *sc_l, None, None, ws_l, out)
    t_loc = median_ms(local, flush)
    pairs = int(((b.expert_ids >= lo) & (b.expert_ids < lo + EL)).sum())
    byt = EL * (FC1_BYTES_PER_EXPERT + FC2_BYTES_PER_EXPERT) + 2 * T * H * 2 + T * K * 6
    res["local_experts"] = {"experts": EL, "pairs": pairs, "ms": round(t_loc, 4),
                            "hbm_frac": byt / (t_loc * 1e-3) / 1e9 / peak}
    del w_l, ws_l

    rs = np.random.default_rng(4)
    beta = dev(rs.uniform(1.0, 8.0, shp.num_experts).astype(np.float32))
    lam = dev(rs.uniform(2.0, 60.0, shp.num_experts).astype(np.float32))
    situ = lambda: api.moe_forward(shp, T, x, ids, rw, *w, qx, *scales, beta, lam, ws, out)
    t_situ = median_ms(situ, flush)
    res["situ_per_expert"] = {"ms": round(t_situ, 4), "vs_plain": t_plain / t_situ}
    return res


def step_bytes(T, n_active):
    """Algorithmic bytes of one forward: weights and block scales of the
    active experts, x read and out written (bf16), ids and route weights."""
    return n_active * (FC1_BYTES_PER_EXPERT + FC2_BYTES_PER_EXPERT) + 2 * T * H * 2 + T * K * 6


def fc1_bytes(T, n_active):
    """Algorithmic bytes of one FC1 launch: W13 codes + block scales of the
    active experts and each token's quantized row (codes + scales) once.  The
    requantized intermediate it writes is activation-requant traffic, which
    counts as overhead, not as algorithmic bytes."""
    return n_active * FC1_BYTES_PER_EXPERT + T * (H // 2 + H // 16)


def fc2_bytes(T, n_active):
    """Algorithmic bytes of one FC2 launch: W2 codes + block scales of the
    active experts.  The intermediate it reads and the fp32 combine
    accumulator are requant and scratch traffic (overhead)."""
    return n_active * FC2_BYTES_PER_EXPERT


KERNEL_BYTES = {"fc1": (fc1_bytes, "n_active*1548288 + T*2016"),
                "fc2": (fc2_bytes, "n_active*774144")}
FLOPS_PER_PAIR = 2 * H * 2 * I + 2 * I * H                        # FC1 + FC2, 8,257,536
KERNEL_FLOPS_PER_PAIR = {"fc1": 2 * H * 2 * I, "fc2": 2 * I * H}


def fp4_peak(sms):
    """Block-scaled FP4 MMA throughput measured on this GPU with the
    library's own microbenchmark (moe_test_mma_peak): every SM issues
    back-to-back M=128, N=256, K=64 kind::mxf4nvf4 MMAs from resident
    operands; CUDA-event time of the launch, best of 5.  Also the tensor
    pipe's cycles per FC1 k-block (four MMAs plus the scale-atom copies that
    FC1 issues with them) for the two FC1 unit shapes."""
    import torch
    from nvfp4_routed_moe_gb300 import api
    cyc = torch.zeros(sms, dtype=torch.int64, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")

    def run(n, mmas, copies, reps=5):
        best, cycles = None, None
        for _ in range(reps + 1):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            api.moe_test_mma_peak(sms, n, mmas, copies, cyc, st)
            b.record()
            torch.cuda.synchronize()
            ms = a.elapsed_time(b)
            c = cyc.cpu().numpy()
            if best is None or ms < best:
                best, cycles = ms, float(np.median(c))
        assert int(st.item()) == 0 and cycles > 0
        return best, cycles

    mmas = 16384
    ms, cyc256 = run(256, mmas, 0)
    flops = 2.0 * 128 * 256 * 64 * mmas * sms
    res = {"tflops": flops / (ms * 1e-3) / 1e12, "unit": "TFLOP/s", "source":
           f"moe_test_mma_peak: {sms} SMs x {mmas} back-to-back M128 N256 K64 kind::mxf4nvf4 scale_vec::4X MMAs, "
           "CUDA events, best of 5", "cycles_per_mma_n256": cyc256 / mmas,
           "sm_mhz_effective": cyc256 / (ms * 1e3)}
    _, c = run(128, 4096, 0)
    res["cycles_per_mma_n128"] = c / 4096
    _, c = run(256, 4096, 12)
    res["fc1_kblock_cycles_pair2"] = c / 1024          # 4 N=256 MMAs + 12 scale-atom copies
    _, c = run(128, 4096, 8)
    res["fc1_kblock_cycles_pair1"] = c / 1024          # 4 N=128 MMAs + 8 scale-atom copies
    del cyc, st
    return res


def cpu_model():
    """The host CPU's model name (lscpu), e.g. an Arm Neoverse core on Grace."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.processor() or platform.machine()


# Sources compiled into the GEMM kernels (the file and everything it includes).
GEMM_SOURCES = ("nvfp4_routed_moe_gb300/csrc/gemm.cu", "nvfp4_routed_moe_gb300/csrc/gemv.cu",
                "nvfp4_routed_moe_gb300/csrc/nvfp4.cuh",
                "nvfp4_routed_moe_gb300/csrc/ptx.cuh", "nvfp4_routed_moe_gb300/csrc/plan.h",
                "include/nvfp4moe.h")


def gemm_sources_sha1():
    """SHA-1 over the GEMM kernels' sources, in GEMM_SOURCES order."""
    h = hashlib.sha1()
    for rel in GEMM_SOURCES:
        h.update(open(os.path.join(ROOT, rel), "rb").read())
    return h.hexdigest()


def traffic_from_profile(kernel, workload):
    """DRAM bytes per launch from the committed ncu summary of this kernel
    and workload, used only while the kernel sources are unchanged since the
    capture."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_kernel_{workload}.md")
    try:
        kv = {}
        for line in open(path).read().splitlines():
            if line.startswith(("gemm_sources_sha1", "dram_bytes_per_launch")) and "=" in line:
                k, v = line.split("=", 1)
                kv[k.strip()] = v.strip().strip("`")
        if kv.get("gemm_sources_sha1") == gemm_sources_sha1():
            return float(kv["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


def job_throughput(ms_local: float, tokens_per_rank: int, steps: int, world: int, device: str = "cuda"):
    """Whole-job throughput of a replicated run: every rank times its own
    steps; the job's time is the slowest rank's (all-reduce MAX when
    world > 1) and the job processed world * tokens_per_rank * steps tokens.
    Returns (max_ms, tokens/s)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms_local], dtype=torch.float64, device=device)
    if world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    ms = float(t.item())
    return ms, world * tokens_per_rank * steps / (ms / 1e3)


class ClockSampler:
    """nvidia-smi clock samples every 200 ms in a background process."""

    def __init__(self, gpu_id: str):
        self.rows = []
        self.marks = {}
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.p = subprocess.Popen(["nvidia-smi", f"--query-gpu={q}", "--format=csv,noheader,nounits",
                                       "-lms", "200", "-i", gpu_id], stdout=subprocess.PIPE,
                                      stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.p = None

    def _read(self):
        for line in self.p.stdout:
            self.rows.append((time.time(), [c.strip() for c in line.split(",")]))

    def mark(self, name):
        self.marks[name] = time.time()

    def stop(self):
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.3)
        self.p.terminate()
        try:
            self.p.wait(timeout=5)
        except Exception:
            self.p.kill()
        t0, t1 = self.marks.get("start", 0), self.marks.get("end", 1e30)
        inside = [r for t, r in self.rows if t0 <= t <= t1 + 0.2]
        window = "timed region"
        if not inside:
            inside = [r for _, r in self.rows]
            window = "whole run (timed region shorter than one sample)"
        sm = [float(r[1]) for r in inside if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in inside if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i in range(4) if len(r) > 5 + i and r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(inside), "window": window}


def cpu_baseline(inp, target_s=12.0, max_tokens=512):
    """The oracle as it stands on a bounded sample (the first n tokens)."""
    import oracle
    from oracle import cases
    oracle.build()
    n, spent, done = 4, 0.0, 0
    t_start = time.time()
    while spent < target_s and done < max_tokens:
        toks = np.arange(done, min(done + n, inp.T))
        t0 = time.time()
        cases.run_oracle(inp, tokens=toks)
        spent += time.time() - t0
        done += len(toks)
        n = min(2 * n, max_tokens - done) if done < max_tokens else 0
        if n <= 0 or done >= inp.T:
            break
    return {"value": done / spent, "unit": "tokens/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"first {done} tokens of the timed workload (same weights and routing), {spent:.1f} s",
            "cpu": cpu_model()}


def cpu_baseline_decode(winp, E):
    """The oracle at decode (T=16, uniform ids) on all host threads and on
    one thread, the second timing the plan asks for at T <= 16."""
    import oracle
    from oracle import cases
    oracle.build()
    b = gen.full(116, T=16, routing="uniform", weights=False, E=E)
    b.w13, b.sf13, b.w2, b.sf2 = winp.w13, winp.sf13, winp.w2, winp.sf2
    b.dXdW13, b.qA, b.dAdW2 = winp.dXdW13, winp.qA, winp.dAdW2
    res = {}
    cores = oracle.num_threads()
    for name, threads, toks in (("all_threads", cores, np.arange(16)), ("one_thread", 1, np.arange(4))):
        oracle.set_num_threads(threads)
        t0 = time.time()
        cases.run_oracle(b, tokens=toks)
        dt = time.time() - t0
        res[name] = {"value": len(toks) / dt, "unit": "tokens/s", "cores": threads,
                     "sample": f"{len(toks)} tokens of the T=16 decode batch, {dt:.2f} s"}
    oracle.set_num_threads(cores)
    return res


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    from oracle import cases
    oracle.build()
    wl = WORKLOADS[args.workload]
    inp = gen.full(0, T=wl["T"], routing=wl["routing"], big_rows_frac=wl["big_rows_frac"], E=wl.get("E"))
    per_step = oracle.num_threads()       # one token per host thread: a step costs about one token's time
    for s in range(args.warmup):
        cases.run_oracle(inp, tokens=np.arange(s * per_step, (s + 1) * per_step) % inp.T)
    t0 = time.time()
    done = 0
    for s in range(args.steps):
        toks = (np.arange(per_step) + (args.warmup + s) * per_step) % inp.T
        cases.run_oracle(inp, tokens=toks)
        done += per_step
    dt = time.time() - t0
    value = done / dt
    sample = f"{per_step} tokens of the {args.workload} workload per step, one per host thread"
    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": {"workload": f"{args.workload}: {wl['text']}", "T": wl["T"]},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": oracle.num_threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="maxbatch", choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-stage-events", action="store_true", help="time the steps without stage events")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.impl == "reference":
        run_reference(args)
        return

    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    from nvfp4_routed_moe_gb300 import api
    from nvfp4_routed_moe_gb300 import build as nvbuild
    if rank == 0 or world == 1:
        nvbuild.build()
    if world > 1:
        dist.barrier()
    api.lib()

    def dev(a, dtype=None):
        a = np.ascontiguousarray(a)
        if a.dtype == np.uint16:
            a = a.view(np.int16)
        t = torch.from_numpy(a)
        return (t.view(dtype) if dtype is not None else t).cuda()

    def barrier():
        if world > 1:
            dist.barrier()

    wl = WORKLOADS[args.workload]
    E = wl.get("E", gen.FULL["E"])
    inp = gen.full(rank, T=wl["T"], routing=wl["routing"], big_rows_frac=wl["big_rows_frac"], weights=False, E=E)
    winp = gen.full(0, T=1, weights=True, E=E)     # same weights on every rank
    shp = api.shape(H, I, E, K)
    sizes = api.moe_prepared_weight_bytes(shp)
    w = [torch.empty(n, dtype=torch.uint8, device="cuda") for n in sizes]
    canon = [dev(winp.w13), dev(winp.sf13), dev(winp.w2), dev(winp.sf2)]
    api.moe_prepare_weights(shp, *canon, *w)
    torch.cuda.synchronize()
    del canon
    torch.cuda.empty_cache()
    scales = [dev(winp.dXdW13), dev(winp.qA), dev(winp.dAdW2)]

    def make_batch(b):
        return dict(x=dev(b.x, torch.bfloat16), ids=dev(b.expert_ids), rw=dev(b.route_weights, torch.bfloat16),
                    qX=dev(np.array([b.qX], np.float32)), T=b.T,
                    n_active=int((np.bincount(b.expert_ids.ravel(), minlength=E) > 0).sum()),
                    pairs=int(((b.expert_ids >= 0) & (b.expert_ids < E)).sum()))

    def forward(bt, ws, out, stream=None):
        api.moe_forward(shp, bt["T"], bt["x"], bt["ids"], bt["rw"], *w, bt["qX"], *scales, None, None, ws, out,
                        stream)

    batch = make_batch(inp)
    T = batch["T"]
    ws = torch.empty(api.moe_workspace_size(shp, T), dtype=torch.uint8, device="cuda")
    api.moe_prepare_workspace(shp, ws, T)
    out = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    for _ in range(args.warmup):
        forward(batch, ws, out)
    torch.cuda.synchronize()
    status = api.moe_read_status(ws)
    if status != (0, 0):
        raise SystemExit(f"device status {status}")

    # ------------------------------------------------------------ timed region
    props = torch.cuda.get_device_properties(local)
    gpu_id = str(getattr(props, "uuid", "")) or str(local)
    if gpu_id and not gpu_id.startswith("GPU-") and len(gpu_id) > 8:
        gpu_id = "GPU-" + gpu_id
    clocks = ClockSampler(gpu_id)
    time.sleep(0.5)
    stage = None
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    clocks.mark("start")
    ev0.record()
    for _ in range(args.steps):
        forward(batch, ws, out)
    ev1.record()
    torch.cuda.synchronize()
    clocks.mark("end")
    barrier()
    ms = ev0.elapsed_time(ev1)
    clk = clocks.stop()
    if not args.no_stage_events:
        # stage breakdown in a separate pass: events recorded between the
        # kernels serialize the chain, so they stay out of the timed steps
        n_stage = min(args.steps, 50)
        api.moe_profile_start(n_stage)
        for _ in range(n_stage):
            forward(batch, ws, out)
        torch.cuda.synchronize()
        stage_ms, ncalls = api.moe_profile_stop()
        stage = {k: v / max(ncalls, 1) for k, v in stage_ms.items()}
    ms, value = job_throughput(ms, T, args.steps, world)
    ms_per_step = ms / args.steps
    launches = api.moe_forward_launch_count(shp, T) * args.steps

    # ------------------------------------------------------------ end to end
    # Every step copies its inputs from pinned host memory and reads its
    # output back, pipelined as a server would run it: step n's input copy
    # (copy-in stream) and step n-1's output copy (copy-out stream) overlap
    # step n's forward (compute stream); inputs and outputs are double-
    # buffered and events order every hand-over.
    x_h = batch["x"].cpu().pin_memory()
    ids_h = batch["ids"].cpu().pin_memory()
    rw_h = batch["rw"].cpu().pin_memory()
    outs_h = [torch.empty((T, H), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    ins = [dict(batch, x=torch.empty_like(batch["x"]), ids=torch.empty_like(batch["ids"]),
                rw=torch.empty_like(batch["rw"])) for _ in range(2)]
    outs = [torch.empty_like(out) for _ in range(2)]
    s_in, s_cmp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()
    in_ready, in_free = [ev(), ev()], [ev(), ev()]
    out_ready, out_free = [ev(), ev()], [ev(), ev()]
    e2e_steps = min(args.steps, 200)

    def e2e_step(n):
        b = n % 2
        with torch.cuda.stream(s_in):
            if n >= 2:
                s_in.wait_event(in_free[b])
            ins[b]["x"].copy_(x_h, non_blocking=True)
            ins[b]["ids"].copy_(ids_h, non_blocking=True)
            ins[b]["rw"].copy_(rw_h, non_blocking=True)
            in_ready[b].record(s_in)
        s_cmp.wait_event(in_ready[b])
        if n >= 2:
            s_cmp.wait_event(out_free[b])
        forward(ins[b], ws, outs[b], stream=s_cmp)
        in_free[b].record(s_cmp)
        out_ready[b].record(s_cmp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(out_ready[b])
            outs_h[b].copy_(outs[b], non_blocking=True)
            out_free[b].record(s_out)

    torch.cuda.synchronize()
    for n in range(2):
        e2e_step(n)
    barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    for n in range(e2e_steps):
        e2e_step(n)
    s_in.wait_stream(s_out)
    e1.record(s_in)
    torch.cuda.synchronize()
    _, e2e_val = job_throughput(e0.elapsed_time(e1), T, e2e_steps, world)
    h2d = x_h.numel() * 2 + ids_h.numel() * 4 + rw_h.numel() * 2
    d2h = outs_h[0].numel() * 2
    last = (e2e_steps - 1) % 2
    assert torch.equal(outs_h[last].view(torch.int16), outs[last].cpu().view(torch.int16))

    # ------------------------------------------------------------ roofline
    peak, peak_src = peaks()
    n_active = batch["n_active"]
    roof_all = {}
    fp4 = fp4_peak(torch.cuda.get_device_properties(local).multi_processor_count) if world == 1 or rank == 0 \
        else None
    pairs = int(batch["pairs"])
    decode_kernels = dict(zip(("fc1", "fc2"), api.moe_forward_kernels(shp, T)))
    for kname, (fn, formula) in KERNEL_BYTES.items():
        b_k = fn(T, n_active)
        kernel = f"{kname}_gemv" if decode_kernels.get(kname) else kname   # the decode kernel or the tcgen05 GEMM
        traffic = traffic_from_profile(kernel, args.workload)
        r = {"kernel": f"{kernel}_kernel", "bound": "hbm", "achieved": None, "peak": peak, "unit": "GB/s",
             "frac": None, "traffic": traffic, "peak_source": peak_src, "bytes_per_launch": b_k,
             "bytes_formula": formula,
             "traffic_over_algorithmic": traffic / b_k if traffic else None}
        if stage:
            ach = b_k / (stage[kname] * 1e-3) / 1e9
            r.update(achieved=ach, frac=ach / peak, ms=stage[kname])
            if fp4:
                tf = pairs * KERNEL_FLOPS_PER_PAIR[kname] / (stage[kname] * 1e-3) / 1e12
                r["tensor"] = {"achieved_tflops": tf, "frac": tf / fp4["tflops"]}
        roof_all[kname] = r
    dominant = max(roof_all, key=lambda k: stage[k] if stage else 0.0)
    roof = roof_all[dominant]
    step_b = step_bytes(T, n_active)
    fwd_roof = {"bytes_per_step": step_b, "achieved": step_b / (ms_per_step * 1e-3) / 1e9}
    fwd_roof["frac"] = fwd_roof["achieved"] / peak
    tensor = None
    if fp4:
        tf = pairs * FLOPS_PER_PAIR / (ms_per_step * 1e-3) / 1e12
        tensor = {"flops_per_step": pairs * FLOPS_PER_PAIR, "achieved_tflops": tf, "peak_tflops": fp4["tflops"],
                  "frac": tf / fp4["tflops"], "peak": fp4}

    # ------------------------------------------------------------ sweep
    sweep = None
    if not args.no_sweep and world == 1:
        sweep = {}
        flush = L2Flush()
        for name, T_s, routing in (("decode1", 1, "uniform"), ("decode8", 8, "uniform"), ("decode16", 16, "uniform"),
                                   ("T32", 32, "uniform"), ("T128", 128, "uniform"), ("T512", 512, "uniform"),
                                   ("T1024", 1024, "uniform"), ("T2048", 2048, "uniform"), ("prefill", 4096, "zipf"),
                                   ("T8192", 8192, "uniform")):
            b = make_batch(gen.full(100 + T_s, T=T_s, routing=routing, weights=False, E=E))
            ws_s = torch.empty(api.moe_workspace_size(shp, T_s), dtype=torch.uint8, device="cuda")
            api.moe_prepare_workspace(shp, ws_s, T_s)
            out_s = torch.empty((T_s, H), dtype=torch.bfloat16, device="cuda")
            for _ in range(3):
                forward(b, ws_s, out_s)
            n_s = 20
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_s)]
            for a, c in evs:
                flush()
                a.record()
                forward(b, ws_s, out_s)
                c.record()
            torch.cuda.synchronize()
            t_ms = statistics.median([a.elapsed_time(c) for a, c in evs])
            # the same forward captured once in a CUDA graph and replayed
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                forward(b, ws_s, out_s)
            for _ in range(3):
                g.replay()
            for a, c in evs:
                flush()
                a.record()
                g.replay()
                c.record()
            torch.cuda.synchronize()
            t_graph = statistics.median([a.elapsed_time(c) for a, c in evs])
            del g
            api.moe_profile_start(n_s)           # stage breakdown in a separate pass
            for _ in range(n_s):
                flush()
                forward(b, ws_s, out_s)
            torch.cuda.synchronize()
            st_ms, nc = api.moe_profile_stop()
            byt = step_bytes(T_s, b["n_active"])
            sweep[name] = {"T": T_s, "ms": round(t_ms, 4), "ms_graph": round(t_graph, 4),
                           "tokens_per_s": T_s / (t_ms * 1e-3),
                           "hbm_frac": byt / (t_ms * 1e-3) / 1e9 / peak, "n_active": b["n_active"],
                           "fc1_ms": round(st_ms["fc1"] / nc, 4), "fc2_ms": round(st_ms["fc2"] / nc, 4),
                           "fc1_hbm_frac": fc1_bytes(T_s, b["n_active"]) / (st_ms["fc1"] / nc * 1e-3) / 1e9 / peak,
                           "fc2_hbm_frac": fc2_bytes(T_s, b["n_active"]) / (st_ms["fc2"] / nc * 1e-3) / 1e9 / peak}
            if fp4:
                sweep[name]["tensor_frac"] = (b["pairs"] * FLOPS_PER_PAIR / (t_ms * 1e-3) / 1e12) / fp4["tflops"]
        sweep["l2_flush"] = "between timed steps: 512 MB written, then 256 MB read (write-backs outside the timed region)"
        sweep["init_routing"] = init_routing_sweep(shp, flush, dev)
        sweep["next_rows"] = next_rows_sweep(shp, flush, dev, w, scales, winp, peak)
        del flush

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        inp_w = gen.full(rank, T=wl["T"], routing=wl["routing"], big_rows_frac=wl["big_rows_frac"], weights=False,
                         E=E)
        inp_w.w13, inp_w.sf13, inp_w.w2, inp_w.sf2 = winp.w13, winp.sf13, winp.w2, winp.sf2
        inp_w.dXdW13, inp_w.qA, inp_w.dAdW2 = winp.dXdW13, winp.qA, winp.dAdW2
        cpu = cpu_baseline(inp_w)
        cpu["decode"] = cpu_baseline_decode(winp, E)

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "nvfp4 (e2m1 x e4m3-scaled, fp32 accumulate, bf16 out)",
                "data": "synthetic",
                "config": {"workload": f"{args.workload}: {wl['text']}", "T": T, "n_active_experts": n_active,
                           "l2": "inputs larger than L2 (2.08 GB of weights read per step)",
                           "parallelism": f"replicas x{world} (data parallel, weak scaling)"},
                "roofline": roof, "roofline_kernels": roof_all, "forward_roofline": fwd_roof, "tensor": tensor,
                "tensor_frac": tensor["frac"] if tensor else None, "stages_ms": stage,
                "cpu_baseline": cpu,
                "e2e": {"value": e2e_val, "unit": "tokens/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                        "steps": e2e_steps, "pipeline": "copy-in, compute and copy-out streams, double-buffered"},
                "gpu_launches": launches, "clocks": clk, "sweep": sweep}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
