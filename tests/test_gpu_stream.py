"""GPU tests of the chunk-ready streaming front end through the C ABI
("[RFC] Chunk-ready symmetric-buffer protocol for streaming MegaMoE inputs",
section "Validation plan"): streamed outputs against the oracle and the
batch-ready forward across partial, zero-token and wrapping chunks;
route and layout published separately; producer and consumer on two streams
ordered by events; repeated CUDA-graph replay; and the bounded waits running
out (a generation that nothing publishes), which must leave a status and no
writes behind."""
import numpy as np
import pytest
import torch

from oracle import cases
from nvfp4_routed_moe_gb300 import api
from nvfp4_routed_moe_gb300 import inputs as gen
from gpu_util import Model, assert_close, dev, out_bits

pytestmark = pytest.mark.gpu

SHORT_WAIT_US = 2000   # waits that are meant to run out give up after 2 ms


class Stream:
    """A ring, a workspace for one chunk and the model's weights."""

    def __init__(self, m: Model, slots: int, tokens_per_slot: int, max_sms: int = 0):
        self.m = m
        self.cfg = api.moe_stream_ring_t(slots, tokens_per_slot, max_sms)
        self.ring = torch.empty(api.moe_stream_ring_size(m.shape, self.cfg), dtype=torch.uint8, device="cuda")
        api.moe_stream_ring_init(m.shape, self.cfg, self.ring)
        self.ws = m.workspace(tokens_per_slot)
        api.moe_prepare_workspace(m.shape, self.ws, tokens_per_slot)

    def begin(self, stream=None):
        api.moe_stream_begin(self.m.shape, self.cfg, self.ring, stream=stream)

    def publish(self, chunk, base, n, x, ids, rw, parts=api.STREAM_ROUTE | api.STREAM_LAYOUT, wait_us=0,
                stream=None):
        sl = slice(base, base + n)
        api.moe_stream_publish(self.m.shape, self.cfg, self.ring, chunk, base, n, parts,
                               x[sl] if n else None, ids[sl] if n else None, rw[sl] if n else None,
                               wait_us=wait_us, stream=stream)

    def forward(self, chunk, out, wait_us=0, stream=None):
        m = self.m
        api.moe_stream_forward(m.shape, self.cfg, self.ring, chunk, m.w13, m.sf13, m.w2, m.sf2, m.qX, m.dXdW13,
                               m.qA, m.dAdW2, None, None, self.ws, out, wait_us=wait_us, stream=stream)


def chunks_of(T, C, zero_tail=True):
    """(base, n) of consecutive chunks of at most C tokens, plus a zero-token chunk."""
    out = [(b, min(C, T - b)) for b in range(0, T, C)]
    return out + [(T, 0)] if zero_tail else out


@pytest.fixture(scope="module")
def tiny300():
    inp = cases.prepare_tiny(2, T=300)
    m = Model(inp)
    x = dev(inp.x, torch.bfloat16)
    ids = dev(inp.expert_ids)
    rw = dev(inp.route_weights, torch.bfloat16)
    return inp, m, x, ids, rw, cases.run_oracle(inp)


def test_streamed_matches_oracle_and_batch(tiny300):
    """Chunks of 128 tokens through a 2-slot ring (partial last chunk of 44,
    then a zero-token chunk): every slot is reused, every output row is
    written once, and the result matches the oracle and the batch forward."""
    inp, m, x, ids, rw, ref = tiny300
    st = Stream(m, slots=2, tokens_per_slot=128)
    out = torch.full((inp.T, inp.H), float("nan"), dtype=torch.bfloat16, device="cuda")
    st.begin()
    for c, (base, n) in enumerate(chunks_of(inp.T, 128)):
        st.publish(c, base, n, x, ids, rw)
        st.forward(c, out)
    torch.cuda.synchronize()
    assert api.moe_read_status(st.ws) == (0, 0)
    assert api.moe_stream_read_status(st.ring) == 0
    assert_close(out_bits(out), ref, "streamed vs oracle")
    batch, _ = m.forward_inputs()
    assert_close(out_bits(out), out_bits(batch), "streamed vs batch")


def test_route_and_layout_published_separately(tiny300):
    """Layout (x) first, route (ids, weights, base, count) second, in separate
    calls; a one-slot ring so every chunk waits for the previous one's release."""
    inp, m, x, ids, rw, ref = tiny300
    st = Stream(m, slots=1, tokens_per_slot=96)
    out = torch.empty((inp.T, inp.H), dtype=torch.bfloat16, device="cuda")
    st.begin()
    for c, (base, n) in enumerate(chunks_of(inp.T, 96, zero_tail=False)):
        st.publish(c, base, n, x, ids, rw, parts=api.STREAM_LAYOUT)
        st.publish(c, base, n, x, ids, rw, parts=api.STREAM_ROUTE)
        st.forward(c, out)
    torch.cuda.synchronize()
    assert api.moe_read_status(st.ws) == (0, 0)
    assert_close(out_bits(out), ref, "separate publishes")


def test_two_streams_ordered_by_events(tiny300):
    """Producer on one stream, forward on another: chunk c's forward waits on
    the event recorded after its publish, and the publish of chunk c reusing a
    slot waits on the event recorded after chunk c - slots' forward."""
    inp, m, x, ids, rw, ref = tiny300
    S, C = 3, 64
    st = Stream(m, slots=S, tokens_per_slot=C)
    out = torch.empty((inp.T, inp.H), dtype=torch.bfloat16, device="cuda")
    prod, cons = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    st.begin(stream=prod)
    parts = chunks_of(inp.T, C)
    published = [torch.cuda.Event() for _ in parts]
    consumed = [torch.cuda.Event() for _ in parts]
    for c, (base, n) in enumerate(parts):
        if c >= S:
            prod.wait_event(consumed[c - S])
        st.publish(c, base, n, x, ids, rw, stream=prod)
        published[c].record(prod)
        cons.wait_event(published[c])
        st.forward(c, out, stream=cons)
        consumed[c].record(cons)
    torch.cuda.synchronize()
    assert api.moe_read_status(st.ws) == (0, 0)
    assert api.moe_stream_read_status(st.ring) == 0
    assert_close(out_bits(out), ref, "two streams")


@pytest.mark.parametrize("max_sms", [8, 100])
def test_two_streams_with_an_sm_budget(tiny300, max_sms):
    """The chunk forwards sized to a budget of SMs (the ring's max_sms), with
    the producer publishing on its own stream into the rest: the same output
    as the batch oracle."""
    inp, m, x, ids, rw, ref = tiny300
    S, C = 2, 64
    st = Stream(m, slots=S, tokens_per_slot=C, max_sms=max_sms)
    out = torch.empty((inp.T, inp.H), dtype=torch.bfloat16, device="cuda")
    prod, cons = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    st.begin(stream=prod)
    parts = chunks_of(inp.T, C)
    published = [torch.cuda.Event() for _ in parts]
    consumed = [torch.cuda.Event() for _ in parts]
    for c, (base, n) in enumerate(parts):
        if c >= S:
            prod.wait_event(consumed[c - S])
        st.publish(c, base, n, x, ids, rw, stream=prod)
        published[c].record(prod)
        cons.wait_event(published[c])
        st.forward(c, out, stream=cons)
        consumed[c].record(cons)
    torch.cuda.synchronize()
    assert api.moe_read_status(st.ws) == (0, 0)
    assert api.moe_stream_read_status(st.ring) == 0
    assert_close(out_bits(out), ref, f"two streams, max_sms={max_sms}")


def test_graph_replay_new_epoch_each_time(tiny300):
    """Begin + every publish and forward captured once and replayed twice with
    new activations in the same buffers: each replay starts a new epoch, so
    no generation of the first replay satisfies the second."""
    inp, m, x, ids, rw, ref = tiny300
    st = Stream(m, slots=2, tokens_per_slot=128)
    xg = x.clone()
    out = torch.empty((inp.T, inp.H), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        st.begin(stream=s)
        for c, (base, n) in enumerate(chunks_of(inp.T, 128)):
            st.publish(c, base, n, xg, ids, rw, stream=s)
            st.forward(c, out, stream=s)
    g.replay()
    torch.cuda.synchronize()
    assert_close(out_bits(out), ref, "replay 1")
    inp2 = gen.tiny(5, inp.T)
    for name in ("w13", "sf13", "w2", "sf2", "dXdW13", "qA", "dAdW2", "expert_ids", "route_weights", "qX"):
        setattr(inp2, name, getattr(inp, name))
    xg.copy_(dev(inp2.x, torch.bfloat16))
    out.fill_(0)
    g.replay()
    torch.cuda.synchronize()
    assert api.moe_read_status(st.ws) == (0, 0)
    assert api.moe_stream_read_status(st.ring) == 0
    assert_close(out_bits(out), cases.run_oracle(inp2), "replay 2")


def test_forward_wait_runs_out_without_publish(tiny300):
    """A chunk that nothing publishes: the forward's bounded wait gives up,
    records MOE_DEVSTAT_STREAM_WAIT, writes no output row and does not mark
    the slot consumed (a later publish of the next occupant then gives up too)."""
    inp, m, x, ids, rw, ref = tiny300
    st = Stream(m, slots=1, tokens_per_slot=64)
    out = torch.zeros((inp.T, inp.H), dtype=torch.bfloat16, device="cuda")
    st.begin()
    st.forward(0, out, wait_us=SHORT_WAIT_US)
    torch.cuda.synchronize()
    status, _ = api.moe_read_status(st.ws)
    assert status & api.DEVSTAT_STREAM_WAIT
    assert not out.view(torch.int16).any()
    st.publish(1, 0, 64, x, ids, rw, wait_us=SHORT_WAIT_US)   # slot 0 still holds unconsumed chunk 0
    torch.cuda.synchronize()
    assert api.moe_stream_read_status(st.ring) == api.STREAM_PRODUCER_TIMEOUT


def test_publish_wait_runs_out_and_copies_nothing(tiny300):
    """Publishing chunk c + slots before chunk c is consumed: the producer's
    bounded wait gives up, the ring status says so, and the slot still holds
    chunk c, whose forward then produces chunk c's rows."""
    inp, m, x, ids, rw, ref = tiny300
    st = Stream(m, slots=2, tokens_per_slot=128)
    out = torch.zeros((inp.T, inp.H), dtype=torch.bfloat16, device="cuda")
    st.begin()
    st.publish(0, 0, 128, x, ids, rw)
    st.publish(1, 128, 128, x, ids, rw)
    st.publish(2, 256, 44, x, ids, rw, wait_us=SHORT_WAIT_US)   # slot 0: chunk 0 not consumed yet
    torch.cuda.synchronize()
    assert api.moe_stream_read_status(st.ring) == api.STREAM_PRODUCER_TIMEOUT
    st.forward(0, out)
    torch.cuda.synchronize()
    assert api.moe_read_status(st.ws) == (0, 0)
    got = out_bits(out)
    assert_close(got[:128], ref[:128], "chunk 0 after the refused publish")
    assert not got[128:].any()


def test_rows_past_the_output_are_refused(tiny300):
    """A chunk whose token base and count run past out_rows: status
    MOE_DEVSTAT_STREAM_BOUNDS and no row written; the slot is released."""
    inp, m, x, ids, rw, ref = tiny300
    st = Stream(m, slots=1, tokens_per_slot=64)
    out = torch.zeros((100, inp.H), dtype=torch.bfloat16, device="cuda")
    st.begin()
    st.publish(0, 60, 64, x, ids, rw)
    st.forward(0, out)
    st.publish(1, 0, 64, x, ids, rw, wait_us=SHORT_WAIT_US)
    st.forward(1, out)
    torch.cuda.synchronize()
    status, _ = api.moe_read_status(st.ws)
    assert status == api.DEVSTAT_STREAM_BOUNDS
    assert api.moe_stream_read_status(st.ring) == 0
    got = out_bits(out)
    assert not got[64:].any()
    assert_close(got[:64], ref[:64], "chunk 1 after the refused chunk")
