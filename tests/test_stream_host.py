"""Host-side checks of the streaming front end's C ABI that need no GPU:
ring sizes, and argument validation that returns before anything touches
the device ("[RFC] Chunk-ready symmetric-buffer protocol for streaming
MegaMoE inputs", section "Fixed-capacity ring": the ring is fixed-capacity
and caller-owned, so every size and index is checked up front)."""
import ctypes

import pytest

from nvfp4_routed_moe_gb300 import api


@pytest.fixture(scope="module")
def L():
    from nvfp4_routed_moe_gb300 import build
    build.build()
    return api.lib()


FULL = api.shape(3584, 384, 896, 16)


def test_ring_size_covers_the_payload(L):
    for S, C in ((1, 1), (2, 128), (4, 4096), (64, 16)):
        n = api.moe_stream_ring_size(FULL, api.moe_stream_ring_t(S, C))
        payload = S * C * (3584 * 2 + 16 * 4 + 16 * 2)
        assert payload + 256 + 64 * S <= n <= payload + 256 + 64 * S + 4 * 256
        assert n % 256 == 0
    sizes = [api.moe_stream_ring_size(FULL, api.moe_stream_ring_t(2, C)) for C in (1, 16, 256, 4096)]
    assert sizes == sorted(sizes)


def test_ring_config_validation(L):
    for S, C, want in ((0, 16, 1), (65, 16, 1), (2, 0, 1), (2, (1 << 31) // 16, 2)):
        with pytest.raises(api.MoeError) as e:
            api.moe_stream_ring_size(FULL, api.moe_stream_ring_t(S, C))
        assert e.value.status == want
    with pytest.raises(api.MoeError) as e:
        api.moe_stream_ring_size(api.shape(3584, 200, 896, 16), api.moe_stream_ring_t(2, 16))
    assert e.value.status == 2
    # the SM budget: non-negative, and no part of the ring's size
    with pytest.raises(api.MoeError) as e:
        api.moe_stream_ring_size(FULL, api.moe_stream_ring_t(2, 16, -1))
    assert e.value.status == 1
    assert api.moe_stream_ring_size(FULL, api.moe_stream_ring_t(2, 16, 96)) == \
        api.moe_stream_ring_size(FULL, api.moe_stream_ring_t(2, 16))


def test_calls_rejected_before_the_device(L):
    cfg = api.moe_stream_ring_t(2, 16)
    n = api.moe_stream_ring_size(FULL, cfg)
    R, p = ctypes.byref(cfg), ctypes.c_void_p(256)
    S = ctypes.byref(FULL)
    assert L.moe_stream_ring_init(S, R, None, n, None) == 1
    assert L.moe_stream_ring_init(S, R, ctypes.c_void_p(257), n, None) == 1          # misaligned
    assert L.moe_stream_ring_init(S, R, p, n - 256, None) == 3                      # too small
    assert L.moe_stream_begin(S, R, p, n - 1, None) == 3
    both = api.STREAM_ROUTE | api.STREAM_LAYOUT
    pub = lambda chunk, base, cnt, parts, x=p, ids=p, w=p: L.moe_stream_publish(
        S, R, p, n, chunk, base, cnt, parts, x, ids, w, 0, None)
    assert pub(-1, 0, 4, both) == 1                        # negative chunk
    assert pub((1 << 32) - 1, 0, 4, both) == 1             # sequence would overflow its 32 bits
    assert pub(0, -1, 4, both) == 1                        # negative token base
    assert pub(0, 0, 17, both) == 1                        # more tokens than a slot holds
    assert pub(0, 0, -1, both) == 1
    assert pub(0, 0, 4, 0) == 1 and pub(0, 0, 4, 4) == 1  # no such parts
    assert pub(0, 0, 4, api.STREAM_LAYOUT, x=None) == 1
    assert pub(0, 0, 4, api.STREAM_LAYOUT, x=ctypes.c_void_p(264)) == 1   # x not 16-byte aligned
    assert pub(0, 0, 4, api.STREAM_ROUTE, ids=None) == 1
    fwd = lambda chunk, ws_bytes, out_rows: L.moe_stream_forward(
        S, R, p, n, chunk, *([p] * 10), p, ws_bytes, p, out_rows, 0, None)
    assert fwd(0, 1 << 30, 0) == 1                         # no output rows
    assert fwd(-1, 1 << 30, 8) == 1
    assert fwd(0, 1024, 8) == 3                            # workspace smaller than one slot's tokens
    assert fwd(0, 1 << 30, 8) == 4                         # workspace not prepared
    assert L.moe_stream_read_status(None, p, None) == 1
