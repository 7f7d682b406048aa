"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every entry point its headers declare, and rejects bad arguments before it
touches the device."""
import ctypes
import os
import re

import pytest

from nvfp4_routed_moe_gb300 import api

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = set()
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        src = open(os.path.join(ROOT, "include", h)).read()
        names |= set(re.findall(r"^\s*(?:moe_status_t|const char\*)\s+(moe_\w+)\(", src, re.M))
    return names


@pytest.fixture(scope="module")
def L():
    from nvfp4_routed_moe_gb300 import build
    build.build()
    return api.lib()


def test_exports_every_declared_symbol(L):
    declared = _declared()
    assert len(declared) >= 15
    for name in declared:
        assert hasattr(L, name), name
    assert declared == set(api.EXPORTED)


def test_status_strings(L):
    for code, name in api.STATUS_NAMES.items():
        assert api.moe_status_string(code) == name


def test_workspace_size_monotone_and_validation(L):
    full = api.shape(3584, 384, 896, 16)
    sizes = [api.moe_workspace_size(full, t) for t in (1, 8, 16, 4096, 16384)]
    assert sizes == sorted(sizes) and sizes[0] > 0
    for bad in (api.shape(3584, 384, 896, 0), api.shape(0, 384, 896, 16)):
        with pytest.raises(api.MoeError) as e:
            api.moe_workspace_size(bad, 16)
        assert e.value.status == 1
    for unsup in (api.shape(3600, 384, 896, 16), api.shape(3584, 200, 896, 16), api.shape(3584, 384, 2048, 16),
                  api.shape(512, 128, 8, 16)):
        with pytest.raises(api.MoeError) as e:
            api.moe_workspace_size(unsup, 16)
        assert e.value.status == 2
    with pytest.raises(api.MoeError):
        api.moe_workspace_size(full, 0)


def test_prepared_weight_bytes_match_page_shapes(L, golden_dir):
    full = api.shape(3584, 384, 896, 16)
    got = api.moe_prepared_weight_bytes(full)
    rows = [l.split() for l in open(os.path.join(golden_dir, "storage_shapes.txt")) if l.strip() and l[0] != "#"]
    assert list(got) == [int(r[-1]) for r in rows]


def test_layout_regions_fit_and_are_aligned(L):
    full = api.shape(3584, 384, 896, 16)
    n = api.moe_workspace_size(full, 4096)
    lay = api.moe_workspace_layout(full, n)
    assert lay.max_tokens >= 4096 and lay.total <= n
    offs = [lay.header, lay.count, lay.cumsum, lay.offs, lay.poffs, lay.sorted_row, lay.gather, lay.row_pos,
            lay.prow_pair, lay.tt_list, lay.xq, lay.sfx, lay.sft, lay.aq, lay.sfa, lay.acc]
    assert offs == sorted(offs) and all(o % 1024 == 0 for o in offs)
    assert lay.padded_rows_max % 128 == 0
    assert lay.padded_rows_max >= 4096 * 16 + 127 * 896


def test_null_and_bad_args_rejected_without_device(L):
    shp = api.shape(512, 128, 32, 4)
    st = L.moe_forward(ctypes.byref(shp), 16, *([None] * 13), None, 0, None, None)
    assert st == 1
    st = L.moe_prepare_workspace(ctypes.byref(shp), None, 0, 16, None)
    assert st == 1
    p = ctypes.c_void_p(256)
    O = api.moe_routing_opts_t
    for opts, want in ((O(0, 0, 0, 3, 1), 1),                          # no such histogram mode
                       (O(0, 0, 0, 0, 0), 1),                          # static int8 without scale / offset
                       (O(0, 0, 0, 0, 2), 1),                          # no such quant mode
                       (O(1, 0, 0, 0, 1), 1),                          # drop_pad without capacity
                       (O(0, 0, 3, 0, 1), 1),                          # bad row_idx_type
                       (O(0, 0, 0, 0, 1, 5, 5), 1),                    # empty expert range
                       (O(0, 0, 0, 0, 1, 4, 33), 1),                   # range past E
                       (O(1, 8, 0, 0, 1, 4, 20), 1),                   # drop/pad needs every expert
                       (O(0, 0, 0, 0, 1, 0, 0, 0, 256, 3), 1),         # smooth scale rows neither 1 nor the range
                       (O(0, 0, 0, 2, 1, 4, 20), 3)):                  # valid options, workspace too small
        st = L.moe_init_routing(ctypes.byref(shp), 16, p, p, ctypes.byref(opts), p, p, p, None, p, 1 << 18, None)
        assert st == want
    assert L.moe_test_mma_fp4(p, p, p, p, 200, 256, p, p, None) == 1
    assert L.moe_test_codec_sweep(0xFFFFFFF0, 100, None, None, None, None) == 1



def test_forward_token_count_alignment_and_capacity_checked_before_launch(L):
    """An empty or negative batch, a misaligned activation pointer, a batch
    larger than the workspace holds and a workspace never prepared are each
    refused on the host with their own status; the (aligned, fake) device
    pointers are never touched."""
    shp = api.shape(512, 128, 32, 4)
    n = api.moe_workspace_size(shp, 64)
    p = ctypes.c_void_p(1 << 20)

    def fwd(T, x=p):
        return L.moe_forward(ctypes.byref(shp), T, x, p, p, p, p, p, p, p, p, p, p, None, None, p, n, p, None)

    assert fwd(0) == 1                                  # empty batch
    assert fwd(-5) == 1
    assert fwd(16, x=ctypes.c_void_p((1 << 20) + 8)) == 1   # x not 16-byte aligned
    assert fwd(1 << 20) == 3                            # more tokens than the workspace holds
    assert fwd(16) == 4                                 # never prepared

def test_forward_kernel_choice(L, monkeypatch):
    """The decode kernels run FC1 up to 32 tokens and FC2 up to 16, the
    tcgen05 GEMMs above; the environment overrides either."""
    full = api.shape(3584, 384, 896, 16)
    assert api.moe_forward_kernels(full, 1) == (True, True)
    assert api.moe_forward_kernels(full, 16) == (True, True)
    assert api.moe_forward_kernels(full, 17) == (True, False)
    assert api.moe_forward_kernels(full, 32) == (True, False)
    assert api.moe_forward_kernels(full, 33) == (False, False)
    assert api.moe_forward_kernels(full, 16384) == (False, False)
    monkeypatch.setenv("NVFP4MOE_FC1_GEMV", "0")
    monkeypatch.setenv("NVFP4MOE_FC2_GEMV", "1")
    assert api.moe_forward_kernels(full, 4096) == (False, True)
    assert api.moe_forward_kernels(full, 8) == (False, True)


def test_launch_count(L):
    assert api.moe_forward_launch_count(api.shape(3584, 384, 896, 16), 1) == 5
    assert api.moe_forward_launch_count(api.shape(3584, 384, 896, 16), 4096) == 7
    assert api.moe_forward_launch_count(api.shape(3584, 384, 896, 16), 16384) == 7
