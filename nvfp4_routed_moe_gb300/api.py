"""ctypes binding of libnvfp4moe.so -- argument marshalling only.

Every function has the name of the C entry point it calls (see
include/nvfp4moe.h, include/nvfp4moe_stream.h and include/nvfp4moe_testing.h).  Tensor arguments are
torch tensors already on the GPU; the binding passes their data pointers,
byte sizes and the current CUDA stream, and raises :class:`MoeError` on a
non-OK status.  No computation happens here, and there is no fallback: if the
library is missing the first call raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "lib", "libnvfp4moe.so")
_lib = None

MOE_OK = 0
STATUS_NAMES = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED", 3: "MOE_ERR_WORKSPACE_TOO_SMALL",
                4: "MOE_ERR_NOT_PREPARED", 5: "MOE_ERR_CUDA", 6: "MOE_ERR_DEVICE_STATUS"}
DEVSTAT_INVALID_EXPERT, DEVSTAT_TIMEOUT, DEVSTAT_BAD_TILE = 1, 2, 4
DEVSTAT_STREAM_WAIT, DEVSTAT_STREAM_BOUNDS, DEVSTAT_NOT_PREPARED = 8, 16, 32
STREAM_ROUTE, STREAM_LAYOUT = 1, 2
STREAM_PRODUCER_TIMEOUT = 1

EXPORTED = ["moe_workspace_size", "moe_prepared_weight_bytes", "moe_prepare_weights", "moe_prepare_workspace",
            "moe_forward", "moe_forward_local_experts", "moe_init_routing", "moe_init_routing_static", "moe_read_status", "moe_status_string", "moe_test_codec_sweep",
            "moe_test_quantize_rows", "moe_test_situ_requant", "moe_test_requant_lanes", "moe_test_mma_fp4", "moe_test_mma_peak",
            "moe_workspace_layout", "moe_forward_launch_count", "moe_forward_kernels", "moe_profile_start", "moe_profile_stop",
            "moe_stream_ring_size", "moe_stream_ring_init", "moe_stream_begin", "moe_stream_publish",
            "moe_stream_forward", "moe_stream_read_status"]


class MoeError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {STATUS_NAMES.get(status, status)}")
        self.status = status


class moe_shape_t(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int32), ("inter", ctypes.c_int32), ("num_experts", ctypes.c_int32),
                ("top_k", ctypes.c_int32)]


class moe_routing_opts_t(ctypes.Structure):
    _fields_ = [("drop_pad", ctypes.c_int32), ("expert_capacity", ctypes.c_int32), ("row_idx_type", ctypes.c_int32),
                ("tokens_num_type", ctypes.c_int32), ("quant_mode", ctypes.c_int32), ("expert_start", ctypes.c_int32),
                ("expert_end", ctypes.c_int32), ("active_num", ctypes.c_int64), ("scale", ctypes.c_void_p),
                ("scale_rows", ctypes.c_int32), ("offset", ctypes.c_void_p), ("available_out", ctypes.c_void_p)]


class moe_ws_layout_t(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in
                ("max_tokens", "pairs_max", "padded_rows_max", "tiles_max", "header", "count", "cumsum", "offs",
                 "poffs", "sorted_row", "gather", "row_pos", "prow_pair", "tt_list", "xq", "sfx", "sft", "aq", "sfa",
                 "acc", "total")]


class moe_stream_ring_t(ctypes.Structure):
    _fields_ = [("num_slots", ctypes.c_int32), ("tokens_per_slot", ctypes.c_int32), ("max_sms", ctypes.c_int32)]


def shape(hidden: int, inter: int, num_experts: int, top_k: int) -> moe_shape_t:
    return moe_shape_t(hidden, inter, num_experts, top_k)


def lib():
    """Load the library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with `python -m nvfp4_routed_moe_gb300.build`")
    L = ctypes.CDLL(LIB_PATH)
    P, i32, i64, u32, f32, sz = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_uint32, ctypes.c_float,
                                 ctypes.c_size_t)
    S = ctypes.POINTER(moe_shape_t)
    R = ctypes.POINTER(moe_stream_ring_t)
    sig = {
        "moe_workspace_size": [S, i64, ctypes.POINTER(sz)],
        "moe_prepared_weight_bytes": [S] + [ctypes.POINTER(sz)] * 4,
        "moe_prepare_weights": [S] + [P] * 8 + [P],
        "moe_prepare_workspace": [S, P, sz, i64, P],
        "moe_forward": [S, i64] + [P] * 13 + [P, sz, P, P],
        "moe_forward_local_experts": [S, i32, i64] + [P] * 13 + [P, sz, P, P],
        "moe_init_routing": [S, i64, P, P, ctypes.POINTER(moe_routing_opts_t), P, P, P, P, P, sz, P],
        "moe_init_routing_static": [S, i64, P, P, ctypes.POINTER(moe_routing_opts_t), P, P, P, P, P],
        "moe_read_status": [P, P, P],
        "moe_test_codec_sweep": [u32, i64, P, P, P, P],
        "moe_test_quantize_rows": [P, i64, i32, P, P, P, P],
        "moe_test_situ_requant": [P, i64, i32, f32, f32, f32, P, P, P, P],
        "moe_test_requant_lanes": [P, i64, i32, f32, P, P, P],
        "moe_test_mma_fp4": [P, P, P, P, i32, i32, P, P, P],
        "moe_test_mma_peak": [i32, i32, i32, i32, i32, P, P, P],
        "moe_workspace_layout": [S, sz, ctypes.POINTER(moe_ws_layout_t)],
        "moe_forward_launch_count": [S, i64, ctypes.POINTER(i32)],
        "moe_forward_kernels": [S, i64, ctypes.POINTER(i32), ctypes.POINTER(i32)],
        "moe_profile_start": [i32],
        "moe_profile_stop": [ctypes.POINTER(ctypes.c_float), ctypes.POINTER(i32)],
        "moe_stream_ring_size": [S, R, ctypes.POINTER(sz)],
        "moe_stream_ring_init": [S, R, P, sz, P],
        "moe_stream_begin": [S, R, P, sz, P],
        "moe_stream_publish": [S, R, P, sz, i64, i64, i32, i32, P, P, P, u32, P],
        "moe_stream_forward": [S, R, P, sz, i64] + [P] * 10 + [P, sz, P, i64, u32, P],
        "moe_stream_read_status": [P, P, P],
    }
    for name, args in sig.items():
        fn = getattr(L, name)
        fn.argtypes = args
        fn.restype = ctypes.c_int
    L.moe_status_string.argtypes = [ctypes.c_int]
    L.moe_status_string.restype = ctypes.c_char_p
    _lib = L
    return L


def _p(t):
    if t is None:
        return None
    if isinstance(t, int):
        return ctypes.c_void_p(t)
    return ctypes.c_void_p(t.data_ptr())


def _nbytes(t) -> int:
    return t.numel() * t.element_size()


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check(st: int, what: str):
    if st != MOE_OK:
        raise MoeError(st, what)


def moe_status_string(status: int) -> str:
    return lib().moe_status_string(status).decode()


def moe_workspace_size(shp: moe_shape_t, max_tokens: int) -> int:
    out = ctypes.c_size_t()
    _check(lib().moe_workspace_size(ctypes.byref(shp), max_tokens, ctypes.byref(out)), "moe_workspace_size")
    return out.value


def moe_prepared_weight_bytes(shp: moe_shape_t):
    v = [ctypes.c_size_t() for _ in range(4)]
    _check(lib().moe_prepared_weight_bytes(ctypes.byref(shp), *[ctypes.byref(x) for x in v]),
           "moe_prepared_weight_bytes")
    return tuple(x.value for x in v)


def moe_prepare_weights(shp, w13, sf13, w2, sf2, w13_out, sf13_out, w2_out, sf2_out, stream=None):
    _check(lib().moe_prepare_weights(ctypes.byref(shp), _p(w13), _p(sf13), _p(w2), _p(sf2), _p(w13_out),
                                     _p(sf13_out), _p(w2_out), _p(sf2_out), _stream(stream)), "moe_prepare_weights")


def moe_prepare_workspace(shp, ws, num_tokens: int, stream=None):
    _check(lib().moe_prepare_workspace(ctypes.byref(shp), _p(ws), _nbytes(ws), num_tokens, _stream(stream)),
           "moe_prepare_workspace")


def moe_forward(shp, num_tokens, x, expert_ids, route_weights, w13, sf13, w2, sf2, qX, dX_dW13, qA, dA_dW2,
                situ_beta, situ_linear_beta, ws, out, stream=None):
    _check(lib().moe_forward(ctypes.byref(shp), num_tokens, _p(x), _p(expert_ids), _p(route_weights), _p(w13),
                             _p(sf13), _p(w2), _p(sf2), _p(qX), _p(dX_dW13), _p(qA), _p(dA_dW2), _p(situ_beta),
                             _p(situ_linear_beta), _p(ws), _nbytes(ws), _p(out), _stream(stream)), "moe_forward")


def moe_forward_local_experts(shp, expert_begin: int, num_tokens: int, x, expert_ids, route_weights, w13, sf13, w2,
                              sf2, qX, dX_dW13, qA, dA_dW2, situ_beta, situ_linear_beta, ws, out, stream=None):
    _check(lib().moe_forward_local_experts(ctypes.byref(shp), expert_begin, num_tokens, _p(x), _p(expert_ids),
                                           _p(route_weights), _p(w13), _p(sf13), _p(w2), _p(sf2), _p(qX),
                                           _p(dX_dW13), _p(qA), _p(dA_dW2), _p(situ_beta), _p(situ_linear_beta),
                                           _p(ws), _nbytes(ws), _p(out), _stream(stream)),
           "moe_forward_local_experts")


def routing_opts(drop_pad=0, expert_capacity=0, row_idx_type=0, tokens_num_type=0, quant_mode=1, expert_start=0,
                 expert_end=0, active_num=0, scale=None, scale_rows=0, offset=None, available_out=None):
    """moe_routing_opts_t with device tensors (or None) for scale, offset, available_out."""
    ptr = lambda t: None if t is None else t.data_ptr()
    return moe_routing_opts_t(drop_pad, expert_capacity, row_idx_type, tokens_num_type, quant_mode, expert_start,
                              expert_end, active_num, ptr(scale), scale_rows, ptr(offset), ptr(available_out))


def moe_init_routing(shp, num_rows, x, expert_ids, opts: moe_routing_opts_t, expanded_x, expanded_row_idx,
                     tokens_cumsum_or_count, expanded_scale, ws, stream=None):
    _check(lib().moe_init_routing(ctypes.byref(shp), num_rows, _p(x), _p(expert_ids), ctypes.byref(opts),
                                  _p(expanded_x), _p(expanded_row_idx), _p(tokens_cumsum_or_count),
                                  _p(expanded_scale), _p(ws), _nbytes(ws), _stream(stream)), "moe_init_routing")


def moe_init_routing_static(shp, num_rows, x, expert_ids, opts: moe_routing_opts_t, expanded_x, expanded_row_idx,
                            tokens_cumsum_or_count, expanded_scale, stream=None):
    _check(lib().moe_init_routing_static(ctypes.byref(shp), num_rows, _p(x), _p(expert_ids), ctypes.byref(opts),
                                         _p(expanded_x), _p(expanded_row_idx), _p(tokens_cumsum_or_count),
                                         _p(expanded_scale), _stream(stream)), "moe_init_routing_static")


def moe_read_status(ws, stream=None):
    """Returns (status_word, skipped_ids) and clears them (synchronizes)."""
    h = (ctypes.c_int32 * 2)()
    st = lib().moe_read_status(_p(ws), ctypes.cast(h, ctypes.c_void_p), _stream(stream))
    if st not in (MOE_OK, 6):
        _check(st, "moe_read_status")
    return int(h[0]), int(h[1])


def moe_test_codec_sweep(start: int, n: int, e2m1_lo, e2m1_hi, e4m3, stream=None):
    _check(lib().moe_test_codec_sweep(start, n, _p(e2m1_lo), _p(e2m1_hi), _p(e4m3), _stream(stream)),
           "moe_test_codec_sweep")


def moe_test_quantize_rows(x, q_per_row, packed, sf, stream=None):
    rows, cols = x.shape
    _check(lib().moe_test_quantize_rows(_p(x), rows, cols, _p(q_per_row), _p(packed), _p(sf), _stream(stream)),
           "moe_test_quantize_rows")


def moe_test_situ_requant(z, inter, qA, beta, lam, a_out, packed, sf, stream=None):
    _check(lib().moe_test_situ_requant(_p(z), z.shape[0], inter, qA, beta, lam, _p(a_out), _p(packed), _p(sf),
                                       _stream(stream)), "moe_test_situ_requant")


def moe_test_requant_lanes(act, qA, packed, sf, stream=None):
    rows, inter = act.shape
    _check(lib().moe_test_requant_lanes(_p(act), rows, inter, qA, _p(packed), _p(sf), _stream(stream)),
           "moe_test_requant_lanes")


def moe_test_mma_fp4(a, sfa_atoms, b, sfb_atoms, n, k, d, status, stream=None):
    _check(lib().moe_test_mma_fp4(_p(a), _p(sfa_atoms), _p(b), _p(sfb_atoms), n, k, _p(d), _p(status),
                                  _stream(stream)), "moe_test_mma_fp4")


def moe_test_mma_peak(grid: int, n: int, mmas: int, copies: int, cycles, status, stream=None, accs: int = 1):
    _check(lib().moe_test_mma_peak(grid, n, mmas, copies, accs, _p(cycles), _p(status), _stream(stream)),
           "moe_test_mma_peak")


def moe_workspace_layout(shp, ws_bytes: int) -> moe_ws_layout_t:
    out = moe_ws_layout_t()
    _check(lib().moe_workspace_layout(ctypes.byref(shp), ws_bytes, ctypes.byref(out)), "moe_workspace_layout")
    return out


def moe_forward_kernels(shp, num_tokens: int):
    """(fc1_decode, fc2_decode): True where the forward runs the decode kernel."""
    a, b = ctypes.c_int32(), ctypes.c_int32()
    _check(lib().moe_forward_kernels(ctypes.byref(shp), num_tokens, ctypes.byref(a), ctypes.byref(b)),
           "moe_forward_kernels")
    return bool(a.value), bool(b.value)


def moe_forward_launch_count(shp, num_tokens: int) -> int:
    out = ctypes.c_int32()
    _check(lib().moe_forward_launch_count(ctypes.byref(shp), num_tokens, ctypes.byref(out)),
           "moe_forward_launch_count")
    return out.value


STAGES = ("routing", "quant_x", "fc1", "fc2", "finalize")


def moe_profile_start(max_calls: int):
    _check(lib().moe_profile_start(max_calls), "moe_profile_start")


def moe_profile_stop():
    """Returns ({stage: summed ms}, calls)."""
    ms = (ctypes.c_float * len(STAGES))()
    calls = ctypes.c_int32()
    _check(lib().moe_profile_stop(ms, ctypes.byref(calls)), "moe_profile_stop")
    return dict(zip(STAGES, [float(v) for v in ms])), calls.value


# ------------------------------------------------------------ streaming front end
def moe_stream_ring_size(shp, ring_cfg: moe_stream_ring_t) -> int:
    out = ctypes.c_size_t()
    _check(lib().moe_stream_ring_size(ctypes.byref(shp), ctypes.byref(ring_cfg), ctypes.byref(out)),
           "moe_stream_ring_size")
    return out.value


def moe_stream_ring_init(shp, ring_cfg: moe_stream_ring_t, ring, stream=None):
    _check(lib().moe_stream_ring_init(ctypes.byref(shp), ctypes.byref(ring_cfg), _p(ring), _nbytes(ring),
                                      _stream(stream)), "moe_stream_ring_init")


def moe_stream_begin(shp, ring_cfg: moe_stream_ring_t, ring, stream=None):
    _check(lib().moe_stream_begin(ctypes.byref(shp), ctypes.byref(ring_cfg), _p(ring), _nbytes(ring),
                                  _stream(stream)), "moe_stream_begin")


def moe_stream_publish(shp, ring_cfg: moe_stream_ring_t, ring, chunk: int, token_base: int, n: int, parts: int,
                       x=None, expert_ids=None, route_weights=None, wait_us: int = 0, stream=None):
    _check(lib().moe_stream_publish(ctypes.byref(shp), ctypes.byref(ring_cfg), _p(ring), _nbytes(ring), chunk,
                                    token_base, n, parts, _p(x), _p(expert_ids), _p(route_weights), wait_us,
                                    _stream(stream)), "moe_stream_publish")


def moe_stream_forward(shp, ring_cfg: moe_stream_ring_t, ring, chunk: int, w13, sf13, w2, sf2, qX, dX_dW13, qA,
                       dA_dW2, situ_beta, situ_linear_beta, ws, out, wait_us: int = 0, stream=None):
    _check(lib().moe_stream_forward(ctypes.byref(shp), ctypes.byref(ring_cfg), _p(ring), _nbytes(ring), chunk,
                                    _p(w13), _p(sf13), _p(w2), _p(sf2), _p(qX), _p(dX_dW13), _p(qA), _p(dA_dW2),
                                    _p(situ_beta), _p(situ_linear_beta), _p(ws), _nbytes(ws), _p(out),
                                    out.shape[0], wait_us, _stream(stream)), "moe_stream_forward")


def moe_stream_read_status(ring, stream=None) -> int:
    """Returns the ring status word (STREAM_* bits) and clears it (synchronizes)."""
    h = ctypes.c_int32()
    _check(lib().moe_stream_read_status(_p(ring), ctypes.cast(ctypes.byref(h), ctypes.c_void_p), _stream(stream)),
           "moe_stream_read_status")
    return int(h.value)
