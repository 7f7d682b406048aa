"""CPU oracle of the routed NVFP4 SiTU MoE forward -- TEST INFRASTRUCTURE.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never imports, links or runs it, and the oracle shares no
code with it.

The arithmetic lives in ``moe_oracle.c`` (plain C, fp64 accumulation, fp32
quantizer steps compiled with ``-ffp-contract=off``); this module only builds
it with gcc and marshals numpy arrays.  Each wrapper names the page passage its
C function follows:

* "Cake SiTU backend" (FlashInfer tutorial): the forward, the six scales,
  ``qX = 1/dX``, ``qA = 1/dA``, default SiTU 4/25, storage shapes.
* "npu_moe_init_routing_v2" (torch_npu), formulas 1-6: routing and init-routing.
* "Nvfp4 Tensor" (TensorRT-Edge-LLM): global scale after block dequantization.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP, no FMA contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fopenmp", "-shared", "-fPIC",
           "-std=c11", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i32, i64, u32, f32 = ctypes.c_int32, ctypes.c_int64, ctypes.c_uint32, ctypes.c_float
        lib.oracle_e2m1_value.restype = ctypes.c_double
        lib.oracle_e2m1_value.argtypes = [ctypes.c_uint8]
        lib.oracle_e2m1_encode.restype = ctypes.c_uint8
        lib.oracle_e2m1_encode.argtypes = [f32]
        lib.oracle_e4m3_value.restype = ctypes.c_double
        lib.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_encode.restype = ctypes.c_uint8
        lib.oracle_e4m3_encode.argtypes = [f32]
        lib.oracle_float_to_bf16.restype = ctypes.c_uint16
        lib.oracle_float_to_bf16.argtypes = [f32]
        lib.oracle_nvfp4_quant_group.restype = None
        lib.oracle_nvfp4_quant_group.argtypes = [P, f32, P, P]
        lib.oracle_nvfp4_quant_rows.restype = None
        lib.oracle_nvfp4_quant_rows.argtypes = [P, i64, i64, P, f32, P, P]
        lib.oracle_nvfp4_dequant_rows.restype = None
        lib.oracle_nvfp4_dequant_rows.argtypes = [P, P, i64, i64, P]
        lib.oracle_routing.restype = i64
        lib.oracle_routing.argtypes = [P, i64, i32, i32, P, P, P, P, P]
        lib.oracle_dynamic_int8_row.restype = None
        lib.oracle_dynamic_int8_row.argtypes = [P, i64, P, P]
        lib.oracle_init_routing.restype = i64
        lib.oracle_init_routing.argtypes = [P, P, i64, i32, i32, i64, i32, i32, i32, i32, i32, P, P, P, P]
        lib.oracle_init_routing_ex.restype = i64
        lib.oracle_init_routing_ex.argtypes = [P, P, i64, i32, i32, i64, i32, i32, i64, i32, i32, i32, i32, i32,
                                               P, i32, P, P, P, P, P]
        lib.oracle_situ.restype = ctypes.c_double
        lib.oracle_situ.argtypes = [ctypes.c_double] * 4
        lib.oracle_moe_forward_tokens.restype = None
        lib.oracle_moe_forward_tokens.argtypes = [i32, i32, i32, i32, P, P, P, P, i64,
                                                  P, P, P, P, P, P, P, P, P, P, P, P, P, P, P, P]
        lib.oracle_situ_requant_rows.restype = None
        lib.oracle_situ_requant_rows.argtypes = [P, i64, i32, f32, f32, f32, P, P, P]
        lib.oracle_e2m1_encode_range.restype = None
        lib.oracle_e2m1_encode_range.argtypes = [u32, i64, P]
        lib.oracle_e4m3_encode_range.restype = None
        lib.oracle_e4m3_encode_range.argtypes = [u32, i64, P]
        lib.oracle_scale_atom_offset.restype = i64
        lib.oracle_scale_atom_offset.argtypes = [i64, i64, i64]
        lib.oracle_num_threads.restype = ctypes.c_int
        lib.oracle_num_threads.argtypes = []
        lib.oracle_set_num_threads.restype = None
        lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
        _lib = lib
        return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def set_num_threads(n: int) -> None:
    """Threads of the oracle's parallel loops from now on."""
    _load().oracle_set_num_threads(int(n))


# --------------------------------------------------------------------- codecs

def e2m1_value(code: int) -> float:
    """Value of a 4-bit E2M1 code (sign in bit 3)."""
    return float(_load().oracle_e2m1_value(code))


def e2m1_encode(v: float) -> int:
    """fp32 -> E2M1, round-to-nearest-even, saturating at 6."""
    return int(_load().oracle_e2m1_encode(v))


def e4m3_value(b: int) -> float:
    return float(_load().oracle_e4m3_value(b))


def e4m3_encode(v: float) -> int:
    """fp32 -> E4M3 (fn), round-to-nearest-even, saturating at 448."""
    return int(_load().oracle_e4m3_encode(v))


def e2m1_encode_range(start: int, n: int) -> np.ndarray:
    out = np.empty(n, np.uint8)
    _load().oracle_e2m1_encode_range(start, n, _ptr(out))
    return out


def e4m3_encode_range(start: int, n: int) -> np.ndarray:
    out = np.empty(n, np.uint8)
    _load().oracle_e4m3_encode_range(start, n, _ptr(out))
    return out


def float_to_bf16_bits(f: float) -> int:
    return int(_load().oracle_float_to_bf16(f))


def scale_atom_offset(m_row: int, k_chunk: int, num_sf_cols: int) -> int:
    """Byte offset of block scale (m_row, k_chunk) in the 128x4 atom layout
    ("Nvfp4 Tensor", block_scale / tileScaleIndex)."""
    return int(_load().oracle_scale_atom_offset(m_row, k_chunk, num_sf_cols))


def to_atom_layout(sf_rows):
    """Scatter a row-major scale matrix [rows, cols] (rows % 128 == 0) into the
    128x4 atom layout, one byte at a time through scale_atom_offset."""
    sf_rows = _c(sf_rows, np.uint8)
    rows, cols = sf_rows.shape
    nkt = (cols + 3) // 4
    out = np.zeros(((rows + 127) // 128) * nkt * 512, np.uint8)
    lib = _load()
    for r in range(rows):
        for c in range(cols):
            out[lib.oracle_scale_atom_offset(r, c, cols)] = sf_rows[r, c]
    return out


# ------------------------------------------------------------ NVFP4 quantizer

def nvfp4_quant_group(v, q: float):
    """Group-16 quantization ("Cake SiTU backend": group-16 NVFP4 with encode
    scale q).  Returns (codes[16] uint8, sf byte)."""
    v = _c(v, np.float32)
    assert v.shape == (16,)
    codes = np.empty(16, np.uint8)
    sf = np.empty(1, np.uint8)
    _load().oracle_nvfp4_quant_group(_ptr(v), float(np.float32(q)), _ptr(codes), _ptr(sf))
    return codes, int(sf[0])


def nvfp4_quant_rows(x, q=None, q_per_row=None):
    """Quantize [rows, cols] fp32 to packed codes [rows, cols/2] and E4M3
    block scales [rows, cols/16] (canonical row-major layout)."""
    x = _c(x, np.float32)
    rows, cols = x.shape
    assert cols % 16 == 0
    packed = np.empty((rows, cols // 2), np.uint8)
    sf = np.empty((rows, cols // 16), np.uint8)
    qpr = None if q_per_row is None else _c(q_per_row, np.float32)
    _load().oracle_nvfp4_quant_rows(_ptr(x), rows, cols, _ptr(qpr), float(np.float32(q or 0.0)),
                                    _ptr(packed), _ptr(sf))
    return packed, sf


def nvfp4_dequant_rows(packed, sf):
    """E2M1(code) * S per element (fp64); the global scale is not applied."""
    packed = _c(packed, np.uint8)
    sf = _c(sf, np.uint8)
    rows = packed.shape[0]
    cols = packed.shape[1] * 2
    out = np.empty((rows, cols), np.float64)
    _load().oracle_nvfp4_dequant_rows(_ptr(packed), _ptr(sf), rows, cols, _ptr(out))
    return out


# -------------------------------------------------------------------- routing

def routing(expert_ids, num_experts: int):
    """keyValueSort / expanded_row_idx / histogram ("npu_moe_init_routing_v2",
    formulas 1-3).  Returns dict with sorted_row (scatter form), sorted_expert,
    gather (gather form), count, cumsum (inclusive), nvalid."""
    ids = _c(expert_ids, np.int32)
    T, k = ids.shape
    P = T * k
    sorted_row = np.empty(max(P, 1), np.int32)
    sorted_expert = np.empty(max(P, 1), np.int32)
    gather = np.empty(max(P, 1), np.int32)
    count = np.empty(num_experts, np.int32)
    cumsum = np.empty(num_experts, np.int32)
    nvalid = _load().oracle_routing(_ptr(ids), T, k, num_experts, _ptr(sorted_row), _ptr(sorted_expert),
                                    _ptr(gather), _ptr(count), _ptr(cumsum))
    return dict(sorted_row=sorted_row[:P], sorted_expert=sorted_expert[:P], gather=gather[:P],
                count=count, cumsum=cumsum, nvalid=int(nvalid))


def dynamic_int8_row(x_bf16_bits):
    """Dynamic int8 quant of one row ("npu_moe_init_routing_v2", formula 4)."""
    x = _c(x_bf16_bits, np.uint16)
    q = np.empty(x.shape[0], np.int8)
    s = np.empty(1, np.float32)
    _load().oracle_dynamic_int8_row(_ptr(x), x.shape[0], _ptr(q), _ptr(s))
    return q, float(s[0])


def init_routing(x_bf16_bits, expert_ids, num_experts: int, *, drop_pad: int = 0, expert_capacity: int = 0,
                 row_idx_type: int = 0, tokens_num_type: int = 0, quant_mode: int = 1):
    """Full init-routing ("npu_moe_init_routing_v2", formulas 1-5).
    Returns (expanded_x, expanded_row_idx, tokens_cumsum_or_count, expanded_scale, nvalid)."""
    x = _c(x_bf16_bits, np.uint16)
    ids = _c(expert_ids, np.int32)
    T, H = x.shape
    k = ids.shape[1]
    P = T * k
    rows = num_experts * expert_capacity if drop_pad else P
    if quant_mode == 1:
        ex = np.zeros((rows, H), np.int8)
        scale = np.zeros(max(rows, 1), np.float32)
    else:
        ex = np.zeros((rows, H), np.uint16)
        scale = None
    ridx = np.empty(max(P, 1), np.int32)
    tok = np.empty(num_experts, np.int32)
    nvalid = _load().oracle_init_routing(_ptr(x), _ptr(ids), T, k, num_experts, H, drop_pad, expert_capacity,
                                         row_idx_type, tokens_num_type, quant_mode, _ptr(ex), _ptr(ridx),
                                         _ptr(tok), _ptr(scale))
    if scale is not None:
        scale = scale[:rows]
    return ex, ridx[:P], tok, scale, int(nvalid)


def init_routing_ex(x_bf16_bits, expert_ids, num_experts: int, *, expert_start: int = 0, expert_end=None,
                    active_num: int = 0, drop_pad: int = 0, expert_capacity: int = 0, row_idx_type: int = 0,
                    tokens_num_type: int = 0, quant_mode: int = 1, scale=None, offset=None):
    """Init-routing with every option of the page's parameter list
    ("npu_moe_init_routing_v2": active_expert_range, active_num,
    expert_tokens_num_type 0/1/2, quant_mode -1/0/1 with scale / offset).
    Returns (expanded_x, expanded_row_idx, tokens_out, expanded_scale,
    available); tokens_out is [end-start] (cumsum or count) or [E, 2]
    (key_value)."""
    x = _c(x_bf16_bits, np.uint16)
    ids = _c(expert_ids, np.int32)
    T, H = x.shape
    k = ids.shape[1]
    P = T * k
    end = num_experts if expert_end is None else expert_end
    R = end - expert_start
    rows = R * expert_capacity if drop_pad else P
    ex = np.zeros((rows, H), np.uint16 if quant_mode == -1 else np.int8)
    want_scale = quant_mode == 1 or (quant_mode == -1 and scale is not None)
    sc_out = np.zeros(max(rows, 1), np.float32) if want_scale else None
    if scale is None:
        sc_in, scale_rows = None, 0
    elif quant_mode == 1:                       # smooth scale rows [1 or end-start, H]
        sc_in = _c(np.asarray(scale, np.float32).reshape(-1, H), np.float32)
        scale_rows = sc_in.shape[0]
    else:                                       # [T] (no quant) or [1] (static)
        sc_in, scale_rows = _c(np.asarray(scale, np.float32).ravel(), np.float32), 1
    off = None if offset is None else _c(np.asarray(offset, np.float32).ravel(), np.float32)
    ridx = np.empty(max(P, 1), np.int32)
    tok = np.zeros(2 * num_experts if tokens_num_type == 2 else max(R, 1), np.int32)
    avail = _load().oracle_init_routing_ex(_ptr(x), _ptr(ids), T, k, num_experts, H, expert_start, end, active_num,
                                           drop_pad, expert_capacity, row_idx_type, tokens_num_type, quant_mode,
                                           _ptr(sc_in), scale_rows, _ptr(off), _ptr(ex), _ptr(ridx), _ptr(tok),
                                           _ptr(sc_out))
    if tokens_num_type == 2:
        tok = tok.reshape(num_experts, 2)
    else:
        tok = tok[:R]
    return ex, ridx[:P], tok, (None if sc_out is None else sc_out[:rows]), int(avail)


# ----------------------------------------------------------------- the forward

def situ(g: float, u: float, beta: float = 4.0, lam: float = 25.0) -> float:
    """(beta*tanh(g/beta)*sigmoid(g)) * (lam*tanh(u/lam)) in fp64 ("Cake SiTU backend")."""
    return float(_load().oracle_situ(g, u, beta, lam))


def situ_requant_rows(z, I: int, qA: float, beta: float = 4.0, lam: float = 25.0):
    """SiTU + NVFP4 requant of fp32 pre-activation rows [rows, 2I] (gate | up)."""
    z = _c(z, np.float32)
    rows = z.shape[0]
    a = np.empty((rows, I), np.float32)
    packed = np.empty((rows, I // 2), np.uint8)
    sf = np.empty((rows, I // 16), np.uint8)
    _load().oracle_situ_requant_rows(_ptr(z), rows, I, float(np.float32(qA)), float(beta), float(lam),
                                     _ptr(a), _ptr(packed), _ptr(sf))
    return a, packed, sf


def moe_forward_tokens(*, H, I, E, k, x, expert_ids, route_weights, tokens, w13, sf13, w2, sf2,
                       qX, dXdW13, qA, dAdW2, beta=None, lam=None, want_intermediates=False):
    """Reference forward for the listed tokens ("Cake SiTU backend": quant X,
    FC1, SiTU, requant, FC2, BF16 weighted finalize).

    x: [T, H] bf16 bits (uint16); expert_ids [T, k] int32; route_weights
    [T, k] bf16 bits; weights in the canonical layout.  Returns out [ntok, H]
    as bf16 bits, and (if asked) z [ntok,k,2I], a [ntok,k,I], aq, asf, y.
    """
    x = _c(x, np.uint16)
    ids = _c(expert_ids, np.int32)
    rw = _c(route_weights, np.uint16)
    toks = _c(tokens, np.int64)
    n = toks.shape[0]
    out = np.empty((n, H), np.uint16)
    z = a = aq = asf = y = None
    if want_intermediates:
        z = np.zeros((n, k, 2 * I), np.float32)
        a = np.zeros((n, k, I), np.float32)
        aq = np.zeros((n, k, I // 2), np.uint8)
        asf = np.zeros((n, k, I // 16), np.uint8)
        y = np.zeros((n, k, H), np.float32)
    qX = _c(np.atleast_1d(qX), np.float32)
    args = [_c(w13, np.uint8), _c(sf13, np.uint8), _c(w2, np.uint8), _c(sf2, np.uint8), qX,
            _c(dXdW13, np.float32), _c(qA, np.float32), _c(dAdW2, np.float32),
            None if beta is None else _c(beta, np.float32), None if lam is None else _c(lam, np.float32)]
    _load().oracle_moe_forward_tokens(H, I, E, k, _ptr(x), _ptr(ids), _ptr(rw), _ptr(toks), n,
                                      *[_ptr(v) for v in args],
                                      _ptr(out), _ptr(z), _ptr(a), _ptr(aq), _ptr(asf), _ptr(y))
    if want_intermediates:
        return out, dict(z=z, a=a, aq=aq, asf=asf, y=y)
    return out
