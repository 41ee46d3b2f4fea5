"""CPU oracle for the MXFP4 lightning-indexer path (test infrastructure).

Only the tests, the smoke check and the benchmark's CPU-baseline leg may import
this package.  It wraps ``oracle.c`` (plain C, fp64) through ctypes and shares
nothing with the CUDA library: no headers, helpers, tables or constants.

Every function states what it computes; the C source cites the pages each step
follows and lists the readings taken where the pages are silent.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
# A test may point the wrapper at a separately compiled variant of oracle.c
# (the mutation test plants mistakes in copies of the source this way).
_OVERRIDE = os.environ.get("IDX_ORACLE_LIB_OVERRIDE")
_lock = threading.Lock()
_lib = None

VAL_BYTES = 64
SCALE_BYTES = 4
HEAD_DIM = 128


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so with gcc (OpenMP, no fast-math)."""
    stale = (not os.path.exists(_LIB_PATH)) or (
        os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
               "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if _OVERRIDE:
            lib = ctypes.CDLL(_OVERRIDE)
        else:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
        P = ctypes.c_void_p
        i64, i32 = ctypes.c_int64, ctypes.c_int32
        lib.oracle_num_threads.restype = ctypes.c_int
        lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_double.restype = ctypes.c_double
        lib.oracle_ue8m0_scale.argtypes = [P, ctypes.c_int]
        lib.oracle_ue8m0_scale.restype = ctypes.c_uint8
        lib.oracle_e2m1_code.argtypes = [ctypes.c_double]
        lib.oracle_e2m1_code.restype = ctypes.c_uint8
        lib.oracle_e2m1_value.argtypes = [ctypes.c_uint8]
        lib.oracle_e2m1_value.restype = ctypes.c_double
        lib.oracle_quant_vec128.argtypes = [P, P, P]
        lib.oracle_quant_vec128.restype = None
        lib.oracle_dequant_vec128.argtypes = [P, P, P]
        lib.oracle_dequant_vec128.restype = None
        lib.oracle_quant_insert.argtypes = [P, i64, i64, P, P, i64, i32]
        lib.oracle_quant_insert.restype = i64
        lib.oracle_quant_q.argtypes = [P, i64, P, P]
        lib.oracle_quant_q.restype = None
        lib.oracle_mqa_logits.argtypes = [P, P, i64, i32, P, P, i64, P, P, P, P, P, i64]
        lib.oracle_mqa_logits.restype = None
        lib.oracle_paged_mqa_logits.argtypes = [P, P, i32, i32, i32, P, i32, P, i32, P, P, P, P, i64]
        lib.oracle_paged_mqa_logits.restype = None
        lib.oracle_topk_rows.argtypes = [P, i64, i64, P, P, i32, P]
        lib.oracle_topk_rows.restype = None
        lib.oracle_gather_k.argtypes = [P, i32, P, i32, P, P, i32, P, P]
        lib.oracle_gather_k.restype = None
        lib.oracle_quant_vec128_f32.argtypes = [P, P, P]
        lib.oracle_quant_vec128_f32.restype = None
        lib.oracle_rope_quant_q.argtypes = [P, P, i64, i32, P, P, i32, P, P, P]
        lib.oracle_rope_quant_q.restype = None
        lib.oracle_kpool_compress.argtypes = [P, P, P, P, i64, i32, P, P]
        lib.oracle_kpool_compress.restype = None
        lib.oracle_kpool_insert.argtypes = [P, P, i64, i32, P, i64, i32]
        lib.oracle_kpool_insert.restype = i64
        _lib = lib
        return lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def num_threads() -> int:
    return int(_load().oracle_num_threads())


# ---------------------------------------------------------------- scalar rules

def bf16_to_float(bits: int) -> float:
    return float(_load().oracle_bf16_to_double(int(bits) & 0xFFFF))


def ue8m0_scale(block) -> int:
    """UE8M0 byte of one block of values (smallest e with amax <= 6*2^e, +127)."""
    x = _c(block, np.float64)
    return int(_load().oracle_ue8m0_scale(_ptr(x), x.size))


def e2m1_code(y: float) -> int:
    """E2M1 code (RNE, ties to even code, saturating, sign kept) of y."""
    return int(_load().oracle_e2m1_code(float(y)))


def e2m1_value(code: int) -> float:
    return float(_load().oracle_e2m1_value(int(code) & 0xF))


# ---------------------------------------------------------------- vector steps

def quant_vec128(x_bf16_bits):
    """One bf16 vector of 128 (as uint16 bits) -> (vals[64] u8, scales[4] u8)."""
    x = _c(x_bf16_bits, np.uint16).reshape(HEAD_DIM)
    v = np.zeros(VAL_BYTES, np.uint8)
    s = np.zeros(SCALE_BYTES, np.uint8)
    _load().oracle_quant_vec128(_ptr(x), _ptr(v), _ptr(s))
    return v, s


def dequant_vec128(vals, scales):
    v = _c(vals, np.uint8).reshape(VAL_BYTES)
    s = _c(scales, np.uint8).reshape(SCALE_BYTES)
    out = np.zeros(HEAD_DIM, np.float64)
    _load().oracle_dequant_vec128(_ptr(v), _ptr(s), _ptr(out))
    return out


def quant_insert(k_bf16_bits, slot_mapping, cache, page_size: int = 64):
    """Quantise rows of k ([N,128] bf16 bits, any row stride >= 128 is flattened
    to a copy) and scatter them into ``cache`` ([num_blocks, page bytes] u8) in
    place.  Returns the number of out-of-range slots (slot -1 is not counted)."""
    k = _c(k_bf16_bits, np.uint16)
    n = k.shape[0] if k.ndim == 2 else 0
    stride = k.shape[1] if k.ndim == 2 else HEAD_DIM
    slots = _c(slot_mapping, np.int64)
    assert cache.dtype == np.uint8 and cache.flags["C_CONTIGUOUS"]
    num_blocks = cache.shape[0]
    return int(_load().oracle_quant_insert(_ptr(k), n, stride, _ptr(slots), _ptr(cache),
                                           num_blocks, page_size))


def quant_q(q_bf16_bits):
    """[..., 128] bf16 bits -> (vals [rows, 64], scales [rows, 4]), rows = prod(...)."""
    q = _c(q_bf16_bits, np.uint16).reshape(-1, HEAD_DIM)
    rows = q.shape[0]
    v = np.zeros((rows, VAL_BYTES), np.uint8)
    s = np.zeros((rows, SCALE_BYTES), np.uint8)
    _load().oracle_quant_q(_ptr(q), rows, _ptr(v), _ptr(s))
    return v, s


def mqa_logits(q_vals, q_scales, H, k_vals, k_scales, weights, row_start, row_end, ld=None,
               fill=np.nan):
    """Prefill logits.  Returns (logits[T, ld], mag[T, ld]) in fp64; columns
    outside [row_start, row_end) hold ``fill``."""
    qv = _c(q_vals, np.uint8)
    qs = _c(q_scales, np.uint8)
    kv = _c(k_vals, np.uint8)
    ks = _c(k_scales, np.uint8)
    w = _c(weights, np.float32)
    rs = _c(row_start, np.int32)
    re = _c(row_end, np.int32)
    T = rs.shape[0]
    S = kv.shape[0] if kv.ndim == 2 else kv.size // VAL_BYTES
    ld = S if ld is None else ld
    logits = np.full((T, ld), fill, np.float64)
    mag = np.full((T, ld), fill, np.float64)
    _load().oracle_mqa_logits(_ptr(qv), _ptr(qs), T, int(H), _ptr(kv), _ptr(ks), S, _ptr(w),
                              _ptr(rs), _ptr(re), _ptr(logits), _ptr(mag), ld)
    return logits, mag


def paged_mqa_logits(q_vals, q_scales, B, next_n, H, cache, block_table, context_lens,
                     weights, ld, page_size=64, fill=np.nan):
    """Decode logits through the block table.  Returns (logits[B*next_n, ld],
    mag[B*next_n, ld]) in fp64; columns past each row's window hold ``fill``."""
    qv = _c(q_vals, np.uint8)
    qs = _c(q_scales, np.uint8)
    c = _c(cache, np.uint8)
    bt = _c(block_table, np.int32)
    cl = _c(context_lens, np.int32)
    w = _c(weights, np.float32)
    max_blocks = bt.shape[1]
    rows = B * next_n
    logits = np.full((rows, ld), fill, np.float64)
    mag = np.full((rows, ld), fill, np.float64)
    _load().oracle_paged_mqa_logits(_ptr(qv), _ptr(qs), int(B), int(next_n), int(H), _ptr(c),
                                    int(page_size), _ptr(bt), int(max_blocks), _ptr(cl), _ptr(w),
                                    _ptr(logits), _ptr(mag), int(ld))
    return logits, mag


def topk_rows(logits, row_start, row_end, k):
    """Top-k per row by (value desc, index asc); indices relative to row_start,
    -1 padded.  ``logits`` is fp64 [rows, ld]."""
    lg = _c(logits, np.float64)
    rs = _c(row_start, np.int32)
    re = _c(row_end, np.int32)
    rows, ld = lg.shape
    out = np.empty((rows, k), np.int32)
    _load().oracle_topk_rows(_ptr(lg), rows, ld, _ptr(rs), _ptr(re), int(k), _ptr(out))
    return out


def gather_k(cache, block_table, seq_lens, out_offsets, total_rows, page_size=64):
    """Copy each sequence's cached tokens into contiguous (vals[total,64], scales[total,4])."""
    c = _c(cache, np.uint8)
    bt = _c(block_table, np.int32)
    sl = _c(seq_lens, np.int32)
    oo = _c(out_offsets, np.int64)
    v = np.zeros((total_rows, VAL_BYTES), np.uint8)
    s = np.zeros((total_rows, SCALE_BYTES), np.uint8)
    _load().oracle_gather_k(_ptr(c), int(page_size), _ptr(bt), int(bt.shape[1]), _ptr(sl),
                            _ptr(oo), int(sl.shape[0]), _ptr(v), _ptr(s))
    return v, s


# ---------------------------------------------------------------- next steps

def quant_vec128_f32(x):
    """One fp32 vector of 128 -> (vals[64] u8, scales[4] u8), the same rules
    applied to the exact fp32 values."""
    xf = _c(x, np.float32).reshape(HEAD_DIM)
    v = np.zeros(VAL_BYTES, np.uint8)
    s = np.zeros(SCALE_BYTES, np.uint8)
    _load().oracle_quant_vec128_f32(_ptr(xf), _ptr(v), _ptr(s))
    return v, s


def rope_quant_q(q_bf16_bits, positions, cos, sin, rot_dim: int):
    """Rotary embedding of query heads then MXFP4 quantisation.
    q [T, H, 128] bf16 bits; positions [T] rows of the tables; cos, sin
    [num_pos, rot_dim / 2] fp32.  The first rot_dim dimensions rotate in pairs
    (2i, 2i+1) by table column i, in fp32 with the order stated in oracle.c.
    Returns (vals [T*H, 64], scales [T*H, 4], rotated fp32 [T*H, 128])."""
    q = _c(q_bf16_bits, np.uint16)
    T, H = q.shape[0], q.shape[1]
    pos = _c(positions, np.int32)
    cs = _c(cos, np.float32)
    sn = _c(sin, np.float32)
    assert rot_dim % 2 == 0 and 0 <= rot_dim <= HEAD_DIM
    assert cs.shape == sn.shape and (rot_dim == 0 or cs.shape[1] == rot_dim // 2)
    assert len(pos) == T and (T == 0 or (pos.min() >= 0 and pos.max() < max(cs.shape[0], 1)))
    v = np.zeros((T * H, VAL_BYTES), np.uint8)
    s = np.zeros((T * H, SCALE_BYTES), np.uint8)
    r = np.zeros((T * H, HEAD_DIM), np.float32)
    _load().oracle_rope_quant_q(_ptr(q), _ptr(pos), T, H, _ptr(cs), _ptr(sn), rot_dim, _ptr(v),
                                _ptr(s), _ptr(r))
    return v, s, r


def kpool_compress(k_bf16_bits, gate, ape, slot_mapping, pool: int):
    """The pooled key of every row that the K-pool insert writes, in fp64:
    kc[p, d] = sum_j softmax_j(gate[p-P+1+j, d] + ape[j, d]) * k[p-P+1+j, d]
    for rows p with slot >= 0 and p >= P - 1 (NaN elsewhere), and beside it the
    tolerance scale mag[p, d] = sum_j w_j |k[p-P+1+j, d]|."""
    k = _c(k_bf16_bits, np.uint16).reshape(-1, HEAD_DIM)
    n = k.shape[0]
    g = _c(gate, np.float32).reshape(n, HEAD_DIM)
    a = _c(ape, np.float32).reshape(pool, HEAD_DIM)
    sl = _c(slot_mapping, np.int64).reshape(n)
    kc = np.zeros((n, HEAD_DIM), np.float64)
    mag = np.zeros((n, HEAD_DIM), np.float64)
    _load().oracle_kpool_compress(_ptr(k), _ptr(g), _ptr(a), _ptr(sl), n, int(pool), _ptr(kc),
                                  _ptr(mag))
    return kc, mag


def kpool_insert(kc32, slot_mapping, pool: int, cache, page_size: int = 64):
    """The write step of the K-pool insert: every row p with slot >= 0 and
    p >= P - 1 (and n >= P) stores the MXFP4 encoding of its pooled fp32
    vector kc32[p] at its slot.  Returns the count of out-of-range slots."""
    kc = _c(kc32, np.float32).reshape(-1, HEAD_DIM)
    sl = _c(slot_mapping, np.int64).reshape(-1)
    assert cache.dtype == np.uint8 and cache.flags["C_CONTIGUOUS"]
    return int(_load().oracle_kpool_insert(_ptr(kc), _ptr(sl), len(sl), int(pool), _ptr(cache),
                                           cache.shape[0], page_size))
