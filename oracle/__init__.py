"""CPU oracle for the CSA/HCA hot path -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never calls it and
shares no code with it; ``oracle.c`` is written independently from the pages
(see its header for the citations and the row formats).

Every function takes and returns numpy arrays.  Stored inputs are passed in the
form the GPU path receives them: ``float64``/``float32`` arrays, ``uint16``
arrays holding bfloat16 bit patterns, or ``uint8`` arrays of mixed-precision
FP8 rows (last axis = bytes per row).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

F64, F32, BF16, FP8M = 0, 1, 2, 3
OK, BAD_INDEX, BAD_WINDOW, BAD_ARG = 0, 1, 2, 3


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (plain gcc, IEEE arithmetic, OpenMP)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(
            ["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-std=c11",
             "-Wall", "-Wno-unknown-pragmas", "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        _declare(_lib)
    return _lib


_vp, _i32, _i64, _dbl = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double


def _declare(L):
    L.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
    L.oracle_e4m3_decode.restype = _dbl
    L.oracle_e4m3_encode.argtypes = [ctypes.c_float]
    L.oracle_e4m3_encode.restype = ctypes.c_uint8
    L.oracle_f32_to_bf16.argtypes = [ctypes.c_float]
    L.oracle_f32_to_bf16.restype = ctypes.c_uint16
    L.oracle_fp8m_row_bytes.argtypes = [_i32]
    L.oracle_fp8m_row_bytes.restype = _i64
    L.oracle_row_bytes.argtypes = [_i32, _i32]
    L.oracle_row_bytes.restype = _i64
    L.oracle_read_row.argtypes = [_vp, _i32, _i32, _i64, _vp]
    L.oracle_read_row.restype = None
    L.oracle_pack_fp8_rows.argtypes = [_vp, _i64, _i32, _vp]
    L.oracle_pack_fp8_rows.restype = None
    L.oracle_store_rows.argtypes = [_vp, _i64, _i32, _i32, _vp]
    L.oracle_store_rows.restype = None
    L.oracle_rmsnorm.argtypes = [_vp, _i32, _dbl, _vp]
    L.oracle_rmsnorm.restype = None
    L.oracle_rope.argtypes = [_vp, _i32, _i32, _dbl, _dbl]
    L.oracle_rope.restype = None
    L.oracle_compress.argtypes = [_vp, _i32, _i64, _i32, _i64, _i32, _vp, _vp, _i32, _dbl, _dbl, _vp]
    L.oracle_compress.restype = _i32
    L.oracle_n_complete.argtypes = [_i64, _i32]
    L.oracle_n_complete.restype = _i64
    L.oracle_index_scores.argtypes = [_vp, _i32, _vp, _i32, _i32, _vp, _i32, _i64, _vp]
    L.oracle_index_scores.restype = None
    L.oracle_pack_idx_keys_fp8.argtypes = [_vp, _i64, _i32, _vp, _vp]
    L.oracle_pack_idx_keys_fp8.restype = None
    L.oracle_index_scores_fp8.argtypes = [_vp, _i32, _vp, _i32, _i32, _vp, _vp, _i64, _vp]
    L.oracle_index_scores_fp8.restype = None
    L.oracle_e2m1_decode.argtypes = [ctypes.c_uint8]
    L.oracle_e2m1_decode.restype = _dbl
    L.oracle_e2m1_encode.argtypes = [_dbl]
    L.oracle_e2m1_encode.restype = ctypes.c_uint8
    L.oracle_pack_idx_keys_fp4.argtypes = [_vp, _i64, _i32, _vp, _vp]
    L.oracle_pack_idx_keys_fp4.restype = None
    L.oracle_index_scores_fp4.argtypes = [_vp, _i32, _vp, _i32, _i32, _vp, _vp, _i64, _vp]
    L.oracle_index_scores_fp4.restype = None
    L.oracle_topk.argtypes = [_vp, _i64, _i32, _vp, _vp]
    L.oracle_topk.restype = _i64
    L.oracle_attend_rows.argtypes = [_vp, _i32, _i32, _i32, _i64, _vp, _i64, _vp, _dbl, _i32,
                                     _dbl, _dbl, _i32, _vp, _vp, _vp]
    L.oracle_attend_rows.restype = None
    L.oracle_attend_query.argtypes = [_vp, _i32, _i32, _i32, _i64, _i32, _vp, _i32, _i64, _vp,
                                      _i32, _vp, _i64, _i64, _i32, _vp, _dbl, _i32, _dbl, _dbl,
                                      _i32, _vp, _vp]
    L.oracle_attend_query.restype = _i32
    L.oracle_index_topk_batch.argtypes = [_i32, _vp, _i32, _vp, _i32, _i32, _vp, _i32, _i64, _vp,
                                          _vp, _i32, _i32, _vp, _vp]
    L.oracle_index_topk_batch.restype = _i32
    L.oracle_attend_batch.argtypes = [_i32, _vp, _i32, _i32, _i32, _vp, _vp, _i32, _vp, _i32, _i64,
                                      _vp, _i32, _vp, _vp, _i64, _i32, _vp, _dbl, _i32, _dbl,
                                      _dbl, _i32, _vp, _vp]
    L.oracle_attend_batch.restype = _i32


# --------------------------------------------------------------------------
# helpers
# --------------------------------------------------------------------------

def _ptr(a):
    return None if a is None else a.ctypes.data_as(_vp)


def fmt_of(a: np.ndarray) -> int:
    """Storage format of a stored-input array."""
    if a.dtype == np.float64:
        return F64
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:
        return BF16
    if a.dtype == np.uint8:
        return FP8M
    raise TypeError("unsupported stored dtype %s" % a.dtype)


def _c(a, dtype=None):
    if dtype is not None:
        a = np.asarray(a, dtype=dtype)
    return np.ascontiguousarray(a)


def row_bytes(fmt: int, D: int) -> int:
    return int(lib().oracle_row_bytes(fmt, D))


def fp8m_row_bytes(D: int) -> int:
    return int(lib().oracle_fp8m_row_bytes(D))


# --------------------------------------------------------------------------
# number formats
# --------------------------------------------------------------------------

def e4m3_decode(code: int) -> float:
    return float(lib().oracle_e4m3_decode(int(code)))


def e4m3_encode(x: float) -> int:
    return int(lib().oracle_e4m3_encode(float(x)))


def f32_to_bf16_bits(x: float) -> int:
    return int(lib().oracle_f32_to_bf16(float(x)))


def pack_fp8_rows(x: np.ndarray) -> np.ndarray:
    """float32 [..., D] -> uint8 [..., row_bytes] mixed-precision rows."""
    x = _c(x, np.float32)
    D = x.shape[-1]
    n = x.size // D
    out = np.zeros(x.shape[:-1] + (fp8m_row_bytes(D),), dtype=np.uint8)
    lib().oracle_pack_fp8_rows(_ptr(x), n, D, _ptr(out))
    return out


def store_rows(x: np.ndarray, fmt: int) -> np.ndarray:
    """float64 [..., D] -> rows stored in `fmt` (float32, bf16 bits or FP8 rows)."""
    x = _c(x, np.float64)
    D = x.shape[-1]
    n = x.size // D
    if fmt == F64:
        return x.copy()
    if fmt == F32:
        out = np.empty(x.shape, dtype=np.float32)
    elif fmt == BF16:
        out = np.empty(x.shape, dtype=np.uint16)
    else:
        out = np.zeros(x.shape[:-1] + (fp8m_row_bytes(D),), dtype=np.uint8)
    lib().oracle_store_rows(_ptr(x), n, D, fmt, _ptr(out))
    return out


def read_rows(a: np.ndarray, D: int) -> np.ndarray:
    """Stored rows -> float64 [n, D]."""
    a = _c(a)
    fmt = fmt_of(a)
    rb = row_bytes(fmt, D)
    n = a.nbytes // rb
    out = np.empty((n, D), dtype=np.float64)
    for r in range(n):
        lib().oracle_read_row(_ptr(a), fmt, D, r, out[r].ctypes.data_as(_vp))
    return out


# --------------------------------------------------------------------------
# the method
# --------------------------------------------------------------------------

def rmsnorm(x: np.ndarray, eps: float = 1e-6) -> np.ndarray:
    x = _c(x, np.float64)
    out = np.empty_like(x)
    lib().oracle_rmsnorm(_ptr(x), x.shape[-1], eps, _ptr(out))
    return out


def rope(x: np.ndarray, pos: float, rope_dims: int = 64, base: float = 10000.0) -> np.ndarray:
    out = _c(x, np.float64).copy()
    lib().oracle_rope(_ptr(out), out.shape[-1], rope_dims, base, float(pos))
    return out


def compress(kv: np.ndarray, pos0: int, m: int, w_z, bias, rope_dims=64, base=10000.0,
             eps=1e-6) -> np.ndarray:
    """kv stored [T, D] -> float64 [T//m, D] compressed, normed, roped entries."""
    kv = _c(kv)
    D = kv.shape[-1] if fmt_of(kv) != FP8M else None
    if D is None:
        raise TypeError("raw kv is not stored as FP8 rows")
    T = kv.shape[0]
    w_z = _c(w_z, np.float64)
    bias = _c(bias, np.float64)
    assert w_z.shape == (D,) and bias.shape == (m,)
    out = np.zeros((T // m, D), dtype=np.float64)
    st = lib().oracle_compress(_ptr(kv), fmt_of(kv), T, D, int(pos0), m, _ptr(w_z), _ptr(bias),
                               rope_dims, base, eps, _ptr(out))
    if st != OK:
        raise ValueError("oracle_compress: status %d" % st)
    return out


def n_complete(i: int, m: int) -> int:
    return int(lib().oracle_n_complete(int(i), m))


def index_scores(q: np.ndarray, w, keys: np.ndarray) -> np.ndarray:
    """q stored [HI, dI], w [HI], keys stored [n, dI] -> float64 scores [n]."""
    q = _c(q)
    keys = _c(keys)
    HI, dI = q.shape
    w = _c(w, np.float64)
    n = keys.shape[0]
    out = np.empty(n, dtype=np.float64)
    lib().oracle_index_scores(_ptr(q), fmt_of(q), _ptr(w), HI, dI, _ptr(keys), fmt_of(keys), n,
                              _ptr(out))
    return out


def pack_idx_keys_fp8(x: np.ndarray):
    """float32 keys [n, dI] -> (E4M3 codes uint8 [n, dI], float32 scales [n]),
    one scale per key row."""
    x = _c(x, np.float32)
    n, dI = x.shape
    codes = np.empty((n, dI), dtype=np.uint8)
    scales = np.empty(n, dtype=np.float32)
    lib().oracle_pack_idx_keys_fp8(_ptr(x), n, dI, _ptr(codes), _ptr(scales))
    return codes, scales


def index_scores_fp8(q: np.ndarray, w, codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """q stored [HI, dI] (its heads quantised to FP8 inside), w [HI], FP8 keys
    (codes [n, dI], scales [n]) -> float64 scores [n]."""
    q = _c(q)
    HI, dI = q.shape
    w = _c(w, np.float64)
    codes = _c(codes, np.uint8)
    scales = _c(scales, np.float32)
    n = codes.shape[0]
    out = np.empty(n, dtype=np.float64)
    lib().oracle_index_scores_fp8(_ptr(q), fmt_of(q), _ptr(w), HI, dI, _ptr(codes), _ptr(scales), n,
                                  _ptr(out))
    return out


def e2m1_decode(code: int) -> float:
    """E2M1 (FP4) code 0..15 -> value."""
    return float(lib().oracle_e2m1_decode(int(code)))


def e2m1_encode(x: float) -> int:
    """value -> E2M1 code (nearest, ties to the even code, saturating at 6)."""
    return int(lib().oracle_e2m1_encode(float(x)))


def pack_idx_keys_fp4(x: np.ndarray):
    """float32 keys [n, dI] (dI a multiple of 32) -> (E2M1 codes uint8
    [n, dI/2], two dims a byte, the even dim in the low nibble; scale bytes
    uint8 [n, dI/32], block scale 2^(byte - 127))."""
    x = _c(x, np.float32)
    n, dI = x.shape
    assert dI % 32 == 0
    codes = np.empty((n, dI // 2), dtype=np.uint8)
    scales = np.empty((n, dI // 32), dtype=np.uint8)
    lib().oracle_pack_idx_keys_fp4(_ptr(x), n, dI, _ptr(codes), _ptr(scales))
    return codes, scales


def decode_idx_keys_fp4(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """FP4 keys -> float64 values [n, dI] (the oracle's decoder, element by element)."""
    codes = _c(codes, np.uint8)
    scales = _c(scales, np.uint8)
    n, half = codes.shape
    out = np.empty((n, 2 * half), dtype=np.float64)
    for b in range(n):
        for d in range(2 * half):
            byte = int(codes[b, d // 2])
            c = (byte >> 4) if d & 1 else (byte & 15)
            out[b, d] = e2m1_decode(c) * 2.0 ** (int(scales[b, d // 32]) - 127)
    return out


def index_scores_fp4(q: np.ndarray, w, codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """q stored [HI, dI] (its heads quantised to E4M3 inside), w [HI], FP4 keys
    (codes [n, dI/2], scale bytes [n, dI/32]) -> float64 scores [n]."""
    q = _c(q)
    HI, dI = q.shape
    w = _c(w, np.float64)
    codes = _c(codes, np.uint8)
    scales = _c(scales, np.uint8)
    n = codes.shape[0]
    out = np.empty(n, dtype=np.float64)
    lib().oracle_index_scores_fp4(_ptr(q), fmt_of(q), _ptr(w), HI, dI, _ptr(codes), _ptr(scales), n,
                                  _ptr(out))
    return out


def topk(scores: np.ndarray, k: int):
    """-> (idx int32 [k] in rank order padded with -1, selected scores [k])."""
    s = _c(scores, np.float64)
    idx = np.empty(k, dtype=np.int32)
    sel = np.empty(k, dtype=np.float64)
    lib().oracle_topk(_ptr(s), s.shape[0], k, _ptr(idx), _ptr(sel))
    return idx, sel


def attend_rows(q: np.ndarray, i: int, rows: np.ndarray, sink, scale=None, rope_dims=64,
                base=10000.0, eps=1e-6, derotate=True, return_weights=False):
    """q stored [H, D]; rows float64 [J, D] -> (out [H, D], lse [H] (, weights [H, J]))."""
    q = _c(q)
    H, D = q.shape
    rows = _c(rows, np.float64).reshape(-1, D)
    J = rows.shape[0]
    sink = _c(np.broadcast_to(np.asarray(sink, dtype=np.float64), (H,)))
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    out = np.empty((H, D), dtype=np.float64)
    lse = np.empty(H, dtype=np.float64)
    wts = np.empty((H, J), dtype=np.float64) if return_weights else None
    lib().oracle_attend_rows(_ptr(q), fmt_of(q), H, D, int(i), _ptr(rows), J, _ptr(sink), scale,
                             rope_dims, base, eps, int(derotate), _ptr(out), _ptr(lse), _ptr(wts))
    return (out, lse, wts) if return_weights else (out, lse)


def attend_query(q, i, m, cache, D, idx, window, win_pos0, W, sink, scale=None, rope_dims=64,
                 base=10000.0, eps=1e-6, derotate=True):
    """One query: CSA when idx is given, HCA (all complete blocks) when idx is None."""
    q = _c(q)
    H = q.shape[0]
    cache = _c(cache)
    window = _c(window)
    kv_fmt = fmt_of(cache)
    assert fmt_of(window) == kv_fmt
    rb = row_bytes(kv_fmt, D)
    n_cap = cache.nbytes // rb
    n_win = window.nbytes // rb
    if idx is not None:
        idx = _c(idx, np.int32)
    k = 0 if idx is None else idx.shape[0]
    sink = _c(np.broadcast_to(np.asarray(sink, dtype=np.float64), (H,)))
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    out = np.empty((H, D), dtype=np.float64)
    lse = np.empty(H, dtype=np.float64)
    st = lib().oracle_attend_query(_ptr(q), fmt_of(q), H, D, int(i), m, _ptr(cache), kv_fmt, n_cap,
                                   _ptr(idx), k, _ptr(window), int(win_pos0), n_win, W, _ptr(sink),
                                   scale, rope_dims, base, eps, int(derotate), _ptr(out), _ptr(lse))
    if st != OK:
        raise ValueError("oracle_attend_query: status %d" % st)
    return out, lse


def index_topk_batch(q, w, keys, seq, pos, m, k):
    """q stored [Q, HI, dI]; w [Q, HI]; keys stored [B, n_cap, dI]; seq/pos [Q]."""
    q = _c(q)
    keys = _c(keys)
    Q, HI, dI = q.shape
    n_cap = keys.shape[1]
    w = _c(w, np.float64)
    seq = _c(seq, np.int32)
    pos = _c(pos, np.int64)
    idx = np.empty((Q, k), dtype=np.int32)
    sc = np.empty((Q, k), dtype=np.float64)
    st = lib().oracle_index_topk_batch(Q, _ptr(q), fmt_of(q), _ptr(w), HI, dI, _ptr(keys),
                                       fmt_of(keys), n_cap, _ptr(seq), _ptr(pos), m, k, _ptr(idx),
                                       _ptr(sc))
    if st != OK:
        raise ValueError("oracle_index_topk_batch: status %d" % st)
    return idx, sc


def attend_batch(q, seq, pos, m, cache, D, idx, window, win_pos0, W, sink, scale=None,
                 rope_dims=64, base=10000.0, eps=1e-6, derotate=True):
    """q stored [Q, H, D]; cache stored [B, n_cap, ...]; window stored [B, n_win, ...]."""
    q = _c(q)
    Q, H = q.shape[0], q.shape[1]
    cache = _c(cache)
    window = _c(window)
    kv_fmt = fmt_of(cache)
    B = cache.shape[0]
    rb = row_bytes(kv_fmt, D)
    n_cap = cache.nbytes // (rb * B)
    n_win = window.nbytes // (rb * B)
    seq = _c(seq, np.int32)
    pos = _c(pos, np.int64)
    win_pos0 = _c(np.broadcast_to(np.asarray(win_pos0, dtype=np.int64), (B,)))
    if idx is not None:
        idx = _c(idx, np.int32)
    k = 0 if idx is None else idx.shape[1]
    sink = _c(np.broadcast_to(np.asarray(sink, dtype=np.float64), (H,)))
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    out = np.empty((Q, H, D), dtype=np.float64)
    lse = np.empty((Q, H), dtype=np.float64)
    st = lib().oracle_attend_batch(Q, _ptr(q), fmt_of(q), H, D, _ptr(seq), _ptr(pos), m,
                                   _ptr(cache), kv_fmt, n_cap, _ptr(idx), k, _ptr(window),
                                   _ptr(win_pos0), n_win, W, _ptr(sink), scale, rope_dims, base,
                                   eps, int(derotate), _ptr(out), _ptr(lse))
    if st != OK:
        raise ValueError("oracle_attend_batch: status %d" % st)
    return out, lse


# --------------------------------------------------------------------------
# grouped output projection
# --------------------------------------------------------------------------
def grouped_out_proj(o: np.ndarray, w: np.ndarray, G: int) -> np.ndarray:
    """Grouped output projection ["DeepSeek-V4百万上下文时代的开源宣言" §三.2 CSA
    "Step 4: Grouped Output Projection" (the 512-dim heads are projected in
    groups, which cuts the cost)]: the H heads form G consecutive groups of
    H/G; group g's concatenated head outputs x_g (H/G * D values) are
    projected by its own matrix, out[:, g*d_g:(g+1)*d_g] = x_g . W_g^T.
    o: stored attention outputs [Q, H, D]; w: stored weights [G, d_g, H/G*D]
    (row n of W_g is output n's weights).  Returns float64 [Q, G*d_g]."""
    x = read_act(o)
    Q, H, D = x.shape
    assert H % G == 0
    wt = read_act(w)
    Gw, d_g, K = wt.shape
    assert Gw == G and K == H // G * D
    xg = x.reshape(Q, G, K)
    out = np.empty((Q, G * d_g), dtype=np.float64)
    for g in range(G):
        out[:, g * d_g:(g + 1) * d_g] = xg[:, g, :] @ wt[g].T
    return out


def read_act(a: np.ndarray) -> np.ndarray:
    """Stored activations (bf16 bits as uint16, float32 or float64) -> float64."""
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)
