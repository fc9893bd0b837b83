"""Python binding of libcsa: the DeepSeek-V4 CSA/HCA attention hot path on B300.

Every function has the name and argument order of its C counterpart in
``include/csa.h`` and does argument marshalling only: torch tensors become
device pointers, the stream defaults to torch's current stream, and a non-OK
status raises :class:`CsaError`.  All computation happens in the CUDA kernels
of ``libcsa.so``; there is no fallback of any kind -- importing works without a
GPU, but every call needs the built library and a CUDA device.
"""
from __future__ import annotations

import ctypes
import os

import torch

__all__ = [
    "CsaError", "CsaParams", "F32", "BF16", "FP8_MIXED", "OP_INDEX_TOPK", "OP_INDEX_TOPK_FP8", "OP_INDEX_TOPK_FP4", "OP_ATTEND",
    "OP_HCA_ATTEND", "params", "lib", "csa_row_bytes", "csa_cache_pack", "csa_compress", "csa_append", "csa_decode_append", "csa_index_keys_pack", "csa_index_score_fp8", "csa_index_topk_fp8",
    "csa_index_keys_fp4_bytes", "csa_index_keys_pack_fp4", "csa_index_score_fp4", "csa_index_topk_fp4",
    "csa_index_topk", "csa_index_score", "csa_topk_select", "csa_launch_count", "csa_test_withhold_indexer_loads", "csa_index_topk_noalloc", "csa_attend", "hca_attend", "csa_grouped_out_proj", "csa_grouped_out_proj_ws_bytes", "csa_workspace_bytes", "csa_workspace_init",
    "csa_check_status", "csa_last_device_bits", "csa_status_string", "csa_last_error",
    "workspace", "LIB_PATH",
]

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libcsa.so")

F32, BF16, FP8_MIXED = 0, 1, 2
OP_INDEX_TOPK, OP_ATTEND, OP_HCA_ATTEND, OP_INDEX_TOPK_FP8, OP_INDEX_TOPK_FP4 = 1, 2, 3, 4, 5
_FMT = {"f32": F32, "bf16": BF16, "fp8m": FP8_MIXED}


class CsaError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str):
        self.status = status
        super().__init__("%s: %s: %s" % (where, detail, _status_name(status)))


class CsaParams(ctypes.Structure):
    _fields_ = [
        ("head_dim", ctypes.c_int32),
        ("rope_dims", ctypes.c_int32),
        ("rope_base", ctypes.c_float),
        ("norm_eps", ctypes.c_float),
        ("softmax_scale", ctypes.c_float),
        ("ratio", ctypes.c_int32),
        ("topk", ctypes.c_int32),
        ("window", ctypes.c_int32),
        ("derotate_output", ctypes.c_int32),
        ("act_format", ctypes.c_int32),
        ("kv_format", ctypes.c_int32),
        ("batch_invariant", ctypes.c_int32),
    ]


def params(head_dim: int, ratio: int, topk: int = 0, window: int = 128, act="bf16", kv="bf16",
           rope_dims: int = 64, rope_base: float = 10000.0, norm_eps: float = 1e-6,
           softmax_scale: float = 0.0, derotate_output: bool = True,
           batch_invariant: bool = False) -> CsaParams:
    return CsaParams(head_dim, rope_dims, rope_base, norm_eps, softmax_scale, ratio, topk, window,
                     int(bool(derotate_output)), _FMT.get(act, act), _FMT.get(kv, kv),
                     int(bool(batch_invariant)))


_lib = None
_vp, _i32, _i64, _sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t


def lib() -> ctypes.CDLL:
    """The loaded libcsa.so; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError("libcsa.so is not built (python -m long_context_compressed_17_b300.build)")
        L = ctypes.CDLL(LIB_PATH)
        P = ctypes.POINTER(CsaParams)
        sigs = {
            "csa_row_bytes": (_i64, [_i32, _i32]),
            "csa_cache_pack": (_i32, [P, _vp, _i64, _vp, _vp]),
            "csa_compress": (_i32, [P, _vp, _i32, _i64, _i64, _i64, _vp, _vp, _vp, _i64, _vp]),
            "csa_append": (_i32, [P, _vp, _i32, _i64, _i64, _vp, _vp, _vp, _i64, _vp, _i64, _vp]),
            "csa_decode_append": (_i32, [P, _vp, _i32, _vp, _vp, _vp, _vp, _vp, _i64, _vp, _i64, _vp, _sz,
                                         _vp]),
            "csa_index_keys_pack": (_i32, [P, _vp, _i64, _i32, _vp, _vp, _vp]),
            "csa_index_score_fp8": (_i32, [P, _vp, _vp, _i32, _i32, _vp, _vp, _i64, _i32, _i32, _vp,
                                           _vp, _i64, _vp, _sz, _vp]),
            "csa_index_topk_fp8": (_i32, [P, _vp, _vp, _i32, _i32, _vp, _vp, _i64, _i32, _i32, _vp,
                                          _vp, _vp, _vp, _sz, _vp]),
            "csa_index_keys_fp4_bytes": (_i64, [_i64]),
            "csa_index_keys_pack_fp4": (_i32, [P, _vp, _i32, _i64, _i32, _vp, _vp]),
            "csa_index_score_fp4": (_i32, [P, _vp, _vp, _i32, _i32, _vp, _i64, _i32, _i32, _vp, _vp, _i64, _vp,
                                           _sz, _vp]),
            "csa_index_topk_fp4": (_i32, [P, _vp, _vp, _i32, _i32, _vp, _i64, _i32, _i32, _vp, _vp, _vp, _vp,
                                          _sz, _vp]),
            "csa_index_topk": (_i32, [P, _vp, _vp, _i32, _i32, _vp, _i64, _i32, _i32, _vp, _vp,
                                      _vp, _vp, _sz, _vp]),
            "csa_attend": (_i32, [P, _vp, _i32, _i32, _i32, _vp, _vp, _i64, _vp, _vp, _i64, _vp,
                                  _vp, _vp, _vp, _vp, _sz, _vp]),
            "hca_attend": (_i32, [P, _vp, _i32, _i32, _i32, _vp, _vp, _i64, _vp, _i64, _vp, _vp,
                                  _vp, _vp, _vp, _sz, _vp]),
            "csa_index_score": (_i32, [P, _vp, _vp, _i32, _i32, _vp, _i64, _i32, _i32, _vp, _vp,
                                       _i64, _vp, _sz, _vp]),
            "csa_topk_select": (_i32, [P, _vp, _i64, _i64, _i32, _vp, _vp, _vp, _vp]),
            "csa_launch_count": (ctypes.c_uint64, []),
            "csa_test_withhold_indexer_loads": (_i32, [_i32]),
            "csa_index_topk_noalloc": (_i32, [P, _vp, _vp, _i32, _i32, _vp, _i64, _i32, _i32, _vp,
                                              _vp, _vp, _vp, _vp]),
            "csa_grouped_out_proj": (_i32, [_vp, _i32, _i32, _i32, _i32, _vp, _i32, _vp, _vp, _sz, _vp]),
            "csa_grouped_out_proj_ws_bytes": (_sz, [_i32, _i32, _i32]),
            "csa_workspace_bytes": (_sz, [P, _i32, _i32, _i32, _i32, _i32, _i64, _i64]),
            "csa_workspace_init": (_i32, [_vp, _sz, _vp]),
            "csa_check_status": (_i32, [_vp, _vp]),
            "csa_last_device_bits": (ctypes.c_uint32, []),
            "csa_status_string": (ctypes.c_char_p, [_i32]),
            "csa_last_error": (ctypes.c_char_p, []),
        }
        for name, (res, args) in sigs.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _status_name(s: int) -> str:
    try:
        return lib().csa_status_string(s).decode()
    except Exception:  # pragma: no cover
        return str(s)


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return ctypes.c_void_p(t)
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        if not torch.cuda.is_available():
            return ctypes.c_void_p(0)  # the call fails in the library, not here
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _check(status: int, where: str):
    if status != 0:
        raise CsaError(status, where, lib().csa_last_error().decode())


# ----------------------------------------------------------------------- ABI
def csa_row_bytes(kv_format: int, head_dim: int) -> int:
    return int(lib().csa_row_bytes(_FMT.get(kv_format, kv_format), head_dim))


def csa_cache_pack(p, src, n_rows, dst, stream=None):
    _check(lib().csa_cache_pack(ctypes.byref(p), _ptr(src), n_rows, _ptr(dst), _stream(stream)),
           "csa_cache_pack")


def csa_append(p, kv_new, B, kv_seq_stride, pos0, w_z, bias, entry_out, out_seq_stride, win_out,
               win_seq_stride, stream=None):
    _check(lib().csa_append(ctypes.byref(p), _ptr(kv_new), B, kv_seq_stride, pos0, _ptr(w_z),
                            _ptr(bias), _ptr(entry_out), out_seq_stride, _ptr(win_out),
                            win_seq_stride, _stream(stream)), "csa_append")


def csa_decode_append(p, kv_tok, B, pos, raw_ring, w_z, bias, cache, n_cap, window, n_win, ws, ws_bytes,
                      stream=None):
    _check(lib().csa_decode_append(ctypes.byref(p), _ptr(kv_tok), B, _ptr(pos), _ptr(raw_ring), _ptr(w_z),
                                   _ptr(bias), _ptr(cache), n_cap, _ptr(window), n_win, _ptr(ws), ws_bytes,
                                   _stream(stream)), "csa_decode_append")


def csa_compress(p, kv_raw, B, T, kv_seq_stride, pos0, w_z, bias, out, out_seq_stride,
                 stream=None):
    _check(lib().csa_compress(ctypes.byref(p), _ptr(kv_raw), B, T, kv_seq_stride, pos0,
                              _ptr(w_z), _ptr(bias), _ptr(out), out_seq_stride, _stream(stream)),
           "csa_compress")


def csa_index_topk(p, q_idx, w_idx, n_idx_heads, idx_dim, keys, n_cap, B, Q, q_pos, topk_idx,
                   topk_score, ws, ws_bytes, stream=None):
    _check(lib().csa_index_topk(ctypes.byref(p), _ptr(q_idx), _ptr(w_idx), n_idx_heads, idx_dim,
                                _ptr(keys), n_cap, B, Q, _ptr(q_pos), _ptr(topk_idx),
                                _ptr(topk_score), _ptr(ws), ws_bytes, _stream(stream)),
           "csa_index_topk")


def csa_index_keys_pack(p, keys, n_rows, idx_dim, codes, scales, stream=None):
    _check(lib().csa_index_keys_pack(ctypes.byref(p), _ptr(keys), n_rows, idx_dim, _ptr(codes),
                                     _ptr(scales), _stream(stream)), "csa_index_keys_pack")


def csa_index_score_fp8(p, q_idx, w_idx, n_idx_heads, idx_dim, key_codes, key_scales, n_cap, B, Q,
                        q_pos, scores, ld_scores, ws, ws_bytes, stream=None):
    _check(lib().csa_index_score_fp8(ctypes.byref(p), _ptr(q_idx), _ptr(w_idx), n_idx_heads,
                                     idx_dim, _ptr(key_codes), _ptr(key_scales), n_cap, B, Q,
                                     _ptr(q_pos), _ptr(scores), ld_scores, _ptr(ws), ws_bytes,
                                     _stream(stream)), "csa_index_score_fp8")


def csa_index_topk_fp8(p, q_idx, w_idx, n_idx_heads, idx_dim, key_codes, key_scales, n_cap, B, Q,
                       q_pos, topk_idx, topk_score, ws, ws_bytes, stream=None):
    _check(lib().csa_index_topk_fp8(ctypes.byref(p), _ptr(q_idx), _ptr(w_idx), n_idx_heads, idx_dim,
                                    _ptr(key_codes), _ptr(key_scales), n_cap, B, Q, _ptr(q_pos),
                                    _ptr(topk_idx), _ptr(topk_score), _ptr(ws), ws_bytes,
                                    _stream(stream)), "csa_index_topk_fp8")


def csa_index_keys_fp4_bytes(n_cap: int) -> int:
    return int(lib().csa_index_keys_fp4_bytes(n_cap))


def csa_index_keys_pack_fp4(p, keys, B, n_cap, idx_dim, pack, stream=None):
    _check(lib().csa_index_keys_pack_fp4(ctypes.byref(p), _ptr(keys), B, n_cap, idx_dim, _ptr(pack),
                                         _stream(stream)), "csa_index_keys_pack_fp4")


def csa_index_score_fp4(p, q_idx, w_idx, n_idx_heads, idx_dim, key_pack, n_cap, B, Q, q_pos, scores, ld_scores,
                        ws, ws_bytes, stream=None):
    _check(lib().csa_index_score_fp4(ctypes.byref(p), _ptr(q_idx), _ptr(w_idx), n_idx_heads, idx_dim,
                                     _ptr(key_pack), n_cap, B, Q, _ptr(q_pos), _ptr(scores), ld_scores, _ptr(ws),
                                     ws_bytes, _stream(stream)), "csa_index_score_fp4")


def csa_index_topk_fp4(p, q_idx, w_idx, n_idx_heads, idx_dim, key_pack, n_cap, B, Q, q_pos, topk_idx, topk_score,
                       ws, ws_bytes, stream=None):
    _check(lib().csa_index_topk_fp4(ctypes.byref(p), _ptr(q_idx), _ptr(w_idx), n_idx_heads, idx_dim,
                                    _ptr(key_pack), n_cap, B, Q, _ptr(q_pos), _ptr(topk_idx), _ptr(topk_score),
                                    _ptr(ws), ws_bytes, _stream(stream)), "csa_index_topk_fp4")


def csa_index_score(p, q_idx, w_idx, n_idx_heads, idx_dim, keys, n_cap, B, Q, q_pos, scores,
                    ld_scores, ws, ws_bytes, stream=None):
    _check(lib().csa_index_score(ctypes.byref(p), _ptr(q_idx), _ptr(w_idx), n_idx_heads, idx_dim,
                                 _ptr(keys), n_cap, B, Q, _ptr(q_pos), _ptr(scores), ld_scores,
                                 _ptr(ws), ws_bytes, _stream(stream)),
           "csa_index_score")


def csa_topk_select(p, scores, ld_scores, n_cap, Q, q_pos, topk_idx, topk_score, stream=None):
    _check(lib().csa_topk_select(ctypes.byref(p), _ptr(scores), ld_scores, n_cap, Q, _ptr(q_pos),
                                 _ptr(topk_idx), _ptr(topk_score), _stream(stream)),
           "csa_topk_select")


def csa_index_topk_noalloc(p, q_idx, w_idx, n_idx_heads, idx_dim, keys, n_cap, B, Q, q_pos,
                           topk_idx, topk_score, status, stream=None):
    """csa_index_topk without a workspace, for callers that cannot allocate
    device memory (its scores live in a fixed scratch array inside the library;
    see include/csa.h for the size limit and the ordering rule)."""
    _check(lib().csa_index_topk_noalloc(ctypes.byref(p), _ptr(q_idx), _ptr(w_idx), n_idx_heads,
                                        idx_dim, _ptr(keys), n_cap, B, Q, _ptr(q_pos),
                                        _ptr(topk_idx), _ptr(topk_score), _ptr(status),
                                        _stream(stream)),
           "csa_index_topk_noalloc")


def csa_launch_count() -> int:
    return int(lib().csa_launch_count())


def csa_test_withhold_indexer_loads(on: bool):
    _check(lib().csa_test_withhold_indexer_loads(int(bool(on))), "csa_test_withhold_indexer_loads")


def csa_attend(p, q, H, B, Q, q_pos, cache, n_cap, topk_idx, window, n_win, win_pos0, sink, out,
               lse, ws, ws_bytes, stream=None):
    _check(lib().csa_attend(ctypes.byref(p), _ptr(q), H, B, Q, _ptr(q_pos), _ptr(cache), n_cap,
                            _ptr(topk_idx), _ptr(window), n_win, _ptr(win_pos0), _ptr(sink),
                            _ptr(out), _ptr(lse), _ptr(ws), ws_bytes, _stream(stream)),
           "csa_attend")


def hca_attend(p, q, H, B, Q, q_pos, cache, n_cap, window, n_win, win_pos0, sink, out, lse, ws,
               ws_bytes, stream=None):
    _check(lib().hca_attend(ctypes.byref(p), _ptr(q), H, B, Q, _ptr(q_pos), _ptr(cache), n_cap,
                            _ptr(window), n_win, _ptr(win_pos0), _ptr(sink), _ptr(out), _ptr(lse),
                            _ptr(ws), ws_bytes, _stream(stream)),
           "hca_attend")


def csa_grouped_out_proj_ws_bytes(Q, G, d_g):
    return lib().csa_grouped_out_proj_ws_bytes(Q, G, d_g)


def csa_grouped_out_proj(o, Q, H, D, G, w, d_g, out, ws, ws_bytes, stream=None):
    _check(lib().csa_grouped_out_proj(_ptr(o), Q, H, D, G, _ptr(w), d_g, _ptr(out), _ptr(ws), ws_bytes,
                                      _stream(stream)), "csa_grouped_out_proj")


def csa_workspace_bytes(p, op, B, Q, H, n_idx_heads, n_cap, n_win) -> int:
    return int(lib().csa_workspace_bytes(ctypes.byref(p), op, B, Q, H, n_idx_heads, n_cap, n_win))


def csa_workspace_init(ws, ws_bytes, stream=None):
    _check(lib().csa_workspace_init(_ptr(ws), ws_bytes, _stream(stream)), "csa_workspace_init")


def csa_check_status(ws, stream=None):
    _check(lib().csa_check_status(_ptr(ws), _stream(stream)), "csa_check_status")


def csa_last_device_bits() -> int:
    return int(lib().csa_last_device_bits())


def csa_status_string(s: int) -> str:
    return lib().csa_status_string(s).decode()


def csa_last_error() -> str:
    return lib().csa_last_error().decode()


# ------------------------------------------------------------------ plumbing
def workspace(nbytes: int, device="cuda", stream=None) -> torch.Tensor:
    """A device buffer of `nbytes` (at least 256) with its status word zeroed."""
    ws = torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)
    csa_workspace_init(ws, ws.numel(), stream)
    return ws
