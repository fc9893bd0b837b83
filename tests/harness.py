"""Run one workload through the CUDA library and through the oracle, and compare.

Test infrastructure: imported by the tests, by ``__graft_entry__.smoke()`` and
by the CPU-baseline leg of ``bench.py``.  The GPU side goes through the public
binding only; the oracle side sees the identical stored input bits.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import workloads
from workloads import Workload

# Tolerances fixed for this hot path: bf16 inputs with fp32 accumulation
# compare within max-abs 2e-2 and mean-abs 2e-3; the fp32 workload within
# 1e-4; top-k sets are exact except between blocks whose oracle scores are
# within 1e-6 (relative) of the selection threshold.
TOL = {"bf16": (2e-2, 2e-3), "f32": (1e-4, 1e-4)}
LSE_TOL = {"bf16": 2e-2, "f32": 1e-4}
NEAR_TIE_REL = 1e-6

_ORC_FMT = {"f32": oracle.F32, "bf16": oracle.BF16, "fp8m": oracle.FP8M}


def cfg_of(w: Workload):
    from long_context_compressed_17_b300.pipeline import LayerConfig
    return LayerConfig(D=w.D, H=w.H, m=w.m, W=w.W, topk=w.topk if w.kind != "hca_decode" else 0,
                       H_I=w.H_I, d_I=w.d_I, act=w.act, kv=w.kv_fmt, rope_base=w.rope_base,
                       eps=w.eps)


# ------------------------------------------------------------------ GPU side
def gpu_pack(w: Workload, x: torch.Tensor) -> torch.Tensor:
    """Stored rows on the device (FP8 rows packed by the library)."""
    import long_context_compressed_17_b300 as L
    if w.kv_fmt != "fp8m":
        return x.clone()
    cfg = cfg_of(w)
    out = cfg.empty_rows(*x.shape[:-1], device=x.device)
    L.csa_cache_pack(cfg.params(), x.contiguous(), x.numel() // w.D, out)
    return out


def gpu_decode(w: Workload, inp: dict, append: bool = True) -> dict:
    """Decode step on the GPU for every sequence of the workload."""
    import long_context_compressed_17_b300 as L
    from long_context_compressed_17_b300.pipeline import DecodeLayer
    cfg = cfg_of(w)
    cache = gpu_pack(w, inp["cache"])
    window = gpu_pack(w, inp["window"])
    layer = DecodeLayer(cfg, w.B, w.n_cap, w.W, device=cache.device)
    if append:
        lens = w.lengths
        rb = cfg.row_bytes
        p, p1 = cfg.params(), cfg.params(ratio=1)
        act_rb = inp["kv_new"].element_size() * w.D
        for b, Lb in enumerate(lens):
            kv_b = inp["kv_new"][b]
            if Lb % w.m == 0 and Lb >= w.m:
                L.csa_compress(p, kv_b, 1, w.m, w.m, Lb - w.m, inp["w_z"], inp["bias"],
                               cache.data_ptr() + (b * w.n_cap + Lb // w.m - 1) * rb, w.n_cap)
            wr = (Lb - 1) - int(inp["win_pos0"][b])
            L.csa_compress(p1, kv_b.data_ptr() + (w.m - 1) * act_rb, 1, 1, 1, Lb - 1, inp["w_z"],
                           inp["bias"], window.data_ptr() + (b * w.W + wr) * rb, w.W)
    kw = {}
    if w.kind == "csa_decode":
        kw = dict(q_idx=inp["q_idx"], w_idx=inp["w_idx"], keys=inp["keys"])
    out, lse = layer.attend(inp["q"], cache, window, inp["q_pos"], inp["win_pos0"], inp["sink"],
                            **kw)
    torch.cuda.synchronize()
    L.csa_check_status(layer.ws)
    res = dict(out=out, lse=lse, cache=cache, window=window, layer=layer)
    if w.kind == "csa_decode":
        res.update(topk_idx=layer.topk_idx, topk_score=layer.topk_score)
    return res


def gpu_prefill(w: Workload, inp: dict) -> dict:
    import long_context_compressed_17_b300 as L
    from long_context_compressed_17_b300.pipeline import PrefillLayer
    cfg = cfg_of(w)
    layer = PrefillLayer(cfg, w.T_cached, w.T_new, device=inp["q"].device)
    if w.T_cached:
        layer.load_cached_rows(gpu_pack(w, inp["cache_old"]))
    layer.compress(inp["kv_raw"], inp["w_z"], inp["bias"])
    out, lse = layer.attend(inp["q"], inp["q_idx"], inp["w_idx"], inp["keys"], inp["q_pos"],
                            inp["sink"])
    torch.cuda.synchronize()
    L.csa_check_status(layer.ws)
    return dict(out=out, lse=lse, cache=layer.cache, window=layer.window,
                topk_idx=layer.topk_idx, topk_score=layer.topk_score, layer=layer)


# --------------------------------------------------------------- oracle side
def np_stored(t):
    return workloads.to_numpy_stored(t)


def oracle_stored_rows(w: Workload, x: torch.Tensor) -> np.ndarray:
    """Rows in the stored format, quantised by the oracle for FP8."""
    a = np_stored(x)
    if w.kv_fmt == "fp8m":
        return oracle.pack_fp8_rows(a.astype(np.float32))
    return a


def oracle_decode_state(w: Workload, inp: dict, seqs, append=True):
    """Per-sequence stored cache/window after the oracle's own append step."""
    fmt = _ORC_FMT[w.kv_fmt]
    w_z = np_stored(inp["w_z"]).astype(np.float64)
    bias = np_stored(inp["bias"]).astype(np.float64)
    state = {}
    for b in seqs:
        Lb = w.lengths[b]
        cache = oracle_stored_rows(w, inp["cache"][b])
        window = oracle_stored_rows(w, inp["window"][b])
        if append:
            kv_b = np_stored(inp["kv_new"][b])
            if Lb % w.m == 0 and Lb >= w.m:
                e = oracle.compress(kv_b, Lb - w.m, w.m, w_z, bias, w.rope_dims, w.rope_base, w.eps)
                cache[Lb // w.m - 1] = oracle.store_rows(e, fmt)[0]
            wr = (Lb - 1) - int(inp["win_pos0"][b])
            r = oracle.compress(kv_b[w.m - 1:], Lb - 1, 1, w_z, bias[:1], w.rope_dims,
                                w.rope_base, w.eps)
            window[wr] = oracle.store_rows(r, fmt)[0]
        state[b] = (cache, window)
    return state


def oracle_prefill_state(w: Workload, inp: dict):
    fmt = _ORC_FMT[w.kv_fmt]
    w_z = np_stored(inp["w_z"]).astype(np.float64)
    bias = np_stored(inp["bias"]).astype(np.float64)
    kv_raw = np_stored(inp["kv_raw"])
    raw_pos0 = inp["raw_pos0"]
    off = w.T_cached - raw_pos0
    new = oracle.compress(kv_raw[off:], w.T_cached, w.m, w_z, bias, w.rope_dims, w.rope_base, w.eps)
    rows = [oracle_stored_rows(w, inp["cache_old"])] if w.T_cached else []
    rows.append(oracle.store_rows(new, fmt))
    cache = np.concatenate(rows, axis=0)
    win = oracle.compress(kv_raw, raw_pos0, 1, w_z, bias[:1], w.rope_dims, w.rope_base, w.eps)
    window = oracle.store_rows(win, fmt)
    return cache, window


# ----------------------------------------------------------------- compare
def max_mean_abs(a, b):
    d = np.abs(np.asarray(a, np.float64) - np.asarray(b, np.float64))
    return float(d.max()) if d.size else 0.0, float(d.mean()) if d.size else 0.0


def assert_close(got, ref, act, what):
    mx, mn = max_mean_abs(got, ref)
    tmax, tmean = TOL[act]
    assert mx <= tmax and mn <= tmean, "%s: max-abs %.3g (tol %g), mean-abs %.3g (tol %g)" % (
        what, mx, tmax, mn, tmean)
    return mx, mn


def check_topk_set(gpu_idx, orc_scores, k, what=""):
    """GPU set vs the exact top-k of the oracle's scores (lower index on ties).
    Blocks may differ only where both scores lie within NEAR_TIE_REL of the
    k-th largest oracle score.  Returns True when the sets are identical."""
    n = orc_scores.shape[0]
    kk = min(k, n)
    g = np.asarray(gpu_idx)
    assert np.all(g[kk:] == -1), "%s: padding after %d selected" % (what, kk)
    gs = g[:kk]
    assert np.all((gs >= 0) & (gs < n)), "%s: index out of range" % what
    assert len(set(gs.tolist())) == kk, "%s: duplicate indices" % what
    assert np.all(np.diff(gs) > 0), "%s: not in ascending index order" % what
    ref_idx, _ = oracle.topk(orc_scores, k)
    rs = set(ref_idx[:kk].tolist())
    diff = rs.symmetric_difference(gs.tolist())
    if not diff:
        return True
    thr = np.sort(orc_scores)[::-1][kk - 1]
    band = NEAR_TIE_REL * max(abs(thr), 1e-30)
    bad = [b for b in diff if abs(orc_scores[b] - thr) > band]
    assert not bad, "%s: %d blocks differ beyond near-ties, e.g. %s (thr %.9g)" % (
        what, len(bad), [(b, orc_scores[b]) for b in bad[:4]], thr)
    return False
