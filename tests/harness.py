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
                       eps=w.eps, scale=w.softmax_scale)


def _scale(w: Workload):
    return w.softmax_scale if w.softmax_scale > 0 else None


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
    """Decode step on the GPU for every sequence of the workload, through the
    decode layer: the state (raw ring, cache, window ring) is laid out from the
    seeded inputs, csa_decode_append adds every sequence's newest token (its
    window row, and its block's entry where it completes one), then the
    indexer / top-k and the attention run with the ring window."""
    from long_context_compressed_17_b300.pipeline import DecodeLayer, ring_order
    import long_context_compressed_17_b300 as L
    cfg = cfg_of(w)
    cache = gpu_pack(w, inp["cache"])
    lens = torch.tensor(w.lengths, dtype=torch.int64)
    window = ring_order(gpu_pack(w, inp["window"]), inp["win_pos0"].cpu(), w.W)
    # the newest block's raw tokens (positions L-m .. L-1) in their ring slots
    raw_ring = ring_order(inp["kv_new"], (lens - w.m).tolist(), w.m)
    layer = DecodeLayer(cfg, w.B, w.n_cap, w.W, device=cache.device)
    if append:
        kv_tok = inp["kv_new"][:, w.m - 1].contiguous()
        layer.append(kv_tok, inp["q_pos"], inp["w_z"], inp["bias"], raw_ring, cache, window)
    kw = {}
    if w.kind == "csa_decode":
        kw = dict(q_idx=inp["q_idx"], w_idx=inp["w_idx"], keys=inp["keys"])
    out, lse = layer.attend(inp["q"], cache, window, inp["q_pos"], None, inp["sink"], **kw)
    torch.cuda.synchronize()
    L.csa_check_status(layer.ws)
    res = dict(out=out, lse=lse, cache=cache, window=window, raw_ring=raw_ring, layer=layer)
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


# ----------------------------------------------------------- parity drivers
def _to_cuda(inp):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}


def _e4m3_midpoints():
    vals = np.array(sorted(oracle.e4m3_decode(c) for c in range(127)))  # the non-negative finite codes
    return (vals[:-1] + vals[1:]) / 2


_E4M3_MIDS = None
# A code decided from the GPU's float32 compressor output may differ from the
# oracle's (decided from its double output rounded to float32) only where the
# value lies within float32 noise of a rounding midpoint.  Stored rows are
# RMS-normalised (magnitudes of order 1) and the compressor's float32 error
# is absolute as much as relative (the pooled sum cancels), so the noise bound
# of a value v is NOISE * (|v| + 1/4): ~5e-7 at zero, far below a bfloat16 or
# E4M3 step.  Window rows quantised to E4M3 often sit exactly on a midpoint
# (x/scale = 448 kv_d / max|kv| is a ratio of bfloat16 numbers), which the
# noise then decides; a row may hold up to MAX_NEAR_MID_PER_ROW such values.
NOISE = 2.0 ** -19
MAX_NEAR_MID_PER_ROW = 16
NEAR_MID_COUNTS = []  # exceptions seen by check_stored_rows (reported by the tests)


def _noise(v):
    return NOISE * (np.abs(np.asarray(v, np.float64)) + 0.25)


def _bf16_round(x):
    """bfloat16 RNE of float64 values (through float32), as float64."""
    t = torch.from_numpy(np.asarray(x, np.float64)).to(torch.float32).to(torch.bfloat16)
    return t.to(torch.float64).numpy()


def _e4m3_round(x):
    """E4M3 RNE with saturation of float64 values (through float32), as float64."""
    t = torch.from_numpy(np.clip(np.asarray(x, np.float64), -448.0, 448.0)).to(torch.float32)
    return t.to(torch.float8_e4m3fn).to(torch.float64).numpy()


def _within_rounding(got, ref, tol, rnd):
    """got (decoded stored values) is the rounding of some value within tol
    of ref: rnd(ref - tol) <= got <= rnd(ref + tol)."""
    return (got >= rnd(ref - tol)) & (got <= rnd(ref + tol))


def check_stored_rows(w, gpu_rows, ref_rows, what):
    """GPU-written cache rows vs the oracle's stored form of its own (double)
    compressor output.  fp32 rows: within float32 accumulation noise.  bf16 and
    FP8 rows: every stored code is the rounding of a value within float32 noise
    of the oracle's value (so it equals the oracle's code except where that
    value lies within the noise of a rounding midpoint, or is so small that the
    noise spans a step); at most MAX_NEAR_MID_PER_ROW codes of a row differ from
    the oracle's, and the count is recorded in NEAR_MID_COUNTS."""
    ref = np.asarray(ref_rows, np.float64).reshape(-1, w.D)
    g = np_stored(gpu_rows).reshape(ref.shape[0], -1)
    if w.kv_fmt == "f32":
        got = g.view(np.float32).astype(np.float64)
        assert np.all(np.abs(got - ref) <= 1e-5 + 1e-6 * np.abs(ref)), "%s: worst %.3g" % (
            what, np.abs(got - ref).max())
        return 0
    o = oracle.store_rows(ref, _ORC_FMT[w.kv_fmt]).reshape(g.shape)
    ref32 = ref.astype(np.float32).astype(np.float64)
    n_exc = 0
    for r in range(g.shape[0]):
        if w.kv_fmt == "bf16":
            gv = (g[r].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
            ok = _within_rounding(gv, ref32[r], _noise(ref32[r]), _bf16_round)
            assert ok.all(), "%s row %d: %d bf16 values beyond float32 noise, e.g. dim %d (%.9g vs %.9g)" % (
                what, r, int((~ok).sum()), int(np.argmin(ok)), gv[np.argmin(ok)], ref[r, np.argmin(ok)])
            n = int((g[r] != o[r]).sum())
        else:
            nf = w.D - 64
            gs = g[r, nf + 128:nf + 128 + 4 * (nf // 64)].view(np.float32).astype(np.float64)
            os_ = o[r, nf + 128:nf + 128 + 4 * (nf // 64)].view(np.float32).astype(np.float64)
            amax = np.abs(ref32[r, :nf]).reshape(-1, 64).max(axis=1)
            assert np.all(np.abs(gs - os_) <= _noise(amax) / 448.0), "%s row %d: group scales differ" % (what, r)
            sc = np.repeat(os_, 64)
            q = ref32[r, :nf] / sc
            # the quotient's noise: the value's, over the scale, plus the scale's own
            tol = (_noise(ref32[r, :nf]) + np.abs(q) * np.repeat(_noise(amax), 64) / 448.0) / sc
            gq = np.array([oracle.e4m3_decode(int(c)) for c in g[r, :nf]])
            ok = _within_rounding(gq, q, tol, _e4m3_round)
            assert ok.all(), "%s row %d: %d E4M3 codes beyond float32 noise, e.g. dim %d" % (
                what, r, int((~ok).sum()), int(np.argmin(ok)))
            gr = (g[r, nf:nf + 128].view(np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
            rok = _within_rounding(gr, ref32[r, nf:], _noise(ref32[r, nf:]), _bf16_round)
            assert rok.all(), "%s row %d: rotated dims beyond float32 noise" % (what, r)
            assert np.all(g[r, nf + 128 + 4 * (nf // 64):] == 0), "%s row %d: padding" % (what, r)
            n = int((g[r, :nf + 128] != o[r, :nf + 128]).sum())
        assert n <= MAX_NEAR_MID_PER_ROW, "%s row %d: %d codes differ from the oracle's" % (what, r, n)
        n_exc += n
    NEAR_MID_COUNTS.append((what, g.shape[0], n_exc))
    return n_exc


# ---------------------------------------------------------------- decode
def decode_parity(w, seqs=None, gen_device="cpu", append=True, mutate=None):
    """Decode step on the GPU vs the oracle.  `mutate(inp)` may rewrite the
    generated inputs in place before either side sees them."""
    inp = _to_cuda(workloads.generate(w, device=gen_device))
    if mutate is not None:
        mutate(inp)
    res = gpu_decode(w, inp, append=append)
    seqs = list(range(w.B)) if seqs is None else seqs
    fmt = {"f32": oracle.F32, "bf16": oracle.BF16, "fp8m": oracle.FP8M}[w.kv_fmt]
    w_z = np_stored(inp["w_z"]).astype(np.float64)
    bias = np_stored(inp["bias"]).astype(np.float64)
    sink = np_stored(inp["sink"]).astype(np.float64)
    stats = []
    for b in seqs:
        Lb = w.lengths[b]
        i, n_av = Lb - 1, Lb // w.m
        q = np_stored(inp["q"][b])
        # the append step: the newest block's entry and the newest window row
        ent = None
        kv_b = np_stored(inp["kv_new"][b])
        if append and Lb % w.m == 0 and Lb >= w.m:
            ent = oracle.compress(kv_b, Lb - w.m, w.m, w_z, bias, w.rope_dims, w.rope_base, w.eps)
            check_stored_rows(w, res["cache"][b, n_av - 1], ent, "appended entry seq %d" % b)
        wr = i - int(inp["win_pos0"][b])   # the oracle's window is linear
        gr = i % w.W                       # the GPU's is a ring
        wrow = oracle.compress(kv_b[w.m - 1:], i, 1, w_z, bias[:1], w.rope_dims, w.rope_base, w.eps)
        if append:
            check_stored_rows(w, res["window"][b, gr], wrow, "window row seq %d" % b)
        window = oracle_stored_rows(w, inp["window"][b])
        if append:
            window[wr] = _appended(w, res["window"][b, gr], wrow, fmt)
        same = True
        if w.kind == "csa_decode":
            g_idx = res["topk_idx"][b].cpu().numpy()
            scores = oracle.index_scores(np_stored(inp["q_idx"][b]),
                                         np_stored(inp["w_idx"][b]).astype(np.float64),
                                         np_stored(inp["keys"][b, :n_av]))
            same = check_topk_set(g_idx, scores, w.topk, "seq %d" % b)
            kk = min(w.topk, n_av)
            g_sc = res["topk_score"][b, :kk].cpu().numpy().astype(np.float64)
            assert np.allclose(g_sc, scores[g_idx[:kk]], rtol=1e-4, atol=1e-4), "scores seq %d" % b
            need = np.unique(g_idx[:kk])
        else:
            need = np.arange(n_av)
        # compact cache: only the rows this query reads, stored like the GPU's
        rows = inp["cache"][b][torch.as_tensor(need, device=inp["cache"].device, dtype=torch.long)]
        cache_c = oracle_stored_rows(w, rows)
        if ent is not None and (n_av - 1) in set(need.tolist()):
            cache_c[int(np.searchsorted(need, n_av - 1))] = _appended(w, res["cache"][b, n_av - 1],
                                                                     ent, fmt)
        if w.kind == "csa_decode":
            out_o, lse_o = _attend_compact(w, q, i, cache_c, np.arange(len(need)), window,
                                           int(inp["win_pos0"][b]), sink)
        else:
            out_o, lse_o = oracle.attend_query(q, i, w.m, cache_c, w.D, None, window,
                                               int(inp["win_pos0"][b]), w.W, sink,
                                               rope_dims=w.rope_dims, base=w.rope_base, eps=w.eps,
                       scale=_scale(w))
        out_g = res["out"][b].float().cpu().numpy()
        mx, mn = assert_close(out_g, out_o, w.act, "out seq %d" % b)
        lse_g = res["lse"][b].cpu().numpy()
        assert np.max(np.abs(lse_g - lse_o)) <= LSE_TOL[w.act], "lse seq %d" % b
        stats.append((b, same, mx, mn))
    return stats


def _appended(w, gpu_row, ref_row, fmt):
    """The stored row an appended entry is attended from on the oracle side.
    An E4M3 code is decided by rounding the compressor's output, which the GPU
    holds in fp32 and the oracle in fp64: a value within rounding noise of a
    code midpoint may land one E4M3 step (1/8 relative) apart, which the row
    check allows there and nowhere else.  For FP8 rows the attention is
    therefore checked given the GPU's stored row (itself checked code by code
    against the oracle's); for the other formats the oracle's own rounding is
    used."""
    if w.kv_fmt == "fp8m":
        return np_stored(gpu_row)
    return oracle.store_rows(ref_row, fmt)[0]


def _attend_compact(w, q, i, cache_c, idx_c, window, win_pos0, sink):
    """CSA attention over the rows idx_c of a compact cache: the rows are the
    selected blocks, so the query attends to exactly those plus the window."""
    D = w.D
    rows = oracle.read_rows(cache_c, D)[idx_c]
    lo = max(0, i - w.W + 1)
    wrows = oracle.read_rows(window, D)[lo - win_pos0:i + 1 - win_pos0] if w.W else np.zeros((0, D))
    allrows = np.concatenate([rows, wrows], axis=0)
    return oracle.attend_rows(q, i, allrows, sink, rope_dims=w.rope_dims, base=w.rope_base,
                              eps=w.eps, scale=_scale(w))



# ---------------------------------------------------------------- prefill
def prefill_parity(w, sample=None, gen_device="cpu"):
    inp = _to_cuda(workloads.generate(w, device=gen_device))
    res = gpu_prefill(w, inp)
    cache_o, window_o = oracle_prefill_state(w, inp)
    n_old = w.T_cached // w.m
    # compressor outputs (new entries, window rows) against the oracle's
    w_z = np_stored(inp["w_z"]).astype(np.float64)
    bias = np_stored(inp["bias"]).astype(np.float64)
    kv_raw = np_stored(inp["kv_raw"])
    off = w.T_cached - inp["raw_pos0"]
    new = oracle.compress(kv_raw[off:], w.T_cached, w.m, w_z, bias, w.rope_dims, w.rope_base, w.eps)
    check_stored_rows(w, res["cache"][n_old:], new, "compressed entries")
    win = oracle.compress(kv_raw, inp["raw_pos0"], 1, w_z, bias[:1], w.rope_dims, w.rope_base, w.eps)
    check_stored_rows(w, res["window"], win, "window rows")
    qs = list(range(w.T_new)) if sample is None else sample
    q = np_stored(inp["q"])
    q_idx = np_stored(inp["q_idx"])
    w_idx = np_stored(inp["w_idx"]).astype(np.float64)
    keys = np_stored(inp["keys"])
    sink = np_stored(inp["sink"]).astype(np.float64)
    g_idx = res["topk_idx"].cpu().numpy()
    out_g = res["out"].float().cpu().numpy()
    lse_g = res["lse"].cpu().numpy()
    n_same = 0
    for t in qs:
        i = w.T_cached + t
        n_av = (i + 1) // w.m
        scores = oracle.index_scores(q_idx[t], w_idx[t], keys[:n_av])
        n_same += check_topk_set(g_idx[t], scores, w.topk, "query %d" % t)
    # attention for the sampled queries, given the GPU's indices (and, for FP8
    # rows, the GPU's stored rows: see _appended)
    if w.kv_fmt == "fp8m":
        cache_o = np_stored(res["cache"])[:cache_o.shape[0]]
        window_o = np_stored(res["window"])[:window_o.shape[0]]
    seq = np.zeros(len(qs), np.int32)
    pos = np.array([w.T_cached + t for t in qs], np.int64)
    out_o, lse_o = oracle.attend_batch(q[qs], seq, pos, w.m, cache_o[None], w.D, g_idx[qs],
                                       window_o[None], inp["raw_pos0"], w.W, sink,
                                       rope_dims=w.rope_dims, base=w.rope_base, eps=w.eps,
                       scale=_scale(w))
    assert_close(out_g[qs], out_o, w.act, "prefill out")
    assert np.max(np.abs(lse_g[qs] - lse_o)) <= LSE_TOL[w.act]
    # end to end (the oracle's own selection) for the queries whose sets agree
    return n_same, len(qs)


