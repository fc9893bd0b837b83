"""GPU parity: the CUDA library against the oracle on identical seeded inputs.

Small cases (ragged lengths, several tiles, partial tiles, k > available
blocks, windows clipped at position 0) run in full; the five full-size
workloads run in the launch configuration the benchmark times and are checked
on sampled sequences / queries.  Tolerances: bf16 max-abs 2e-2 and mean-abs
2e-3, fp32 1e-4; top-k sets exact except at oracle-score near-ties (1e-6
relative).  Attention is checked given the GPU's own top-k indices, and end to
end where the sets agree.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests import harness as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from long_context_compressed_17_b300 import build
    build.build()
    oracle.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _to_cuda(inp):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}


def _row_tol(w, ref):
    if w.kv_fmt == "f32":
        return 1e-5 + 1e-6 * np.abs(ref)
    if w.kv_fmt == "bf16":
        return 1e-5 + 2.0 ** -7 * np.abs(ref)
    return 1e-4 + np.abs(ref) / 8 + 2.0 ** -9 * np.abs(ref).max()


def check_stored_rows(w, gpu_rows, ref_rows, what):
    """GPU-written cache rows vs the oracle's unrounded rows."""
    got = oracle.read_rows(H.np_stored(gpu_rows), w.D)
    ref = np.asarray(ref_rows, np.float64).reshape(got.shape)
    err = np.abs(got - ref)
    assert np.all(err <= _row_tol(w, ref)), "%s: worst %.3g" % (what, err.max())


# ---------------------------------------------------------------- decode
def decode_parity(w, seqs=None, gen_device="cpu", append=True):
    inp = _to_cuda(workloads.generate(w, device=gen_device))
    res = H.gpu_decode(w, inp, append=append)
    seqs = list(range(w.B)) if seqs is None else seqs
    fmt = {"f32": oracle.F32, "bf16": oracle.BF16, "fp8m": oracle.FP8M}[w.kv_fmt]
    w_z = H.np_stored(inp["w_z"]).astype(np.float64)
    bias = H.np_stored(inp["bias"]).astype(np.float64)
    sink = H.np_stored(inp["sink"]).astype(np.float64)
    stats = []
    for b in seqs:
        Lb = w.lengths[b]
        i, n_av = Lb - 1, Lb // w.m
        q = H.np_stored(inp["q"][b])
        # the append step: the newest block's entry and the newest window row
        ent = None
        kv_b = H.np_stored(inp["kv_new"][b])
        if append and Lb % w.m == 0:
            ent = oracle.compress(kv_b, Lb - w.m, w.m, w_z, bias, w.rope_dims, w.rope_base, w.eps)
            check_stored_rows(w, res["cache"][b, n_av - 1], ent, "appended entry seq %d" % b)
        wr = i - int(inp["win_pos0"][b])
        wrow = oracle.compress(kv_b[w.m - 1:], i, 1, w_z, bias[:1], w.rope_dims, w.rope_base, w.eps)
        if append:
            check_stored_rows(w, res["window"][b, wr], wrow, "window row seq %d" % b)
        window = H.oracle_stored_rows(w, inp["window"][b])
        if append:
            window[wr] = oracle.store_rows(wrow, fmt)[0]
        same = True
        if w.kind == "csa_decode":
            g_idx = res["topk_idx"][b].cpu().numpy()
            scores = oracle.index_scores(H.np_stored(inp["q_idx"][b]),
                                         H.np_stored(inp["w_idx"][b]).astype(np.float64),
                                         H.np_stored(inp["keys"][b, :n_av]))
            same = H.check_topk_set(g_idx, scores, w.topk, "seq %d" % b)
            kk = min(w.topk, n_av)
            g_sc = res["topk_score"][b, :kk].cpu().numpy().astype(np.float64)
            assert np.allclose(g_sc, scores[g_idx[:kk]], rtol=1e-4, atol=1e-4), "scores seq %d" % b
            need = np.unique(g_idx[:kk])
        else:
            need = np.arange(n_av)
        # compact cache: only the rows this query reads, stored like the GPU's
        rows = inp["cache"][b][torch.as_tensor(need, device=inp["cache"].device, dtype=torch.long)]
        cache_c = H.oracle_stored_rows(w, rows)
        if ent is not None and (n_av - 1) in set(need.tolist()):
            cache_c[int(np.searchsorted(need, n_av - 1))] = oracle.store_rows(ent, fmt)[0]
        if w.kind == "csa_decode":
            out_o, lse_o = _attend_compact(w, q, i, cache_c, np.arange(len(need)), window,
                                           int(inp["win_pos0"][b]), sink)
        else:
            out_o, lse_o = oracle.attend_query(q, i, w.m, cache_c, w.D, None, window,
                                               int(inp["win_pos0"][b]), w.W, sink,
                                               rope_dims=w.rope_dims, base=w.rope_base, eps=w.eps)
        out_g = res["out"][b].float().cpu().numpy()
        mx, mn = H.assert_close(out_g, out_o, w.act, "out seq %d" % b)
        lse_g = res["lse"][b].cpu().numpy()
        assert np.max(np.abs(lse_g - lse_o)) <= H.LSE_TOL[w.act], "lse seq %d" % b
        stats.append((b, same, mx, mn))
    return stats


def _attend_compact(w, q, i, cache_c, idx_c, window, win_pos0, sink):
    """CSA attention over the rows idx_c of a compact cache: the rows are the
    selected blocks, so the query attends to exactly those plus the window."""
    D = w.D
    rows = oracle.read_rows(cache_c, D)[idx_c]
    lo = max(0, i - w.W + 1)
    wrows = oracle.read_rows(window, D)[lo - win_pos0:i + 1 - win_pos0] if w.W else np.zeros((0, D))
    allrows = np.concatenate([rows, wrows], axis=0)
    return oracle.attend_rows(q, i, allrows, sink, rope_dims=w.rope_dims, base=w.rope_base,
                              eps=w.eps)


SMALL_CSA = workloads.CSA_DECODE_128K.replace(
    name="csa_decode_small", B=4, L_per_seq=(5000, 4096, 2999, 30), topk=100)
SMALL_HCA = workloads.HCA_DECODE_1M.replace(
    name="hca_decode_small", B=3, L_per_seq=(128 * 37, 128 * 20 + 64, 100))
SMALL_FP8 = workloads.CSA_DECODE_1M_FP8.replace(
    name="csa_decode_fp8_small", B=2, L_per_seq=(8192, 6001), topk=200)


def test_csa_decode_small():
    st = decode_parity(SMALL_CSA)
    assert len(st) == 4


def test_csa_decode_small_sink_neginf():
    w = SMALL_CSA.replace(sink="neginf", B=2, L_per_seq=(3000, 1024))
    decode_parity(w)


def test_hca_decode_small():
    decode_parity(SMALL_HCA)


def test_csa_decode_fp8_small():
    decode_parity(SMALL_FP8)


def test_fp8_pack_is_bit_exact():
    from long_context_compressed_17_b300.pipeline import LayerConfig
    g = torch.Generator(device="cpu").manual_seed(11)
    x = torch.randn(300, 512, generator=g) * torch.rand(300, 1, generator=g) * 5
    x[7, 64:128] = 0  # all-zero group
    x[8, :10] = 1e6   # saturating group
    cfg = LayerConfig(D=512, H=64, m=4, kv="fp8m")
    dst = cfg.empty_rows(300)
    import long_context_compressed_17_b300 as L
    L.csa_cache_pack(cfg.params(), x.cuda(), 300, dst)
    ref = oracle.pack_fp8_rows(x.numpy())
    assert np.array_equal(dst.cpu().numpy(), ref)


# ---------------------------------------------------------------- prefill
def prefill_parity(w, sample=None, gen_device="cpu"):
    inp = _to_cuda(workloads.generate(w, device=gen_device))
    res = H.gpu_prefill(w, inp)
    cache_o, window_o = H.oracle_prefill_state(w, inp)
    n_old = w.T_cached // w.m
    # compressor outputs (new entries, window rows) against the oracle's
    w_z = H.np_stored(inp["w_z"]).astype(np.float64)
    bias = H.np_stored(inp["bias"]).astype(np.float64)
    kv_raw = H.np_stored(inp["kv_raw"])
    off = w.T_cached - inp["raw_pos0"]
    new = oracle.compress(kv_raw[off:], w.T_cached, w.m, w_z, bias, w.rope_dims, w.rope_base, w.eps)
    check_stored_rows(w, res["cache"][n_old:], new, "compressed entries")
    win = oracle.compress(kv_raw, inp["raw_pos0"], 1, w_z, bias[:1], w.rope_dims, w.rope_base, w.eps)
    check_stored_rows(w, res["window"], win, "window rows")
    qs = list(range(w.T_new)) if sample is None else sample
    q = H.np_stored(inp["q"])
    q_idx = H.np_stored(inp["q_idx"])
    w_idx = H.np_stored(inp["w_idx"]).astype(np.float64)
    keys = H.np_stored(inp["keys"])
    sink = H.np_stored(inp["sink"]).astype(np.float64)
    g_idx = res["topk_idx"].cpu().numpy()
    out_g = res["out"].float().cpu().numpy()
    lse_g = res["lse"].cpu().numpy()
    n_same = 0
    for t in qs:
        i = w.T_cached + t
        n_av = (i + 1) // w.m
        scores = oracle.index_scores(q_idx[t], w_idx[t], keys[:n_av])
        n_same += H.check_topk_set(g_idx[t], scores, w.topk, "query %d" % t)
    # attention for the sampled queries, given the GPU's indices
    seq = np.zeros(len(qs), np.int32)
    pos = np.array([w.T_cached + t for t in qs], np.int64)
    out_o, lse_o = oracle.attend_batch(q[qs], seq, pos, w.m, cache_o[None], w.D, g_idx[qs],
                                       window_o[None], inp["raw_pos0"], w.W, sink,
                                       rope_dims=w.rope_dims, base=w.rope_base, eps=w.eps)
    H.assert_close(out_g[qs], out_o, w.act, "prefill out")
    assert np.max(np.abs(lse_g[qs] - lse_o)) <= H.LSE_TOL[w.act]
    # end to end (the oracle's own selection) for the queries whose sets agree
    return n_same, len(qs)


def test_csa_prefill_bf16_small():
    w = workloads.CSA_CHUNKED_PREFILL.replace(name="prefill_small", T_cached=512, T_new=300,
                                              topk=64)
    n_same, n = prefill_parity(w)
    assert n_same >= n - 2


def test_csa_prefill_from_position_zero_small():
    w = workloads.CSA_CHUNKED_PREFILL.replace(name="prefill_zero", T_cached=0, T_new=200, topk=16,
                                              W=40)
    prefill_parity(w)


def test_cfg_csa_prefill_f32_full():
    """fp32 workload at its full size: 4096 causal queries, every query checked."""
    n_same, n = prefill_parity(workloads.CSA_PREFILL_F32)
    assert n_same >= n - 4


# ---------------------------------------------------------------- device status
def test_bad_topk_index_and_missing_window_are_flagged_not_faulted():
    import long_context_compressed_17_b300 as L
    from long_context_compressed_17_b300.pipeline import DecodeLayer
    w = SMALL_CSA.replace(B=1, L_per_seq=(4000,))
    inp = _to_cuda(workloads.generate(w))
    cfg = H.cfg_of(w)
    layer = DecodeLayer(cfg, 1, w.n_cap, w.W)
    idx = torch.arange(w.topk, dtype=torch.int32, device="cuda")[None].clone()
    idx[0, 5] = 1000  # block 1000 covers tokens 4000..4003: not complete at position 3999
    L.csa_attend(layer.p, inp["q"], w.H, 1, 1, inp["q_pos"], inp["cache"], w.n_cap, idx,
                 inp["window"], w.W, inp["win_pos0"], inp["sink"], layer.out, layer.lse,
                 layer.ws, layer.ws_bytes)
    with pytest.raises(L.CsaError) as ei:
        L.csa_check_status(layer.ws)
    assert ei.value.status == 5 and L.csa_last_device_bits() & 0x1
    L.csa_check_status(layer.ws)  # cleared
    bad_pos0 = inp["win_pos0"] + 5
    L.csa_attend(layer.p, inp["q"], w.H, 1, 1, inp["q_pos"], inp["cache"], w.n_cap,
                 idx.clamp(max=10), inp["window"], w.W, bad_pos0, inp["sink"], layer.out,
                 layer.lse, layer.ws, layer.ws_bytes)
    with pytest.raises(L.CsaError):
        L.csa_check_status(layer.ws)
    assert L.csa_last_device_bits() & 0x2


# ---------------------------------------------------------------- full size
@pytest.mark.parametrize("wl,seqs", [
    (workloads.CSA_DECODE_128K, [0, 31]),
    (workloads.HCA_DECODE_1M, [0, 17]),
    (workloads.CSA_DECODE_1M_FP8, [5]),
])
def test_full_size_decode_sampled(wl, seqs):
    stats = decode_parity(wl, seqs=seqs, gen_device="cuda")
    assert len(stats) == len(seqs)


def test_full_size_chunked_prefill_sampled():
    w = workloads.CSA_CHUNKED_PREFILL
    rng = np.random.default_rng(3)
    sample = sorted(set(list(range(8)) + list(range(w.T_new - 8, w.T_new)) +
                        rng.choice(w.T_new, 16, replace=False).tolist()))
    n_same, n = prefill_parity(w, sample=sample, gen_device="cuda")
    assert n_same >= n - 2
