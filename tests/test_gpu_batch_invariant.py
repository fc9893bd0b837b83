"""Batch invariance [gitcode §5.3 "批次不变且确定性内核"].

With the batch_invariant params flag a query's attention output and lse are
bit-identical whether it runs alone, in a larger batch, at another place in
the batch, among other queries, or again; they still match the oracle within
the bf16 tolerance.  The lightning indexer's decode kernel (one query per
MMA) and its prefill kernel (four queries per MMA) give bit-identical scores
for the same query, with bf16 and with E4M3 keys.  The top-k is exact and the
compressor works per block, so the whole step inherits the property.
"""
import numpy as np
import pytest
import torch

import oracle
from tests import harness as H

pytestmark = pytest.mark.gpu

D, NH, W = 512, 64, 128


@pytest.fixture(scope="module")
def L():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from long_context_compressed_17_b300 import build
    build.build()
    oracle.build()
    import long_context_compressed_17_b300 as pkg
    return pkg


def _state(L, g, B, n_cap, lengths, m, k, kv, qps=1):
    """Per-sequence decode (qps = 1) or prefill-like state on the host."""
    Q = B * qps
    q = torch.randn(Q, NH, D, generator=g).to(torch.bfloat16)
    q_pos = torch.tensor([lengths[b] - qps + j for b in range(B) for j in range(qps)], dtype=torch.int64)
    win_pos0 = torch.tensor([max(0, lengths[b] - qps + 1 - W) for b in range(B)], dtype=torch.int64)
    n_win = W + qps - 1
    cache_f = torch.randn(B, n_cap, D, generator=g)
    win_f = torch.randn(B, n_win, D, generator=g)
    p = L.params(D, m, topk=k, kv=kv, batch_invariant=True)
    if kv == "bf16":
        cache, window = cache_f.to(torch.bfloat16), win_f.to(torch.bfloat16)
    else:
        rb = L.csa_row_bytes(kv, D)
        cache = torch.empty(B, n_cap, rb, dtype=torch.uint8, device="cuda")
        window = torch.empty(B, n_win, rb, dtype=torch.uint8, device="cuda")
        L.csa_cache_pack(p, cache_f.cuda(), B * n_cap, cache)
        L.csa_cache_pack(p, win_f.cuda(), B * n_win, window)
        torch.cuda.synchronize()
        cache, window = cache.cpu(), window.cpu()
    idx = None
    if k:
        idx = torch.full((Q, k), -1, dtype=torch.int32)
        for qq in range(Q):
            n = min((int(q_pos[qq]) + 1) // m, n_cap)
            sel = torch.randperm(n, generator=g)[:min(k, n)].sort().values
            idx[qq, :sel.numel()] = sel.to(torch.int32)
    sink = torch.randn(NH, generator=g)
    return dict(q=q, q_pos=q_pos, win_pos0=win_pos0, cache=cache, window=window, idx=idx, sink=sink,
                p=p, n_cap=n_cap, n_win=n_win, qps=qps, m=m, k=k, kv=kv)


def _pick(st, seqs):
    """The sub-batch of sequences `seqs` (in that order), all their queries."""
    qps = st["qps"]
    qs = [b * qps + j for b in seqs for j in range(qps)]
    sub = dict(st)
    sub["q"] = st["q"][qs]
    sub["q_pos"] = st["q_pos"][qs]
    sub["win_pos0"] = st["win_pos0"][seqs]
    sub["cache"] = st["cache"][seqs]
    sub["window"] = st["window"][seqs]
    sub["idx"] = None if st["idx"] is None else st["idx"][qs]
    return sub, qs


def _attend(L, st):
    """Runs the attention on a fresh device copy; returns (out bits int16, lse)."""
    B = st["cache"].shape[0]
    Q = st["q"].shape[0]
    c = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in st.items()}
    out = torch.empty(Q, NH, D, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(Q, NH, dtype=torch.float32, device="cuda")
    sparse = st["k"] > 0
    op = L.OP_ATTEND if sparse else L.OP_HCA_ATTEND
    nb = L.csa_workspace_bytes(st["p"], op, B, Q, NH, 0, st["n_cap"], st["n_win"])
    ws = L.workspace(nb)
    if sparse:
        L.csa_attend(st["p"], c["q"], NH, B, Q, c["q_pos"], c["cache"], st["n_cap"], c["idx"], c["window"],
                     st["n_win"], c["win_pos0"], c["sink"], out, lse, ws, nb)
    else:
        L.hca_attend(st["p"], c["q"], NH, B, Q, c["q_pos"], c["cache"], st["n_cap"], c["window"],
                     st["n_win"], c["win_pos0"], c["sink"], out, lse, ws, nb)
    torch.cuda.synchronize()
    L.csa_check_status(ws)
    return out.cpu().view(torch.int16), lse.cpu()


def _same(full, sub, qs, what):
    o_f, l_f = full
    o_s, l_s = sub
    for j, qq in enumerate(qs):
        assert torch.equal(o_s[j], o_f[qq]), "%s: out of query %d differs" % (what, qq)
        assert torch.equal(l_s[j].view(torch.int32), l_f[qq].view(torch.int32)), "%s: lse of query %d" % (what, qq)


def _oracle_check(st, res, qs):
    out = res[0].view(torch.bfloat16).float().numpy()
    lse = res[1].numpy()
    for qq in qs:
        b = qq // st["qps"]
        idx = None if st["idx"] is None else st["idx"][qq].numpy()
        ref, rl = oracle.attend_query(H.np_stored(st["q"][qq]), int(st["q_pos"][qq]), st["m"],
                                      H.np_stored(st["cache"][b]), D, idx, H.np_stored(st["window"][b]),
                                      int(st["win_pos0"][b]), W, st["sink"].numpy().astype(np.float64))
        H.assert_close(out[qq], ref, "bf16", "query %d out" % qq)
        assert np.max(np.abs(lse[qq] - rl)) <= H.LSE_TOL["bf16"], "query %d lse" % qq


def _invariance(L, st, B, what):
    full = _attend(L, st)
    again = _attend(L, st)
    _same(full, again, list(range(st["q"].shape[0])), what + ": rerun")
    orders = [list(range(B))[::-1], [B - 1], [0], [B // 2, 1, B - 2]]
    for seqs in orders:
        sub, qs = _pick(st, seqs)
        _same(full, _attend(L, sub), qs, "%s: sequences %s" % (what, seqs[:4]))
    _oracle_check(st, full, [0, st["q"].shape[0] // 2, st["q"].shape[0] - 1])
    return full


@pytest.mark.parametrize("kv", ["bf16", "fp8m"])
def test_csa_decode_bit_identical_in_any_batch(L, kv):
    """18 tiles per query (k = 1024 + W): splits of 2 tiles, 9 partials."""
    g = torch.Generator(device="cpu").manual_seed(71)
    B = 24
    lengths = [int(x) for x in torch.randint(100, 16384, (B,), generator=g)]
    lengths[3] = 40  # no complete block of 4 beyond the first ten: short list
    st = _state(L, g, B, 4096, lengths, 4, 1024, kv)
    full = _invariance(L, st, B, "csa " + kv)
    # among other queries: sequences 5 and 9 inside a batch of fresh ones
    g2 = torch.Generator(device="cpu").manual_seed(72)
    other = _state(L, g2, 6, 4096, [9000] * 6, 4, 1024, kv)
    mix = dict(st)
    for key in ("q", "q_pos", "win_pos0", "cache", "window", "idx"):
        a, b = st[key], other[key]
        mix[key] = torch.cat([b[:3], a[5:6], b[3:], a[9:10]])
    res = _attend(L, mix)
    _same(full, (res[0][[3, 7]], res[1][[3, 7]]), [5, 9], "csa %s: among other queries" % kv)


def test_hca_decode_bit_identical_in_any_batch(L):
    """34 tiles per query: splits of 4 tiles; ragged last split (2 tiles)."""
    g = torch.Generator(device="cpu").manual_seed(73)
    B = 12
    lengths = [int(x) for x in torch.randint(2000, 128 * 2048, (B,), generator=g)]
    st = _state(L, g, B, 2048, lengths, 128, 0, "bf16")
    _invariance(L, st, B, "hca")


def test_hca_long_list_sixteen_tile_splits(L):
    """130 tiles per query (the 1M-context HCA shape: 8192 blocks): splits of 16."""
    g = torch.Generator(device="cpu").manual_seed(74)
    B = 5
    lengths = [128 * 8192, 128 * 8000 + 5, 128 * 700, 128 * 64, 200]
    st = _state(L, g, B, 8192, lengths, 128, 0, "bf16")
    _invariance(L, st, B, "hca long")


def test_prefill_queries_bit_identical_in_any_grouping(L):
    """Eight queries per sequence: the same query alone, with its sequence's
    other queries, or with a second sequence gives the same bits."""
    g = torch.Generator(device="cpu").manual_seed(75)
    st = _state(L, g, 2, 2048, [7000, 5003], 4, 256, "bf16", qps=8)
    full = _attend(L, st)
    sub, qs = _pick(st, [1])
    _same(full, _attend(L, sub), qs, "prefill: second sequence alone")
    # the last four queries of sequence 0 as a batch of their own
    four = dict(st, qps=4, q=st["q"][4:8], q_pos=st["q_pos"][4:8], idx=st["idx"][4:8],
                win_pos0=st["win_pos0"][:1], cache=st["cache"][:1], window=st["window"][:1])
    _same(full, _attend(L, four), [4, 5, 6, 7], "prefill: four queries")
    one = dict(st, qps=1, q=st["q"][6:7], q_pos=st["q_pos"][6:7], idx=st["idx"][6:7],
               win_pos0=st["win_pos0"][:1], cache=st["cache"][:1], window=st["window"][:1])
    _same(full, _attend(L, one), [6], "prefill: one query")
    _oracle_check(st, full, [0, 9, 15])


# ----------------------------------------------------------------- indexer
def _scores(L, fp8, q_idx, w_idx, keys_dev, scales_dev, n_cap, q_pos, B):
    Q = q_idx.shape[0]
    p = L.params(D, 4, topk=64)
    ld = (n_cap + 127) // 128 * 128
    sc = torch.empty(Q, ld, dtype=torch.float32, device="cuda")
    if fp8:
        nb = 256 + 2 * 256 + Q * 64 * 128 + Q * 64 * 4
        ws = L.workspace(nb)
        L.csa_index_score_fp8(p, q_idx.cuda(), w_idx.cuda(), 64, 128, keys_dev, scales_dev, n_cap, B, Q,
                              q_pos.cuda(), sc, ld, ws, nb)
    else:
        ws = L.workspace(256)
        L.csa_index_score(p, q_idx.cuda(), w_idx.cuda(), 64, 128, keys_dev, n_cap, B, Q, q_pos.cuda(),
                          sc, ld, ws, 256)
    torch.cuda.synchronize()
    L.csa_check_status(ws)
    return sc.cpu()[:, :n_cap]


@pytest.mark.parametrize("fp8", [False, True])
def test_indexer_decode_and_prefill_kernels_agree_bitwise(L, fp8):
    g = torch.Generator(device="cpu").manual_seed(76)
    n_cap = 3000
    keys = (torch.randn(1, n_cap, 128, generator=g) * 2).to(torch.bfloat16)
    q_idx = torch.randn(8, 64, 128, generator=g).to(torch.bfloat16)
    w_idx = torch.rand(8, 64, generator=g)
    q_pos = torch.tensor([11999 - 7 + j for j in range(8)], dtype=torch.int64)
    p = L.params(D, 4, topk=64)
    if fp8:
        kd = torch.empty(1, n_cap, 128, dtype=torch.uint8, device="cuda")
        sd = torch.empty(1, n_cap, dtype=torch.float32, device="cuda")
        L.csa_index_keys_pack(p, keys.cuda(), n_cap, 128, kd, sd)
    else:
        kd, sd = keys.cuda(), None
    grouped = _scores(L, fp8, q_idx, w_idx, kd, sd, n_cap, q_pos, 1)       # 8 per sequence: 4 per MMA
    for j in range(8):
        alone = _scores(L, fp8, q_idx[j:j + 1], w_idx[j:j + 1], kd, sd, n_cap, q_pos[j:j + 1], 1)
        assert torch.equal(alone[0].view(torch.int32), grouped[j].view(torch.int32)), "query %d" % j
