"""Oracle pins: multi-query core attention with window, sink and output -i RoPE.

Pages: "DeepSeek-V4百万上下文时代的开源宣言" §三.2 CSA "Step 3: Core Attention
Multi-Query Attention", HCA "对所有压缩 KV 做 dense attention", and
"四项关键 Trick" (Q/KV Normalization, Partial RoPE with output RoPE at -i,
Sliding Window of 128 raw tokens, Attention Sink); "DeepSeek-V4 技术报告深度解析"
§2.1.4.

Pins: reduction to library softmax attention (top-k = every complete block,
window off, sink -inf); closed forms with one row; the sink's weight deficit;
relative-position invariance under a shift of all positions; permutation
invariance; the window's exact extent; causality errors.
"""
import math

import numpy as np
import pytest
import torch

from tests.test_oracle_norm_rope_compress import rms_closed, rope_complex


def sdpa(qp, rows, scale):
    """torch's scaled_dot_product_attention in float64 (one query token)."""
    q = torch.tensor(qp)[None, :, None, :]              # [1, H, 1, D]
    kv = torch.tensor(rows)[None, None].expand(1, qp.shape[0], -1, -1)
    o = torch.nn.functional.scaled_dot_product_attention(q, kv, kv, scale=scale)
    return o[0, :, 0].numpy()


def prep_q(q, i):
    return np.stack([rope_complex(rms_closed(qh), i) for qh in q])


def test_attend_rows_reduces_to_library_softmax_attention(orc):
    rng = np.random.default_rng(0)
    H, D, J, i = 6, 128, 37, 1234
    q = rng.standard_normal((H, D))
    rows = rng.standard_normal((J, D))
    out, lse = orc.attend_rows(q, i, rows, sink=-np.inf, derotate=False)
    ref = sdpa(prep_q(q, i), rows, 1.0 / math.sqrt(D))
    assert np.allclose(out, ref, atol=1e-12)
    logits = prep_q(q, i) @ rows.T / math.sqrt(D)
    assert np.allclose(lse, np.log(np.exp(logits).sum(1)), atol=1e-12)


def test_csa_topk_all_window_off_is_dense_attention_over_entries(orc):
    rng = np.random.default_rng(1)
    H, D, m, n_cap, i = 4, 128, 4, 30, 4 * 25 + 2   # 25 complete blocks
    q = rng.standard_normal((H, D)).astype(np.float32)
    cache = rng.standard_normal((n_cap, D)).astype(np.float32)
    window = np.zeros((1, D), dtype=np.float32)
    idx = np.arange(25, dtype=np.int32)[::-1].copy()  # every complete block, any order
    out, lse = orc.attend_query(q, i, m, cache, D, idx, window, win_pos0=0, W=0, sink=-np.inf,
                                derotate=False)
    ref = sdpa(prep_q(q.astype(np.float64), i), cache[:25].astype(np.float64), 1 / math.sqrt(D))
    assert np.allclose(out, ref, atol=1e-12)
    # HCA over the same blocks is the same computation
    out2, _ = orc.attend_query(q, i, m, cache, D, None, window, 0, 0, -np.inf, derotate=False)
    assert np.allclose(out2, out, atol=1e-13)


def test_single_row_with_sink_closed_form(orc):
    rng = np.random.default_rng(2)
    H, D, i = 3, 128, 77
    q = rng.standard_normal((H, D))
    e = rng.standard_normal((1, D))
    sink = np.array([-1.0, 0.0, 2.5])
    out, lse, wts = orc.attend_rows(q, i, e, sink, derotate=False, return_weights=True)
    l = prep_q(q, i) @ e[0] / math.sqrt(D)
    a = 1.0 / (1.0 + np.exp(sink - l))       # e^l / (e^s + e^l)
    assert np.allclose(wts[:, 0], a, atol=1e-14)
    assert np.allclose(out, a[:, None] * e, atol=1e-13)
    assert np.allclose(lse, np.logaddexp(sink, l), atol=1e-13)


def test_sink_weight_deficit_and_limits(orc):
    rng = np.random.default_rng(3)
    H, D, J = 5, 128, 50
    q = rng.standard_normal((H, D))
    rows = rng.standard_normal((J, D))
    sink = rng.standard_normal(H)
    out, lse, wts = orc.attend_rows(q, 9, rows, sink, derotate=False, return_weights=True)
    assert np.allclose(wts.sum(1), 1.0 - np.exp(sink - lse), atol=1e-14)
    assert np.all(wts.sum(1) <= 1.0)
    o0, _, w0 = orc.attend_rows(q, 9, rows, -np.inf, derotate=False, return_weights=True)
    assert np.allclose(w0.sum(1), 1.0, atol=1e-14)
    o_big, _ = orc.attend_rows(q, 9, rows, 1e4, derotate=False)
    assert np.max(np.abs(o_big)) < 1e-100


def test_output_derotation_closed_form(orc):
    """One row e = RoPE(x, p) and no sink: o = e, and RoPE(o, -i) = RoPE(x, p - i)."""
    rng = np.random.default_rng(4)
    H, D, p, i = 2, 512, 1000, 1300
    x = rms_closed(rng.standard_normal(D))
    e = rope_complex(x, p)[None]
    q = rng.standard_normal((H, D))
    out, _ = orc.attend_rows(q, i, e, -np.inf, derotate=True)
    ref = rope_complex(x, p - i)
    assert np.allclose(out, np.stack([ref] * H), atol=1e-10)


def test_shift_of_all_positions_leaves_output_and_lse_unchanged(orc):
    """Relative-only RoPE: entries compressed at positions shifted by delta (a
    multiple of m) and a query shifted by delta give the same logits; with the
    output -i rotation the outputs are unchanged too."""
    rng = np.random.default_rng(5)
    H, D, m, T = 4, 128, 4, 64
    kv = rng.standard_normal((T, D))
    w_z, bias = rng.standard_normal(D) * 0.02, rng.standard_normal(m) * 0.1
    q = rng.standard_normal((H, D))
    sink = rng.standard_normal(H)
    res = []
    for delta in (0, 4, 1000, 65536):
        ent = orc.compress(kv, delta, m, w_z, bias)
        win = orc.compress(kv, delta, 1, w_z, bias[:1])
        i = delta + T - 1
        rows = np.concatenate([ent[[2, 7, 11]], win[-16:]])
        res.append(orc.attend_rows(q, i, rows, sink, derotate=True))
        res_raw = orc.attend_rows(q, i, rows, sink, derotate=False)
        if delta == 0:
            first_raw = res_raw
    for out, lse in res[1:]:
        assert np.allclose(out, res[0][0], atol=1e-9)
        assert np.allclose(lse, res[0][1], atol=1e-9)
    # without the output rotation the absolute position leaks into the output
    assert not np.allclose(res_raw[0], first_raw[0], atol=1e-3)


def test_permutation_invariance(orc):
    rng = np.random.default_rng(6)
    q = rng.standard_normal((3, 128))
    rows = rng.standard_normal((40, 128))
    perm = rng.permutation(40)
    a = orc.attend_rows(q, 5, rows, 0.3)
    b = orc.attend_rows(q, 5, rows[perm], 0.3)
    assert np.allclose(a[0], b[0], atol=1e-13) and np.allclose(a[1], b[1], atol=1e-13)


@pytest.mark.parametrize("i,W", [(100, 5), (3, 8), (0, 128), (200, 128), (50, 1)])
def test_window_covers_exactly_the_last_W_positions(orc, i, W):
    rng = np.random.default_rng(i + W)
    H, D, m = 2, 128, 4
    q = rng.standard_normal((H, D)).astype(np.float32)
    n_win, win_pos0 = 300, 0
    window = rng.standard_normal((n_win, D)).astype(np.float32)
    cache = rng.standard_normal((80, D)).astype(np.float32)
    no_idx = np.full(4, -1, dtype=np.int32)
    out, lse = orc.attend_query(q, i, m, cache, D, no_idx, window, win_pos0, W, sink=0.5)
    lo = max(0, i - W + 1)
    ref, ref_lse = orc.attend_rows(q, i, window[lo:i + 1].astype(np.float64), 0.5)
    assert np.allclose(out, ref, atol=1e-13) and np.allclose(lse, ref_lse, atol=1e-13)
    # closed form for the window's size: with a sink of -inf and all-equal rows the
    # output is that row, and the log-normaliser is logit + log(count)
    same = np.tile(window[:1], (n_win, 1))
    out1, lse1 = orc.attend_query(q, i, m, cache, D, no_idx, same, win_pos0, W, -np.inf,
                                  derotate=False)
    l = prep_q(q.astype(np.float64), i) @ same[0].astype(np.float64) / math.sqrt(D)
    assert np.allclose(lse1, l + math.log(i - lo + 1), atol=1e-12)


def test_window_rows_are_found_by_position(orc):
    rng = np.random.default_rng(7)
    H, D, i, W = 2, 128, 1000, 16
    q = rng.standard_normal((H, D)).astype(np.float32)
    window = rng.standard_normal((W, D)).astype(np.float32)
    cache = rng.standard_normal((300, D)).astype(np.float32)
    out, _ = orc.attend_query(q, i, 4, cache, D, np.array([-1], np.int32), window, i - W + 1, W, 0.0)
    ref, _ = orc.attend_rows(q, i, window.astype(np.float64), 0.0)
    assert np.allclose(out, ref, atol=1e-13)
    with pytest.raises(ValueError):  # position i is not in a buffer that starts at i-W+2
        orc.attend_query(q, i, 4, cache, D, np.array([-1], np.int32), window, i - W + 2, W, 0.0)


def test_csa_rejects_incomplete_block(orc):
    rng = np.random.default_rng(8)
    q = rng.standard_normal((2, 128)).astype(np.float32)
    cache = rng.standard_normal((10, 128)).astype(np.float32)
    window = np.zeros((1, 128), np.float32)
    # position 10 with m = 4: blocks 0, 1 complete; block 2 (tokens 8..11) is not
    orc.attend_query(q, 10, 4, cache, 128, np.array([1, 0], np.int32), window, 0, 0, 0.0)
    with pytest.raises(ValueError):
        orc.attend_query(q, 10, 4, cache, 128, np.array([2], np.int32), window, 0, 0, 0.0)


def test_no_rows_and_no_sink_gives_zero_output(orc):
    q = np.ones((2, 128))
    out, lse = orc.attend_rows(q, 0, np.zeros((0, 128)), -np.inf)
    assert np.all(out == 0) and np.all(np.isneginf(lse))
    out, lse = orc.attend_rows(q, 0, np.zeros((0, 128)), 1.5)
    assert np.all(out == 0) and np.allclose(lse, 1.5)


def test_attend_batch_equals_single_queries(orc):
    rng = np.random.default_rng(9)
    B, H, D, m, n_cap, W, k, n_win = 2, 3, 128, 4, 40, 8, 5, 12
    q = rng.standard_normal((3, H, D)).astype(np.float32)
    cache = rng.standard_normal((B, n_cap, D)).astype(np.float32)
    window = rng.standard_normal((B, n_win, D)).astype(np.float32)
    pos = np.array([159, 157, 155])
    seq = np.array([0, 1, 1])
    win_pos0 = np.array([148, 146])
    idx = np.array([[0, 5, 39, -1, 2], [3, 4, -1, -1, 24], [1, 2, 3, 38, 0]], np.int32)
    sink = rng.standard_normal(H)
    out, lse = orc.attend_batch(q, seq, pos, m, cache, D, idx, window, win_pos0, W, sink)
    for j in range(3):
        o1, l1 = orc.attend_query(q[j], pos[j], m, cache[seq[j]], D, idx[j], window[seq[j]],
                                  win_pos0[seq[j]], W, sink)
        assert np.array_equal(out[j], o1) and np.array_equal(lse[j], l1)
    with pytest.raises(ValueError):  # W = 16: query 0 needs 144..159, the buffer starts at 148
        orc.attend_batch(q, seq, pos, m, cache, D, idx, window, win_pos0, 16, sink)
