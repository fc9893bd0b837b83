"""Oracle pins: lightning indexer score and top-k selection.

Pages: "DeepSeek-V4百万上下文时代的开源宣言" §三.2, CSA "Step 2: Lightning
Indexer Top-K 选择"; "DeepSeek-V4 技术报告深度解析" §2.1.1.  Score of block b
for one query: sum_h w_h relu(q_h . k_b) over causally complete blocks; keep
the top k, ties to the lower index.
"""
import numpy as np
import pytest


def test_indexer_hand_computed_example(orc):
    # q_0 = (1, 0), q_1 = (0, 1), w = (1, 2); keys k_0..k_3 below.
    # k_0 = (1, 1):  1*relu(1)  + 2*relu(1)  = 3
    # k_1 = (-1, 2): 1*relu(-1) + 2*relu(2)  = 4
    # k_2 = (3, -1): 1*relu(3)  + 2*relu(-1) = 3
    # k_3 = (0, 0):  0
    q = np.array([[1.0, 0.0], [0.0, 1.0]])
    keys = np.array([[1.0, 1.0], [-1.0, 2.0], [3.0, -1.0], [0.0, 0.0]])
    s = orc.index_scores(q, [1.0, 2.0], keys)
    assert s.tolist() == [3.0, 4.0, 3.0, 0.0]
    idx, sel = orc.topk(s, 2)
    assert idx.tolist() == [1, 0]  # 4, then the tie at 3 goes to the lower index
    idx, _ = orc.topk(s, 3)
    assert idx.tolist() == [1, 0, 2]


def test_indexer_all_nonpositive_dots_give_exact_zero_ties(orc):
    rng = np.random.default_rng(0)
    HI, dI, n = 4, 16, 50
    q = np.abs(rng.standard_normal((HI, dI)))
    keys = -np.abs(rng.standard_normal((n, dI)))  # every q_h . k_b < 0
    s = orc.index_scores(q, rng.random(HI), keys)
    assert np.all(s == 0.0)
    idx, _ = orc.topk(s, 7)
    assert idx.tolist() == list(range(7))


def test_indexer_linear_in_head_weights(orc):
    rng = np.random.default_rng(1)
    q = rng.standard_normal((8, 32))
    keys = rng.standard_normal((100, 32))
    w1, w2 = rng.random(8), rng.random(8)
    s1 = orc.index_scores(q, w1, keys)
    s2 = orc.index_scores(q, w2, keys)
    s12 = orc.index_scores(q, w1 + w2, keys)
    assert np.allclose(s12, s1 + s2, rtol=1e-13, atol=1e-13)
    # one head with unit weight is relu of the dot product
    e0 = np.zeros(8)
    e0[3] = 1.0
    s3 = orc.index_scores(q, e0, keys)
    assert np.allclose(s3, np.maximum(keys @ q[3], 0.0), rtol=1e-13, atol=1e-14)


def test_indexer_reads_bf16_storage(orc):
    import torch
    rng = np.random.default_rng(2)
    q = rng.standard_normal((4, 64)).astype(np.float32)
    keys = rng.standard_normal((30, 64)).astype(np.float32)
    qb = torch.tensor(q).to(torch.bfloat16)
    kb = torch.tensor(keys).to(torch.bfloat16)
    bits = lambda t: t.view(torch.int16).numpy().view(np.uint16)
    w = rng.random(4)
    s_bits = orc.index_scores(bits(qb), w, bits(kb))
    s_f64 = orc.index_scores(qb.double().numpy(), w, kb.double().numpy())
    assert np.array_equal(s_bits, s_f64)


def _brute_topk(s, k):
    order = sorted(range(len(s)), key=lambda b: (-s[b], b))[:k]
    return order + [-1] * (k - len(order))


@pytest.mark.parametrize("n,k", [(0, 4), (3, 8), (40, 8), (200, 64), (1000, 1)])
def test_topk_matches_brute_force_with_ties(orc, n, k):
    rng = np.random.default_rng(n * 31 + k)
    s = rng.integers(0, 6, n).astype(np.float64)  # many exact ties
    idx, sel = orc.topk(s, k)
    assert idx.tolist() == _brute_topk(s.tolist(), k)
    nsel = min(n, k)
    assert np.array_equal(sel[:nsel], s[idx[:nsel]])
    assert np.all(np.isneginf(sel[nsel:]))


def test_index_topk_batch_causality(orc):
    """Only blocks whose last token is at or before the query are scored: a
    huge key in the first incomplete block is never selected."""
    rng = np.random.default_rng(3)
    m, n_cap, HI, dI = 4, 20, 2, 8
    q = np.abs(rng.standard_normal((3, HI, dI)))
    w = np.ones((3, HI))
    keys = np.abs(rng.standard_normal((1, n_cap, dI))) * 0.01
    keys[0, 5] = 100.0  # block 5 = tokens 20..23, complete from position 23 on
    pos = np.array([21, 22, 23])
    idx, _ = orc.index_topk_batch(q, w, keys, seq=[0, 0, 0], pos=pos, m=m, k=3)
    assert 5 not in idx[0] and 5 not in idx[1]
    assert idx[2][0] == 5
    # n_complete((i+1)//m): position 2 sees no block, position 3 sees one
    assert orc.n_complete(2, 4) == 0 and orc.n_complete(3, 4) == 1
    idx, _ = orc.index_topk_batch(q[:2], w[:2], keys, seq=[0, 0], pos=np.array([2, 3]), m=m, k=2)
    assert idx[0].tolist() == [-1, -1] and idx[1].tolist() == [0, -1]


def test_index_topk_batch_equals_single_query_path(orc):
    rng = np.random.default_rng(4)
    B, n_cap, HI, dI, m, k = 2, 64, 4, 16, 4, 10
    q = rng.standard_normal((3, HI, dI))
    w = rng.random((3, HI))
    keys = rng.standard_normal((B, n_cap, dI))
    seq, pos = np.array([0, 1, 1]), np.array([255, 100, 17])
    idx, _ = orc.index_topk_batch(q, w, keys, seq, pos, m, k)
    for j in range(3):
        n = orc.n_complete(pos[j], m)
        s = orc.index_scores(q[j], w[j], keys[seq[j], :n])
        assert idx[j].tolist() == _brute_topk(s.tolist(), k)
