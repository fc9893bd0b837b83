"""GPU parity of the FP4 lightning indexer ["DeepSeek-V4 技术报告深度解析"
§2.1.1, §3.2]: the key packer bit-exact against the oracle (codes, block
exponents, the 14-binade threshold, the tile layout and its all-zero padding keys),
and the scores and top-k sets of csa_index_topk_fp4 / csa_index_score_fp4
against the oracle's FP4 scores (its exact top-k), in decode (one query per
sequence) and prefill-like (four queries per MMA) shapes, ragged and at the
headline decode size."""
import numpy as np
import pytest
import torch

import oracle
from tests import harness as H

pytestmark = pytest.mark.gpu

TILE = 8704


@pytest.fixture(scope="module")
def L():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from long_context_compressed_17_b300 import build
    build.build()
    oracle.build()
    import long_context_compressed_17_b300 as pkg
    return pkg


def _keys(g, shape):
    x = torch.randn(*shape, generator=g) * torch.rand(*shape[:-1], 1, generator=g) * 4
    return x.to(torch.bfloat16)


def _unpack(pack, B, n_cap):
    """GPU tiles -> (codes [B, n_cap, 64], exponent bytes [B, n_cap, 4]) and the padding bytes."""
    n_tiles = (n_cap + 127) // 128
    t = pack.reshape(B, n_tiles, TILE)
    codes = t[:, :, :128 * 64].reshape(B, n_tiles * 128, 64)
    exps = t[:, :, 128 * 64:].reshape(B, n_tiles * 128, 4)
    return codes[:, :n_cap], exps[:, :n_cap], codes[:, n_cap:], exps[:, n_cap:]


def _pack(L, p, keys):
    B, n_cap = keys.shape[0], keys.shape[1]
    nb = L.csa_index_keys_fp4_bytes(n_cap)
    assert nb == (n_cap + 127) // 128 * TILE
    pack = torch.full((B, nb), 0xA5, dtype=torch.uint8, device="cuda")  # padding must be rewritten
    L.csa_index_keys_pack_fp4(p, keys.cuda(), B, n_cap, 128, pack)
    torch.cuda.synchronize()
    return pack


def test_key_pack_is_bit_exact(L):
    g = torch.Generator(device="cpu").manual_seed(71)
    B, n_cap = 2, 300  # a ragged last tile
    keys = _keys(g, (B, n_cap, 128))
    keys[0, 3] = 0                          # an all-zero key
    keys[0, 4, 32:64] = 0                   # an all-zero block
    keys[1, 9, 5] = 3.0e4                   # a block whose scale is far above the others
    keys[1, 10, 96:] *= 2.0 ** -40          # a block far below: raised to the threshold
    keys[1, 11, 7] = -0.0
    keys[0, 200, 64:96] = 1e-39             # bfloat16 subnormals
    p = L.params(512, 4, topk=64)
    pack = _pack(L, p, keys)
    codes, exps, pad_c, pad_e = _unpack(pack.cpu().numpy(), B, n_cap)
    for b in range(B):
        rc, rs = oracle.pack_idx_keys_fp4(keys[b].float().numpy())
        assert np.array_equal(codes[b], rc), "codes of sequence %d" % b
        assert np.array_equal(exps[b], rs), "exponents of sequence %d" % b
    assert np.all(pad_c == 0) and np.all(pad_e == 127)  # all-zero keys (scale 1)
    # the threshold was exercised
    es = exps[1, 10].astype(int) - 127
    assert es[3] == es[:3].max() - 14


def _run(L, B, qps, n_cap, lengths, k, m=4, seed=72, sample=None):
    g = torch.Generator(device="cpu").manual_seed(seed)
    Q = B * qps
    q_idx = torch.randn(Q, 64, 128, generator=g).to(torch.bfloat16)
    w_idx = torch.rand(Q, 64, generator=g)
    keys = _keys(g, (B, n_cap, 128))
    q_pos = torch.tensor([lengths[b] - qps + j for b in range(B) for j in range(qps)], dtype=torch.int64)
    p = L.params(512, m, topk=k)
    pack = _pack(L, p, keys)
    nb = L.csa_workspace_bytes(p, L.OP_INDEX_TOPK_FP4, B, Q, 64, 64, n_cap, 128)
    ws = L.workspace(nb)
    idx = torch.empty(Q, k, dtype=torch.int32, device="cuda")
    sc = torch.empty(Q, k, dtype=torch.float32, device="cuda")
    L.csa_index_topk_fp4(p, q_idx.cuda(), w_idx.cuda(), 64, 128, pack, n_cap, B, Q, q_pos.cuda(), idx, sc, ws, nb)
    # the scoring half on its own: every score of every query
    ld = (n_cap + 127) // 128 * 128
    scores_g = torch.empty(Q, ld, dtype=torch.float32, device="cuda")
    L.csa_index_score_fp4(p, q_idx.cuda(), w_idx.cuda(), 64, 128, pack, n_cap, B, Q, q_pos.cuda(), scores_g, ld,
                          ws, nb)
    torch.cuda.synchronize()
    L.csa_check_status(ws)
    gi, gs, sg = idx.cpu().numpy(), sc.cpu().numpy(), scores_g.cpu().numpy()
    codes, exps, _, _ = _unpack(pack.cpu().numpy(), B, n_cap)
    qn = H.np_stored(q_idx)
    wn = w_idx.numpy().astype(np.float64)
    same = 0
    qs = range(Q) if sample is None else sample
    for q in qs:
        b = q // qps
        n = (int(q_pos[q]) + 1) // m
        scores = oracle.index_scores_fp4(qn[q], wn[q], codes[b, :n], exps[b, :n])
        assert np.allclose(sg[q, :n], scores, rtol=1e-4, atol=1e-4), "scores of query %d" % q
        assert np.all(np.isneginf(sg[q, n:n_cap]))
        same += H.check_topk_set(gi[q], scores, k, "query %d" % q)
        kk = min(k, n)
        assert np.allclose(gs[q, :kk], scores[gi[q, :kk]], rtol=1e-4, atol=1e-4), "scores of query %d" % q
    return same, len(list(qs))


def test_decode_ragged(L):
    same, n = _run(L, B=4, qps=1, n_cap=6000, lengths=[24000, 17001, 4000, 700], k=512)
    assert same >= n - 1


def test_four_queries_per_mma(L):
    same, n = _run(L, B=2, qps=8, n_cap=3000, lengths=[12000, 9000], k=256)
    assert same >= n - 2


def test_headline_decode_size_sampled(L):
    same, n = _run(L, B=32, qps=1, n_cap=32768, lengths=[131072] * 32, k=1024, sample=[0, 17, 31])
    assert same >= n - 1
