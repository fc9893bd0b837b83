"""GPU parity of the E4M3 lightning indexer: the key packer bit-exact against
the oracle, and the top-k sets (and scores) of csa_index_topk_fp8 against the
oracle's exact top-k of its FP8 scores, in decode (one query per sequence)
and prefill-like (four queries per MMA) shapes, ragged and at the headline
decode size."""
import numpy as np
import pytest
import torch

import oracle
from tests import harness as H

pytestmark = pytest.mark.gpu


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


def test_key_pack_is_bit_exact(L):
    g = torch.Generator(device="cpu").manual_seed(51)
    keys = _keys(g, (700, 128))
    keys[3] = 0
    keys[9, 5] = 3.0e4
    p = L.params(512, 4, topk=64)
    codes = torch.empty(700, 128, dtype=torch.uint8, device="cuda")
    scales = torch.empty(700, dtype=torch.float32, device="cuda")
    L.csa_index_keys_pack(p, keys.cuda(), 700, 128, codes, scales)
    torch.cuda.synchronize()
    rc, rs = oracle.pack_idx_keys_fp8(keys.float().numpy())
    assert np.array_equal(codes.cpu().numpy(), rc)
    assert np.array_equal(scales.cpu().numpy(), rs)


def _run(L, B, qps, n_cap, lengths, k, m=4, seed=52, sample=None):
    g = torch.Generator(device="cpu").manual_seed(seed)
    Q = B * qps
    q_idx = torch.randn(Q, 64, 128, generator=g).to(torch.bfloat16)
    w_idx = torch.rand(Q, 64, generator=g)
    keys = _keys(g, (B, n_cap, 128))
    # query positions: each sequence's queries end at its length
    q_pos = torch.tensor([lengths[b] - qps + j for b in range(B) for j in range(qps)], dtype=torch.int64)
    p = L.params(512, m, topk=k)
    codes = torch.empty(B, n_cap, 128, dtype=torch.uint8, device="cuda")
    scales = torch.empty(B, n_cap, dtype=torch.float32, device="cuda")
    L.csa_index_keys_pack(p, keys.cuda(), B * n_cap, 128, codes, scales)
    nb = L.csa_workspace_bytes(p, L.OP_INDEX_TOPK_FP8, B, Q, 64, 64, n_cap, 128)
    ws = L.workspace(nb)
    idx = torch.empty(Q, k, dtype=torch.int32, device="cuda")
    sc = torch.empty(Q, k, dtype=torch.float32, device="cuda")
    L.csa_index_topk_fp8(p, q_idx.cuda(), w_idx.cuda(), 64, 128, codes, scales, n_cap, B, Q,
                         q_pos.cuda(), idx, sc, ws, nb)
    torch.cuda.synchronize()
    L.csa_check_status(ws)
    gi, gs = idx.cpu().numpy(), sc.cpu().numpy()
    c_np, s_np = codes.cpu().numpy(), scales.cpu().numpy()
    qn = H.np_stored(q_idx)
    wn = w_idx.numpy().astype(np.float64)
    same = 0
    qs = range(Q) if sample is None else sample
    for q in qs:
        b = q // qps
        n = (int(q_pos[q]) + 1) // m
        scores = oracle.index_scores_fp8(qn[q], wn[q], c_np[b, :n], s_np[b, :n])
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
    same, n = _run(L, B=32, qps=1, n_cap=32768, lengths=[131072] * 32, k=1024, sample=[0, 13, 31])
    assert same >= n - 1
