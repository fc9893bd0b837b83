"""GPU top-k selection against the oracle's exact selection (score
descending, lower block index on ties), bit-exact, on score matrices built to
stress it: heavy exact ties (small integers, +0 and -0), several chunks with a
ragged last chunk, a single chunk, many queries at once, and k larger than the
number of complete blocks."""
import numpy as np
import pytest
import torch

import oracle

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


def _scores(rng, Q, n_cap, n_av):
    s = rng.integers(-3, 40, size=(Q, n_cap)).astype(np.float32)
    s[:, ::7] = 0.0
    s[:, 3::11] = -0.0
    for q in range(Q):
        s[q, n_av[q]:] = -np.inf  # blocks not yet complete, as the indexer writes them
    return s


def _check(L, s, n_av, m, k):
    Q, n_cap = s.shape
    ld = (n_cap + 127) // 128 * 128
    dev = torch.full((Q, ld), float("nan"), dtype=torch.float32, device="cuda")
    dev[:, :n_cap] = torch.from_numpy(s).cuda()
    # a query at the last token of block n-1 sees exactly n complete blocks
    q_pos = torch.tensor([n * m - 1 for n in n_av], dtype=torch.int64, device="cuda")
    idx = torch.full((Q, k), -7, dtype=torch.int32, device="cuda")
    sc = torch.zeros(Q, k, dtype=torch.float32, device="cuda")
    p = L.params(512, m, topk=k)
    L.csa_topk_select(p, dev, ld, n_cap, Q, q_pos, idx, sc)
    torch.cuda.synchronize()
    gi, gs = idx.cpu().numpy(), sc.cpu().numpy()
    for q in range(Q):
        n = n_av[q]
        kk = min(k, n)
        ref, _ = oracle.topk(s[q, :n].astype(np.float64), k)
        want = np.sort(np.asarray(ref[:kk]))
        assert np.array_equal(gi[q, :kk], want), "query %d: selection differs" % q
        assert np.all(gi[q, kk:] == -1), "query %d: padding" % q
        np.testing.assert_array_equal(gs[q, :kk], s[q, want])


@pytest.mark.parametrize("k", [1024, 2048])
def test_topk_several_chunks_ragged_ties(L, k):
    rng = np.random.default_rng(5)
    n_av = [40000, 25001, 9000, 300]
    _check(L, _scores(rng, 4, 40000, n_av), n_av, 4, k)


def test_topk_many_queries_one_chunk_each(L):
    rng = np.random.default_rng(6)
    Q = 400
    n_av = list(rng.integers(500, 20000, size=Q))
    _check(L, _scores(rng, Q, 20000, n_av), n_av, 4, 1024)


def test_topk_one_million_blocks(L):
    rng = np.random.default_rng(7)
    n_av = [262144, 200000]
    _check(L, _scores(rng, 2, 262144, n_av), n_av, 4, 1024)


def test_topk_continuous_scores_at_the_chunk_boundary(L):
    """Distinct float scores; 32768 blocks fit one chunk, 32769 need two."""
    rng = np.random.default_rng(8)
    n_av = [32768, 32769, 32767]
    s = (rng.standard_normal((3, 32769)) * 30 + 150).astype(np.float32)
    for q in range(3):
        s[q, n_av[q]:] = -np.inf
    _check(L, s, n_av, 4, 1024)


def test_topk_all_scores_equal(L):
    """One distinct key: the lowest indices are kept."""
    n_av = [5000, 70000]
    s = np.full((2, 70000), 2.5, dtype=np.float32)
    s[0, 5000:] = -np.inf
    _check(L, s, n_av, 4, 1024)
