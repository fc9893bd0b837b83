"""csa_index_topk_noalloc: the indexer + top-k step for callers that cannot
allocate device memory (a plug-in whose host framework owns every device
allocation, or a latency-critical path that cannot risk the synchronisation an
allocation may cause).  Its scores live in a scratch array inside the library,
so the checks here are: it agrees with csa_index_topk (which uses a caller
workspace) on three calls in a row with different shapes (the last one large
enough for the chunked selection), it rejects requests
larger than the scratch, and it reports device status through its own output.

This file is named to be collected last.
"""
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from long_context_compressed_17_b300 import build
    build.build()
    import long_context_compressed_17_b300 as pkg
    return pkg


def _inputs(w):
    inp = {k: (v.cuda() if isinstance(v, torch.Tensor) else v)
           for k, v in workloads.generate(w).items()}
    return inp


def _with_workspace(L, w, p, inp):
    nb = L.csa_workspace_bytes(p, L.OP_INDEX_TOPK, w.B, w.Q, w.H, w.H_I, w.n_cap, w.W)
    ws = L.workspace(nb)
    idx = torch.empty(w.Q, w.topk, dtype=torch.int32, device="cuda")
    sc = torch.empty(w.Q, w.topk, dtype=torch.float32, device="cuda")
    L.csa_index_topk(p, inp["q_idx"], inp["w_idx"], w.H_I, w.d_I, inp["keys"], w.n_cap, w.B, w.Q,
                     inp["q_pos"], idx, sc, ws, ws.numel())
    torch.cuda.synchronize()
    L.csa_check_status(ws)
    return idx, sc


def _without(L, w, p, inp, q_pos=None):
    idx = torch.full((w.Q, w.topk), -7, dtype=torch.int32, device="cuda")
    sc = torch.zeros(w.Q, w.topk, dtype=torch.float32, device="cuda")
    status = torch.full((4,), 0xFFFF, dtype=torch.int32, device="cuda")
    L.csa_index_topk_noalloc(p, inp["q_idx"], inp["w_idx"], w.H_I, w.d_I, inp["keys"], w.n_cap,
                             w.B, w.Q, inp["q_pos"] if q_pos is None else q_pos, idx, sc, status)
    torch.cuda.synchronize()
    return idx, sc, int(status[0].item())


CALLS = [
    workloads.CSA_DECODE_128K.replace(name="noalloc_a", B=3, L_per_seq=(5000, 4096, 2999),
                                      topk=100),
    workloads.CSA_DECODE_128K.replace(name="noalloc_b", seed=7, B=2, L_per_seq=(3001, 777),
                                      topk=50, H_I=32),
    # more than 32768 blocks: the selection runs in chunks whose candidates are
    # written over the scores (here the shared scratch) and merged
    workloads.CSA_DECODE_128K.replace(name="noalloc_c", seed=8, B=2, L_per_seq=(160000, 140001),
                                      topk=1024),
]


def test_noalloc_matches_workspace_entry_point_on_calls_in_a_row(L):
    for w in CALLS:  # calls in a row: the second smaller than the first, the third chunked
        p = L.params(w.D, w.m, topk=w.topk, window=w.W, act=w.act, kv=w.kv_fmt)
        inp = _inputs(w)
        ref_idx, ref_sc = _with_workspace(L, w, p, inp)
        idx, sc, status = _without(L, w, p, inp)
        assert status == 0
        assert torch.equal(idx, ref_idx), w.name
        # same kernels on the same inputs: scores agree exactly (tolerance kept for clarity)
        assert torch.allclose(sc, ref_sc, rtol=1e-6, atol=0), w.name


def test_noalloc_rejects_requests_beyond_the_scratch(L):
    w = CALLS[0]
    p = L.params(w.D, w.m, topk=w.topk)
    n_cap = 4194304 // 2 + 1  # two queries need more than 4194304 scores after padding to 128
    fake = 1 << 20            # never dereferenced: the size check fails first
    with pytest.raises(L.CsaError) as ei:
        L.csa_index_topk_noalloc(p, fake, fake, 64, 128, fake, n_cap, 2, 2, fake, fake, None,
                                 None)
    assert ei.value.status == 1 and "scratch" in L.csa_last_error()


def test_noalloc_reports_device_status(L):
    w = CALLS[1]
    p = L.params(w.D, w.m, topk=w.topk, window=w.W)
    inp = _inputs(w)
    far = inp["q_pos"].clone()
    far[0] = 4 * w.n_cap + 100  # more complete blocks than the cache holds
    _, _, status = _without(L, w, p, inp, q_pos=far)
    assert status & 0x4
    _, _, status = _without(L, w, p, inp)  # cleared by the next call
    assert status == 0
