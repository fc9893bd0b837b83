"""Failure detection on the GPU without a fault: a bounded wait that runs out.

Every wait inside the tensor-core kernels gives up after 2 s of wall time,
sets CSA_DEV_TIMEOUT in the caller's status word and makes every role of the
kernel leave its loop, with nothing in flight and TMEM freed.  Here the test
hook csa_test_withhold_indexer_loads keeps the lightning indexer's producer
from issuing any copy, so its MMA warps wait for tiles that never come.  The
kernel must end on its own within a few seconds, report the timeout through
csa_check_status, and leave the context usable: the next call, hook off, must
match the oracle.
"""
import time

import numpy as np
import pytest
import torch

import oracle
import workloads
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


def test_bounded_wait_expires_then_the_next_call_is_correct(L):
    w = workloads.CSA_DECODE_128K.replace(name="timeout", B=2, L_per_seq=(4096, 3001), topk=64)
    inp = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in workloads.generate(w).items()}
    p = L.params(w.D, w.m, topk=w.topk, window=w.W)
    ld = (w.n_cap + 127) // 128 * 128
    scores = torch.empty(w.Q, ld, dtype=torch.float32, device="cuda")
    ws = L.workspace(256)

    def score():
        L.csa_index_score(p, inp["q_idx"], inp["w_idx"], w.H_I, w.d_I, inp["keys"], w.n_cap, w.B, w.Q,
                          inp["q_pos"], scores, ld, ws, ws.numel())

    torch.cuda.synchronize()
    L.csa_test_withhold_indexer_loads(True)
    try:
        t0 = time.time()
        score()
        torch.cuda.synchronize()
        dt = time.time() - t0
    finally:
        L.csa_test_withhold_indexer_loads(False)
    with pytest.raises(L.CsaError) as ei:
        L.csa_check_status(ws)
    assert ei.value.status == 5
    assert L.csa_last_device_bits() & 0x8, "CSA_DEV_TIMEOUT expected"
    assert 1.5 <= dt < 30.0, dt  # the 2 s bound, not a hang
    L.csa_check_status(ws)       # cleared

    # the context is intact: the same call, hook off, scores as the oracle does
    score()
    torch.cuda.synchronize()
    L.csa_check_status(ws)
    got = scores.cpu().numpy()
    for b in range(w.B):
        n_av = w.lengths[b] // w.m
        ref = oracle.index_scores(H.np_stored(inp["q_idx"][b]), H.np_stored(inp["w_idx"][b]).astype(np.float64),
                                  H.np_stored(inp["keys"][b, :n_av]))
        assert np.allclose(got[b, :n_av], ref, rtol=1e-4, atol=1e-4)
        assert np.all(np.isneginf(got[b, n_av:w.n_cap]))
