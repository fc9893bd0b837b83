"""Consecutive decode steps over a ragged batch through DecodeLayer.step.

Every step appends each sequence's newest token (csa_decode_append: its raw-
ring slot, its window row in the window ring and, when it completes a block,
the block's cache entry) and attends at its position.  The loop runs at least
twice around the 128-row window ring, and every step is checked against the
oracle, which keeps its own state (rows by position, from its own compressor
["DeepSeek-V4百万上下文时代的开源宣言" §三.2 CSA "Step 1: KV 压缩"; 四项关键
Trick "Sliding Window"]): the window row and entry written (strict row
check), the top-k set (CSA), and the outputs and lse (bf16 tolerances).
"""
import numpy as np
import pytest
import torch

import oracle
from tests import harness as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from long_context_compressed_17_b300 import build
    build.build()
    oracle.build()


class _Spec:
    def __init__(self, kind, kv, m, steps, L0, topk=64):
        self.kind, self.kv_fmt, self.m, self.steps, self.L0 = kind, kv, m, steps, L0
        self.topk = topk if kind == "csa" else 0
        self.D, self.H, self.W, self.H_I, self.d_I = 512, 64, 128, 64, 128
        self.act, self.rope_dims, self.rope_base, self.eps = "bf16", 64, 10000.0, 1e-6
        self.softmax_scale = 0.0
        self.B = len(L0)


CASES = [
    _Spec("csa", "bf16", 4, 260, (1021, 514)),
    # 70+ complete blocks: the tensor-core attention; a dozen: the CUDA-core one
    _Spec("hca", "bf16", 128, 260, (128 * 70 + 37, 128 * 66 + 100)),
    _Spec("hca", "bf16", 128, 140, (128 * 9 + 37, 128 * 4 + 100)),
    _Spec("csa", "fp8m", 4, 140, (2050, 777)),
]


def _bits(t):
    return H.np_stored(t)


@pytest.mark.parametrize("sp", CASES, ids=["csa_bf16", "hca_bf16", "hca_bf16_few_blocks", "csa_fp8"])
def test_decode_loop_ring_ragged(sp):
    import long_context_compressed_17_b300 as L
    from long_context_compressed_17_b300.pipeline import DecodeLayer, LayerConfig, ring_order
    B, D, Hh, W, m = sp.B, sp.D, sp.H, sp.W, sp.m
    L0 = np.array(sp.L0)
    Lmax = int(L0.max()) + sp.steps
    n_cap = Lmax // m + 1
    g = torch.Generator(device="cpu").manual_seed(1234 + m)
    rnd = lambda *s: torch.randn(*s, generator=g)
    raw = rnd(B, Lmax, D).to(torch.bfloat16)                    # raw tokens of every position
    cache0 = rnd(B, n_cap, D)                                   # stand-ins for entries stored earlier
    win0 = rnd(B, W, D)                                         # window rows of positions L0-W .. L0-1
    keys = rnd(B, n_cap, sp.d_I).to(torch.bfloat16)
    sink = rnd(Hh)
    w_z = rnd(D) * 0.02
    bias = rnd(m) * 0.1
    if sp.kv_fmt == "bf16":
        cache0, win0 = cache0.to(torch.bfloat16), win0.to(torch.bfloat16)
    cfg = LayerConfig(D=D, H=Hh, m=m, W=W, topk=sp.topk, H_I=sp.H_I, d_I=sp.d_I, kv=sp.kv_fmt)
    layer = DecodeLayer(cfg, B, n_cap, W)
    # GPU state: the same draws, packed by the library for FP8 rows; window and
    # raw tokens of the current block laid out as rings
    cache = H.gpu_pack(sp, cache0.cuda())
    window = ring_order(H.gpu_pack(sp, win0.cuda()), (L0 - W).tolist(), W)
    raw_ring = torch.zeros(B, m, D, dtype=torch.bfloat16, device="cuda")
    for b in range(B):
        for p in range(int(L0[b]) - int(L0[b]) % m, int(L0[b])):
            raw_ring[b, p % m] = raw[b, p].cuda()
    # oracle state: stored rows by entry / by position
    fmt = H._ORC_FMT[sp.kv_fmt]
    cache_o = [H.oracle_stored_rows(sp, cache0[b]) for b in range(B)]
    win_o = [{int(L0[b]) - W + r: H.oracle_stored_rows(sp, win0[b, r:r + 1])[0] for r in range(W)}
             for b in range(B)]
    raw_np = _bits(raw)
    w_z_np = w_z.numpy().astype(np.float64)
    bias_np = bias.numpy().astype(np.float64)
    sink_np = sink.numpy().astype(np.float64)
    dev = {k: v.cuda() for k, v in dict(keys=keys, sink=sink, w_z=w_z, bias=bias).items()}
    worst = 0.0
    for t in range(sp.steps):
        pos = torch.tensor(L0 + t, dtype=torch.int64)
        q = rnd(B, Hh, D).to(torch.bfloat16)
        q_idx = rnd(B, sp.H_I, sp.d_I).to(torch.bfloat16)
        w_idx = torch.rand(B, sp.H_I, generator=g)
        kv_tok = raw[torch.arange(B), pos].contiguous()
        out, lse = layer.step(kv_tok.cuda(), pos.cuda(), dev["w_z"], dev["bias"], raw_ring, q.cuda(), cache,
                              window, dev["sink"], q_idx=q_idx.cuda(), w_idx=w_idx.cuda(), keys=dev["keys"])
        torch.cuda.synchronize()
        L.csa_check_status(layer.ws)
        out_g, lse_g = out.float().cpu().numpy(), lse.cpu().numpy()
        idx_g = layer.topk_idx.cpu().numpy() if sp.topk else None
        for b in range(B):
            p = int(pos[b])
            # the window row written this step
            wrow = oracle.compress(raw_np[b, p:p + 1], p, 1, w_z_np, bias_np[:1], sp.rope_dims,
                                   sp.rope_base, sp.eps)
            H.check_stored_rows(sp, window[b, p % W], wrow, "step %d seq %d window row" % (t, b))
            win_o[b][p] = _bits(window[b, p % W]) if sp.kv_fmt == "fp8m" else oracle.store_rows(wrow, fmt)[0]
            win_o[b].pop(p - W, None)
            # the entry of the block this token completes
            if (p + 1) % m == 0:
                e = (p + 1) // m - 1
                ent = oracle.compress(raw_np[b, p + 1 - m:p + 1], p + 1 - m, m, w_z_np, bias_np, sp.rope_dims,
                                      sp.rope_base, sp.eps)
                H.check_stored_rows(sp, cache[b, e], ent, "step %d seq %d entry %d" % (t, b, e))
                cache_o[b][e] = _bits(cache[b, e]) if sp.kv_fmt == "fp8m" else oracle.store_rows(ent, fmt)[0]
            lo = max(0, p - W + 1)
            win_lin = np.stack([win_o[b][r] for r in range(lo, p + 1)])
            n_av = (p + 1) // m
            qb = _bits(q[b])
            if sp.topk:
                scores = oracle.index_scores(_bits(q_idx[b]), w_idx[b].numpy().astype(np.float64),
                                             _bits(keys[b, :n_av]))
                H.check_topk_set(idx_g[b], scores, sp.topk, "step %d seq %d" % (t, b))
                sel = idx_g[b][idx_g[b] >= 0]
                rows = np.concatenate([oracle.read_rows(cache_o[b][sel], D), oracle.read_rows(win_lin, D)])
                out_o, lse_o = oracle.attend_rows(qb, p, rows, sink_np, rope_dims=sp.rope_dims,
                                                  base=sp.rope_base, eps=sp.eps)
            else:
                out_o, lse_o = oracle.attend_query(qb, p, m, cache_o[b][:n_av], D, None, win_lin, lo, W,
                                                   sink_np, rope_dims=sp.rope_dims, base=sp.rope_base,
                                                   eps=sp.eps)
            mx, _ = H.assert_close(out_g[b], out_o, "bf16", "step %d seq %d out" % (t, b))
            assert np.max(np.abs(lse_g[b] - lse_o)) <= H.LSE_TOL["bf16"], "step %d seq %d lse" % (t, b)
            worst = max(worst, mx)
    n_exc = sum(c for what, n, c in H.NEAR_MID_COUNTS if what.startswith("step"))
    print("decode loop %s/%s: %d steps x %d sequences, worst max-abs %.3g, near-midpoint codes %d"
          % (sp.kind, sp.kv_fmt, sp.steps, B, worst, n_exc))
