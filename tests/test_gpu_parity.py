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
from tests.harness import _to_cuda, decode_parity, prefill_parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from long_context_compressed_17_b300 import build
    build.build()
    oracle.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


SMALL_CSA = workloads.CSA_DECODE_128K.replace(
    name="csa_decode_small", B=4, L_per_seq=(5000, 4096, 2999, 30), topk=100)
SMALL_HCA = workloads.HCA_DECODE_1M.replace(
    name="hca_decode_small", B=3, L_per_seq=(128 * 37, 128 * 20 + 64, 100))
SMALL_FP8 = workloads.CSA_DECODE_1M_FP8.replace(
    name="csa_decode_fp8_small", B=2, L_per_seq=(8192, 6001), topk=200)


def test_csa_decode_small():
    st = decode_parity(SMALL_CSA)
    assert len(st) == 4


@pytest.mark.parametrize("B", [37, 75, 148, 149])
def test_csa_decode_tile_deals(B):
    """Batches around the SM count: with no more queries than SMs each query's
    tiles are split over its own CTAs (37: four CTAs a query, one tile each;
    75: one or two CTAs a query; 148: every query whole in one CTA), beyond it
    (149) the tiles of all queries are dealt in balanced ranges that cut
    queries; the combine follows either deal.  Sampled sequences."""
    w = SMALL_CSA.replace(name="csa_decode_deal_%d" % B, B=B,
                          L_per_seq=tuple(600 + 37 * b for b in range(B)), topk=100)
    decode_parity(w, seqs=sorted({0, 1, B // 2, B - 2, B - 1}))


def test_csa_decode_small_sink_neginf():
    w = SMALL_CSA.replace(sink="neginf", B=2, L_per_seq=(3000, 1024))
    decode_parity(w)


def test_hca_decode_small():
    decode_parity(SMALL_HCA)


SMALL_HCA_TILES = workloads.HCA_DECODE_1M.replace(
    name="hca_decode_tiles", B=3, L_per_seq=(128 * 300, 128 * 170 + 64, 128 * 129 - 1))


def test_hca_decode_several_tiles():
    """Caches of 300, 170 and 128 blocks: several 128-row tiles, a ragged last tile."""
    decode_parity(SMALL_HCA_TILES)


def test_hca_decode_query_cost_deal():
    """Six sequences of 100 to 160 cache tiles on the SMs: each query's tiles
    span several CTAs, and a CTA whose range starts a query takes five tiles
    fewer than one that does not (a query's start counted as five tiles);
    ragged lengths leave the shorter queries' last tiles dead.  Every
    sequence checked."""
    L = (128 * 64 * 160, 128 * 64 * 150 + 100, 128 * 9000, 128 * 64 * 100 + 7, 128 * 64 * 131 - 1, 128 * 64 * 120)
    w = workloads.HCA_DECODE_1M.replace(name="hca_decode_cost_deal", B=6, L_per_seq=L)
    assert len(decode_parity(w)) == 6


def _ramp_toward_q(inp, t_max):
    """Every query head is 1 on dims 0..127 and 0 elsewhere (unrotated dims), so
    its normalised form is exactly 2 there -- exact in bf16 as well.  Cache
    row j gains t_max * j / n along u = that direction / sqrt(128).  Its logit
    is then about scale * 2 * sqrt(128) * t_j plus noise, climbing along the
    row list, so the running softmax reference is raised several times per
    query; the output stays of order 1."""
    dev = inp["q"].device
    D = inp["q"].shape[-1]
    q = torch.zeros(D, device=dev)
    q[:128] = 1.0
    inp["q"].copy_(q.expand_as(inp["q"]).to(inp["q"].dtype))
    u = q / 128 ** 0.5
    n = inp["cache"].shape[1]
    t = t_max * torch.arange(n, device=dev, dtype=torch.float32) / n
    inp["cache"].copy_((inp["cache"].float() + t[None, :, None] * u).to(inp["cache"].dtype))


def test_hca_decode_growing_logits_rescale():
    # softmax scale 3/sqrt(D): 4 cache tiles whose maxima climb by ~9 nats each
    w = SMALL_HCA_TILES.replace(name="hca_ramp", B=2, L_per_seq=(128 * 500, 128 * 380),
                                softmax_scale=3.0 / 512 ** 0.5)
    decode_parity(w, mutate=lambda inp: _ramp_toward_q(inp, 12.0))


def test_csa_decode_growing_logits_rescale():
    # the selected blocks are listed in index order, so their logits climb too
    w = SMALL_CSA.replace(name="csa_ramp", B=2, L_per_seq=(20000, 9001), topk=600,
                          softmax_scale=3.0 / 512 ** 0.5)
    decode_parity(w, mutate=lambda inp: _ramp_toward_q(inp, 12.0))


def test_hca_decode_fp8_small():
    """FP8 rows on the tensor-core path, in both dequantised layouts: a 37-block
    capacity (fewer stored rows than tile rows: every stored row) and a
    128-block one (the rows of each query's tiles)."""
    decode_parity(SMALL_HCA.replace(name="hca_fp8_small", kv_fmt="fp8m"))
    decode_parity(SMALL_HCA.replace(name="hca_fp8_rows", kv_fmt="fp8m", B=2,
                                    L_per_seq=(128 * 128, 128 * 50 + 3)))


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


def test_csa_prefill_bf16_small():
    w = workloads.CSA_CHUNKED_PREFILL.replace(name="prefill_small", T_cached=512, T_new=300,
                                              topk=64)
    n_same, n = prefill_parity(w)
    assert n_same >= n - 2


def test_csa_prefill_fp8_small():
    w = workloads.CSA_CHUNKED_PREFILL.replace(name="prefill_fp8_small", kv_fmt="fp8m",
                                              T_cached=512, T_new=300, topk=64)
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


@pytest.mark.parametrize("m,kv", [(4, "bf16"), (128, "bf16"), (4, "fp8m"), (128, "fp8m")])
def test_append_matches_two_compress_calls(m, kv):
    """csa_append (one launch) writes the same bits as csa_compress over the
    block plus csa_compress with ratio 1 over its last token."""
    import long_context_compressed_17_b300 as L
    from long_context_compressed_17_b300.pipeline import LayerConfig
    B, D, n_cap, n_win = 5, 512, 40, 16
    cfg = LayerConfig(D=D, H=64, m=m, kv=kv)
    g = torch.Generator(device="cpu").manual_seed(21 + m)
    kv_new = (torch.randn(B, m, D, generator=g) * 2).to(torch.bfloat16).cuda()
    w_z = (torch.randn(D, generator=g) * 0.02).cuda()
    bias = (torch.randn(m, generator=g) * 0.1).cuda()
    pos0 = 37 * m
    e, wr = 11, 9
    outs = []
    for fused in (True, False):
        cache = cfg.empty_rows(B, n_cap)
        window = cfg.empty_rows(B, n_win)
        rb = cache.shape[-1] * cache.element_size()
        if fused:
            L.csa_append(cfg.params(), kv_new, B, m, pos0, w_z, bias, cache.data_ptr() + e * rb,
                         n_cap, window.data_ptr() + wr * rb, n_win)
        else:
            L.csa_compress(cfg.params(), kv_new, B, m, m, pos0, w_z, bias,
                           cache.data_ptr() + e * rb, n_cap)
            L.csa_compress(cfg.params(ratio=1), kv_new[:, m - 1:].data_ptr(), B, 1, m,
                           pos0 + m - 1, w_z, bias, window.data_ptr() + wr * rb, n_win)
        torch.cuda.synchronize()
        outs.append((cache.cpu(), window.cpu()))
    assert torch.equal(outs[0][0], outs[1][0]), "entries differ"
    assert torch.equal(outs[0][1], outs[1][1]), "window rows differ"
    assert outs[0][0][:, e].abs().sum() > 0 and outs[0][1][:, wr].abs().sum() > 0


@pytest.mark.parametrize("m,kv", [(4, "bf16"), (128, "bf16"), (4, "fp8m"), (128, "fp8m")])
def test_decode_append_matches_the_fused_append(m, kv):
    """csa_decode_append over a ragged batch: sequences whose newest token
    completes a block get the same entry and window row bits as csa_append
    over that block; the others get only their window row (and raw-ring slot),
    their cache entries untouched."""
    import long_context_compressed_17_b300 as L
    from long_context_compressed_17_b300.pipeline import DecodeLayer, LayerConfig
    B, D, n_cap, n_win = 4, 512, 40, 128
    cfg = LayerConfig(D=D, H=64, m=m, kv=kv)
    g = torch.Generator(device="cpu").manual_seed(31 + m)
    blk = (torch.randn(B, m, D, generator=g) * 2).to(torch.bfloat16).cuda()
    w_z = (torch.randn(D, generator=g) * 0.02).cuda()
    bias = (torch.randn(m, generator=g) * 0.1).cuda()
    # sequences 0 and 2 complete block 11 / 30; 1 and 3 stop inside a block
    pos = torch.tensor([12 * m - 1, 7 * m + 2, 31 * m - 1, 3 * m], dtype=torch.int64)
    layer = DecodeLayer(cfg, B, n_cap, n_win)
    raw_ring, cache, window = layer.new_state()
    for b in range(B):  # the block's tokens before the newest one, in their ring slots
        p0 = int(pos[b]) - int(pos[b]) % m
        for t in range(p0, int(pos[b])):
            raw_ring[b, t % m] = blk[b, t - p0]
    kv_tok = torch.stack([blk[b, int(pos[b]) % m] for b in range(B)]).contiguous()
    layer.append(kv_tok, pos.cuda(), w_z, bias, raw_ring, cache, window)
    torch.cuda.synchronize()
    L.csa_check_status(layer.ws)
    rb = cache.shape[-1] * cache.element_size()
    for b in range(B):
        t = int(pos[b])
        assert torch.equal(raw_ring[b, t % m], blk[b, t % m]), "raw ring slot"
        win_ref = cfg.empty_rows(1, 1)
        if (t + 1) % m == 0:
            ent_ref = cfg.empty_rows(1, 1)
            L.csa_append(cfg.params(), blk[b:b + 1], 1, m, t + 1 - m, w_z, bias, ent_ref, 1, win_ref, 1)
            torch.cuda.synchronize()
            assert torch.equal(cache[b, (t + 1) // m - 1].cpu(), ent_ref[0, 0].cpu()), "entry seq %d" % b
            assert int((cache[b].view(torch.uint8) != 0).any(dim=-1).sum()) == 1
        else:
            L.csa_compress(cfg.params(ratio=1), kv_tok[b:b + 1], 1, 1, 1, t, w_z, bias, win_ref, 1)
            torch.cuda.synchronize()
            assert not bool((cache[b].view(torch.uint8) != 0).any()), "no entry for an incomplete block"
        assert torch.equal(window[b, t % n_win].cpu(), win_ref[0, 0].cpu()), "window row seq %d" % b
    assert rb > 0


def test_decode_append_flags_a_position_beyond_the_cache():
    import long_context_compressed_17_b300 as L
    from long_context_compressed_17_b300.pipeline import DecodeLayer, LayerConfig
    cfg = LayerConfig(D=512, H=64, m=4)
    layer = DecodeLayer(cfg, 2, 8, 128)
    raw_ring, cache, window = layer.new_state()
    tok = torch.randn(2, 512, device="cuda").to(torch.bfloat16)
    pos = torch.tensor([8 * 4 + 3, 5], dtype=torch.int64, device="cuda")  # entry 8 of an 8-entry cache
    layer.append(tok, pos, torch.zeros(512, device="cuda"), torch.zeros(4, device="cuda"), raw_ring, cache,
                 window)
    with pytest.raises(L.CsaError):
        L.csa_check_status(layer.ws)
    assert L.csa_last_device_bits() & 0x4
    assert not bool((cache.view(torch.uint8) != 0).any())
    assert bool((window[1, 5].view(torch.uint8) != 0).any())  # the other sequence proceeds


@pytest.mark.parametrize("kv", ["bf16", "fp8m"])
def test_decode_step_with_side_stream_append_matches_sequential(kv):
    """DecodeLayer.step runs the CSA append on a side stream beside the
    indexer and top-k; outputs, cache and window rows equal those of the
    sequential append-then-attend, bit for bit (a ragged batch, two of whose
    sequences complete a block)."""
    from long_context_compressed_17_b300.pipeline import DecodeLayer, ring_order
    w = SMALL_CSA.replace(name="csa_step_overlap", B=4, L_per_seq=(8192, 8191, 4096, 3001), kv_fmt=kv)
    inp = _to_cuda(workloads.generate(w))
    cfg = H.cfg_of(w)
    lens = torch.tensor(w.lengths, dtype=torch.int64)
    kv_tok = inp["kv_new"][:, w.m - 1].contiguous()
    res = []
    for overlapped in (False, True):
        cache = H.gpu_pack(w, inp["cache"])
        window = ring_order(H.gpu_pack(w, inp["window"]), inp["win_pos0"].cpu(), w.W)
        raw_ring = ring_order(inp["kv_new"], (lens - w.m).tolist(), w.m)
        layer = DecodeLayer(cfg, w.B, w.n_cap, w.W)
        if overlapped:
            out, lse = layer.step(kv_tok, inp["q_pos"], inp["w_z"], inp["bias"], raw_ring, inp["q"], cache,
                                  window, inp["sink"], q_idx=inp["q_idx"], w_idx=inp["w_idx"], keys=inp["keys"])
        else:
            layer.append(kv_tok, inp["q_pos"], inp["w_z"], inp["bias"], raw_ring, cache, window)
            out, lse = layer.attend(inp["q"], cache, window, inp["q_pos"], None, inp["sink"],
                                    q_idx=inp["q_idx"], w_idx=inp["w_idx"], keys=inp["keys"])
        torch.cuda.synchronize()
        import long_context_compressed_17_b300 as L
        L.csa_check_status(layer.ws)
        res.append([t.clone() for t in (out, lse, cache, window, layer.topk_idx)])
    for a, b, what in zip(res[0], res[1], ("out", "lse", "cache", "window", "topk_idx")):
        assert torch.equal(a.view(torch.uint8) if a.dtype != torch.uint8 else a,
                           b.view(torch.uint8) if b.dtype != torch.uint8 else b), what
