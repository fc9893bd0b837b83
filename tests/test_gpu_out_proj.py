"""GPU parity of the grouped output projection ["DeepSeek-V4百万上下文时代的开源
宣言" §三.2 CSA "Step 4: Grouped Output Projection"] against the oracle:
decode-sized (32 queries, narrow tiles streaming the weights; unsplit, and
with K split over four CTAs a group whose float32 products are summed in the
workspace), prefill-sized with a ragged last query tile (wide tiles), and a
small odd shape.  Every bf16
output must be the rounding of a value within float32 accumulation noise of
the oracle's double result (so it equals the rounded oracle except near a
rounding midpoint), and the outputs meet the bf16 tolerances."""
import numpy as np
import pytest
import torch

import oracle
from tests import harness as hn

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from long_context_compressed_17_b300 import build
    build.build()
    import long_context_compressed_17_b300 as pkg
    return pkg


def _case(L, Q, H, D, G, d_g, seed, split=False):
    g = torch.Generator(device="cpu").manual_seed(seed)
    K = H // G * D
    o = torch.randn(Q, H, D, generator=g).to(torch.bfloat16)
    w = (torch.randn(G, d_g, K, generator=g) / K ** 0.5).to(torch.bfloat16)
    out = torch.full((Q, G * d_g), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = L.workspace(L.csa_grouped_out_proj_ws_bytes(Q, G, d_g) if split else 256)
    L.csa_grouped_out_proj(o.cuda(), Q, H, D, G, w.cuda(), d_g, out, ws, ws.numel())
    torch.cuda.synchronize()
    L.csa_check_status(ws)
    ref = oracle.grouped_out_proj(hn.np_stored(o), hn.np_stored(w), G)
    got = out.float().cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(got))
    hn.assert_close(got, ref, "bf16", "grouped projection")
    # every output is the bf16 rounding of a value within float32 accumulation
    # noise of the oracle's (4 sqrt(K) 2^-24 sum |x w|): it equals the rounded
    # oracle except where the oracle's value lies that close to a midpoint
    absum = oracle.grouped_out_proj(np.abs(hn.np_stored(o.float())), np.abs(hn.np_stored(w.float())), G)
    tol = 4.0 * (H // G * D) ** 0.5 * 2.0 ** -24 * absum
    assert np.all(hn._within_rounding(got, ref, tol, hn._bf16_round)), "outputs beyond float32 noise"
    ref_b = hn._bf16_round(ref)
    n_diff = int((got != ref_b).sum())
    assert n_diff <= 0.01 * got.size
    return n_diff


def test_decode_sized(L):
    _case(L, Q=32, H=64, D=512, G=8, d_g=512, seed=91)


def test_decode_sized_split_k(L):
    _case(L, Q=32, H=64, D=512, G=8, d_g=512, seed=94, split=True)
    _case(L, Q=7, H=8, D=128, G=2, d_g=128, seed=95, split=True)  # K = 512: one step a CTA


def test_prefill_sized_with_a_ragged_tile(L):
    _case(L, Q=300, H=64, D=512, G=8, d_g=512, seed=92)


def test_small_odd_shape(L):
    _case(L, Q=5, H=8, D=128, G=2, d_g=64, seed=93)
