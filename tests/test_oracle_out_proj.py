"""Pins of the oracle's grouped output projection ["DeepSeek-V4百万上下文时代的
开源宣言" §三.2 CSA "Step 4: Grouped Output Projection"]: the heads projected
in G groups, each by its own matrix.  Checked against a dense projection with
the block-diagonal weight assembled explicitly, a one-hot closed form, the two
extreme group counts, and invariance under a permutation of a group's heads
with their weight rows."""
import numpy as np

import oracle


def _draw(rng, Q, H, D, G, d_g):
    o = rng.standard_normal((Q, H, D))
    w = rng.standard_normal((G, d_g, H // G * D)) / np.sqrt(H // G * D)
    return o, w


def test_equals_dense_projection_with_block_diagonal_weight():
    rng = np.random.default_rng(81)
    Q, H, D, G, d_g = 5, 8, 16, 4, 6
    o, w = _draw(rng, Q, H, D, G, d_g)
    K = H // G * D
    full = np.zeros((H * D, G * d_g))
    for g in range(G):
        full[g * K:(g + 1) * K, g * d_g:(g + 1) * d_g] = w[g].T
    want = o.reshape(Q, H * D) @ full
    assert np.allclose(oracle.grouped_out_proj(o, w, G), want, rtol=1e-12, atol=1e-12)


def test_one_hot_head_output_selects_one_weight_row_of_its_group():
    rng = np.random.default_rng(82)
    Q, H, D, G, d_g = 1, 8, 4, 2, 3
    _, w = _draw(rng, Q, H, D, G, d_g)
    for h, d in [(0, 0), (3, 2), (4, 1), (7, 3)]:
        o = np.zeros((1, H, D))
        o[0, h, d] = 2.5
        g = h // (H // G)
        col = (h - g * (H // G)) * D + d
        want = np.zeros(G * d_g)
        want[g * d_g:(g + 1) * d_g] = 2.5 * w[g, :, col]
        assert np.array_equal(oracle.grouped_out_proj(o, w, G)[0], want)


def test_one_group_is_a_dense_projection_and_h_groups_project_each_head():
    rng = np.random.default_rng(83)
    Q, H, D, d = 3, 4, 8, 5
    o = rng.standard_normal((Q, H, D))
    w1 = rng.standard_normal((1, d, H * D))
    assert np.allclose(oracle.grouped_out_proj(o, w1, 1), o.reshape(Q, -1) @ w1[0].T, rtol=1e-12)
    wh = rng.standard_normal((H, d, D))
    got = oracle.grouped_out_proj(o, wh, H)
    for h in range(H):
        assert np.allclose(got[:, h * d:(h + 1) * d], o[:, h, :] @ wh[h].T, rtol=1e-12)


def test_permuting_a_groups_heads_with_their_weight_rows_changes_nothing():
    rng = np.random.default_rng(84)
    Q, H, D, G, d_g = 4, 8, 8, 2, 5
    o, w = _draw(rng, Q, H, D, G, d_g)
    perm = np.array([2, 0, 3, 1])  # heads of group 0
    o2 = o.copy()
    o2[:, :4] = o[:, perm]
    w2 = w.copy()
    blocks = w[0].reshape(d_g, 4, D)
    w2[0] = blocks[:, perm].reshape(d_g, 4 * D)
    assert np.allclose(oracle.grouped_out_proj(o2, w2, G), oracle.grouped_out_proj(o, w, G), rtol=1e-12)


def test_reads_bf16_bits_exactly():
    import torch
    rng = np.random.default_rng(85)
    o = rng.standard_normal((2, 4, 8)).astype(np.float32)
    w = rng.standard_normal((2, 3, 16)).astype(np.float32)
    ob = torch.from_numpy(o).to(torch.bfloat16)
    wb = torch.from_numpy(w).to(torch.bfloat16)
    got = oracle.grouped_out_proj(ob.view(torch.int16).numpy().view(np.uint16),
                                  wb.view(torch.int16).numpy().view(np.uint16), 2)
    want = oracle.grouped_out_proj(ob.double().numpy(), wb.double().numpy(), 2)
    assert np.array_equal(got, want)
