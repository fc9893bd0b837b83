"""Pins of the oracle's FP8 indexer keys (one float32 scale per key row,
E4M3 codes) and of the indexer score over them: the packer against torch's
float8_e4m3fn cast, the score against the float32 indexer on inputs that
FP8 represents exactly, scale equivariance, and an all-zero row."""
import numpy as np
import torch

import oracle


def _representable_rows(rng, n, dI):
    """Rows of E4M3 grid values whose amax is exactly 448 (scale 1)."""
    codes = rng.integers(0, 126, size=(n, dI)).astype(np.uint8)
    codes |= (rng.integers(0, 2, size=(n, dI)) << 7).astype(np.uint8)
    vals = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float32).numpy()
    vals[:, 0] = 448.0 * np.where(rng.integers(0, 2, size=n) > 0, 1.0, -1.0)
    return vals.astype(np.float32)


def test_pack_matches_torch_cast():
    rng = np.random.default_rng(41)
    x = (rng.standard_normal((300, 128)) * rng.uniform(0.01, 50, size=(300, 1))).astype(np.float32)
    x[5] = 0.0
    codes, scales = oracle.pack_idx_keys_fp8(x)
    amax = np.abs(x).max(axis=1)
    want_scales = np.where(amax == 0, np.float32(1.0), (amax / np.float32(448.0)).astype(np.float32))
    assert np.array_equal(scales, want_scales.astype(np.float32))
    q = torch.from_numpy(x) / torch.from_numpy(scales)[:, None]          # float32 division
    ref = q.clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(codes, ref)


def test_scores_reduce_to_the_float32_indexer_when_fp8_is_exact():
    rng = np.random.default_rng(42)
    HI, dI, n = 8, 128, 64
    keys = _representable_rows(rng, n, dI)
    q = _representable_rows(rng, HI, dI)
    w = rng.uniform(0, 1, size=HI)
    codes, scales = oracle.pack_idx_keys_fp8(keys)
    assert np.all(scales == 1.0)
    got = oracle.index_scores_fp8(q, w, codes, scales)
    want = oracle.index_scores(q, w, keys)
    assert np.array_equal(got, want)
    assert np.count_nonzero(want) > n // 2


def test_scores_scale_with_a_key_row():
    rng = np.random.default_rng(43)
    HI, dI, n = 4, 128, 16
    keys = rng.standard_normal((n, dI)).astype(np.float32)
    q = rng.standard_normal((HI, dI)).astype(np.float32)
    w = rng.uniform(0, 1, size=HI)
    codes, scales = oracle.pack_idx_keys_fp8(keys)
    base = oracle.index_scores_fp8(q, w, codes, scales)
    keys2 = keys.copy()
    keys2[3] *= 8.0                       # a power of two: same codes, scale x 8
    codes2, scales2 = oracle.pack_idx_keys_fp8(keys2)
    assert np.array_equal(codes2, codes) and scales2[3] == scales[3] * 8
    got = oracle.index_scores_fp8(q, w, codes2, scales2)
    assert got[3] == base[3] * 8 and np.array_equal(np.delete(got, 3), np.delete(base, 3))


def test_all_zero_key_row_scores_zero():
    q = np.ones((2, 128), np.float32)
    keys = np.zeros((3, 128), np.float32)
    keys[1, 7] = -2.0
    codes, scales = oracle.pack_idx_keys_fp8(keys)
    assert scales[0] == 1.0 and not codes[0].any()
    s = oracle.index_scores_fp8(q, np.array([0.5, 0.25]), codes, scales)
    assert s[0] == 0.0 and s[1] == 0.0 and s[2] == 0.0   # relu of a negative dot is 0


def test_scores_scale_with_a_query_head():
    rng = np.random.default_rng(44)
    HI, dI, n = 4, 128, 16
    keys = rng.standard_normal((n, dI)).astype(np.float32)
    q = rng.standard_normal((HI, dI)).astype(np.float32)
    codes, scales = oracle.pack_idx_keys_fp8(keys)
    only = np.zeros(HI)
    only[2] = 1.0                        # the score of head 2 alone
    base = oracle.index_scores_fp8(q, only, codes, scales)
    q2 = q.copy()
    q2[2] *= 4.0                         # same codes, head scale x 4
    got = oracle.index_scores_fp8(q2, only, codes, scales)
    assert np.array_equal(got, base * 4) and np.count_nonzero(base) > 0
