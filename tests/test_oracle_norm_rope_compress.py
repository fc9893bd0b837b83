"""Oracle pins: Q/KV RMSNorm, partial RoPE and the block compressor.

Pages: "DeepSeek-V4百万上下文时代的开源宣言" §三.2, CSA "Step 1: KV 压缩" and
"四项关键 Trick" (Q/KV Normalization, Partial RoPE on the last 64 dims);
"DeepSeek-V4 技术报告深度解析" §2.1.4.

Independent forms used here: RoPE as multiplication of complex pairs by
exp(i p theta_j) (the RoFormer definition), RMSNorm through its closed-form
norm, pooling through closed forms for special blocks.
"""
import math

import numpy as np
import pytest


def rope_complex(x, pos, R=64, base=10000.0):
    x = np.array(x, dtype=np.float64)
    D = x.shape[-1]
    z = x[..., D - R::2] + 1j * x[..., D - R + 1::2]
    theta = base ** (-np.arange(R // 2) * 2.0 / R)
    z = z * np.exp(1j * pos * theta)
    out = x.copy()
    out[..., D - R::2] = z.real
    out[..., D - R + 1::2] = z.imag
    return out


def rms_closed(x, eps=1e-6):
    x = np.asarray(x, dtype=np.float64)
    return x / math.sqrt(float(np.mean(x * x)) + eps)


# ---------------------------------------------------------------- RMSNorm
def test_rmsnorm_norm_closed_form(orc):
    rng = np.random.default_rng(0)
    for D in (64, 128, 512):
        x = rng.standard_normal(D) * 3.0
        y = orc.rmsnorm(x, 1e-6)
        ms = np.mean(x * x)
        assert abs(np.dot(y, y) - D * ms / (ms + 1e-6)) < 1e-9 * D
        # direction preserved: y is a positive multiple of x
        c = y / x
        assert np.allclose(c, c[0], rtol=1e-13) and c[0] > 0


def test_rmsnorm_constant_vector_and_eps(orc):
    y = orc.rmsnorm(np.full(8, 0.5), 0.25)
    assert np.allclose(y, 0.5 / math.sqrt(0.25 + 0.25), rtol=1e-15)
    y = orc.rmsnorm(np.zeros(16), 1e-6)
    assert np.all(y == 0)


# ---------------------------------------------------------------- RoPE
def test_rope_matches_complex_rotation(orc):
    rng = np.random.default_rng(1)
    for D in (128, 512):
        for pos in (0, 1, 7, 4095, 131071, 1048575, -3):
            x = rng.standard_normal(D)
            # both sides round pos * theta_j in double: error grows like |pos| * 1e-16
            tol = 1e-12 + 1e-15 * abs(pos)
            assert np.allclose(orc.rope(x, pos), rope_complex(x, pos), rtol=0, atol=tol)


def test_rope_unit_vectors_closed_form(orc):
    D = 128
    e = np.zeros(D)
    e[D - 64] = 1.0
    y = orc.rope(e, 1)
    assert abs(y[D - 64] - math.cos(1.0)) < 1e-15 and abs(y[D - 63] - math.sin(1.0)) < 1e-15
    e = np.zeros(D)
    e[D - 2] = 1.0
    th = 10000.0 ** (-62.0 / 64.0)
    y = orc.rope(e, 1000)
    assert abs(y[D - 2] - math.cos(1000 * th)) < 1e-13 and abs(y[D - 1] - math.sin(1000 * th)) < 1e-13


def test_rope_leaves_leading_dims_and_norm(orc):
    rng = np.random.default_rng(2)
    x = rng.standard_normal(512)
    y = orc.rope(x, 12345)
    assert np.array_equal(y[:448], x[:448])
    assert abs(np.linalg.norm(y) - np.linalg.norm(x)) < 1e-12
    assert np.allclose(orc.rope(y, -12345), x, atol=1e-12)


def test_rope_inner_product_is_relative(orc):
    rng = np.random.default_rng(3)
    a, b = rng.standard_normal(128), rng.standard_normal(128)
    for p, q in ((10, 3), (100000, 99990), (5, 5)):
        lhs = np.dot(orc.rope(a, p), orc.rope(b, q))
        rhs = np.dot(orc.rope(a, p - q), b)
        assert abs(lhs - rhs) < 1e-10


# ---------------------------------------------------------------- compressor
def test_compress_m1_is_norm_then_rope_at_own_position(orc):
    rng = np.random.default_rng(4)
    T, D = 9, 128
    kv = rng.standard_normal((T, D)).astype(np.float32)
    w_z, bias = rng.standard_normal(D) * 0.02, rng.standard_normal(1) * 0.1
    out = orc.compress(kv, pos0=37, m=1, w_z=w_z, bias=bias)
    for t in range(T):
        ref = rope_complex(rms_closed(kv[t].astype(np.float64)), 37 + t)
        assert np.allclose(out[t], ref, atol=1e-12)


def test_compress_identical_tokens_positions_block_last_token(orc):
    """A block of identical tokens pools to that token whatever the weights, so
    the output pins the RoPE position to the block's last token."""
    rng = np.random.default_rng(5)
    m, D, nb, pos0 = 4, 128, 3, 8
    base_rows = rng.standard_normal((nb, D))
    kv = np.repeat(base_rows, m, axis=0)
    out = orc.compress(kv, pos0, m, rng.standard_normal(D), rng.standard_normal(m))
    for b in range(nb):
        ref = rope_complex(rms_closed(base_rows[b]), pos0 + b * m + m - 1)
        assert np.allclose(out[b], ref, atol=1e-12)


def test_compress_two_token_block_closed_form(orc):
    """m = 2: alpha_1 = logistic(z_1 - z_2), z_t = kv_t . w_z + bias[t mod 2]."""
    rng = np.random.default_rng(6)
    D = 128
    kv = rng.standard_normal((4, D))
    w_z = rng.standard_normal(D) * 0.3
    bias = np.array([0.7, -0.4])
    out = orc.compress(kv, 6, 2, w_z, bias)
    for b in range(2):
        k1, k2 = kv[2 * b], kv[2 * b + 1]
        z1 = float(k1 @ w_z) + 0.7
        z2 = float(k2 @ w_z) - 0.4
        a1 = 1.0 / (1.0 + math.exp(-(z1 - z2)))
        c = a1 * k1 + (1.0 - a1) * k2
        ref = rope_complex(rms_closed(c), 6 + 2 * b + 1)
        assert np.allclose(out[b], ref, atol=1e-11)


def test_compress_bias_slot_selects_token(orc):
    """A dominant bias on slot s selects token s of every block (t mod m with
    absolute positions, blocks aligned to multiples of m)."""
    rng = np.random.default_rng(7)
    m, D, nb = 4, 128, 3
    kv = rng.standard_normal((nb * m, D))
    w_z = rng.standard_normal(D) * 0.02
    for s in range(m):
        bias = np.zeros(m)
        bias[s] = 1000.0
        out = orc.compress(kv, 4 * m, m, w_z, bias)
        for b in range(nb):
            ref = rope_complex(rms_closed(kv[b * m + s]), 4 * m + b * m + m - 1)
            assert np.allclose(out[b], ref, atol=1e-11)


def test_compress_zero_scores_is_mean_pooling(orc):
    rng = np.random.default_rng(8)
    m, D = 128, 512
    kv = rng.standard_normal((2 * m, D)).astype(np.float32)
    out = orc.compress(kv, 0, m, np.zeros(D), np.zeros(m))
    for b in range(2):
        c = kv[b * m:(b + 1) * m].astype(np.float64).mean(0)
        assert np.allclose(out[b], rope_complex(rms_closed(c), b * m + m - 1), atol=1e-12)


def test_compress_drops_partial_block_and_rejects_misaligned_start(orc):
    rng = np.random.default_rng(9)
    kv = rng.standard_normal((10, 64))
    assert orc.compress(kv, 0, 4, np.zeros(64), np.zeros(4)).shape == (2, 64)
    with pytest.raises(ValueError):
        orc.compress(kv, 2, 4, np.zeros(64), np.zeros(4))
