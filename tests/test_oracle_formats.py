"""Oracle pins: number formats of the mixed-precision cache.

The cache stores the non-RoPE dims as FP8 E4M3 with one float32 scale per 64
dims and the 64 RoPE dims as bfloat16 ["DeepSeek-V4 技术报告深度解析"
§2.1.4 "KV 缓存精度"].  The oracle's encoder/decoder are written from the OCP
FP8 definition; here they are pinned to PyTorch's independent implementation
of the same formats.
"""
import numpy as np
import pytest
import torch


def test_e4m3_decode_all_codes_match_torch(orc):
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([orc.e4m3_decode(c) for c in range(256)])
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert nan.sum() == 2  # S.1111.111 only
    assert np.array_equal(ref[~nan], got[~nan])
    assert orc.e4m3_decode(0x7E) == 448.0
    assert orc.e4m3_decode(0x01) == 2.0 ** -9  # smallest subnormal


def _torch_e4m3(x):
    t = torch.tensor(x, dtype=torch.float32).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy()


def test_e4m3_encode_matches_torch_rne_in_range(orc):
    rng = np.random.default_rng(0)
    vals = [orc.e4m3_decode(c) for c in range(127)]
    mids = [(a + b) / 2 for a, b in zip(vals[:-1], vals[1:])]  # exact ties
    xs = np.concatenate([
        rng.standard_normal(3000) * 50, rng.standard_normal(500) * 0.01,
        np.array(vals), -np.array(vals), np.array(mids), -np.array(mids),
        np.array([2.0 ** -10, 3 * 2.0 ** -11, 460.0, -463.9])]).astype(np.float32)
    xs = xs[np.abs(xs) <= 464.0]
    ref = _torch_e4m3(xs)
    got = np.array([orc.e4m3_encode(float(x)) for x in xs], dtype=np.uint8)
    # torch keeps the sign of zero for tiny negatives as we do
    assert np.array_equal(ref, got), xs[ref != got][:10]


def test_e4m3_encode_saturates(orc):
    assert orc.e4m3_encode(470.0) == 0x7E
    assert orc.e4m3_encode(1e6) == 0x7E
    assert orc.e4m3_encode(-1e6) == 0xFE
    assert orc.e4m3_encode(464.0) == 0x7E  # tie between 448 and 480 -> even -> 448


def test_bf16_rounding_matches_torch(orc):
    rng = np.random.default_rng(1)
    xs = rng.standard_normal(2000).astype(np.float32)
    # exact ties: bit pattern with the low half 0x8000
    ties = (rng.integers(0, 2 ** 31, 200, dtype=np.uint32) & 0x7FFF0000 | 0x8000).view(np.float32)
    ties = ties[np.isfinite(ties)]
    xs = np.concatenate([xs, ties])
    ref = torch.tensor(xs).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([orc.f32_to_bf16_bits(float(x)) for x in xs], dtype=np.uint16)
    assert np.array_equal(ref, got)


def test_fp8_row_layout_and_roundtrip(orc):
    D = 512
    rng = np.random.default_rng(2)
    x = rng.standard_normal((5, D)).astype(np.float32)
    x[3, 64:128] = 0.0  # an all-zero group takes scale 1
    rows = orc.pack_fp8_rows(x)
    assert rows.shape == (5, 608) and orc.fp8m_row_bytes(D) == 608
    assert (448 + 128 + 28) == 604  # algorithmic bytes; the rest is zero padding
    assert np.all(rows[:, 604:] == 0)
    scales = rows[:, 576:604].copy().view(np.float32)
    amax = np.abs(x[:, :448].reshape(5, 7, 64)).max(-1)
    exp_scales = np.where(amax == 0, np.float32(1), (amax / np.float32(448)).astype(np.float32))
    assert np.array_equal(scales, exp_scales)
    assert scales[3, 1] == 1.0 and np.all(rows[3, 64:128] == 0)
    dec = orc.read_rows(rows, D)
    # RoPE dims: bf16 of the value
    ref_rope = torch.tensor(x[:, 448:]).to(torch.bfloat16).double().numpy()
    assert np.array_equal(dec[:, 448:], ref_rope)
    # FP8 dims: torch's e4m3 cast of x/scale, times scale
    q = (x[:, :448].reshape(5, 7, 64) / scales[:, :, None]).astype(np.float32)
    ref_fp8 = torch.tensor(q).to(torch.float8_e4m3fn).double().numpy() * scales[:, :, None]
    assert np.array_equal(dec[:, :448], ref_fp8.reshape(5, 448))
    # each group's largest magnitude survives exactly up to the scale rounding
    err = np.abs(dec[:, :448] - x[:, :448]).reshape(5, 7, 64).max(-1)
    assert np.all(err <= amax / 16 + 1e-12)  # 3 mantissa bits: half-ulp <= 2^-4 relative


def test_read_rows_bf16_and_f32(orc):
    x = np.random.default_rng(3).standard_normal((4, 64)).astype(np.float32)
    assert np.array_equal(orc.read_rows(x, 64), x.astype(np.float64))
    bits = torch.tensor(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(orc.read_rows(bits, 64), torch.tensor(x).to(torch.bfloat16).double().numpy())
