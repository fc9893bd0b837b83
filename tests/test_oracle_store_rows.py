"""Oracle pin: storing compressor outputs in the cache formats.

The compressor's outputs (double in the oracle) enter the cache in its storage
format ["DeepSeek-V4 技术报告深度解析" §2.1.4 "KV 缓存精度": the RoPE dims in
BF16, the other dims in FP8].  The oracle first rounds each value to float32
(what the compressor kernel holds) and then stores the float32 row: bfloat16
by round-to-nearest-even, or the mixed FP8/BF16 row quantiser.  These tests pin
that composition against torch's own casts, on values chosen so that a
shortcut (rounding the double straight to bfloat16, quantising the double
instead of its float32 value, or quantising another row) gives other bits.
"""
import numpy as np
import torch


def _double_rounding_cases():
    """Doubles whose float32 value is an exact bfloat16 midpoint, so that
    round-to-nearest-even then lands on the even neighbour while the direct
    rounding of the double goes to the odd one: just above a midpoint whose
    lower neighbour is even, just below one whose lower neighbour is odd."""
    xs = []
    for e in (-3, 0, 5):
        for m in range(0, 128, 9):  # bfloat16 mantissa of the lower neighbour
            lo = (1.0 + m / 128.0) * 2.0 ** e
            mid = lo + 2.0 ** (e - 8)       # halfway to the next bfloat16 value
            eps = 2.0 ** (e - 31)           # below half a float32 ulp of mid
            x = mid + eps if m % 2 == 0 else mid - eps
            xs += [x, -x]
    return np.array(xs, dtype=np.float64)


def _direct_bf16(x):
    """Round-to-nearest of a double straight to the bfloat16 grid (exact in
    double: the grid step is a power of two and no case is a tie)."""
    out = []
    for v in x:
        e = np.floor(np.log2(abs(v)))
        step = 2.0 ** (e - 7)
        r = np.round(v / step) * step
        f = torch.tensor(r, dtype=torch.float64).to(torch.float32)  # exact: r is on the grid
        out.append(f.to(torch.bfloat16).view(torch.int16).item() & 0xFFFF)
    return np.array(out, dtype=np.uint16)


def test_bf16_storage_is_float32_then_rne(orc):
    x = _double_rounding_cases()
    got = orc.store_rows(x.reshape(1, -1), orc.BF16).reshape(-1)
    ref = torch.tensor(x, dtype=torch.float64).to(torch.float32).to(torch.bfloat16).view(torch.int16)
    ref = ref.numpy().view(np.uint16)
    assert np.array_equal(got, ref)
    # the cases tell the two roundings apart: rounding the double straight to
    # bfloat16 gives the other neighbour on every one of them
    assert np.all(_direct_bf16(x) != ref)


def test_f32_storage_is_the_float32_rounding(orc):
    rng = np.random.default_rng(3)
    x = rng.standard_normal((5, 128))
    got = orc.store_rows(x, orc.F32)
    assert got.dtype == np.float32 and np.array_equal(got, x.astype(np.float32))


def _fp8_rows_with_float32_sensitive_values(D=512, n=6, seed=11):
    """Rows whose values sit so close to an E4M3 code midpoint (relative to the
    group scale) that dividing the double or its float32 value decide
    different codes, plus plain N(0,1) rows."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((n, D))
    for r in range(n):
        for g0 in range(0, D - 64, 64):
            amax = np.abs(x[r, g0:g0 + 64]).max()
            scale = np.float32(np.float32(amax) / np.float32(448.0))
            # value = scale * (1.0625 + tiny): 1.0625 is halfway between the E4M3
            # codes 1.0 and 1.125, and the tiny offset is lost in float32
            x[r, g0 + 5] = float(scale) * (1.0625 + 2.0 ** -40)
    return x


def test_fp8_storage_packs_the_float32_rows(orc):
    D = 512
    x = _fp8_rows_with_float32_sensitive_values(D)
    got = orc.store_rows(x, orc.FP8M)
    ref = orc.pack_fp8_rows(x.astype(np.float32))
    assert got.shape == ref.shape == (x.shape[0], orc.fp8m_row_bytes(D))
    assert np.array_equal(got, ref)
    # each row is its own: a permutation of the inputs permutes the rows
    perm = np.array([3, 0, 5, 1, 4, 2])
    assert np.array_equal(orc.store_rows(x[perm], orc.FP8M), ref[perm])
    assert not np.array_equal(ref[perm], ref)


def test_fp8_storage_codes_follow_torch_e4m3_of_the_float32_quotient(orc):
    # The stored codes are torch's RNE E4M3 cast of float32(x) / float32(scale),
    # and the float32 rounding of x decides codes on the planted midpoints.
    D = 512
    x = _fp8_rows_with_float32_sensitive_values(D)
    rows = orc.store_rows(x, orc.FP8M)
    nf = D - 64
    xf = torch.tensor(x.astype(np.float32))
    for r in range(x.shape[0]):
        scales = np.frombuffer(rows[r, nf + 128:nf + 128 + 4 * (nf // 64)].tobytes(), dtype=np.float32)
        for g in range(nf // 64):
            blk = xf[r, 64 * g:64 * (g + 1)]
            sc = (blk.abs().max() / torch.tensor(448.0, dtype=torch.float32)).to(torch.float32)
            assert scales[g] == sc.item()
            codes = (blk / sc).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
            assert np.array_equal(rows[r, 64 * g:64 * (g + 1)], codes)
        # the planted value of group 0 rounds down (to the even code 1.0) from
        # float32, while its double quotient lies above the midpoint
        q64 = x[r, 5] / float(scales[0])
        assert q64 > 1.0625 and orc.e4m3_decode(int(rows[r, 5])) == 1.0
        # the rotated dims are bfloat16 RNE of the float32 values
        rope = np.frombuffer(rows[r, nf:nf + 128].tobytes(), dtype=np.uint16)
        ref = xf[r, nf:].to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(rope, ref)
