"""Pins of the oracle's FP4 indexer keys ([gitcode] §2.1.1 and §3.2: the
indexer's QK path in FP4 with 1 x 32 sub-blocks, converting to E4M3 without
loss while the sub-block scales stay within E4M3's range): E2M1 codes with one
power-of-two scale per 32 dims.  The code values are checked against torch's
E4M3 grid, the encoder against a different formulation of the same rounding
(half-to-even on the value's own spacing), the block-scale rule against grid
values it must reproduce, the score against the float32 indexer on inputs FP4
holds exactly, and the pages' lossless FP4 -> E4M3 conversion against the FP8
oracle."""
import math

import numpy as np
import torch

import oracle


def _e4m3_values():
    v = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float32).numpy()
    return v[np.isfinite(v)]


def test_e2m1_values_are_the_one_mantissa_bit_points_of_e4m3_up_to_6():
    vals = np.array([oracle.e2m1_decode(c) for c in range(16)])
    # every code value is an E4M3 value (round trip through torch's cast)
    back = torch.from_numpy(vals.astype(np.float32)).to(torch.float8_e4m3fn).to(torch.float32).numpy()
    assert np.array_equal(back, vals.astype(np.float32))
    # sign symmetry
    assert all(oracle.e2m1_decode(c | 8) == -oracle.e2m1_decode(c) for c in range(8))
    # the positive values: 0, and the E4M3 values in (0, 6] that are whole
    # multiples of their spacing 2^(max(floor(log2 v), 0) - 1) (one mantissa
    # bit from 1 up; 0.5 steps below 1, where the subnormals sit)
    e4 = _e4m3_values()
    want = {0.0} | {float(v) for v in e4
                    if 0.0 < v <= 6.0 and (v / 2.0 ** (max(math.floor(math.log2(v)), 0) - 1)).is_integer()}
    assert {float(x) for x in vals[:8]} == want
    assert list(vals[:8]) == sorted(vals[:8])  # codes ordered by value


def _half_even_reference(x):
    """Nearest E2M1 value by rounding |x| to a multiple of its own spacing
    (0.5 below 2, 2^(floor(log2 |x|) - 1) above), half to even, then
    saturating at 6."""
    a = abs(x)
    if a >= 8.0:
        r = 6.0
    else:
        ulp = 0.5 if a < 2.0 else 2.0 ** (math.floor(math.log2(a)) - 1)
        r = min(6.0, float(np.round(a / ulp)) * ulp)
    return math.copysign(r, x) if r != 0.0 else 0.0


def test_e2m1_encoder_matches_half_even_rounding_on_the_value_spacing():
    rng = np.random.default_rng(61)
    xs = list(rng.uniform(-9, 9, 4000)) + list(rng.standard_normal(2000) * 0.7)
    # every grid value, every midpoint between neighbours, and their neighbours
    grid = [oracle.e2m1_decode(c) for c in range(8)]
    mids = [(a + b) / 2 for a, b in zip(grid, grid[1:])] + [7.0]
    for v in grid + mids:
        for t in (v, np.nextafter(v, -np.inf), np.nextafter(v, np.inf)):
            xs += [t, -t]
    for x in xs:
        got = oracle.e2m1_decode(oracle.e2m1_encode(x))
        assert got == _half_even_reference(x) or (got == 0.0 and _half_even_reference(x) == 0.0), x


def _grid_keys(rng, n, dI, kmin=-6, kmax=4):
    """Keys whose every 32-dim block is E2M1 grid values times 2^k, the block's
    largest magnitude 4 or 6 times 2^k and a 0.5 * 2^k among them: the block
    scale rule must give exactly 2^k and reproduce every value."""
    x = np.empty((n, dI), dtype=np.float32)
    ks = rng.integers(kmin, kmax + 1, size=(n, dI // 32))
    grid = np.array([oracle.e2m1_decode(c) for c in range(16)])
    for b in range(n):
        for j in range(dI // 32):
            blk = rng.choice(grid, size=32)
            blk[0] = rng.choice([4.0, 6.0, -4.0, -6.0])
            blk[1] = rng.choice([0.5, -0.5])
            blk = np.clip(blk, -6.0, 6.0)
            x[b, j * 32:(j + 1) * 32] = blk * 2.0 ** ks[b, j]
    return x, ks


def test_block_scale_reproduces_grid_values_exactly():
    rng = np.random.default_rng(62)
    x, ks = _grid_keys(rng, 40, 128)
    codes, scales = oracle.pack_idx_keys_fp4(x)
    assert np.array_equal(scales.astype(np.int64) - 127, ks)
    assert np.array_equal(oracle.decode_idx_keys_fp4(codes, scales), x.astype(np.float64))


def test_block_maximum_lands_in_four_to_eight_and_zero_blocks():
    rng = np.random.default_rng(63)
    x = (rng.standard_normal((50, 128)) * np.exp2(rng.integers(-12, 12, size=(50, 1)))).astype(np.float32)
    x[3, 32:64] = 0.0  # an all-zero block
    codes, scales = oracle.pack_idx_keys_fp4(x)
    for b in range(50):
        for j in range(4):
            amax = float(np.abs(x[b, j * 32:(j + 1) * 32]).max())
            e = int(scales[b, j]) - 127
            if amax == 0.0:
                assert e == 0
                continue
            assert 4.0 <= amax / 2.0 ** e < 8.0
    assert np.all(codes[3, 16:32] == 0)


def _representable_queries(rng, HI, dI):
    """E4M3 grid values whose row maximum is exactly 448 (query scale 1)."""
    e4 = _e4m3_values()
    q = rng.choice(e4[np.abs(e4) <= 448], size=(HI, dI)).astype(np.float32)
    q[:, 0] = 448.0
    return q


def test_fp4_scores_equal_the_float32_indexer_on_exact_inputs():
    rng = np.random.default_rng(64)
    HI, dI, n = 4, 128, 24
    keys, _ = _grid_keys(rng, n, dI)
    q = _representable_queries(rng, HI, dI)
    w = rng.uniform(0, 1, size=HI)
    codes, scales = oracle.pack_idx_keys_fp4(keys)
    got = oracle.index_scores_fp4(q, w, codes, scales)
    want = oracle.index_scores(q, w, keys)
    assert np.allclose(got, want, rtol=1e-12, atol=0.0)


def _to_e4m3_per_key(decoded):
    """FP4 key values -> E4M3 codes with one power-of-two scale per key (the
    largest block scale), through torch's cast; returns codes, scales and
    whether every value survived."""
    n, dI = decoded.shape
    codes = np.empty((n, dI), dtype=np.uint8)
    scales = np.empty(n, dtype=np.float32)
    exact = True
    for b in range(n):
        amax = np.abs(decoded[b]).max()
        e = math.floor(math.log2(amax)) - 2 if amax > 0 else 0
        S = 2.0 ** e
        c = torch.from_numpy((decoded[b] / S).astype(np.float32)).to(torch.float8_e4m3fn)
        codes[b] = c.view(torch.uint8).numpy()
        scales[b] = S
        exact &= bool(np.array_equal(c.to(torch.float32).numpy().astype(np.float64) * S, decoded[b]))
    return codes, scales, exact


def test_fp4_to_e4m3_is_lossless_while_block_scales_stay_within_eight_binades():
    rng = np.random.default_rng(65)
    HI, dI, n = 4, 128, 30
    # block magnitudes spread over at most 2^8 within a key
    spread = rng.integers(0, 9, size=(n, dI // 32))
    x = (rng.standard_normal((n, dI)) * np.repeat(np.exp2(-spread), 32, axis=1)).astype(np.float32)
    codes4, scales4 = oracle.pack_idx_keys_fp4(x)
    dec = oracle.decode_idx_keys_fp4(codes4, scales4)
    es = scales4.astype(np.int64) - 127
    assert np.all(es.max(axis=1) - es.min(axis=1) <= 8)
    codes8, scales8, exact = _to_e4m3_per_key(dec)
    assert exact
    q = rng.standard_normal((HI, dI)).astype(np.float32)
    w = rng.uniform(0, 1, size=HI)
    s4 = oracle.index_scores_fp4(q, w, codes4, scales4)
    s8 = oracle.index_scores_fp8(q, w, codes8, scales8)
    assert np.array_equal(s4, s8)
    # beyond the range the conversion loses the smallest block's values
    y = x.copy()
    y[:, 96:] *= 2.0 ** -14
    c4, sc4 = oracle.pack_idx_keys_fp4(y)
    assert not _to_e4m3_per_key(oracle.decode_idx_keys_fp4(c4, sc4))[2]


def _block_exponents(x, dI=128):
    """floor(log2 amax) - 2 per 32-dim block (None for an all-zero block)."""
    out = []
    for j in range(dI // 32):
        amax = float(np.abs(x[j * 32:(j + 1) * 32]).max())
        out.append(None if amax == 0.0 else math.floor(math.log2(amax)) - 2)
    return out


def test_packer_keeps_block_scales_within_fourteen_binades_of_the_largest():
    """A block far below the key's largest gets the exponent E - 14, and its
    codes are the half-even roundings of its values on that coarser grid."""
    rng = np.random.default_rng(66)
    n, dI = 30, 128
    x = rng.standard_normal((n, dI)).astype(np.float32)
    drop = rng.integers(15, 30, size=n)           # binades block 3 sits below the others
    x[:, 96:] *= np.exp2(-drop)[:, None].astype(np.float32)
    x[5, 64:96] = 0.0                              # an all-zero block keeps exponent 0
    codes, scales = oracle.pack_idx_keys_fp4(x)
    for b in range(n):
        ref = _block_exponents(x[b])
        E = max(e for e in ref if e is not None)
        es = scales[b].astype(int) - 127
        for j, e in enumerate(ref):
            want = 0 if e is None else max(e, E - 14)
            assert es[j] == want, (b, j, es[j], want)
        assert es[3] == E - 14  # the dropped block was raised
        for d in range(96, 128):
            c = (int(codes[b, d // 2]) >> 4) if d & 1 else (int(codes[b, d // 2]) & 15)
            got = oracle.e2m1_decode(c)
            want = _half_even_reference(float(x[b, d]) / 2.0 ** es[3])
            assert got == want or (got == 0.0 and want == 0.0), (b, d)


def _to_e4m3_centred(codes4, scales4):
    """The conversion the FP4 indexer kernel makes: every key's FP4 values to
    E4M3 codes with one power-of-two scale per key, 2^(E - 6) for E the
    largest exponent of its nonzero blocks (through torch's cast); returns
    codes, scales and whether every value survived."""
    dec = oracle.decode_idx_keys_fp4(codes4, scales4)
    n, dI = dec.shape
    codes = np.empty((n, dI), dtype=np.uint8)
    scales = np.empty(n, dtype=np.float32)
    exact = True
    es = scales4.astype(np.int64) - 127
    for b in range(n):
        nz = [j for j in range(dI // 32) if np.any(dec[b, j * 32:(j + 1) * 32] != 0.0)]
        E = max(es[b, j] for j in nz) if nz else 6
        S = 2.0 ** (E - 6)
        c = torch.from_numpy((dec[b] / S).astype(np.float32)).to(torch.float8_e4m3fn)
        codes[b] = c.view(torch.uint8).numpy()
        scales[b] = S
        exact &= bool(np.array_equal(c.to(torch.float32).numpy().astype(np.float64) * S, dec[b]))
    return codes, scales, exact


def test_every_packed_key_converts_to_e4m3_without_loss():
    """Keys with sub-block scale spreads from 0 to 30 binades (the packer
    keeps them within 14): the centred per-key E4M3 conversion is exact, and
    the FP8 oracle over the converted keys gives the FP4 oracle's scores bit
    for bit."""
    rng = np.random.default_rng(67)
    HI, dI, n = 8, 128, 60
    spread = rng.integers(0, 31, size=(n, dI // 32))
    x = (rng.standard_normal((n, dI)) * np.repeat(np.exp2(-spread.astype(np.float64)), 32, axis=1)).astype(np.float32)
    x[7, :32] = 0.0
    codes4, scales4 = oracle.pack_idx_keys_fp4(x)
    es = scales4.astype(np.int64) - 127
    assert np.all(es.max(axis=1) - es.min(axis=1) <= 14 + 127)  # zero blocks keep exponent 0
    codes8, scales8, exact = _to_e4m3_centred(codes4, scales4)
    assert exact
    q = rng.standard_normal((HI, dI)).astype(np.float32)
    w = rng.uniform(0, 1, size=HI)
    assert np.array_equal(oracle.index_scores_fp4(q, w, codes4, scales4),
                          oracle.index_scores_fp8(q, w, codes8, scales8))
