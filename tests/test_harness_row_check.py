"""The stored-row check the GPU parity tests use (tests/harness.py
check_stored_rows) accepts the oracle's own rows and rejects a single code
moved one step away from where float32 noise could put it, in bf16 rows and
in FP8/BF16 rows (E4M3 codes, rotated dims)."""
import numpy as np
import pytest
import torch

import oracle
from tests import harness as H


class _W:
    def __init__(self, kv):
        self.kv_fmt, self.D = kv, 512


def _rows(seed=0):
    return np.random.default_rng(seed).standard_normal((4, 512))


def test_accepts_the_oracles_own_rows(orc):
    ref = _rows()
    bf = oracle.store_rows(ref, oracle.BF16)
    assert H.check_stored_rows(_W("bf16"), torch.from_numpy(bf.view(np.int16)).view(torch.bfloat16), ref, "t") == 0
    f8 = oracle.store_rows(ref, oracle.FP8M)
    assert H.check_stored_rows(_W("fp8m"), torch.from_numpy(f8), ref, "t") == 0


@pytest.mark.parametrize("where", [3, 100, 447])
def test_rejects_one_e4m3_code_off(orc, where):
    ref = _rows(1)
    f8 = oracle.store_rows(ref, oracle.FP8M)
    f8[2, where] = (int(f8[2, where]) & 0x80) | min(0x7E, (int(f8[2, where]) & 0x7F) + 1)
    with pytest.raises(AssertionError):
        H.check_stored_rows(_W("fp8m"), torch.from_numpy(f8), ref, "t")


def test_rejects_one_bf16_step_off_and_a_rotated_dim_off(orc):
    ref = _rows(2)
    bf = oracle.store_rows(ref, oracle.BF16)
    bf[1, 40] += 1
    with pytest.raises(AssertionError):
        H.check_stored_rows(_W("bf16"), torch.from_numpy(bf.view(np.int16)).view(torch.bfloat16), ref, "t")
    f8 = oracle.store_rows(ref, oracle.FP8M)
    rope = f8[0, 448:576].view(np.uint16).copy()
    rope[5] += 1
    f8[0, 448:576] = rope.view(np.uint8)
    with pytest.raises(AssertionError):
        H.check_stored_rows(_W("fp8m"), torch.from_numpy(f8), ref, "t")


def test_rejects_a_scale_off(orc):
    ref = _rows(3)
    f8 = oracle.store_rows(ref, oracle.FP8M)
    sc = f8[0, 576:604].view(np.float32).copy()
    sc[2] *= 1.01
    f8[0, 576:604] = sc.view(np.uint8)
    with pytest.raises(AssertionError):
        H.check_stored_rows(_W("fp8m"), torch.from_numpy(f8), ref, "t")
