"""Seeded synthetic workloads shared by the tests, the smoke check and the benchmark.

This module only draws random numbers and stores them in the input dtypes; it
holds none of the method's arithmetic (no normalisation, rotation, pooling,
scoring or quantisation).  Both the CUDA path and the oracle receive the
identical bits produced here.

Shapes and distributions follow the pages' 1M-context workloads:
  * q, raw kv, indexer q and keys, cached rows: N(0, 1)
  * indexer head weights w: U(0, 1)
  * pooling weight w_z: N(0, 0.02); per-slot pooling bias: N(0, 0.1)
  * sink logits: N(0, 1) (0.0 for the fp32 prefill workload)
Cached compressed rows of a decode workload are N(0, 1) draws standing in for
rows that were already normalised and rotated when they were appended.
For the mixed-precision cache the draws are float32 values before
quantisation; each side quantises them itself.
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass
from typing import Optional

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    kind: str            # "csa_decode" | "hca_decode" | "csa_prefill"
    act: str             # "f32" | "bf16": q, raw kv, indexer q/keys, outputs
    kv_fmt: str          # "f32" | "bf16" | "fp8m": stored compressed/window rows
    seed: int
    B: int
    D: int
    H: int
    m: int
    W: int
    L: int = 0           # decode: context length including the current token
    L_per_seq: Optional[tuple] = None   # decode: ragged lengths (overrides L)
    T_cached: int = 0    # prefill: tokens already in the cache
    T_new: int = 0       # prefill: new query tokens
    H_I: int = 0
    d_I: int = 0
    topk: int = 0
    sink: str = "normal"  # "normal" | "zero" | "neginf"
    rope_dims: int = 64
    rope_base: float = 10000.0
    eps: float = 1e-6
    softmax_scale: float = 0.0  # <= 0: 1/sqrt(D)
    idx_fmt: str = "bf16"  # "bf16" | "fp8": E4M3 codes + a scale per key | "fp4": E2M1 codes + 4 block exponents

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)

    @property
    def lengths(self):
        if self.kind == "csa_prefill":
            return (self.T_cached + self.T_new,)
        if self.L_per_seq is not None:
            return tuple(self.L_per_seq)
        return (self.L,) * self.B

    @property
    def n_cap(self) -> int:
        """Compressed-entry capacity per sequence."""
        return max(self.lengths) // self.m

    @property
    def Q(self) -> int:
        return self.T_new if self.kind == "csa_prefill" else self.B


# The five workloads the pages' 1M-context setting is measured on.
CSA_PREFILL_F32 = Workload(
    name="csa_prefill_f32_4k", kind="csa_prefill", act="f32", kv_fmt="f32", seed=0, B=1, D=128,
    H=8, m=4, W=128, T_cached=0, T_new=4096, H_I=4, d_I=64, topk=64, sink="zero")
CSA_DECODE_128K = Workload(
    name="csa_decode_bf16_b32_128k", kind="csa_decode", act="bf16", kv_fmt="bf16", seed=1, B=32,
    D=512, H=64, m=4, W=128, L=131072, H_I=64, d_I=128, topk=1024)
HCA_DECODE_1M = Workload(
    name="hca_decode_bf16_b32_1m", kind="hca_decode", act="bf16", kv_fmt="bf16", seed=2, B=32,
    D=512, H=64, m=128, W=128, L=1048576)
CSA_CHUNKED_PREFILL = Workload(
    name="csa_chunked_prefill_bf16_64k_8k", kind="csa_prefill", act="bf16", kv_fmt="bf16", seed=3,
    B=1, D=512, H=64, m=4, W=128, T_cached=65536, T_new=8192, H_I=64, d_I=128, topk=1024)
CSA_DECODE_1M_FP8 = Workload(
    name="csa_decode_fp8cache_b8_1m", kind="csa_decode", act="bf16", kv_fmt="fp8m", seed=4, B=8,
    D=512, H=64, m=4, W=128, L=1048576, H_I=64, d_I=128, topk=1024)

FULL = [CSA_PREFILL_F32, CSA_DECODE_128K, HCA_DECODE_1M, CSA_CHUNKED_PREFILL, CSA_DECODE_1M_FP8]
# The headline decode shape with the indexer keys in E4M3 (the keys are the
# same N(0,1) draws; each side quantises them itself).
CSA_DECODE_128K_FP8IDX = CSA_DECODE_128K.replace(name="csa_decode_fp8idx_b32_128k", idx_fmt="fp8")
# ... and with FP4 indexer keys (E2M1 codes, one power-of-two scale per 32 dims).
CSA_DECODE_128K_FP4IDX = CSA_DECODE_128K.replace(name="csa_decode_fp4idx_b32_128k", idx_fmt="fp4")
EXTRA = [CSA_DECODE_128K_FP8IDX, CSA_DECODE_128K_FP4IDX]
BY_NAME = {w.name: w for w in FULL + EXTRA}


def _gen(seed: int, stream: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed * 1_000_003 + stream)
    return g


def _normal(shape, seed, stream, device, std=1.0):
    g = _gen(seed, stream, device)
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32) * std


def _uniform(shape, seed, stream, device):
    g = _gen(seed, stream, device)
    return torch.rand(shape, generator=g, device=device, dtype=torch.float32)


def _act(x: torch.Tensor, act: str) -> torch.Tensor:
    return x.to(torch.bfloat16) if act == "bf16" else x


def _kv(x: torch.Tensor, kv_fmt: str) -> torch.Tensor:
    # fp8m rows stay float32 here: quantisation is part of the method
    return x.to(torch.bfloat16) if kv_fmt == "bf16" else x


# stream ids: one independent generator per tensor
_S_Q, _S_QI, _S_WI, _S_KEYS, _S_CACHE, _S_WIN, _S_KVNEW, _S_WZ, _S_BIAS, _S_SINK = range(10)


def generate(w: Workload, device="cpu") -> dict:
    """All inputs of one workload as torch tensors on `device`.

    decode (csa/hca): q [B,H,D], cache [B,n_cap,D], window [B,W,D] with row r at
      position win_pos0[b]+r, kv_new [B,m,D] raw tokens of the newest block
      (positions L_b-m .. L_b-1), q_pos [B] = L_b-1, win_pos0 [B];
      csa adds q_idx [B,H_I,d_I], w_idx [B,H_I], keys [B,n_cap,d_I].
    prefill: q [T_new,H,D], cache_old [T_cached//m, D] rows already in the cache,
      kv_raw [n_raw,D] raw tokens from position raw_pos0 up to the last query,
      q_idx [T_new,H_I,d_I], w_idx [T_new,H_I], keys [n_cap,d_I],
      q_pos [T_new] = T_cached .. T_cached+T_new-1.
    common: w_z [D], bias [m], sink [H].
    """
    s, dev = w.seed, device
    out = {}
    if w.sink == "normal":
        out["sink"] = _normal((w.H,), s, _S_SINK, dev)
    elif w.sink == "zero":
        out["sink"] = torch.zeros(w.H, device=dev)
    else:
        out["sink"] = torch.full((w.H,), float("-inf"), device=dev)
    out["w_z"] = _normal((w.D,), s, _S_WZ, dev, std=0.02)
    out["bias"] = _normal((w.m,), s, _S_BIAS, dev, std=0.1)
    if w.kind in ("csa_decode", "hca_decode"):
        lens = torch.tensor(w.lengths, dtype=torch.int64)
        out["q"] = _act(_normal((w.B, w.H, w.D), s, _S_Q, dev), w.act)
        out["cache"] = _kv(_normal((w.B, w.n_cap, w.D), s, _S_CACHE, dev), w.kv_fmt)
        out["window"] = _kv(_normal((w.B, w.W, w.D), s, _S_WIN, dev), w.kv_fmt)
        out["kv_new"] = _act(_normal((w.B, w.m, w.D), s, _S_KVNEW, dev), w.act)
        out["q_pos"] = (lens - 1).to(dev)
        out["win_pos0"] = torch.clamp(lens - w.W, min=0).to(dev)
        if w.kind == "csa_decode":
            out["q_idx"] = _act(_normal((w.B, w.H_I, w.d_I), s, _S_QI, dev), w.act)
            out["w_idx"] = _uniform((w.B, w.H_I), s, _S_WI, dev)
            out["keys"] = _act(_normal((w.B, w.n_cap, w.d_I), s, _S_KEYS, dev), w.act)
    else:
        assert w.T_cached % w.m == 0
        raw_pos0 = max(0, w.T_cached - (w.W - 1))
        n_raw = w.T_cached + w.T_new - raw_pos0
        out["q"] = _act(_normal((w.T_new, w.H, w.D), s, _S_Q, dev), w.act)
        out["cache_old"] = _kv(_normal((w.T_cached // w.m, w.D), s, _S_CACHE, dev), w.kv_fmt)
        out["kv_raw"] = _act(_normal((n_raw, w.D), s, _S_KVNEW, dev), w.act)
        out["raw_pos0"] = raw_pos0
        out["q_idx"] = _act(_normal((w.T_new, w.H_I, w.d_I), s, _S_QI, dev), w.act)
        out["w_idx"] = _uniform((w.T_new, w.H_I), s, _S_WI, dev)
        out["keys"] = _act(_normal((w.n_cap, w.d_I), s, _S_KEYS, dev), w.act)
        out["q_pos"] = torch.arange(w.T_cached, w.T_cached + w.T_new, dtype=torch.int64,
                                    device=dev)
    return out


def to_numpy_stored(t: torch.Tensor):
    """Tensor -> numpy array in the oracle's stored form (bf16 as uint16 bits)."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view("uint16")
    if t.dtype == torch.uint8:
        return t.numpy()
    return t.numpy()
