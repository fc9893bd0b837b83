"""Call order of one CSA or HCA attention layer on top of the C ABI.

These helpers own no arithmetic: they allocate device buffers with torch and
issue the C-ABI calls in the order the layer needs them.

Decode step (one new token per sequence; every sequence has its own length).
The decode state of B sequences is three caller-owned device buffers:
  raw_ring [B, m, D]   raw tokens of each sequence's current block (position p
                       in slot p mod m)
  cache    [B, n_cap]  compressed entries in the cache row format
  window   [B, n_win]  window rows, a ring (position p at row p mod n_win)
  1. append: csa_decode_append stores the newest token kv_tok [B, D] (at
     positions pos [B]) in its raw-ring slot, writes its window row and, for
     every sequence whose token completes a block, pools the block into its
     cache entry (one launch).
  2. CSA: csa_index_topk then csa_attend; HCA: hca_attend (ring window).
Prefill (one sequence, a chunk of new tokens after `T_cached` cached ones):
  csa_compress over the chunk (ratio=m) and over the window tokens (ratio=1),
  then csa_index_topk and csa_attend for every new token (linear window).
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

from . import (BF16, F32, FP8_MIXED, OP_ATTEND, OP_HCA_ATTEND, OP_INDEX_TOPK, csa_attend, csa_index_score,
               csa_topk_select,
               csa_compress, csa_decode_append, csa_index_topk, csa_row_bytes, csa_workspace_bytes,
               hca_attend, params, workspace)

_ACT_DTYPE = {F32: torch.float32, BF16: torch.bfloat16}


def _fmt(x):
    return {"f32": F32, "bf16": BF16, "fp8m": FP8_MIXED}.get(x, x)


@dataclass
class LayerConfig:
    D: int
    H: int
    m: int
    W: int = 128
    topk: int = 0          # 0: HCA layer
    H_I: int = 0
    d_I: int = 0
    act: str = "bf16"
    kv: str = "bf16"
    rope_base: float = 10000.0
    eps: float = 1e-6
    derotate: bool = True
    scale: float = 0.0     # softmax scale; <= 0: 1/sqrt(D)
    batch_invariant: bool = False  # attention splits fixed per query (bit-identical in any batch)

    @property
    def sparse(self) -> bool:
        return self.topk > 0

    def params(self, ratio=None):
        return params(self.D, self.m if ratio is None else ratio, self.topk, self.W, self.act,
                      self.kv, rope_base=self.rope_base, norm_eps=self.eps,
                      softmax_scale=self.scale, derotate_output=self.derotate,
                      batch_invariant=self.batch_invariant)

    @property
    def row_bytes(self) -> int:
        return csa_row_bytes(_fmt(self.kv), self.D)

    def empty_rows(self, *shape, device="cuda"):
        """Device buffer of stored cache/window rows [*shape, D] in the kv format."""
        if _fmt(self.kv) == FP8_MIXED:
            return torch.zeros(*shape, self.row_bytes, dtype=torch.uint8, device=device)
        dt = torch.float32 if _fmt(self.kv) == F32 else torch.bfloat16
        return torch.zeros(*shape, self.D, dtype=dt, device=device)


def ring_order(rows: torch.Tensor, first_pos, n: int) -> torch.Tensor:
    """Rows [B, n, ...] holding positions first_pos[b] + r (r = 0 .. n-1) laid out
    as a ring of n rows: position p at row p mod n (a permutation per sequence)."""
    out = torch.empty_like(rows)
    for b in range(rows.shape[0]):
        shift = int(first_pos[b]) % n
        out[b] = torch.roll(rows[b], shifts=shift, dims=0)
    return out


class DecodeLayer:
    """Buffers and calls of one decode step for B sequences of any lengths."""

    def __init__(self, cfg: LayerConfig, B: int, n_cap: int, n_win: int = 0, device="cuda"):
        self.cfg, self.B, self.n_cap = cfg, B, n_cap
        self.n_win = n_win if n_win > 0 else cfg.W
        self.p = cfg.params()
        act = _ACT_DTYPE[_fmt(cfg.act)]
        self.act_dtype = act
        self.out = torch.empty(B, cfg.H, cfg.D, dtype=act, device=device)
        self.lse = torch.empty(B, cfg.H, dtype=torch.float32, device=device)
        nb = 0
        if cfg.sparse:
            self.topk_idx = torch.empty(B, cfg.topk, dtype=torch.int32, device=device)
            self.topk_score = torch.empty(B, cfg.topk, dtype=torch.float32, device=device)
            # a decode step's indexer scores (the step scores and selects in two calls)
            self.ld = (n_cap + 127) // 128 * 128
            self.scores = torch.empty(B, self.ld, dtype=torch.float32, device=device)
            nb = csa_workspace_bytes(self.p, OP_INDEX_TOPK, B, B, cfg.H, cfg.H_I, n_cap, self.n_win)
            nb = max(nb, csa_workspace_bytes(self.p, OP_ATTEND, B, B, cfg.H, cfg.H_I, n_cap, self.n_win))
        else:
            nb = csa_workspace_bytes(self.p, OP_HCA_ATTEND, B, B, cfg.H, 0, n_cap, self.n_win)
        self.ws = workspace(nb, device)
        self.ws_bytes = self.ws.numel()
        self._side = torch.cuda.Stream(device=device) if cfg.sparse else None
        self._fork, self._join = torch.cuda.Event(), torch.cuda.Event()

    def new_state(self, device="cuda"):
        """Zeroed decode state: (raw_ring [B, m, D], cache [B, n_cap], window [B, n_win])."""
        cfg = self.cfg
        raw_ring = torch.zeros(self.B, cfg.m, cfg.D, dtype=self.act_dtype, device=device)
        return raw_ring, cfg.empty_rows(self.B, self.n_cap, device=device), \
            cfg.empty_rows(self.B, self.n_win, device=device)

    def append(self, kv_tok, pos, w_z, bias, raw_ring, cache, window, stream=None):
        """kv_tok [B, D]: each sequence's newest raw token, at positions pos [B]."""
        csa_decode_append(self.p, kv_tok, self.B, pos, raw_ring, w_z, bias, cache, self.n_cap, window,
                          self.n_win, self.ws, self.ws_bytes, stream)

    def step(self, kv_tok, pos, w_z, bias, raw_ring, q, cache, window, sink, q_idx=None, w_idx=None,
             keys=None):
        """One decode step on the current stream: append the newest tokens,
        then attend at their positions.  For CSA the append feeds only the
        attention, so it runs on a side stream beside the top-k (whose CTAs
        leave room for it on every SM; beside the indexer it would hold the
        indexer's CTAs back) and the attention waits for both; HCA attends to
        the new entries, so it appends first."""
        if not self.cfg.sparse:
            self.append(kv_tok, pos, w_z, bias, raw_ring, cache, window)
            return self.attend(q, cache, window, pos, None, sink)
        cfg = self.cfg
        main = torch.cuda.current_stream()
        csa_index_score(self.p, q_idx, w_idx, cfg.H_I, cfg.d_I, keys, self.n_cap, self.B, self.B, pos,
                        self.scores, self.ld, self.ws, self.ws_bytes, main)
        self._fork.record(main)
        self._side.wait_event(self._fork)
        self.append(kv_tok, pos, w_z, bias, raw_ring, cache, window, stream=self._side)
        self._join.record(self._side)
        csa_topk_select(self.p, self.scores, self.ld, self.n_cap, self.B, pos, self.topk_idx, self.topk_score,
                        main)
        main.wait_event(self._join)
        return self.attend(q, cache, window, pos, None, sink, stream=main, selected=True)

    def index_topk(self, q_idx, w_idx, keys, q_pos, stream=None):
        cfg = self.cfg
        csa_index_topk(self.p, q_idx, w_idx, cfg.H_I, cfg.d_I, keys, self.n_cap, self.B, self.B,
                       q_pos, self.topk_idx, self.topk_score, self.ws, self.ws_bytes, stream)

    def attend(self, q, cache, window, q_pos, win_pos0, sink, q_idx=None, w_idx=None, keys=None,
               stream=None, selected=False):
        """CSA: index and select (unless `selected`: topk_idx holds this step's
        selection), then attend; HCA: attend to every complete block.
        win_pos0 None: the window is a ring (position p at row p mod n_win)."""
        cfg = self.cfg
        if cfg.sparse:
            if not selected:
                self.index_topk(q_idx, w_idx, keys, q_pos, stream)
            csa_attend(self.p, q, cfg.H, self.B, self.B, q_pos, cache, self.n_cap, self.topk_idx,
                       window, self.n_win, win_pos0, sink, self.out, self.lse, self.ws,
                       self.ws_bytes, stream)
        else:
            hca_attend(self.p, q, cfg.H, self.B, self.B, q_pos, cache, self.n_cap, window,
                       self.n_win, win_pos0, sink, self.out, self.lse, self.ws, self.ws_bytes,
                       stream)
        return self.out, self.lse


class PrefillLayer:
    """Buffers and calls of a chunked prefill of one sequence (CSA)."""

    def __init__(self, cfg: LayerConfig, T_cached: int, T_new: int, device="cuda"):
        assert cfg.sparse and T_cached % cfg.m == 0
        self.cfg, self.T_cached, self.T_new = cfg, T_cached, T_new
        self.n_cap = (T_cached + T_new) // cfg.m
        self.raw_pos0 = max(0, T_cached - (cfg.W - 1))
        self.n_win = T_cached + T_new - self.raw_pos0
        self.p = cfg.params()
        self.p1 = cfg.params(ratio=1)
        act = _ACT_DTYPE[_fmt(cfg.act)]
        self.cache = cfg.empty_rows(self.n_cap, device=device)
        self.window = cfg.empty_rows(self.n_win, device=device)
        self.win_pos0 = torch.tensor([self.raw_pos0], dtype=torch.int64, device=device)
        self.out = torch.empty(T_new, cfg.H, cfg.D, dtype=act, device=device)
        self.lse = torch.empty(T_new, cfg.H, dtype=torch.float32, device=device)
        self.topk_idx = torch.empty(T_new, cfg.topk, dtype=torch.int32, device=device)
        self.topk_score = torch.empty(T_new, cfg.topk, dtype=torch.float32, device=device)
        nb = max(csa_workspace_bytes(self.p, OP_INDEX_TOPK, 1, T_new, cfg.H, cfg.H_I, self.n_cap,
                                     self.n_win),
                 csa_workspace_bytes(self.p, OP_ATTEND, 1, T_new, cfg.H, cfg.H_I, self.n_cap,
                                     self.n_win))
        self.ws = workspace(nb, device)
        self.ws_bytes = self.ws.numel()

    def load_cached_rows(self, rows):
        """Copy already-stored rows of the cached prefix into the cache."""
        n = self.T_cached // self.cfg.m
        if n:
            self.cache[:n].copy_(rows)

    def compress(self, kv_raw, w_z, bias, stream=None):
        """kv_raw [n_win, D]: raw tokens from raw_pos0 to the last new token."""
        cfg = self.cfg
        rb = self.cache.element_size() * self.cache.shape[-1]
        n_old = self.T_cached // cfg.m
        off = self.T_cached - self.raw_pos0
        act_rb = kv_raw.element_size() * kv_raw.shape[-1]
        csa_compress(self.p, kv_raw.data_ptr() + off * act_rb, 1, self.T_new, self.T_new,
                     self.T_cached, w_z, bias, self.cache.data_ptr() + n_old * rb, self.n_cap,
                     stream)
        csa_compress(self.p1, kv_raw, 1, self.n_win, self.n_win, self.raw_pos0, w_z, bias,
                     self.window, self.n_win, stream)

    def attend(self, q, q_idx, w_idx, keys, q_pos, sink, stream=None):
        cfg = self.cfg
        csa_index_topk(self.p, q_idx, w_idx, cfg.H_I, cfg.d_I, keys, self.n_cap, 1, self.T_new,
                       q_pos, self.topk_idx, self.topk_score, self.ws, self.ws_bytes, stream)
        csa_attend(self.p, q, cfg.H, 1, self.T_new, q_pos, self.cache, self.n_cap, self.topk_idx,
                   self.window, self.n_win, self.win_pos0, sink, self.out, self.lse, self.ws,
                   self.ws_bytes, stream)
        return self.out, self.lse
