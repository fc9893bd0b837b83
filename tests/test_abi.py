"""The C-ABI library: it loads without a GPU, exports every entry point the
header declares, and rejects invalid arguments on the host before launching
anything (these checks never touch device memory, so fake aligned addresses
are safe here)."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "csa.h")


@pytest.fixture(scope="module")
def L():
    from long_context_compressed_17_b300 import build
    build.build()
    import long_context_compressed_17_b300 as pkg
    return pkg


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\**\s+([a-z_0-9]+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("csa_compress", "csa_append", "csa_index_topk", "csa_attend", "hca_attend", "csa_cache_pack",
              "csa_workspace_bytes", "csa_workspace_init", "csa_check_status",
              "csa_status_string", "csa_last_error", "csa_row_bytes"):
        assert n in names, n


def test_library_exports_every_declared_symbol(L):
    lib = ctypes.CDLL(L.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing
    out = subprocess.run(["nm", "-D", "--defined-only", L.LIB_PATH], capture_output=True,
                         text=True).stdout
    exported = set(line.split()[-1] for line in out.splitlines() if " T " in line)
    for n in declared_functions():
        assert n in exported, n


def test_library_has_no_unresolved_symbols_of_its_own(L):
    out = subprocess.run(["nm", "-D", "--undefined-only", L.LIB_PATH], capture_output=True,
                         text=True).stdout
    own = [line for line in out.splitlines() if "csa" in line]
    assert not own, own


def test_library_holds_sm103a_code(L):
    out = subprocess.run(["cuobjdump", "--list-elf", L.LIB_PATH], capture_output=True, text=True)
    assert "sm_103a" in out.stdout, out.stdout + out.stderr


def test_row_bytes(L):
    assert L.csa_row_bytes("bf16", 512) == 1024
    assert L.csa_row_bytes("f32", 128) == 512
    assert L.csa_row_bytes("fp8m", 512) == 608   # 448 E4M3 + 64 bf16 + 7 scales + pad
    assert L.csa_row_bytes("fp8m", 128) == 208
    assert L.csa_row_bytes("bf16", 100) == -1


FAKE = 1 << 20  # aligned, never dereferenced: validation fails before any launch


def _attend_args(L, p, **over):
    a = dict(p=p, q=FAKE, H=64, B=2, Q=2, q_pos=FAKE, cache=FAKE, n_cap=100, topk_idx=FAKE,
             window=FAKE, n_win=128, win_pos0=FAKE, sink=FAKE, out=FAKE, lse=None, ws=FAKE,
             ws_bytes=1 << 40, stream=0)
    a.update(over)
    return a


def _status_of(fn, **kw):
    from long_context_compressed_17_b300 import CsaError
    with pytest.raises(CsaError) as ei:
        fn(**kw)
    return ei.value.status


def test_attend_validation(L):
    p = L.params(512, 4, topk=64)
    bad = {
        "null q": dict(q=None),
        "misaligned q": dict(q=FAKE + 2),
        "Q not multiple of B": dict(Q=3),
        "null sink": dict(sink=None),
        "null topk": dict(topk_idx=None),
        "H not multiple of 8": dict(H=12),
        "negative n_cap": dict(n_cap=-1),
    }
    for what, over in bad.items():
        st = _status_of(L.csa_attend, **_attend_args(L, p, **over))
        assert st in (1, 2), what
    assert _status_of(L.csa_attend, **_attend_args(L, p, H=12)) == 2
    assert _status_of(L.csa_attend, **_attend_args(L, p, ws_bytes=100)) == 4
    assert "workspace" in L.csa_last_error()


def test_params_validation(L):
    from long_context_compressed_17_b300 import CsaError
    cases = [
        (L.params(100, 4, topk=8), 2),                    # head_dim
        (L.params(512, 4, topk=0), 1),                    # topk
        (L.params(512, 0, topk=8), 1),                    # ratio
        (L.params(512, 4, topk=8, rope_dims=32), 2),      # rope dims
        (L.params(512, 4, topk=8, act="f32", kv="bf16"), 2),
        (L.params(512, 4, topk=8, window=5000), 1),
        (L.params(512, 4, topk=8, norm_eps=float("nan")), 1),
    ]
    for p, want in cases:
        st = _status_of(L.csa_attend, **_attend_args(L, p))
        assert st == want, (p.head_dim, p.topk, p.ratio, st)


def test_index_topk_validation(L):
    p = L.params(512, 4, topk=1024)
    base = dict(p=p, q_idx=FAKE, w_idx=FAKE, n_idx_heads=64, idx_dim=128, keys=FAKE, n_cap=1000,
                B=2, Q=4, q_pos=FAKE, topk_idx=FAKE, topk_score=None, ws=FAKE, ws_bytes=1 << 40)
    assert _status_of(L.csa_index_topk, **dict(base, idx_dim=96)) == 2
    assert _status_of(L.csa_index_topk, **dict(base, n_idx_heads=65)) == 2
    assert _status_of(L.csa_index_topk, **dict(base, Q=3)) == 1
    assert _status_of(L.csa_index_topk, **dict(base, q_pos=None)) == 1
    assert _status_of(L.csa_index_topk, **dict(base, ws_bytes=1000)) == 4
    assert _status_of(L.csa_index_topk, **dict(base, p=L.params(512, 4, topk=5000))) == 1


def test_compress_validation(L):
    p = L.params(512, 4)
    base = dict(p=p, kv_raw=FAKE, B=2, T=16, kv_seq_stride=16, pos0=8, w_z=FAKE, bias=FAKE,
                out=FAKE, out_seq_stride=4)
    assert _status_of(L.csa_compress, **dict(base, pos0=6)) == 1       # not a multiple of m
    assert _status_of(L.csa_compress, **dict(base, kv_seq_stride=8)) == 1
    assert _status_of(L.csa_compress, **dict(base, out_seq_stride=3)) == 1
    assert _status_of(L.csa_compress, **dict(base, w_z=FAKE + 4)) == 1


def test_append_validation(L):
    p = L.params(512, 4)
    base = dict(p=p, kv_new=FAKE, B=2, kv_seq_stride=4, pos0=8, w_z=FAKE, bias=FAKE,
                entry_out=FAKE, out_seq_stride=4, win_out=FAKE, win_seq_stride=128)
    assert _status_of(L.csa_append, **dict(base, pos0=6)) == 1       # not a multiple of m
    assert _status_of(L.csa_append, **dict(base, kv_seq_stride=3)) == 1
    assert _status_of(L.csa_append, **dict(base, win_out=None)) == 1
    assert _status_of(L.csa_append, **dict(base, entry_out=FAKE + 8)) == 1  # not 16-byte aligned
    assert _status_of(L.csa_append, **dict(base, B=-1)) == 1


def test_zero_sized_requests_are_no_ops(L):
    p = L.params(512, 4, topk=8)
    # Q = 0 and T < m return CSA_OK without touching any pointer or the device
    L.csa_attend(**_attend_args(L, p, Q=0, q=None, out=None))
    L.csa_compress(p, None, 1, 3, 3, 0, None, None, None, 1)


def test_workspace_sizes(L):
    p = L.params(512, 4, topk=1024)
    n = L.csa_workspace_bytes(p, L.OP_INDEX_TOPK, 32, 32, 64, 64, 32768, 128)
    assert n >= 256 + 32 * 32768 * 4
    assert L.csa_workspace_bytes(p, L.OP_ATTEND, 32, 32, 64, 64, 32768, 128) > 256
    assert L.csa_workspace_bytes(p, 99, 32, 32, 64, 64, 32768, 128) == 0


def _al(x):
    return (x + 255) // 256 * 256


def _inv_splits(T):
    """Fixed splits of a T-tile list: one every s tiles, s the largest power of
    two <= T/8 clamped to [2, 16] (the documented batch-invariant rule)."""
    import math
    s = min(16, max(2, 2 ** math.floor(math.log2(T / 8))))
    return -(-T // s)


def test_attend_workspace_partial_counts_and_wide_fallback(L):
    """Tensor-core ranges (bf16, D = 512, 64 heads, k = 1024, W = 128: 18 tiles
    a query): at Q = 32 on 148 SMs the ranges are query-aligned, 4 or 5 CTAs
    a query, so 5 partial slots, plus one int32 partial count per query.  At
    Q*(18 + 5) >= 2^31 tile units the planner hands the call to the CUDA-core
    kernel: one split of all 1152 rows, no partial counts."""
    import torch
    if torch.cuda.is_available() and torch.cuda.get_device_properties(0).multi_processor_count != 148:
        pytest.skip("the expected ranges assume 148 SMs")
    p = L.params(512, 4, topk=1024, window=128)
    Q = 32
    want = 256 + _al(Q * 5 * 64 * 512 * 4) + _al(Q * 5 * 64 * 2 * 4) + _al(Q * 4)
    assert L.csa_workspace_bytes(p, L.OP_ATTEND, Q, Q, 64, 0, 32768, 128) == want
    Q = (1 << 31) // 23 + 1
    want = 256 + _al(Q * 64 * 512 * 4) + _al(Q * 64 * 2 * 4)
    assert L.csa_workspace_bytes(p, L.OP_ATTEND, Q, Q, 64, 0, 32768, 128) == want


@pytest.mark.parametrize("k,W,n_cap,Q,B", [(1024, 128, 32768, 32, 32), (1024, 128, 4096, 5, 5),
                                           (64, 0, 4096, 3, 3), (100, 128, 4096, 8, 2)])
def test_batch_invariant_csa_workspace_follows_the_split_rule(L, k, W, n_cap, Q, B):
    """Tensor-core path (bf16, D = 512, 64 heads): ceil(k/64) + ceil(W/64)
    tiles, one partial per fixed split for every query, whatever Q."""
    p = L.params(512, 4, topk=k, window=W, batch_invariant=True)
    S = _inv_splits(-(-k // 64) + -(-W // 64))
    want = 256 + _al(Q * S * 64 * 512 * 4) + _al(Q * S * 64 * 2 * 4)
    assert L.csa_workspace_bytes(p, L.OP_ATTEND, B, Q, 64, 0, n_cap, 128) == want


@pytest.mark.parametrize("n_cap,Q", [(8192, 32), (2048, 12), (100, 1), (64, 7)])
def test_batch_invariant_hca_workspace_follows_the_split_rule(L, n_cap, Q):
    p = L.params(512, 128, window=128, batch_invariant=True)
    S = _inv_splits(-(-n_cap // 64) + 2)
    want = 256 + _al(Q * S * 64 * 512 * 4) + _al(Q * S * 64 * 2 * 4)
    assert L.csa_workspace_bytes(p, L.OP_HCA_ATTEND, Q, Q, 64, 0, n_cap, 128) == want


def test_batch_invariant_cuda_core_splits_follow_the_rule(L):
    """fp32, D = 128, 8 heads: the list of k + W rows in splits of 64*s rows."""
    import math
    for k, W, Q in [(64, 128, 4096), (1000, 128, 3), (20, 0, 1)]:
        p = L.params(128, 4, topk=k, window=W, act="f32", kv="f32", batch_invariant=True)
        n = k + W
        T = -(-n // 64)
        s = min(16, max(2, 2 ** math.floor(math.log2(T / 8))))
        S = -(-n // (64 * s))
        want = 256 + _al(Q * S * 8 * 128 * 4) + _al(Q * S * 8 * 2 * 4)
        assert L.csa_workspace_bytes(p, L.OP_ATTEND, Q, Q, 8, 0, 4096, 128) == want, (k, W, Q)


def test_index_topk_fp8_validation(L):
    import torch
    p = L.params(512, 4, topk=64)
    base = dict(p=p, q_idx=FAKE, w_idx=FAKE, n_idx_heads=64, idx_dim=128, key_codes=FAKE,
                key_scales=FAKE, n_cap=1024, B=2, Q=2, q_pos=FAKE, topk_idx=FAKE, topk_score=None,
                ws=FAKE, ws_bytes=1 << 30)
    assert _status_of(L.csa_index_topk_fp8, **dict(base, idx_dim=64)) == 2      # unsupported
    assert _status_of(L.csa_index_topk_fp8, **dict(base, n_idx_heads=32)) == 2
    assert _status_of(L.csa_index_topk_fp8, **dict(base, n_cap=100)) == 2       # < one key tile
    assert _status_of(L.csa_index_topk_fp8, **dict(base, Q=3)) == 1             # Q % B
    assert _status_of(L.csa_index_topk_fp8, **dict(base, key_scales=None)) == 1
    assert _status_of(L.csa_index_topk_fp8, **dict(base, ws_bytes=1024)) == 4   # workspace
    assert _status_of(L.csa_index_keys_pack, p=p, keys=FAKE, n_rows=4, idx_dim=64, codes=FAKE,
                      scales=FAKE) == 2
    # the E4M3 workspace adds the query codes and weights to the bf16 one
    a = L.csa_workspace_bytes(p, L.OP_INDEX_TOPK, 2, 8, 64, 64, 4096, 128)
    b = L.csa_workspace_bytes(p, L.OP_INDEX_TOPK_FP8, 2, 8, 64, 64, 4096, 128)
    assert b >= a + 8 * 64 * 128 + 8 * 64 * 4


def test_batch_invariant_attend_needs_its_own_workspace(L):
    """A workspace sized for the balanced splits is too small for the fixed
    ones at the decode shape (32 queries of 18 tiles: at most a few CTAs meet a
    query, 9 fixed splits each): the call is refused before any launch."""
    base = L.params(512, 4, topk=1024)
    inv = L.params(512, 4, topk=1024, batch_invariant=True)
    n_def = L.csa_workspace_bytes(base, L.OP_ATTEND, 32, 32, 64, 0, 32768, 128)
    n_inv = L.csa_workspace_bytes(inv, L.OP_ATTEND, 32, 32, 64, 0, 32768, 128)
    assert n_inv > n_def
    kw = _attend_args(L, inv, B=32, Q=32, n_cap=32768, ws_bytes=n_def)
    assert _status_of(L.csa_attend, **kw) == 4  # CSA_ERR_WORKSPACE


def test_noalloc_refuses_an_oversized_selection_before_any_launch(L):
    # fits the static scratch (1 x 4194304 scores) but not the top-k merge's shared
    # memory (128 chunks x 1024 candidates): refused before the status word is cleared
    p = L.params(512, 4, topk=1024)
    n0 = L.csa_launch_count()
    with pytest.raises(L.CsaError) as ei:
        L.csa_index_topk_noalloc(p, FAKE, FAKE, 64, 128, FAKE, 4194304, 1, 1, FAKE, FAKE, None, None)
    assert ei.value.status == 2 and "shared memory" in L.csa_last_error()
    assert L.csa_launch_count() == n0


def test_ring_window_needs_room_for_the_window(L):
    # win_pos0 NULL: the window buffer is a ring and must hold W rows
    p = L.params(512, 4, topk=64, window=128)
    n0 = L.csa_launch_count()
    assert _status_of(L.csa_attend, **_attend_args(L, p, win_pos0=None, n_win=100)) == 1
    assert "ring" in L.csa_last_error()
    assert L.csa_launch_count() == n0


def test_workspace_covers_both_window_layouts(L):
    # one workspace size serves the linear and the ring window (a ring of more
    # than W rows is read in more tiles)
    p = L.params(512, 4, topk=1024, window=128)
    a = L.csa_workspace_bytes(p, L.OP_ATTEND, 2, 2, 64, 64, 4096, 128)
    b = L.csa_workspace_bytes(p, L.OP_ATTEND, 2, 2, 64, 64, 4096, 512)
    assert b >= a > 0


def test_decode_append_validation(L):
    p = L.params(512, 4)
    base = dict(p=p, kv_tok=FAKE, B=2, pos=FAKE, raw_ring=FAKE, w_z=FAKE, bias=FAKE, cache=FAKE,
                n_cap=100, window=FAKE, n_win=128, ws=FAKE, ws_bytes=256)
    n0 = L.csa_launch_count()
    assert _status_of(L.csa_decode_append, **dict(base, pos=None)) == 1
    assert _status_of(L.csa_decode_append, **dict(base, raw_ring=None)) == 1   # m > 1 needs the ring
    assert _status_of(L.csa_decode_append, **dict(base, kv_tok=FAKE + 4)) == 1
    assert _status_of(L.csa_decode_append, **dict(base, ws_bytes=100)) == 4
    assert _status_of(L.csa_decode_append, **dict(base, B=-1)) == 1
    # a block too large to stage: 1024 fp32 tokens of 512 dims
    big = L.params(512, 1024, act="f32", kv="f32")
    assert _status_of(L.csa_decode_append, **dict(base, p=big)) == 2
    assert L.csa_launch_count() == n0


def test_grouped_out_proj_validation(L):
    n0 = L.csa_launch_count()
    base = dict(o=FAKE, Q=4, H=64, D=512, G=8, w=FAKE, d_g=512, out=FAKE, ws=FAKE, ws_bytes=256)
    assert _status_of(L.csa_grouped_out_proj, **dict(base, G=7)) == 2      # H % G
    assert _status_of(L.csa_grouped_out_proj, **dict(base, d_g=100)) == 2  # d_g % 64
    assert _status_of(L.csa_grouped_out_proj, **dict(base, o=FAKE + 8)) == 1
    assert _status_of(L.csa_grouped_out_proj, **dict(base, ws_bytes=16)) == 4
    # decode-sized calls may use float32 sums in the workspace; larger ones need the status word only
    assert L.csa_grouped_out_proj_ws_bytes(32, 8, 512) == 256 + 4 * 32 * 8 * 512
    assert L.csa_grouped_out_proj_ws_bytes(129, 8, 512) == 256
    assert L.csa_grouped_out_proj_ws_bytes(-1, 8, 512) == 0
    assert L.csa_launch_count() == n0
