"""Host simulation of the top-k kernels' vector shared-memory accesses.

The selection kernels read and write their keys in shared memory with
16-byte accesses (four keys at a time) and read the cluster partners'
histogram pairs and totals with 8-byte accesses.  This test re-derives, on the
host, every index those accesses use for the shapes the kernels accept, and
checks that each 16-byte access starts on a multiple of four keys and stays
inside the keys the CTA holds (within its dynamic shared-memory allocation),
and that the 8-byte accesses start on even words.  It restates the kernels'
index arithmetic (warp ranges of sweep_seg keys, 128 keys per warp step, four
per lane; the cluster's slice bounds rounded down to multiples of four; the
allocation sizes of the launcher), so a change there must be mirrored here.
"""
import random

K_THREADS = 1024
K_WARPS = K_THREADS // 32
K_CHUNK = 32768
K_BINS = 2048
CLUSTER_CS = 4
CLUSTER_MIN_KEYS = 4096


def sweep_seg(n):
    return ((n + K_WARPS - 1) // K_WARPS + 127) & ~127


def check_sweeps(n, alloc_keys):
    """Every load4 of the sweeps over keys[0, n): 16-byte loads only when all
    four keys exist; every such load aligned and inside the allocation."""
    seg = sweep_seg(n)
    assert seg % 128 == 0
    for warp in range(K_WARPS):
        i0 = warp * seg
        i1 = min(n, i0 + seg)
        for r in range(i0, i1, 128):
            for lane in range(32):
                i = r + 4 * lane
                if i + 3 < i1:            # the vector path
                    assert i % 4 == 0
                    assert i + 4 <= n <= alloc_keys
                else:                      # scalar path: keys below i1 only
                    for e in range(4):
                        if i + e < i1:
                            assert i + e < n


def check_load_keys(n, alloc_keys):
    """load_keys: 16-byte stores of keys 4j .. 4j+3 for j < n // 4, the rest one by one."""
    n4 = n // 4
    assert 4 * n4 <= n <= alloc_keys
    # the batched loop visits j0 + u*1024 < n4 only
    for j in (0, n4 - 1) if n4 else ():
        assert 4 * j + 3 < n


def round16(b):
    return (b + 15) & ~15


def chunk_alloc_keys(n_cap):
    n = n_cap if n_cap < K_CHUNK else K_CHUNK
    return round16(max(n, 1) * 4) // 4


def test_single_cta_sweeps_are_aligned_and_in_bounds():
    rng = random.Random(5)
    sizes = sorted(set([1, 2, 3, 4, 5, 31, 127, 128, 129, 130, 4095, 4096, 4097, 8191, 16384, 32767,
                        K_CHUNK] + [rng.randrange(1, K_CHUNK + 1) for _ in range(40)]))
    for n_cap in sizes:
        alloc = chunk_alloc_keys(n_cap)
        for n in {n_cap, max(1, n_cap - 1), max(1, n_cap // 2 + 1)}:
            check_sweeps(n, alloc)
            check_load_keys(n, alloc)


def test_merge_sweeps_are_aligned_and_in_bounds():
    # the merge CTA holds ceil(n / C) * k candidates (at most 40960 keys)
    for nch, k in [(2, 1024), (3, 1024), (10, 4096), (40, 1024), (5, 1), (7, 13)]:
        C = nch * k
        if C > 40960:
            continue
        alloc = round16(C * 4) // 4
        check_sweeps(C, alloc)


def test_cluster_slices_are_aligned_and_in_bounds():
    rng = random.Random(9)
    caps = sorted(set([CLUSTER_MIN_KEYS, 4097, 5000, 8192, 32767, K_CHUNK] +
                      [rng.randrange(CLUSTER_MIN_KEYS, K_CHUNK + 1) for _ in range(30)]))
    for n_cap in caps:
        alloc = round16((n_cap // CLUSTER_CS + 4) * 4) // 4
        for n in {n_cap, n_cap - 3, (n_cap * 2) // 3 + 1}:
            if n < 1:
                continue
            bnd = [n if r == CLUSTER_CS else (r * n // CLUSTER_CS) & ~3 for r in range(CLUSTER_CS + 1)]
            for r in range(CLUSTER_CS):
                lo, nc = bnd[r], bnd[r + 1] - bnd[r]
                assert lo % 4 == 0          # the slice's global loads start 16-byte aligned
                assert 0 <= nc <= alloc, (n_cap, n, r, nc, alloc)
                check_sweeps(nc, alloc) if nc > 0 else None
                check_load_keys(nc, alloc)


def test_cluster_pair_reads_are_8_byte_aligned():
    # digit search: thread t reads bins b1 = 2046 - 2t (even) and b0 = b1 + 1 as one 8-byte
    # pair from a 16-byte aligned histogram; the totals pair ctot sits at an 8-byte offset
    for tid in range(K_THREADS):
        b0 = K_BINS - 1 - 2 * tid
        b1 = b0 - 1
        assert b1 >= 0 and b1 % 2 == 0 and b0 == b1 + 1
        assert (b1 * 4) % 8 == 0
