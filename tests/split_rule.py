"""The key-range split rule of the FP8 attention plan, restated for the tests.

A call's work items (one per 128-query tile of a (segment, head)) are N; on a
GPU with S SMs the last wave holds r = N mod S items.  When 0 < r <= S / 2,
each of those items is cut into k = min(S / r, MAX_K, MAX_PARTS / r) parts,
further limited to the key tiles (256 keys) of the segments involved; k < 2
means no split.  Records are in longest-first order (up to 2048 segments).
"""

import numpy as np

BN = 256            # keys per tile
ROWS = 128          # queries per work item
MAX_K = 4           # parts per item at most
MAX_PARTS = 160     # split CTAs at most


def expected_split(seqlens, H, n_sm):
    """(total items, first split item, parts per item) as the plan decides them."""
    cu = np.concatenate([[0], np.cumsum(seqlens)]).astype(np.int64)
    n = len(seqlens)
    order = sorted(range(n), key=lambda b: (-seqlens[b], b)) if n <= 2048 else list(range(n))
    first, recs = 0, []
    for b in order:
        nq = -(-seqlens[b] // ROWS)
        recs.append((first, int(cu[b]), int(cu[b + 1]), nq))
        first += nq * H
    N = first
    r = N % n_sm
    if r == 0 or 2 * r > n_sm:
        return N, N, 1
    k = min(n_sm // r, MAX_K, MAX_PARTS // r)
    for f, s, e, nq in reversed(recs):
        if nq == 0:
            continue
        if f + nq * H <= N - r:
            break
        k = min(k, (e - (s & ~15) + BN - 1) // BN)
    return (N, N - r, k) if k >= 2 else (N, N, 1)


