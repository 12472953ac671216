"""KV relocation oracle (test infrastructure only: the product never imports it).

The second, "live" tier of KV defragmentation moves each request's scattered
prefix rows into contiguous rows and rewrites the indices that point at them
[The Art of Knowing When to Stop: Deferring Tier 1 Defrag, §"The Decision:
Why Tier 1 Defrag Gets Deferred"].  Written out row by row: for request b
and prefix key j, row kv_indices[kv_indptr[b] + j] is copied to row
dst_start[b] + j, and the index becomes dst_start[b] + j.  Destination rows
are free rows (no source row lies in a destination block), so the copies
commute.  A key whose source or destination row is outside the pool is left
as it was and reported.
"""

from __future__ import annotations

from typing import Tuple

import numpy as np


def relocate(pool: np.ndarray, kv_indptr, kv_indices, dst_start, batch: int) -> Tuple[np.ndarray, np.ndarray, bool]:
    """Returns (new pool, new indices, whether some key was out of range).

    `pool` is any array with one row per pool row (bf16 rows as uint16, for
    instance); the inputs are not modified.
    """
    pool_rows = pool.shape[0]
    new_pool = pool.copy()
    new_idx = np.array(kv_indices, dtype=np.int64).copy()
    bad = False
    for b in range(batch):
        start, end = int(kv_indptr[b]), int(kv_indptr[b + 1])
        for k in range(start, end):
            src = int(kv_indices[k])
            dst = int(dst_start[b]) + (k - start)
            if not (0 <= src < pool_rows and 0 <= dst < pool_rows):
                bad = True
                continue
            new_pool[dst] = pool[src]
            new_idx[k] = dst
    return new_pool, new_idx.astype(np.int32), bad
