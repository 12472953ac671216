"""Seeded synthetic inputs for MLA tree-verify attention.

This module only draws numbers and lays them out in the argument formats of
the verify call; it holds none of the attention arithmetic.  Both the CUDA
path (through the C-ABI) and the CPU oracle consume what it produces.

Shapes follow the verify step of speculative decoding over a paged latent KV
cache with page_size=1 [Custom sm_120 Verify Kernel, §"The Bottleneck:
Triton's Scattered KV Access at 14 GB/s"]: every pool row is one token, 512
latent values followed by 64 RoPE values, stored as bf16.  Prefix rows are
addressed through ``kv_indptr``/``kv_indices`` and the draft tokens' rows
through ``out_cache_loc`` [Capture Safety to MoE Ceiling, §"The Architecture
of Capture Safety"; Custom sm_120 Verify Kernel, §"The Debugging Gauntlet"].
The tree-visibility mask is packed LSB-first, row-major over
``[q_len, prefix + q_len]`` per request, with ``mask_indptr[b]`` holding the
bit offset of request ``b`` (B entries, not B+1) [Custom sm_120 Verify
Kernel, §"The Debugging Gauntlet", bugs 2 and 3].

Recipe: ``numpy.random.default_rng(seed)`` (PCG64); values ~ N(0,1) drawn in
float32 then rounded to bf16 (round-to-nearest-even); draw order: pool,
q_nope, q_rope, prefix lengths, indices, trees.
"""

from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Sequence

import numpy as np

D_LATENT = 512
D_ROPE = 64
D_ROW = D_LATENT + D_ROPE


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest-even) and return the raw uint16 bits."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    flat_in = x.reshape(-1).view(np.uint32)
    flat_out = out.reshape(-1)
    step = 1 << 24
    for s in range(0, flat_in.size, step):
        u = flat_in[s:s + step]
        lsb = (u >> 16) & np.uint32(1)
        r = (u + np.uint32(0x7FFF) + lsb) >> 16
        # NaN stays NaN (quiet bit set); finite overflow rounds to inf as in IEEE.
        nan = (u & np.uint32(0x7FFFFFFF)) > np.uint32(0x7F800000)
        r = np.where(nan, (u >> 16) | np.uint32(0x40), r)
        flat_out[s:s + step] = r.astype(np.uint16)
    return out


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def normal_bf16(rng: np.random.Generator, shape, chunk_rows: int = 1 << 16) -> np.ndarray:
    """N(0,1) float32 draws rounded to bf16 bits, drawn row-chunk by row-chunk."""
    shape = tuple(shape)
    out = np.empty(shape, dtype=np.uint16)
    if len(shape) == 0 or shape[0] == 0:
        return out
    rows = shape[0]
    for s in range(0, rows, chunk_rows):
        e = min(rows, s + chunk_rows)
        out[s:e] = f32_to_bf16_bits(rng.standard_normal((e - s,) + shape[1:], dtype=np.float32))
    return out


def random_tree(rng: np.random.Generator, T: int) -> np.ndarray:
    """Draft tree: node 0 is the root, node i>0 has a parent uniform in 0..i-1."""
    parent = np.full(T, -1, dtype=np.int32)
    for i in range(1, T):
        parent[i] = rng.integers(0, i)
    return parent


def chain_tree(T: int) -> np.ndarray:
    parent = np.arange(-1, T - 1, dtype=np.int32)
    return parent


def tree_visibility(parent: np.ndarray) -> np.ndarray:
    """[T, T] bool: node i sees node j iff j is i or an ancestor of i."""
    T = parent.shape[0]
    vis = np.zeros((T, T), dtype=bool)
    for i in range(T):
        j = i
        while j >= 0:
            vis[i, j] = True
            j = int(parent[j])
    return vis


def pack_bits_lsb(bits: np.ndarray) -> np.ndarray:
    """Pack a flat bool array LSB-first into bytes (bit k -> byte k//8, bit k%8)."""
    return np.packbits(np.asarray(bits, dtype=np.uint8).reshape(-1), bitorder="little")


def build_mask(prefix_lens: Sequence[int], parents: Sequence[np.ndarray], T,
               prefix_visible: Optional[List[np.ndarray]] = None):
    """Dense per-request visibility rows -> (packed bytes, bit offsets, dense list).

    Request b contributes a row-major [T_b, P_b + T_b] block (T an int, or one
    draft-token count per request); the first P_b columns are prefix tokens
    (visible unless ``prefix_visible`` says otherwise), the last T_b columns
    follow the draft tree.
    """
    Ts = [int(t) for t in T] if hasattr(T, "__len__") else [int(T)] * len(prefix_lens)
    dense = []
    offsets = np.zeros(len(prefix_lens), dtype=np.int64)
    total = 0
    for b, P in enumerate(prefix_lens):
        Tb = Ts[b]
        L = P + Tb
        m = np.zeros((Tb, L), dtype=bool)
        if prefix_visible is None:
            m[:, :P] = True
        else:
            m[:, :P] = prefix_visible[b]
        m[:, P:] = tree_visibility(parents[b])
        dense.append(m)
        offsets[b] = total
        total += Tb * L
    flat = np.concatenate([d.reshape(-1) for d in dense]) if dense else np.zeros(0, bool)
    packed = pack_bits_lsb(flat)
    if packed.size == 0:
        packed = np.zeros(1, dtype=np.uint8)
    return packed, offsets, dense


def sorted_free_list_rows(rng: np.random.Generator, n: int, pool_rows: int,
                          mean_run: int = 256, mean_gap: int = 256) -> np.ndarray:
    """Ascending runs of contiguous rows (geometric lengths) separated by geometric gaps."""
    rows = np.empty(n, dtype=np.int64)
    filled = 0
    span_est = int(n * (1 + mean_gap / mean_run)) + 4 * mean_run
    start = int(rng.integers(0, max(1, pool_rows - span_est)))
    cur = start
    while filled < n:
        run = int(rng.geometric(1.0 / mean_run))
        run = min(run, n - filled)
        if cur + run > pool_rows:
            raise ValueError("pool too small for the sorted free-list layout")
        rows[filled:filled + run] = np.arange(cur, cur + run)
        filled += run
        cur += run + int(rng.geometric(1.0 / mean_gap))
    return rows


def place_rows(rng: np.random.Generator, layout: str, n: int, pool_rows: int) -> np.ndarray:
    """Physical rows for n logical keys: "scattered" (sample without replacement),
    "sorted" (sorted free list with runs), or "contiguous" (one run)."""
    if layout == "scattered":
        return rng.permutation(pool_rows)[:n].astype(np.int64)
    if layout == "sorted":
        return sorted_free_list_rows(rng, n, pool_rows)
    if layout == "contiguous":
        start = int(rng.integers(0, pool_rows - n + 1))
        return np.arange(start, start + n, dtype=np.int64)
    raise ValueError(layout)


@dataclasses.dataclass(frozen=True)
class VerifyConfig:
    name: str
    B: int
    H: int
    T: int
    prefix: object  # int, or (lo, hi) for a uniform ragged draw per request
    pool_rows: int
    nsplit: int
    tree: str = "random"  # "random" | "chain"
    layout: str = "scattered"  # "scattered" | "sorted"
    needle: bool = False
    seed: int = 0
    T_range: Optional[tuple] = None  # (lo, hi): per-request draft-token counts T_b ~ U[lo, hi]; T = hi

    @property
    def sm_scale(self) -> float:
        return 1.0 / math.sqrt(192.0)


# The five workloads and the regression cases.  Sizes follow the pages'
# deployment (9-token draft trees, 64 heads on one GPU or 8 per TP8 rank,
# contexts from 256 to 185k tokens).
CONFIGS = {
    "tiny": VerifyConfig("tiny", B=1, H=16, T=4, prefix=256, pool_rows=4096, nsplit=4, tree="chain"),
    "short4k": VerifyConfig("short4k", B=1, H=64, T=9, prefix=4096, pool_rows=262144, nsplit=16),
    "mid64k": VerifyConfig("mid64k", B=1, H=64, T=9, prefix=65536, pool_rows=1048576, nsplit=64),
    "mid64k_sorted": VerifyConfig("mid64k_sorted", B=1, H=64, T=9, prefix=65536, pool_rows=1048576,
                                  nsplit=64, layout="sorted"),
    "long185k_h8": VerifyConfig("long185k_h8", B=1, H=8, T=9, prefix=185000, pool_rows=1048576, nsplit=64),
    "batch16_ragged": VerifyConfig("batch16_ragged", B=16, H=64, T=9, prefix=(1024, 32768),
                                   pool_rows=1048576, nsplit=16),
    # regression: 21 prefix + 9 draft tokens (the extend-layout bug)
    "reg_p21": VerifyConfig("reg_p21", B=1, H=64, T=9, prefix=21, pool_rows=4096, nsplit=4),
    # regression: two requests, mask_indptr has B entries
    "reg_b2": VerifyConfig("reg_b2", B=2, H=16, T=9, prefix=(100, 700), pool_rows=8192, nsplit=8),
    # peaked softmax: a few planted keys score far above the rest
    "needle64k": VerifyConfig("needle64k", B=1, H=64, T=9, prefix=65536, pool_rows=1048576, nsplit=64,
                              needle=True),
    # T = 1 decode on the verify kernels, and per-request draft-token counts
    "decode_b16": VerifyConfig("decode_b16", B=16, H=64, T=1, prefix=(1024, 32768), pool_rows=1048576,
                               nsplit=16),
    # decode on one tensor-parallel shard (8 heads): the CUDA-core kernel's shape
    "decode_h8_b16": VerifyConfig("decode_h8_b16", B=16, H=8, T=1, prefix=(1024, 32768), pool_rows=1048576,
                                  nsplit=16),
    "varlen_b16": VerifyConfig("varlen_b16", B=16, H=64, T=16, prefix=(1024, 32768), pool_rows=1048576,
                               nsplit=16, T_range=(1, 16)),
}


def prefix_lengths(cfg: VerifyConfig, rng: np.random.Generator) -> np.ndarray:
    if isinstance(cfg.prefix, tuple):
        lo, hi = cfg.prefix
        return rng.integers(lo, hi + 1, size=cfg.B).astype(np.int64)
    return np.full(cfg.B, int(cfg.prefix), dtype=np.int64)


def make_workload(cfg: VerifyConfig, seed: Optional[int] = None, layout: Optional[str] = None,
                  prefix_override: Optional[Sequence[int]] = None) -> dict:
    """Draw one verify-call input set for ``cfg`` (all arrays on the host)."""
    seed = cfg.seed if seed is None else seed
    if cfg.T_range is not None:
        rng = np.random.default_rng(seed + 1)
        P = prefix_lengths(cfg, rng) if prefix_override is None else np.asarray(prefix_override, np.int64)
        T_list = rng.integers(cfg.T_range[0], cfg.T_range[1] + 1, size=cfg.B)
        wl = varlen_workload(cfg.B, cfg.H, T_list.tolist(), P.tolist(), cfg.pool_rows, seed, cfg.nsplit,
                             tree=cfg.tree, layout=cfg.layout if layout is None else layout)
        wl["cfg"] = cfg
        wl["T"] = int(cfg.T_range[1])  # the plan's q_len bounds every T_b
        return wl
    layout = cfg.layout if layout is None else layout
    rng = np.random.default_rng(seed)
    B, H, T = cfg.B, cfg.H, cfg.T

    pool = normal_bf16(rng, (cfg.pool_rows, D_ROW))
    q_nope = normal_bf16(rng, (B * T, H, D_LATENT))
    q_rope = normal_bf16(rng, (B * T, H, D_ROPE))
    if prefix_override is not None:
        P = np.asarray(prefix_override, dtype=np.int64)
        assert P.shape == (B,)
    else:
        P = prefix_lengths(cfg, rng)
    n_rows = int(P.sum()) + B * T
    if n_rows > cfg.pool_rows:
        raise ValueError("pool smaller than the rows one call addresses")

    phys = place_rows(rng, layout, n_rows, cfg.pool_rows)

    kv_indptr = np.zeros(B + 1, dtype=np.int64)
    kv_indptr[1:] = np.cumsum(P)
    prefix_phys = phys[: int(P.sum())]
    draft_phys = phys[int(P.sum()):]
    kv_indices = prefix_phys.astype(np.int32)
    out_cache_loc = draft_phys.astype(np.int32)

    parents = []
    for _ in range(B):
        parents.append(chain_tree(T) if cfg.tree == "chain" else random_tree(rng, T))
    custom_mask, mask_indptr, dense = build_mask(P.tolist(), parents, T)

    wl = dict(
        cfg=cfg, seed=seed, layout=layout,
        B=B, H=H, T=T, pool_rows=cfg.pool_rows, nsplit=cfg.nsplit, sm_scale=cfg.sm_scale,
        prefix_lens=P, pool=pool, q_nope=q_nope, q_rope=q_rope,
        kv_indptr=kv_indptr.astype(np.int32), kv_indices=kv_indices, out_cache_loc=out_cache_loc,
        custom_mask=custom_mask, mask_indptr=mask_indptr.astype(np.int32),
        parents=parents, dense_mask=dense,
    )
    if cfg.needle:
        plant_needles(wl, np.random.default_rng(seed + 7))
    return wl


def logical_rows(wl: dict) -> np.ndarray:
    """Physical pool row of every (request, key position) in call order."""
    out = []
    for b in range(wl["B"]):
        s, e = int(wl["kv_indptr"][b]), int(wl["kv_indptr"][b + 1])
        out.append(wl["kv_indices"][s:e])
        out.append(wl["out_cache_loc"][b * wl["T"]:(b + 1) * wl["T"]])
    return np.concatenate(out).astype(np.int64)


def relayout(wl: dict, layout: str, seed: int) -> dict:
    """Same logical KV rows and queries, placed at new physical rows.

    Rows that the call does not address are refilled from an independent
    stream, so only the addressed values are shared between the two layouts.
    """
    rng = np.random.default_rng(seed)
    old_rows = logical_rows(wl)
    n = old_rows.size
    new_rows = place_rows(rng, layout, n, wl["pool_rows"])
    pool = normal_bf16(np.random.default_rng(seed + 1), wl["pool"].shape)
    pool[new_rows] = wl["pool"][old_rows]
    out = dict(wl)
    out["layout"] = layout
    out["pool"] = pool
    P = wl["prefix_lens"]
    pos = 0
    kv_idx, ocl = [], []
    for b in range(wl["B"]):
        kv_idx.append(new_rows[pos:pos + int(P[b])])
        pos += int(P[b])
        ocl.append(new_rows[pos:pos + wl["T"]])
        pos += wl["T"]
    out["kv_indices"] = np.concatenate(kv_idx).astype(np.int32) if kv_idx else np.zeros(0, np.int32)
    out["out_cache_loc"] = np.concatenate(ocl).astype(np.int32)
    return out


def plant_needles(wl: dict, rng: np.random.Generator, per_request: int = 4,
                  q_shift: float = 8.0, k_len: float = 35.0):
    """Plant a few prefix keys that score far above the rest for every query.

    A random unit direction e in the 64-dim RoPE space is added (times
    ``q_shift``) to every query's RoPE part, and the RoPE part of the planted
    key rows is set to ``k_len * e``.  Their scores rise by about
    q_shift * k_len * sm_scale (~20 natural-log units at the default scale)
    while their 512 latent (value) entries stay N(0,1), so the softmax is
    peaked and |O| ~ 1.
    """
    T = wl["T"]
    e = rng.standard_normal(D_ROPE)
    e /= np.linalg.norm(e)
    qr = bf16_bits_to_f32(wl["q_rope"]).astype(np.float64)
    needle_rows = []
    for b in range(wl["B"]):
        P = int(wl["prefix_lens"][b])
        if P == 0:
            continue
        qr[b * T:(b + 1) * T] += q_shift * e
        js = rng.choice(P, size=min(per_request, P), replace=False)
        base = int(wl["kv_indptr"][b])
        for j in js:
            row = int(wl["kv_indices"][base + int(j)])
            wl["pool"][row, D_LATENT:] = f32_to_bf16_bits((k_len * e).astype(np.float32))
            needle_rows.append(row)
    wl["q_rope"] = f32_to_bf16_bits(qr.astype(np.float32))
    wl["needle_rows"] = np.asarray(needle_rows, dtype=np.int64)


def with_free_block(wl: dict, seed: int) -> dict:
    """Inputs of a KV relocation: the call's rows moved clear of a free block.

    Same logical rows and queries as ``wl`` (uniform q_len), but every row the
    call addresses is placed, scattered, at rows >= sum(P_b), so rows
    [0, sum(P_b)) are free; ``dst_start[b]`` = kv_indptr[b] - kv_indptr[0] is
    the contiguous destination of request b's prefix.  Unaddressed rows are
    refilled from an independent stream.
    """
    assert "qo_indptr" not in wl
    rng = np.random.default_rng(seed)
    old_rows = logical_rows(wl)
    n = old_rows.size
    free = int(np.asarray(wl["prefix_lens"]).sum())
    if free + n > wl["pool_rows"]:
        raise ValueError("pool too small for a free block beside the call's rows")
    new_rows = free + rng.choice(wl["pool_rows"] - free, size=n, replace=False)
    pool = normal_bf16(np.random.default_rng(seed + 1), wl["pool"].shape)
    pool[new_rows] = wl["pool"][old_rows]
    out = dict(wl)
    out["pool"] = pool
    P = wl["prefix_lens"]
    pos = 0
    kv_idx, ocl = [], []
    for b in range(wl["B"]):
        kv_idx.append(new_rows[pos:pos + int(P[b])])
        pos += int(P[b])
        ocl.append(new_rows[pos:pos + wl["T"]])
        pos += wl["T"]
    out["kv_indices"] = np.concatenate(kv_idx).astype(np.int32) if kv_idx else np.zeros(0, np.int32)
    out["out_cache_loc"] = np.concatenate(ocl).astype(np.int32)
    out["dst_start"] = (wl["kv_indptr"][:-1] - wl["kv_indptr"][0]).astype(np.int32)
    return out


def tiny_workload(B: int, H: int, T: int, prefix_lens: Sequence[int], pool_rows: int, seed: int,
                  tree: str = "random", nsplit: int = 2) -> dict:
    """Small ad-hoc workload (same recipe) for oracle pins and edge cases."""
    cfg = VerifyConfig("adhoc", B=B, H=H, T=T, prefix=0, pool_rows=pool_rows, nsplit=nsplit, tree=tree,
                       seed=seed)
    return make_workload(cfg, seed=seed, prefix_override=list(prefix_lens))


def varlen_workload(B: int, H: int, T_list: Sequence[int], prefix_lens: Sequence[int], pool_rows: int,
                    seed: int, nsplit: int = 2, tree: str = "random", layout: str = "scattered") -> dict:
    """A verify call whose requests have their own draft-token counts T_b.

    Token rows of request b are qo_indptr[b] .. qo_indptr[b+1]-1 (qo_indptr =
    [0, cumsum(T_b)]); its draft rows are out_cache_loc[qo_indptr[b] + t] and
    its mask block is [T_b, P_b + T_b].  The query buffers hold B * max(T_b)
    token rows (the tail past qo_indptr[B] is padding a device kernel may
    read but never uses); ``T`` is max(T_b), the plan's q_len.
    """
    rng = np.random.default_rng(seed)
    Ts = np.asarray([int(t) for t in T_list], dtype=np.int64)
    assert Ts.shape == (B,) and (Ts >= 0).all()
    T = max(1, int(Ts.max()) if B else 1)
    pool = normal_bf16(rng, (pool_rows, D_ROW))
    q_nope = normal_bf16(rng, (B * T, H, D_LATENT))
    q_rope = normal_bf16(rng, (B * T, H, D_ROPE))
    P = np.asarray(prefix_lens, dtype=np.int64)
    n_tok = int(Ts.sum())
    n_rows = int(P.sum()) + n_tok
    if n_rows > pool_rows:
        raise ValueError("pool smaller than the rows one call addresses")
    phys = place_rows(rng, layout, n_rows, pool_rows)
    kv_indptr = np.zeros(B + 1, dtype=np.int64)
    kv_indptr[1:] = np.cumsum(P)
    qo_indptr = np.zeros(B + 1, dtype=np.int64)
    qo_indptr[1:] = np.cumsum(Ts)
    kv_indices = phys[: int(P.sum())].astype(np.int32)
    out_cache_loc = np.zeros(B * T, dtype=np.int32)  # capacity B*T, padding rows name pool row 0
    out_cache_loc[:n_tok] = phys[int(P.sum()):]
    parents = [chain_tree(int(t)) if tree == "chain" else random_tree(rng, int(t)) for t in Ts]
    custom_mask, mask_indptr, dense = build_mask(P.tolist(), parents, Ts.tolist())
    cfg = VerifyConfig("varlen", B=B, H=H, T=T, prefix=0, pool_rows=pool_rows, nsplit=nsplit, tree=tree,
                       layout=layout, seed=seed)
    return dict(
        cfg=cfg, seed=seed, layout=layout,
        B=B, H=H, T=T, T_list=Ts, qo_indptr=qo_indptr.astype(np.int32), n_tokens=n_tok,
        pool_rows=pool_rows, nsplit=nsplit, sm_scale=cfg.sm_scale,
        prefix_lens=P, pool=pool, q_nope=q_nope, q_rope=q_rope,
        kv_indptr=kv_indptr.astype(np.int32), kv_indices=kv_indices, out_cache_loc=out_cache_loc,
        custom_mask=custom_mask, mask_indptr=mask_indptr.astype(np.int32),
        parents=parents, dense_mask=dense,
    )
