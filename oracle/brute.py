"""Brute-force enumeration of MLA tree-verify attention (test infrastructure).

Pure Python, tiny inputs only.  Unlike the C oracle it never reads the packed
mask: visibility comes straight from the draft tree (parent array), with the
prefix visible to every draft token, and every sum is taken with
``math.fsum``.  Agreement with the C oracle therefore pins the mask decoding
(bit order, row stride prefix + q_len, per-request bit offsets) and the
two-array row selection [Custom sm_120 Verify Kernel, §"The Debugging
Gauntlet"; Capture Safety to MoE Ceiling, §"The Architecture of Capture
Safety"].
"""

from __future__ import annotations

import math
import struct
from typing import Optional, Sequence


def _bf16(u: int) -> float:
    return struct.unpack("<f", struct.pack("<I", (int(u) & 0xFFFF) << 16))[0]


def _ancestors_and_self(parent, i):
    out = set()
    j = i
    while j >= 0:
        out.add(j)
        j = int(parent[j])
    return out


def brute_verify(wl: dict, rows: Optional[Sequence[int]] = None):
    """Return (list of 512-lists, list of LSE) for the selected output rows."""
    B, H, T = wl["B"], wl["H"], wl["T"]
    scale = float(wl["sm_scale"])
    pool = wl["pool"]
    qn, qr = wl["q_nope"], wl["q_rope"]
    # request b's tokens: token rows q0[b] .. q0[b] + Tb[b] - 1
    if wl.get("qo_indptr") is not None:
        qo = [int(x) for x in wl["qo_indptr"]]
        q0 = qo[:-1]
        Tb = [qo[b + 1] - qo[b] for b in range(B)]
    else:
        q0 = [b * T for b in range(B)]
        Tb = [T] * B
    owner = {}
    for b in range(B):
        for i in range(Tb[b]):
            owner[q0[b] + i] = (b, i)
    if rows is None:
        rows = range(sum(Tb) * H)
    outs, lses = [], []
    for r in rows:
        r = int(r)
        h = r % H
        b, i = owner[r // H]
        P = int(wl["kv_indptr"][b + 1]) - int(wl["kv_indptr"][b])
        seen = _ancestors_and_self(wl["parents"][b], i)
        q = [_bf16(x) for x in qn[q0[b] + i, h]] + [_bf16(x) for x in qr[q0[b] + i, h]]
        scores, vals = [], []
        for j in range(P + Tb[b]):
            if j < P:
                row = int(wl["kv_indices"][int(wl["kv_indptr"][b]) + j])
            else:
                if (j - P) not in seen:
                    continue
                row = int(wl["out_cache_loc"][q0[b] + (j - P)])
            k = [_bf16(x) for x in pool[row]]
            scores.append(scale * math.fsum(qa * ka for qa, ka in zip(q, k)))
            vals.append(k[:512])
        if not scores:
            outs.append([0.0] * 512)
            lses.append(-math.inf)
            continue
        m = max(scores)
        w = [math.exp(s - m) for s in scores]
        Z = math.fsum(w)
        outs.append([math.fsum(wj * v[d] for wj, v in zip(w, vals)) / Z for d in range(512)])
        lses.append(m + math.log(Z))
    return outs, lses
