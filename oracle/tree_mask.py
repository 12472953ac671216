"""Tree-mask oracle (test infrastructure only: the product never imports it).

The packed visibility mask of a verify call, from the draft trees' parent
arrays, written out bit by bit with plain loops.  Layout: request b's
row-major [q_len, P_b + q_len] block of bits starts at bit offset
mask_indptr[b] = q_len * sum_{b'<b} (P_b' + q_len); bits are packed
LSB-first within each byte [Custom sm_120 Verify Kernel, §"The Debugging
Gauntlet"].  Bit (i, j) is 1 when j < P_b (every draft token sees the whole
prefix) or when draft node j - P_b is node i or an ancestor of i: a node of
the tree sees itself and its ancestors [Capture Safety to MoE Ceiling,
§"The Architecture of Capture Safety"; the tree semantics are the reading
stated with the inputs].  A parent link outside [-1, node) ends the walk, as
in the device builder's contract.  In a varlen call request b has its own
draft-token count T_b: its block is [T_b, P_b + T_b] and the offsets sum
T_b * (P_b + T_b) (the uniform layout with q_len replaced by T_b).
"""

from __future__ import annotations

import numbers
from typing import List, Sequence, Tuple, Union


def sees(parent: Sequence[int], i: int, d: int) -> bool:
    """True when node d is node i or one of its ancestors."""
    n = i
    while n >= 0:
        if n == d:
            return True
        p = int(parent[n])
        n = p if 0 <= p < n else -1
    return False


def _counts(T: Union[int, Sequence[int]], n: int) -> List[int]:
    """Draft-token count of each request: one q_len for all, or one per request."""
    return [int(T)] * n if isinstance(T, numbers.Integral) else [int(t) for t in T]


def mask_bits(parents: Sequence[Sequence[int]], prefix_lens: Sequence[int],
              T: Union[int, Sequence[int]]) -> Tuple[List[int], List[int]]:
    """Flat list of bits of all requests' blocks and the bit offset of each block.

    T is the q_len of every request, or a list of per-request counts T_b (a
    varlen call): request b's block is then [T_b, P_b + T_b].
    """
    counts = _counts(T, len(prefix_lens))
    bits: List[int] = []
    offsets: List[int] = []
    for b, P in enumerate(prefix_lens):
        offsets.append(len(bits))
        par = parents[b]
        Tb = counts[b]
        for i in range(Tb):
            for j in range(P + Tb):
                if j < P:
                    bits.append(1)
                else:
                    bits.append(1 if sees(par, i, j - P) else 0)
    return bits, offsets


def pack_lsb(bits: Sequence[int]) -> List[int]:
    """Bit k goes to byte k // 8, bit position k % 8 (LSB-first)."""
    out = [0] * ((len(bits) + 7) // 8)
    for k, v in enumerate(bits):
        if v:
            out[k // 8] |= 1 << (k % 8)
    return out


def build(parents: Sequence[Sequence[int]], prefix_lens: Sequence[int],
          T: Union[int, Sequence[int]]) -> Tuple[List[int], List[int]]:
    """(packed mask bytes, mask_indptr) of a verify call (T: q_len, or per-request counts)."""
    bits, offsets = mask_bits(parents, prefix_lens, T)
    return pack_lsb(bits), offsets


def mask_byte(parents: Sequence[Sequence[int]], prefix_lens: Sequence[int], T: int, k: int) -> int:
    """Byte k of the packed mask alone (for sampling large masks)."""
    starts = []
    acc = 0
    for P in prefix_lens:
        starts.append(acc)
        acc += T * (P + T)
    total = acc
    byte = 0
    for e in range(8):
        g = 8 * k + e
        if g >= total:
            break
        b = max(idx for idx, s in enumerate(starts) if s <= g)
        P = prefix_lens[b]
        L = P + T
        i, j = divmod(g - starts[b], L)
        if j < P or sees(parents[b], i, j - P):
            byte |= 1 << e
    return byte
