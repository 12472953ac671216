"""Pins of the tree-mask oracle (CPU only): a hand-worked golden example,
closed forms for chain and star trees, agreement with brute-force attention
that takes visibility from the parent arrays, and planted mistakes that each
fail a pin."""

import json
import os

import numpy as np
import pytest

from oracle import tree_mask as TM
from mla_speculative_decode_tree_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _unpack(packed, nbits):
    return [(packed[k // 8] >> (k % 8)) & 1 for k in range(nbits)]


def test_golden_hand_example():
    with open(os.path.join(GOLDEN, "tree_mask_example.json")) as f:
        g = json.load(f)
    packed, offsets = TM.build(g["parents"], g["prefix_lens"], g["T"])
    assert packed == g["mask_bytes"]
    assert offsets == g["mask_indptr"]
    for k in range(len(packed)):
        assert TM.mask_byte(g["parents"], g["prefix_lens"], g["T"], k) == g["mask_bytes"][k]


@pytest.mark.parametrize("T", [1, 2, 5, 9, 16])
def test_chain_tree_is_lower_triangular(T):
    parents = [list(range(-1, T - 1))]
    bits, _ = TM.mask_bits(parents, [0], T)
    m = np.array(bits).reshape(T, T)
    assert np.array_equal(m, np.tril(np.ones((T, T), dtype=int)))


@pytest.mark.parametrize("T,P", [(1, 0), (4, 3), (9, 7)])
def test_star_tree_sees_root_and_self(T, P):
    parents = [[-1] + [0] * (T - 1)]
    bits, _ = TM.mask_bits(parents, [P], T)
    m = np.array(bits).reshape(T, P + T)
    assert m[:, :P].all()
    expect = np.zeros((T, T), dtype=int)
    expect[:, 0] = 1
    expect[np.arange(T), np.arange(T)] = 1
    assert np.array_equal(m[:, P:], expect)


def test_offsets_closed_form():
    P = [5, 0, 17, 2]
    T = 4
    _, offsets = TM.mask_bits([[-1, 0, 1, 1]] * 4, P, T)
    assert offsets == [0, T * (5 + T), T * (5 + T) + T * (0 + T), T * (5 + T + 0 + T + 17 + T)]


def _tiny_with_oracle_mask(seed, B=2, H=3, T=5, prefix_lens=(7, 3)):
    wl = W.tiny_workload(B=B, H=H, T=T, prefix_lens=list(prefix_lens), pool_rows=512, seed=seed, nsplit=2)
    packed, offsets = TM.build([list(p) for p in wl["parents"]], list(wl["prefix_lens"]), T)
    return wl, np.array(packed, dtype=np.uint8), np.array(offsets, dtype=np.int64)


@pytest.mark.parametrize("seed", [3, 4, 5])
def test_attention_with_oracle_mask_matches_brute_force(oracle_lib, seed):
    """The C oracle reads the packed bits; brute force walks the parents."""
    from oracle import brute
    wl, packed, offsets = _tiny_with_oracle_mask(seed)
    wl = dict(wl, custom_mask=packed, mask_indptr=offsets)
    o, lse = oracle_lib.verify(wl, nthreads=2)
    ob, lb = brute.brute_verify(wl)
    np.testing.assert_allclose(o, np.array(ob), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, np.array(lb), rtol=0, atol=1e-12)


def test_oracle_mask_equals_input_generator_mask():
    wl, packed, offsets = _tiny_with_oracle_mask(9, B=3, T=9, prefix_lens=(0, 12, 40))
    assert np.array_equal(offsets, np.asarray(wl["mask_indptr"], dtype=np.int64))
    n = len(packed)
    assert np.array_equal(packed, np.asarray(wl["custom_mask"], dtype=np.uint8)[:n])


# ---- planted mistakes: each must fail one of the pins above ----------------
def _mutant_build(kind):
    def sees(parent, i, d):
        n = i
        while n >= 0:
            if n == d and not (kind == "no_self" and n == i):
                return True
            n = int(parent[n]) if kind != "parent_of_parent" else (int(parent[int(parent[n])]) if parent[n] >= 0 else -1)
        return False

    def build(parents, prefix_lens, T):
        bits, offsets = [], []
        for b, P in enumerate(prefix_lens):
            offsets.append(len(bits) + (1 if kind == "offset_plus_one" and b > 0 else 0))
            for i in range(T):
                for j in range(P + T):
                    if j < P:
                        bits.append(1)
                    elif kind == "transposed":
                        bits.append(1 if TM.sees(parents[b], j - P, i) else 0)
                    else:
                        bits.append(1 if sees(parents[b], i, j - P) else 0)
        out = [0] * ((len(bits) + 7) // 8)
        for k, v in enumerate(bits):
            if v:
                out[k // 8] |= 1 << ((7 - k % 8) if kind == "msb_first" else (k % 8))
        return out, offsets
    return build


@pytest.mark.parametrize("kind", ["no_self", "parent_of_parent", "offset_plus_one", "transposed", "msb_first"])
def test_planted_mistakes_fail_a_pin(kind, monkeypatch):
    monkeypatch.setattr(TM, "build", _mutant_build(kind))
    failed = 0
    for test in (test_golden_hand_example, lambda: _chain_via_build(9),
                 lambda: _star_via_build(9, 7)):
        try:
            test()
        except AssertionError:
            failed += 1
    assert failed, "mistake %r passed every pin" % kind


def _chain_via_build(T):
    packed, _ = TM.build([list(range(-1, T - 1))], [0], T)
    m = np.array(_unpack(packed, T * T)).reshape(T, T)
    assert np.array_equal(m, np.tril(np.ones((T, T), dtype=int)))


def _star_via_build(T, P):
    packed, _ = TM.build([[-1] + [0] * (T - 1)], [P], T)
    m = np.array(_unpack(packed, T * (P + T))).reshape(T, P + T)
    expect = np.zeros((T, T), dtype=int)
    expect[:, 0] = 1
    expect[np.arange(T), np.arange(T)] = 1
    assert m[:, :P].all() and np.array_equal(m[:, P:], expect)


# ---- varlen calls: per-request draft-token counts T_b ----------------------
def test_varlen_equal_counts_equal_uniform():
    rng = np.random.default_rng(12)
    parents = [list(W.random_tree(rng, 6)) for _ in range(3)]
    assert TM.build(parents, [5, 0, 9], [6, 6, 6]) == TM.build(parents, [5, 0, 9], 6)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_varlen_blocks_are_the_single_request_masks(seed):
    """Request b's block is the one-request mask of (parents_b, P_b, T_b) at
    bit offset sum_{b'<b} T_b' (P_b' + T_b'); a request with T_b = 0 has none."""
    rng = np.random.default_rng(seed)
    B = 5
    Ts = [int(t) for t in rng.integers(0, 10, size=B)]
    Ts[1] = 0
    P = [int(p) for p in rng.integers(0, 40, size=B)]
    parents = [list(W.random_tree(rng, t)) if t else [] for t in Ts]
    bits, offsets = TM.mask_bits(parents, P, Ts)
    acc = 0
    for b in range(B):
        assert offsets[b] == acc
        alone, _ = TM.mask_bits([parents[b]], [P[b]], Ts[b])
        assert bits[acc:acc + len(alone)] == alone
        acc += Ts[b] * (P[b] + Ts[b])
    assert len(bits) == acc


@pytest.mark.parametrize("seed", [6, 7])
def test_varlen_oracle_mask_with_brute_force_attention(oracle_lib, seed):
    """Attention with the oracle's varlen mask (C oracle, reads bits) equals brute
    force that takes visibility from the parent arrays."""
    from oracle import brute
    wl = W.varlen_workload(B=3, H=2, T_list=[4, 0, 7], prefix_lens=[6, 3, 11], pool_rows=256, seed=seed)
    packed, offsets = TM.build([list(p) for p in wl["parents"]], list(wl["prefix_lens"]), list(wl["T_list"]))
    wl = dict(wl, custom_mask=np.array(packed, np.uint8), mask_indptr=np.array(offsets, np.int32))
    o, lse = oracle_lib.verify(wl, nthreads=2)
    ob, lb = brute.brute_verify(wl)
    np.testing.assert_allclose(o, np.array(ob), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, np.array(lb), rtol=0, atol=1e-12)
