"""Pins of the KV relocation oracle (CPU only): a hand-worked example, the
verify result unchanged by relocation (row ids do not enter attention), the
relocated layout contiguous per request, out-of-range keys left alone, and
planted mistakes that fail a pin."""

import numpy as np
import pytest

from oracle import ref
from oracle import relocate as RL
from mla_speculative_decode_tree_gb300 import workloads as W


def test_hand_example():
    # pool row r holds the value 100 + r in every column
    pool = (100 + np.arange(10, dtype=np.uint16))[:, None].repeat(4, axis=1)
    indptr = [0, 3, 5]
    indices = [9, 6, 8, 5, 7]
    dst_start = [0, 3]
    new_pool, new_idx, bad = RL.relocate(pool, indptr, indices, dst_start, 2)
    assert not bad
    assert new_idx.tolist() == [0, 1, 2, 3, 4]
    assert new_pool[:5, 0].tolist() == [109, 106, 108, 105, 107]
    # sources keep their values, untouched rows stay
    assert new_pool[5:, 0].tolist() == [105, 106, 107, 108, 109]
    assert np.array_equal(pool[:, 0], 100 + np.arange(10))  # input not modified


def test_out_of_range_keys_are_left_and_reported():
    pool = np.arange(6, dtype=np.uint16)[:, None]
    new_pool, new_idx, bad = RL.relocate(pool, [0, 2], [4, 9], [0], 1)
    assert bad
    assert new_idx.tolist() == [0, 9]
    assert new_pool[:, 0].tolist() == [4, 1, 2, 3, 4, 5]
    new_pool, new_idx, bad = RL.relocate(pool, [0, 2], [3, 4], [5], 1)  # second destination is row 6
    assert bad and new_idx.tolist() == [5, 4] and new_pool[5, 0] == 3


def _relocated(wl):
    new_pool, new_idx, bad = RL.relocate(wl["pool"], wl["kv_indptr"], wl["kv_indices"], wl["dst_start"], wl["B"])
    assert not bad
    out = dict(wl)
    out["pool"], out["kv_indices"] = new_pool, new_idx
    return out


@pytest.mark.parametrize("case", [dict(B=1, H=4, T=3, P=[37]), dict(B=3, H=2, T=4, P=[12, 0, 21])])
def test_verify_unchanged_and_rows_contiguous(case):
    wl = W.tiny_workload(B=case["B"], H=case["H"], T=case["T"], prefix_lens=case["P"], pool_rows=256, seed=3)
    wl = W.with_free_block(wl, seed=4)
    moved = _relocated(wl)
    o0, l0 = ref.verify(wl)
    o1, l1 = ref.verify(moved)
    assert np.array_equal(o0, o1) and np.array_equal(l0, l1)
    for b in range(wl["B"]):
        s, e = int(wl["kv_indptr"][b]), int(wl["kv_indptr"][b + 1])
        assert moved["kv_indices"][s:e].tolist() == list(range(int(wl["dst_start"][b]), int(wl["dst_start"][b]) + e - s))
        # each moved row carries its source row's values
        assert np.array_equal(moved["pool"][moved["kv_indices"][s:e]], wl["pool"][wl["kv_indices"][s:e]])


def _buggy_relocate(pool, indptr, indices, dst_start, batch, bug):
    """The oracle's relocation with one planted mistake."""
    new_pool, new_idx = pool.copy(), np.array(indices, dtype=np.int64)
    for b in range(batch):
        s, e = int(indptr[b]), int(indptr[b + 1])
        for k in range(s, e):
            src = int(indices[min(k + 1, e - 1)]) if bug == "source" else int(indices[k])
            dst = int(dst_start[b]) + (k - s)
            new_pool[dst + (1 if bug == "copy_dst" else 0)] = pool[src]
            if bug != "no_rewrite":
                new_idx[k] = dst
    return new_pool, new_idx.astype(np.int32)


@pytest.mark.parametrize("bug", ["source", "copy_dst", "no_rewrite"])
def test_planted_mistakes_fail_a_pin(bug):
    wl = W.with_free_block(W.tiny_workload(B=2, H=2, T=2, prefix_lens=[9, 6], pool_rows=128, seed=8), seed=9)
    o_ref, l_ref = ref.verify(wl)
    p, i = _buggy_relocate(wl["pool"], wl["kv_indptr"], wl["kv_indices"], wl["dst_start"], wl["B"], bug)
    moved = dict(wl)
    moved["pool"], moved["kv_indices"] = p, i
    o, l = ref.verify(moved)
    same_result = np.array_equal(o, o_ref) and np.array_equal(l, l_ref)
    contiguous = all(
        i[int(wl["kv_indptr"][b]):int(wl["kv_indptr"][b + 1])].tolist()
        == list(range(int(wl["dst_start"][b]), int(wl["dst_start"][b]) + int(wl["prefix_lens"][b])))
        for b in range(wl["B"]))
    assert not (same_result and contiguous)


def test_free_block_workload_keeps_destinations_free():
    """The relocation inputs: every row the call addresses lies outside the
    destination blocks, and those blocks do not overlap."""
    wl = W.with_free_block(W.tiny_workload(B=4, H=2, T=3, prefix_lens=[50, 0, 17, 200], pool_rows=1024, seed=2),
                           seed=3)
    addressed = set(W.logical_rows(wl).tolist())
    blocks = []
    for b in range(wl["B"]):
        start, n = int(wl["dst_start"][b]), int(wl["prefix_lens"][b])
        blocks.append(set(range(start, start + n)))
    assert all(not (blk & addressed) for blk in blocks)
    for i in range(len(blocks)):
        for j in range(i + 1, len(blocks)):
            assert not (blocks[i] & blocks[j])
    assert all(0 <= r < wl["pool_rows"] for blk in blocks for r in blk)
