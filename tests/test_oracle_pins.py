"""Pins of the CPU oracle to facts outside itself (no GPU).

Each pin checks the oracle against something it does not share code with:
a brute-force enumeration that derives visibility from the draft tree, a
textbook softmax attention evaluated with scipy, exact special cases, closed
forms and invariances the definition implies.  ``test_planted_mistakes``
plants one plausible mistake at a time in the oracle (on the CPU) and checks
that at least one pin fails for each.
"""

import json
import math
import os

import numpy as np
import pytest
from scipy.special import logsumexp, softmax

from mla_speculative_decode_tree_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def f64(bits):
    return W.bf16_bits_to_f32(bits).astype(np.float64)


def oracle_fn(oracle_lib, mutation=0):
    def run(wl, rows=None):
        return oracle_lib.verify(wl, rows=rows, mutation=mutation, nthreads=2)
    return run


# ---------------------------------------------------------------- pins ----
# Each pin returns True when the oracle passes it.

def pin_brute_force(run):
    """Brute-force enumeration (visibility from parents, fsum) agrees to 1e-12."""
    from oracle.brute import brute_verify
    cases = [
        W.tiny_workload(B=2, H=2, T=3, prefix_lens=[5, 9], pool_rows=64, seed=1),
        W.tiny_workload(B=2, H=3, T=4, prefix_lens=[0, 3], pool_rows=64, seed=2, tree="chain"),
        W.tiny_workload(B=3, H=1, T=5, prefix_lens=[7, 1, 4], pool_rows=64, seed=3),
    ]
    for wl in cases:
        o, lse = run(wl)
        bo, blse = brute_verify(wl)
        if not np.allclose(o, np.array(bo), rtol=0, atol=1e-12):
            return False
        if not np.allclose(lse, np.array(blse), rtol=0, atol=1e-12):
            return False
    return True


def pin_textbook_decode(run):
    """q_len=1 with every key visible equals plain softmax(q K^T * scale) V."""
    wl = W.tiny_workload(B=1, H=4, T=1, prefix_lens=[50], pool_rows=256, seed=4)
    o, lse = run(wl)
    rows = np.concatenate([wl["kv_indices"], wl["out_cache_loc"]]).astype(np.int64)
    K = f64(wl["pool"][rows])  # [L, 576]
    for h in range(wl["H"]):
        q = np.concatenate([f64(wl["q_nope"][0, h]), f64(wl["q_rope"][0, h])])
        s = wl["sm_scale"] * (K @ q)
        ref_o = softmax(s) @ K[:, :512]
        if not np.allclose(o[h], ref_o, rtol=0, atol=1e-12):
            return False
        if abs(lse[h] - logsumexp(s)) > 1e-12:
            return False
    return True


def _single_key_workload(seed):
    wl = W.tiny_workload(B=2, H=3, T=4, prefix_lens=[6, 11], pool_rows=128, seed=seed)
    rng = np.random.default_rng(seed + 100)
    dense, pick = [], []
    for b in range(2):
        L = int(wl["prefix_lens"][b]) + wl["T"]
        m = np.zeros((wl["T"], L), dtype=bool)
        js = rng.integers(0, L, size=wl["T"])
        js[0] = L - 1  # a draft key
        js[1] = 0      # the first prefix key
        m[np.arange(wl["T"]), js] = True
        dense.append(m)
        pick.append(js)
    packed = W.pack_bits_lsb(np.concatenate([d.reshape(-1) for d in dense]))
    wl = dict(wl, custom_mask=packed)
    return wl, pick


def pin_single_visible_key(run):
    """One visible key j*: O is that key's 512 latent values exactly, LSE = s_{j*}."""
    wl, pick = _single_key_workload(5)
    o, lse = run(wl)
    H, T = wl["H"], wl["T"]
    for b in range(2):
        P = int(wl["prefix_lens"][b])
        for i in range(T):
            j = int(pick[b][i])
            row = (int(wl["kv_indices"][int(wl["kv_indptr"][b]) + j]) if j < P
                   else int(wl["out_cache_loc"][b * T + j - P]))
            kv = f64(wl["pool"][row])
            for h in range(H):
                r = (b * T + i) * H + h
                if not np.array_equal(o[r], kv[:512]):
                    return False
                q = np.concatenate([f64(wl["q_nope"][b * T + i, h]), f64(wl["q_rope"][b * T + i, h])])
                s = wl["sm_scale"] * math.fsum(q * kv)
                if abs(lse[r] - s) > 1e-12:
                    return False
    return True


def pin_masked_rows_irrelevant(run):
    """Rewriting every pool row a token cannot see leaves that token's output unchanged."""
    wl = W.tiny_workload(B=1, H=2, T=6, prefix_lens=[12], pool_rows=96, seed=6)
    o, lse = run(wl)
    T, H = wl["T"], wl["H"]
    rng = np.random.default_rng(66)
    for i in range(T):
        vis = W.tree_visibility(wl["parents"][0])[i]
        seen = set(int(x) for x in wl["kv_indices"])
        seen |= {int(wl["out_cache_loc"][t]) for t in range(T) if vis[t]}
        pool2 = wl["pool"].copy()
        for row in range(wl["pool_rows"]):
            if row not in seen:
                pool2[row] = W.f32_to_bf16_bits(rng.standard_normal(576, dtype=np.float32) * 3)
        o2, lse2 = run(dict(wl, pool=pool2))
        rs = [i * H + h for h in range(H)]
        if not (np.array_equal(o[rs], o2[rs]) and np.array_equal(lse[rs], lse2[rs])):
            return False
    return True


def pin_layout_invariance(run):
    """Same logical rows stored contiguously or scattered: identical results."""
    # 4096 rows leave room for the sorted free list's runs and gaps (mean 256)
    wl = W.tiny_workload(B=2, H=2, T=4, prefix_lens=[20, 9], pool_rows=4096, seed=7)
    o, lse = run(wl)
    for layout, seed in (("contiguous", 70), ("scattered", 71), ("sorted", 72)):
        wl2 = W.relayout(wl, layout, seed)
        o2, lse2 = run(wl2)
        if not (np.array_equal(o, o2) and np.array_equal(lse, lse2)):
            return False
    return True


def pin_closed_form_uniform(run):
    """q = 0: every score is 0, so O = mean of the visible values, LSE = ln |visible|."""
    wl = W.tiny_workload(B=2, H=2, T=5, prefix_lens=[4, 13], pool_rows=64, seed=8)
    wl = dict(wl, q_nope=np.zeros_like(wl["q_nope"]), q_rope=np.zeros_like(wl["q_rope"]))
    o, lse = run(wl)
    H, T = wl["H"], wl["T"]
    for b in range(2):
        P = int(wl["prefix_lens"][b])
        vis = W.tree_visibility(wl["parents"][b])
        for i in range(T):
            rows = list(wl["kv_indices"][int(wl["kv_indptr"][b]):int(wl["kv_indptr"][b + 1])])
            rows += [wl["out_cache_loc"][b * T + t] for t in range(T) if vis[i, t]]
            V = f64(wl["pool"][np.array(rows, dtype=np.int64)])[:, :512]
            for h in range(H):
                r = (b * T + i) * H + h
                if not np.allclose(o[r], V.mean(axis=0), rtol=0, atol=1e-12):
                    return False
                if abs(lse[r] - math.log(len(rows))) > 1e-12:
                    return False
    return True


def pin_hand_example(run):
    """The golden hand-worked example (closed forms written out below)."""
    g = json.load(open(os.path.join(GOLDEN, "hand_example.json")))
    P, T, H = g["prefix"], g["q_len"], 1
    rows = g["rows"]
    pool = np.zeros((g["pool_rows"], 576), dtype=np.float32)
    for j, r in enumerate(rows):
        pool[r, j] = 1.0
    pool[rows[0], 512] = 2.0
    qn = np.zeros((T, H, 512), dtype=np.float32)
    qr = np.zeros((T, H, 64), dtype=np.float32)
    for t, key in enumerate(("token0", "token1")):
        qn[t, 0, :4] = g[key]["q_nope_head"]
        qr[t, 0, 0] = g[key]["q_rope0"]
    parents = [W.chain_tree(T)]
    packed, offs, _ = W.build_mask([P], parents, T)
    wl = dict(B=1, H=H, T=T, pool_rows=g["pool_rows"], sm_scale=1.0, prefix_lens=np.array([P]),
              pool=W.f32_to_bf16_bits(pool), q_nope=W.f32_to_bf16_bits(qn), q_rope=W.f32_to_bf16_bits(qr),
              kv_indptr=np.array([0, P], np.int32), kv_indices=np.array(rows[:P], np.int32),
              out_cache_loc=np.array(rows[P:], np.int32), custom_mask=packed,
              mask_indptr=offs.astype(np.int32), parents=parents)
    o, lse = run(wl)
    # token 0 sees keys 0,1,2 with scores 1+2*0.5=2, 0, 0.5
    z0 = 1 + math.exp(-2) + math.exp(-1.5)
    exp0 = np.zeros(512)
    exp0[:3] = [1 / z0, math.exp(-2) / z0, math.exp(-1.5) / z0]
    # token 1 sees keys 0..3 with scores 0+2*(-1)=-2, 0, 0, 1
    z1 = 1 + 2 * math.exp(-1) + math.exp(-3)
    exp1 = np.zeros(512)
    exp1[:4] = [math.exp(-3) / z1, math.exp(-1) / z1, math.exp(-1) / z1, 1 / z1]
    ok = np.allclose(o[0], exp0, rtol=0, atol=1e-14) and np.allclose(o[1], exp1, rtol=0, atol=1e-14)
    ok = ok and abs(lse[0] - (2 + math.log(z0))) < 1e-14 and abs(lse[1] - (1 + math.log(z1))) < 1e-14
    return bool(ok)


def pin_extend_layout_case(run):
    """21 prefix + 9 draft tokens from the pages: draft rows and stride 30 matter."""
    from oracle.brute import brute_verify
    g = json.load(open(os.path.join(GOLDEN, "extend_layout_p21_t9.json")))
    wl = W.tiny_workload(B=1, H=2, T=g["q_len"], prefix_lens=[g["prefix"]], pool_rows=128, seed=9)
    assert wl["dense_mask"][0].shape == (g["q_len"], g["mask_row_stride"])
    assert wl["dense_mask"][0].size == g["mask_bits_per_request"]
    o, lse = run(wl)
    bo, blse = brute_verify(wl)
    return bool(np.allclose(o, np.array(bo), rtol=0, atol=1e-12)
                and np.allclose(lse, np.array(blse), rtol=0, atol=1e-12))


PINS = [pin_brute_force, pin_textbook_decode, pin_single_visible_key, pin_masked_rows_irrelevant,
        pin_layout_invariance, pin_closed_form_uniform, pin_hand_example, pin_extend_layout_case]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_oracle_pin(oracle_lib, pin):
    assert pin(oracle_fn(oracle_lib))


def test_split_merge_invariance(oracle_lib):
    """Split-then-merge (the pages' organisation) equals the direct form for any split count."""
    wl = W.tiny_workload(B=2, H=2, T=9, prefix_lens=[300, 41], pool_rows=512, seed=10)
    o, lse = oracle_lib.verify(wl)
    for nsplit, granule, min_chunk in ((1, 1, 1), (2, 1, 1), (3, 128, 128), (3, 64, 128), (7, 1, 1), (16, 128, 128),
                                       (64, 1, 1)):
        o2, lse2 = oracle_lib.verify_split_merge(wl, nsplit, granule, min_chunk)
        np.testing.assert_allclose(o2, o, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse2, lse, rtol=0, atol=1e-12)


def test_empty_visible_set(oracle_lib):
    """Nothing visible (all mask bits 0): O = 0 and LSE = -inf."""
    wl = W.tiny_workload(B=1, H=2, T=3, prefix_lens=[5], pool_rows=32, seed=11)
    wl = dict(wl, custom_mask=np.zeros_like(wl["custom_mask"]))
    o, lse = oracle_lib.verify(wl)
    assert np.all(o == 0) and np.all(np.isneginf(lse))


def test_out_of_range_row_reported(oracle_lib):
    wl = W.tiny_workload(B=1, H=1, T=2, prefix_lens=[4], pool_rows=32, seed=12)
    bad = wl["kv_indices"].copy()
    bad[2] = 32
    with pytest.raises(ValueError):
        oracle_lib.verify(dict(wl, kv_indices=bad))


MUTATIONS = {1: "mask stride P", 2: "draft rows dropped", 3: "mask_indptr of next request",
             4: "rope term dropped", 5: "MSB-first bits", 6: "LSE without max", 7: "no sm_scale",
             8: "values shifted by 64 columns", 9: "draft rows reversed", 10: "softmax sign"}


@pytest.mark.parametrize("mutation", sorted(MUTATIONS), ids=[MUTATIONS[k] for k in sorted(MUTATIONS)])
def test_planted_mistakes(oracle_lib, mutation):
    """Every planted mistake must fail at least one pin."""
    run = oracle_fn(oracle_lib, mutation)
    failed = []
    for pin in PINS:
        try:
            ok = pin(run)
        except (AssertionError, ValueError, FloatingPointError):
            ok = False
        if not ok:
            failed.append(pin.__name__)
    assert failed, "mistake %r passed every pin" % MUTATIONS[mutation]
