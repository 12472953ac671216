"""Pins of the oracle's per-request draft-token counts (qo_indptr), CPU only.

Request b of a varlen call owns token rows qo_indptr[b] .. qo_indptr[b+1]-1,
its draft rows are out_cache_loc[qo_indptr[b] + t] and its mask block is
[T_b, P_b + T_b].  The pins check that against the uniform-T oracle (each
request alone), against brute force over the parent arrays, and against
textbook decode attention for T_b = 1."""

import numpy as np
import pytest
from scipy.special import logsumexp, softmax

from mla_speculative_decode_tree_gb300 import workloads as W
from oracle import brute

H = 4


def _varlen(seed, T_list=(3, 0, 9, 1), prefix=(50, 20, 0, 70), pool_rows=1024):
    return W.varlen_workload(B=len(T_list), H=H, T_list=list(T_list), prefix_lens=list(prefix),
                             pool_rows=pool_rows, seed=seed)


def _request_alone(wl, b):
    """Request b of a varlen call as a one-request uniform call (T = T_b)."""
    qo = wl["qo_indptr"]
    q0, Tb = int(qo[b]), int(qo[b + 1] - qo[b])
    s, e = int(wl["kv_indptr"][b]), int(wl["kv_indptr"][b + 1])
    dense = wl["dense_mask"][b]
    packed = W.pack_bits_lsb(dense.reshape(-1)) if dense.size else np.zeros(1, np.uint8)
    return dict(B=1, H=wl["H"], T=Tb, sm_scale=wl["sm_scale"], pool=wl["pool"],
                q_nope=wl["q_nope"][q0:q0 + Tb], q_rope=wl["q_rope"][q0:q0 + Tb],
                kv_indptr=np.array([0, e - s], np.int32), kv_indices=wl["kv_indices"][s:e],
                out_cache_loc=wl["out_cache_loc"][q0:q0 + Tb], custom_mask=packed,
                mask_indptr=np.zeros(1, np.int32), parents=[wl["parents"][b]], prefix_lens=[e - s])


@pytest.mark.parametrize("seed", [1, 2])
def test_each_request_equals_the_uniform_oracle_alone(oracle_lib, seed):
    wl = _varlen(seed)
    o, lse = oracle_lib.verify(wl, nthreads=2)
    qo = wl["qo_indptr"]
    assert o.shape[0] == int(qo[-1]) * H
    for b in range(wl["B"]):
        Tb = int(qo[b + 1] - qo[b])
        if Tb == 0:
            continue
        one = _request_alone(wl, b)
        o1, l1 = oracle_lib.verify(one, nthreads=2)
        rows = slice(int(qo[b]) * H, int(qo[b + 1]) * H)
        assert np.array_equal(o[rows], o1) and np.array_equal(lse[rows], l1), b


@pytest.mark.parametrize("seed", [3, 4])
def test_varlen_matches_brute_force(oracle_lib, seed):
    wl = _varlen(seed, T_list=(2, 5, 0, 4), prefix=(9, 0, 13, 6), pool_rows=256)
    o, lse = oracle_lib.verify(wl, nthreads=2)
    ob, lb = brute.brute_verify(wl)
    np.testing.assert_allclose(o, np.array(ob), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, np.array(lb), rtol=0, atol=1e-12)


def test_equal_counts_reduce_to_the_uniform_path(oracle_lib):
    wl = _varlen(5, T_list=(4, 4, 4), prefix=(30, 11, 0))
    o, lse = oracle_lib.verify(wl, nthreads=2)
    uni = dict(wl)
    del uni["qo_indptr"]
    uni["T"] = 4
    o2, l2 = oracle_lib.verify(uni, nthreads=2)
    assert np.array_equal(o, o2) and np.array_equal(lse, l2)


def test_decode_t1_is_textbook_attention(oracle_lib):
    """T_b = 1, everything visible: softmax(scale * q.K^T) V and logsumexp."""
    wl = _varlen(6, T_list=(1, 1, 1), prefix=(40, 7, 0))
    o, lse = oracle_lib.verify(wl, nthreads=2)
    pool = W.bf16_bits_to_f32(wl["pool"]).astype(np.float64)
    qn = W.bf16_bits_to_f32(wl["q_nope"]).astype(np.float64)
    qr = W.bf16_bits_to_f32(wl["q_rope"]).astype(np.float64)
    for b in range(3):
        s, e = int(wl["kv_indptr"][b]), int(wl["kv_indptr"][b + 1])
        rows = list(wl["kv_indices"][s:e]) + [int(wl["out_cache_loc"][b])]
        K = pool[rows]
        for h in range(H):
            q = np.concatenate([qn[b, h], qr[b, h]])
            sc = wl["sm_scale"] * (K @ q)
            np.testing.assert_allclose(o[b * H + h], softmax(sc) @ K[:, :512], rtol=0, atol=1e-12)
            assert abs(lse[b * H + h] - logsumexp(sc)) < 1e-12


@pytest.mark.parametrize("nsplit", [1, 3, 16])
def test_varlen_split_merge_identity(oracle_lib, nsplit):
    wl = _varlen(7)
    o, lse = oracle_lib.verify(wl, nthreads=2)
    o2, l2 = oracle_lib.verify_split_merge(wl, nsplit=nsplit, granule=4, min_chunk=4, nthreads=2)
    np.testing.assert_allclose(o2, o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l2, lse, rtol=0, atol=1e-12)


# ---- planted mistakes in the per-request indexing -------------------------
# Each plants one plausible error of the varlen indexing in the C oracle
# (mutation codes of oracle/mla_verify_ref.c) and must fail one of the pins
# above, evaluated on the same workloads.

VARLEN_MUTATIONS = {11: "draft rows at b*T", 12: "query row b*T + i", 13: "mask row stride P_b + T_max"}


def _padded(wl):
    """The workload with its packed mask padded, so a wrong (larger) mask
    stride still reads inside the buffer."""
    pad = np.zeros(wl["B"] * wl["T"] * wl["T"] // 8 + 16, np.uint8)
    return dict(wl, custom_mask=np.concatenate([wl["custom_mask"], pad]))


def _pin_requests_alone(oracle_lib, mutation):
    wl = _padded(_varlen(1))
    o, lse = oracle_lib.verify(wl, nthreads=2, mutation=mutation)
    qo = wl["qo_indptr"]
    for b in range(wl["B"]):
        if int(qo[b + 1] - qo[b]) == 0:
            continue
        one = _request_alone(wl, b)
        o1, l1 = oracle_lib.verify(one, nthreads=2)
        rows = slice(int(qo[b]) * H, int(qo[b + 1]) * H)
        if not (np.array_equal(o[rows], o1) and np.array_equal(lse[rows], l1)):
            return False
    return True


def _pin_brute(oracle_lib, mutation):
    wl = _padded(_varlen(3, T_list=(2, 5, 0, 4), prefix=(9, 0, 13, 6), pool_rows=256))
    o, lse = oracle_lib.verify(wl, nthreads=2, mutation=mutation)
    ob, lb = brute.brute_verify(wl)
    return bool(np.allclose(o, np.array(ob), rtol=0, atol=1e-12) and np.allclose(lse, np.array(lb), rtol=0, atol=1e-12))


def test_varlen_pins_hold_for_the_oracle(oracle_lib):
    assert _pin_requests_alone(oracle_lib, 0) and _pin_brute(oracle_lib, 0)


@pytest.mark.parametrize("mutation", sorted(VARLEN_MUTATIONS), ids=[VARLEN_MUTATIONS[k] for k in sorted(VARLEN_MUTATIONS)])
def test_varlen_planted_mistakes_fail_a_pin(oracle_lib, mutation):
    failed = []
    for pin in (_pin_requests_alone, _pin_brute):
        try:
            ok = pin(oracle_lib, mutation)
        except (AssertionError, ValueError):
            ok = False
        if not ok:
            failed.append(pin.__name__)
    assert failed, "mistake %r passed every varlen pin" % VARLEN_MUTATIONS[mutation]
