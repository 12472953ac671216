"""GPU tree-mask builder (mla_verify_build_tree_mask) against the tree-mask
oracle, bit for bit, and end to end with the verify call."""

import os

import numpy as np
import pytest

from mla_speculative_decode_tree_gb300 import binding as B
from mla_speculative_decode_tree_gb300 import workloads as W
from oracle import tree_mask as TM
from parity_util import bf16_to_f64, compare

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_speculative_decode_tree_gb300 import build
    build.build()


def _gpu_build(plan, parents, prefix_lens, T, capacity=None, fill=0xA5):
    batch = len(prefix_lens)
    indptr = np.concatenate([[0], np.cumsum(prefix_lens)]).astype(np.int32)
    par = torch.from_numpy(np.ascontiguousarray(np.concatenate([np.asarray(p, np.int32) for p in parents])
                                                if batch else np.zeros(1, np.int32))).cuda()
    kvp = torch.from_numpy(indptr).cuda()
    total_bytes = (T * int(sum(p + T for p in prefix_lens)) + 7) // 8
    cap = total_bytes if capacity is None else capacity
    mask = torch.full((max(total_bytes, cap) + 64,), fill, dtype=torch.uint8, device="cuda")
    mip = torch.full((max(batch, 1),), -7, dtype=torch.int32, device="cuda")
    B.mla_verify_build_tree_mask(plan, par, kvp, batch, mask, mip, mask_bytes=cap)
    torch.cuda.synchronize()
    return mask.cpu().numpy(), mip.cpu().numpy()[:batch], total_bytes


def _plan(max_batch, T, max_kv_len):
    return B.mla_verify_plan(max_batch, 16, T, max_kv_len, 4096, 2)


@pytest.mark.parametrize("B_,T,seed", [(1, 1, 0), (1, 4, 1), (3, 9, 2), (4, 16, 3), (2, 64, 4), (5, 7, 5)])
def test_builder_matches_oracle_bit_for_bit(B_, T, seed):
    rng = np.random.default_rng(seed)
    prefix = [int(x) for x in rng.integers(0, 300, size=B_)]
    prefix[0] = 0 if B_ > 1 else prefix[0]  # an empty prefix among the requests
    parents = [W.random_tree(rng, T) if (seed + b) % 3 else W.chain_tree(T) for b in range(B_)]
    plan = _plan(B_, T, max(prefix) + T)
    got, mip, n = _gpu_build(plan, parents, prefix, T)
    ref, offs = TM.build([list(p) for p in parents], prefix, T)
    assert got[:n].tolist() == ref
    assert mip.tolist() == offs
    assert (got[n:] == 0xA5).all(), "bytes past the mask were written"


def test_invalid_parent_links_end_the_walk():
    T = 6
    parents = [np.array([-1, 0, 5, -3, 2, 4], np.int32)]  # 5 >= 2 and -3 are out of range
    prefix = [10]
    got, mip, n = _gpu_build(_plan(1, T, 16), parents, prefix, T)
    ref, offs = TM.build([list(p) for p in parents], prefix, T)
    assert got[:n].tolist() == ref and mip.tolist() == offs


def test_capacity_is_respected():
    T = 9
    rng = np.random.default_rng(7)
    parents = [W.random_tree(rng, T) for _ in range(2)]
    prefix = [100, 57]
    ref, _ = TM.build([list(p) for p in parents], prefix, T)
    cap = len(ref) // 2
    got, _, _ = _gpu_build(_plan(2, T, 200), parents, prefix, T, capacity=cap)
    assert got[:cap].tolist() == ref[:cap]
    assert (got[cap:] == 0xA5).all()


def test_batch_zero_writes_nothing():
    got, _, _ = _gpu_build(_plan(2, 4, 64), [], [], 4)
    assert (got == 0xA5).all()


@pytest.mark.slow
@pytest.mark.parametrize("name", ["short4k", "mid64k", "batch16_ragged"])
def test_full_size_masks(name):
    wl = W.make_workload(W.CONFIGS[name])
    T = wl["T"]
    prefix = [int(p) for p in wl["prefix_lens"]]
    parents = [np.asarray(p, np.int32) for p in wl["parents"]]
    plan = _plan(len(prefix), T, max(prefix) + T)
    got, mip, n = _gpu_build(plan, parents, prefix, T)
    assert np.array_equal(mip, np.asarray(wl["mask_indptr"]))
    assert np.array_equal(got[:n], np.asarray(wl["custom_mask"], np.uint8)[:n])
    rng = np.random.default_rng(11)
    sample = sorted(set(rng.integers(0, n, size=400).tolist()) | {0, n - 1})
    plist = [list(p) for p in parents]
    for k in sample:
        assert got[k] == TM.mask_byte(plist, prefix, T, k), (name, k)


def test_verify_with_device_built_mask_matches_oracle():
    from oracle import ref
    wl = W.tiny_workload(B=2, H=64, T=9, prefix_lens=[700, 129], pool_rows=8192, seed=21, nsplit=4)
    v = B.verifier_for(wl)
    d = B.device_inputs(wl)
    parents = torch.from_numpy(np.concatenate([np.asarray(p, np.int32) for p in wl["parents"]])).cuda()
    mask = torch.zeros_like(d["custom_mask"])
    mip = torch.zeros_like(d["mask_indptr"])
    B.mla_verify_build_tree_mask(v.plan, parents, d["kv_indptr"], 2, mask, mip)
    d = dict(d, custom_mask=mask, mask_indptr=mip)
    o, lse = v.run(d, 2, wl["sm_scale"])
    torch.cuda.synchronize()
    o_ref, lse_ref = ref.verify(wl, nthreads=os.cpu_count() or 4)
    compare(bf16_to_f64(o[: 2 * 9]).reshape(-1, 512), lse[: 2 * 9].cpu().numpy().reshape(-1), o_ref, lse_ref,
            "device-built mask")


def test_builder_and_verify_in_one_graph():
    """Capture mask build + verify once; replay with new trees written in place."""
    from oracle import ref
    T, H = 9, 64
    first = W.tiny_workload(B=2, H=H, T=T, prefix_lens=[300, 41], pool_rows=4096, seed=31, nsplit=4)
    second = W.tiny_workload(B=2, H=H, T=T, prefix_lens=[300, 41], pool_rows=4096, seed=32, nsplit=4)
    v = B.verifier_for(first)
    d = B.device_inputs(first)
    parents = torch.zeros(2 * T, dtype=torch.int32, device="cuda")
    mask = torch.zeros_like(d["custom_mask"])
    mip = torch.zeros_like(d["mask_indptr"])
    stream = torch.cuda.Stream()

    def load(wl):
        parents.copy_(torch.from_numpy(np.concatenate([np.asarray(p, np.int32) for p in wl["parents"]])))
        fresh = B.device_inputs(wl)  # same shapes: same prefix lengths
        for k in ("q_nope", "q_rope", "kv_pool", "kv_indptr", "kv_indices", "out_cache_loc"):
            d[k].copy_(fresh[k])
        torch.cuda.synchronize()

    def call():
        B.mla_verify_build_tree_mask(v.plan, parents, d["kv_indptr"], 2, mask, mip, stream=stream)
        B.mla_verify_run(v.plan, d["q_nope"], d["q_rope"], d["kv_pool"], d["kv_indptr"], d["kv_indices"],
                         d["out_cache_loc"], mask, mip, 2, first["sm_scale"], 4, v.workspace, v.o, v.lse,
                         stream=stream)

    load(first)
    with torch.cuda.stream(stream):
        call()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        call()
    for wl in (second, first):
        load(wl)
        mask.zero_()
        with torch.cuda.stream(stream):
            g.replay()
        torch.cuda.synchronize()
        o_ref, lse_ref = ref.verify(wl, nthreads=os.cpu_count() or 4)
        compare(bf16_to_f64(v.o[: 2 * T]).reshape(-1, 512), v.lse[: 2 * T].cpu().numpy().reshape(-1), o_ref,
                lse_ref, "graph replay")


# ---- varlen calls: per-request draft-token counts ---------------------------
def _gpu_build_varlen(plan, parents, prefix_lens, Ts, fill=0xA5):
    batch = len(prefix_lens)
    indptr = np.concatenate([[0], np.cumsum(prefix_lens)]).astype(np.int32)
    qo = np.concatenate([[0], np.cumsum(Ts)]).astype(np.int32)
    flat = np.concatenate([np.asarray(p, np.int32) for p in parents] + [np.zeros(1, np.int32)])
    total_bytes = (int(sum(t * (p + t) for p, t in zip(prefix_lens, Ts))) + 7) // 8
    mask = torch.full((total_bytes + 64,), fill, dtype=torch.uint8, device="cuda")
    mip = torch.full((max(batch, 1),), -7, dtype=torch.int32, device="cuda")
    B.mla_verify_build_tree_mask_varlen(plan, torch.from_numpy(flat).cuda(), torch.from_numpy(indptr).cuda(),
                                        torch.from_numpy(qo).cuda(), batch, mask, mip, mask_bytes=total_bytes)
    torch.cuda.synchronize()
    return mask.cpu().numpy(), mip.cpu().numpy()[:batch], total_bytes


@pytest.mark.parametrize("seed,Ts,prefix", [
    (0, [3, 0, 9, 1], [500, 40, 0, 1300]),
    (1, [16, 1, 7], [257, 2000, 3]),
    (2, [1] * 12, [int(x) for x in np.random.default_rng(2).integers(0, 400, 12)]),
    (3, [9, 9], [100, 0]),
    (4, [0, 0, 5], [10, 20, 30]),
])
def test_varlen_builder_matches_oracle_bit_for_bit(seed, Ts, prefix):
    rng = np.random.default_rng(seed)
    parents = [W.random_tree(rng, t) if t else np.zeros(0, np.int32) for t in Ts]
    plan = _plan(len(Ts), max(Ts), max(p + t for p, t in zip(prefix, Ts)) + 1)
    got, mip, n = _gpu_build_varlen(plan, parents, prefix, Ts)
    ref, offs = TM.build([list(p) for p in parents], prefix, Ts)
    assert got[:n].tolist() == ref
    assert mip.tolist() == offs
    assert (got[n:] == 0xA5).all(), "bytes past the mask were written"


def test_varlen_verify_with_device_built_mask_is_identical():
    wl = W.varlen_workload(B=4, H=64, T_list=[9, 0, 3, 1], prefix_lens=[800, 50, 2100, 0], pool_rows=8192, seed=5,
                           nsplit=8)
    v = B.verifier_for(wl)
    d = B.device_inputs(wl)
    o0, l0 = v.run(d, wl["B"], wl["sm_scale"])
    o0, l0 = o0.clone(), l0.clone()
    parents = torch.from_numpy(np.concatenate([np.asarray(p, np.int32) for p in wl["parents"]])).cuda()
    mask = torch.zeros_like(d["custom_mask"])
    mip = torch.zeros_like(d["mask_indptr"])
    B.mla_verify_build_tree_mask_varlen(v.plan, parents, d["kv_indptr"], d["qo_indptr"], wl["B"], mask, mip)
    torch.cuda.synchronize()
    n = (int(sum(t * (p + t) for p, t in zip(wl["prefix_lens"], wl["T_list"]))) + 7) // 8
    assert torch.equal(mask[:n], d["custom_mask"][:n]) and torch.equal(mip, d["mask_indptr"])
    o1, l1 = v.run(dict(d, custom_mask=mask, mask_indptr=mip), wl["B"], wl["sm_scale"])
    torch.cuda.synchronize()
    rows = int(wl["qo_indptr"][-1])
    assert torch.equal(o0[:rows].view(torch.int16), o1[:rows].view(torch.int16)) and torch.equal(l0[:rows], l1[:rows])
