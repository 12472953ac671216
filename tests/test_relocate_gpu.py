"""GPU KV relocation (mla_verify_relocate_kv) against the relocation oracle,
bit for bit (pool bytes and rewritten indices), and the verify call's output
bit-identical before and after relocation."""

import numpy as np
import pytest

from mla_speculative_decode_tree_gb300 import binding as B
from mla_speculative_decode_tree_gb300 import workloads as W
from oracle import relocate as RL

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_speculative_decode_tree_gb300 import build
    build.build()


def _relocate_on_gpu(wl, v, d, dst_start=None):
    dst = torch.from_numpy(np.asarray(wl["dst_start"] if dst_start is None else dst_start, np.int32)).cuda()
    B.mla_verify_relocate_kv(v.plan, d["kv_pool"], d["kv_indptr"], d["kv_indices"], dst, wl["B"], v.workspace)
    torch.cuda.synchronize()
    pool = d["kv_pool"].view(torch.int16).cpu().numpy().view(np.uint16)
    idx = d["kv_indices"].cpu().numpy()[: int(wl["kv_indptr"][-1])]
    return pool, idx


CASES = [
    # (B, H, T, prefixes, pool_rows)
    (1, 16, 4, [256], 4096),
    (3, 8, 9, [1000, 0, 77], 8192),
    (4, 64, 9, [5, 130, 2047, 1], 16384),
    (16, 4, 2, [int(x) for x in np.random.default_rng(5).integers(0, 600, 16)], 32768),
]


@pytest.mark.parametrize("case", CASES, ids=[str(i) for i in range(len(CASES))])
def test_relocation_bit_exact(case):
    Bn, H, T, P, pool_rows = case
    wl = W.with_free_block(W.tiny_workload(B=Bn, H=H, T=T, prefix_lens=P, pool_rows=pool_rows, seed=Bn + T), seed=7)
    d = B.device_inputs(wl)
    v = B.verifier_for(wl)
    pool, idx = _relocate_on_gpu(wl, v, d)
    ref_pool, ref_idx, bad = RL.relocate(wl["pool"], wl["kv_indptr"], wl["kv_indices"], wl["dst_start"], wl["B"])
    assert not bad and v.status() == 0
    assert np.array_equal(idx, ref_idx)
    assert np.array_equal(pool, ref_pool)


def test_verify_identical_after_relocation():
    wl = W.with_free_block(W.tiny_workload(B=2, H=64, T=9, prefix_lens=[3000, 1111], pool_rows=16384, seed=11),
                           seed=12)
    d = B.device_inputs(wl)
    v = B.verifier_for(wl)
    o0, l0 = v.run(d, wl["B"], wl["sm_scale"])
    o0, l0 = o0.clone(), l0.clone()
    _relocate_on_gpu(wl, v, d)
    o1, l1 = v.run(d, wl["B"], wl["sm_scale"])
    torch.cuda.synchronize()
    assert torch.equal(o0.view(torch.int16), o1.view(torch.int16)) and torch.equal(l0, l1)
    assert v.status() == 0


def test_out_of_range_keys_are_left_and_reported():
    wl = W.with_free_block(W.tiny_workload(B=2, H=4, T=2, prefix_lens=[40, 30], pool_rows=1024, seed=21), seed=22)
    wl["kv_indices"] = wl["kv_indices"].copy()
    wl["kv_indices"][5] = 5000          # source outside the pool
    dst = wl["dst_start"].copy()
    dst[1] = 1024 + 5                   # request 1's block lies past the pool: its keys stay
    d = B.device_inputs(wl)
    v = B.verifier_for(wl)
    pool, idx = _relocate_on_gpu(wl, v, d, dst_start=dst)
    ref_pool, ref_idx, bad = RL.relocate(wl["pool"], wl["kv_indptr"], wl["kv_indices"], dst, wl["B"])
    assert bad and v.status() == B.MLA_VERIFY_DEV_BAD_ROW
    assert np.array_equal(idx, ref_idx) and np.array_equal(pool, ref_pool)


def test_relocation_in_a_cuda_graph():
    """Captured once, replayed on fresh indices: the call is capture-safe."""
    wl = W.with_free_block(W.tiny_workload(B=2, H=8, T=3, prefix_lens=[500, 300], pool_rows=4096, seed=31), seed=32)
    d = B.device_inputs(wl)
    v = B.verifier_for(wl)
    dst = torch.from_numpy(wl["dst_start"].astype(np.int32)).cuda()
    idx0 = d["kv_indices"].clone()
    stream = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        B.mla_verify_relocate_kv(v.plan, d["kv_pool"], d["kv_indptr"], d["kv_indices"], dst, wl["B"], v.workspace,
                                 stream=stream)
    d["kv_indices"].copy_(idx0)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        g.replay()
    torch.cuda.synchronize()
    ref_pool, ref_idx, _ = RL.relocate(wl["pool"], wl["kv_indptr"], wl["kv_indices"], wl["dst_start"], wl["B"])
    assert np.array_equal(d["kv_indices"].cpu().numpy()[:800], ref_idx)
    assert np.array_equal(d["kv_pool"].view(torch.int16).cpu().numpy().view(np.uint16), ref_pool)
