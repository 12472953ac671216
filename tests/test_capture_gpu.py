"""CUDA-graph capture of a verify call [Capture Safety to MoE Ceiling, §"The
Architecture of Capture Safety"]: the call is captured once, then the device
inputs are rewritten in place -- new prefix lengths (so new chunk bounds),
indices, trees, queries and pool rows -- and the replay must match the oracle
on the new inputs."""

import os

import numpy as np
import pytest

from mla_speculative_decode_tree_gb300 import binding as B
from mla_speculative_decode_tree_gb300 import workloads as W
from parity_util import bf16_to_f64, compare

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_speculative_decode_tree_gb300 import build
    build.build()


def _fill(buf, arr, dtype):
    t = torch.from_numpy(np.ascontiguousarray(arr)).view(dtype)
    buf.zero_()
    buf[: t.numel()].copy_(t.reshape(-1))


@pytest.mark.parametrize("H,flags", [(64, 0), (8, 0), (64, B.MLA_VERIFY_REFETCH_VALUES), (8, B.MLA_VERIFY_REFETCH_VALUES),
                                     (64, B.MLA_VERIFY_FORCE_SIMT)])
def test_capture_then_replay_with_new_inputs(H, flags):
    from oracle import ref
    T, pool_rows, cap = 9, 8192, 2000
    first = W.tiny_workload(B=2, H=H, T=T, prefix_lens=[900, 400], pool_rows=pool_rows, seed=31)
    second = W.tiny_workload(B=2, H=H, T=T, prefix_lens=[1500, 37], pool_rows=pool_rows, seed=32)

    dev = "cuda"
    q_nope = torch.empty((2 * T, H, 512), dtype=torch.bfloat16, device=dev)
    q_rope = torch.empty((2 * T, H, 64), dtype=torch.bfloat16, device=dev)
    kv_pool = torch.empty((pool_rows, 576), dtype=torch.bfloat16, device=dev)
    kv_indptr = torch.empty(3, dtype=torch.int32, device=dev)
    kv_indices = torch.empty(2 * cap, dtype=torch.int32, device=dev)
    out_cache_loc = torch.empty(2 * T, dtype=torch.int32, device=dev)
    mask = torch.empty((2 * T * (cap + T) + 7) // 8, dtype=torch.uint8, device=dev)
    mask_indptr = torch.empty(2, dtype=torch.int32, device=dev)

    def load(wl):
        q_nope.view(torch.int16).copy_(torch.from_numpy(wl["q_nope"].view(np.int16)))
        q_rope.view(torch.int16).copy_(torch.from_numpy(wl["q_rope"].view(np.int16)))
        kv_pool.view(torch.int16).copy_(torch.from_numpy(wl["pool"].view(np.int16)))
        _fill(kv_indptr, wl["kv_indptr"].astype(np.int32), torch.int32)
        _fill(kv_indices, wl["kv_indices"].astype(np.int32), torch.int32)
        _fill(out_cache_loc, wl["out_cache_loc"].astype(np.int32), torch.int32)
        _fill(mask, wl["custom_mask"].astype(np.uint8), torch.uint8)
        _fill(mask_indptr, wl["mask_indptr"].astype(np.int32), torch.int32)
        torch.cuda.synchronize()

    v = B.Verifier(2, H, T, cap + T, pool_rows, 8, flags)
    stream = torch.cuda.Stream()

    def call():
        B.mla_verify_run(v.plan, q_nope, q_rope, kv_pool, kv_indptr, kv_indices, out_cache_loc, mask, mask_indptr,
                         2, first["sm_scale"], 8, v.workspace, v.o, v.lse, stream=stream)

    load(first)
    with torch.cuda.stream(stream):
        call()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        call()
    torch.cuda.synchronize()

    for wl in (first, second, first):
        load(wl)
        v.o.zero_()
        with torch.cuda.stream(stream):
            g.replay()
        torch.cuda.synchronize()
        assert v.status(stream) == 0
        o_ref, lse_ref = ref.verify(wl, nthreads=os.cpu_count() or 4)
        compare(bf16_to_f64(v.o).reshape(-1, 512), v.lse.cpu().numpy().reshape(-1), o_ref, lse_ref,
                "replay prefix=%s" % list(wl["prefix_lens"]))
