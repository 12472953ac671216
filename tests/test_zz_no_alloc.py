"""mla_verify_run_noalloc: the verify call for callers that cannot allocate
device memory (they get no workspace of their own), which runs on a scratch
array built into the library.

Checked through the C ABI against mla_verify_run with a caller-owned
workspace and against the fp64 oracle, on calls in a row with different
inputs (the scratch array keeps the previous call's contents), within the
parity tolerances; also after a call that raised a device status bit, with a
plan that picked its own split count, and with arguments it must reject
before touching the array.  This file sorts last so that a run stopping at
the first failure has run every other test before it.
"""

import numpy as np
import pytest

from mla_speculative_decode_tree_gb300 import binding as B
from mla_speculative_decode_tree_gb300 import workloads as W
from parity_util import bf16_to_f64, compare

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 32 << 20


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_speculative_decode_tree_gb300 import build
    build.build()
    from oracle import ref
    ref.build()


def _outputs(o, lse, n):
    return bf16_to_f64(o[:n]).reshape(-1, 512), lse[:n].cpu().numpy().astype(np.float64).reshape(-1)


def test_noalloc_matches_workspace_call_twice_in_a_row():
    first = W.tiny_workload(B=2, H=64, T=9, prefix_lens=[3000, 700], pool_rows=16384, seed=41, nsplit=8)
    second = W.tiny_workload(B=2, H=64, T=9, prefix_lens=[129, 2500], pool_rows=16384, seed=42, nsplit=8)
    v = B.Verifier(2, 64, 9, 3009, 16384, 8)
    assert v.plan.workspace_bytes <= SCRATCH_BYTES
    o_na = torch.empty_like(v.o)
    lse_na = torch.empty_like(v.lse)
    for wl in (first, second):
        d = B.device_inputs(wl)
        o_ref, lse_ref = v.run(d, 2, wl["sm_scale"])
        B.mla_verify_run_noalloc(v.plan, d["q_nope"], d["q_rope"], d["kv_pool"], d["kv_indptr"], d["kv_indices"],
                                 d["out_cache_loc"], d["custom_mask"], d["mask_indptr"], 2, wl["sm_scale"], 8,
                                 o_na, lse_na)
        torch.cuda.synchronize()
        n = 2 * 9
        # the same kernels on the same inputs: the same bits
        assert torch.equal(o_na[:n].view(torch.int16), o_ref[:n].view(torch.int16)) and torch.equal(lse_na[:n], lse_ref[:n])
        a_o, a_l = _outputs(o_na, lse_na, n)
        r_o, r_l = _outputs(o_ref, lse_ref, n)
        compare(a_o, a_l, r_o, r_l, "noalloc vs workspace, prefix=%s" % list(wl["prefix_lens"]))


def test_noalloc_with_fused_merge_plan():
    """A fused-merge plan on the scratch array: its arrival counters are zeroed
    with the header each call; the results equal the plain plan's, bit for bit,
    over three calls in a row."""
    plain = B.Verifier(2, 64, 9, 3009, 16384, 8)
    fused = B.mla_verify_plan(2, 64, 9, 3009, 16384, 8, B.MLA_VERIFY_FUSED_MERGE)
    assert fused.describe().merge_blocks == 0 and fused.workspace_bytes <= SCRATCH_BYTES
    o_na = torch.empty_like(plain.o)
    lse_na = torch.empty_like(plain.lse)
    for k, P in enumerate(([3000, 700], [129, 2500], [1, 3000])):
        wl = W.tiny_workload(B=2, H=64, T=9, prefix_lens=P, pool_rows=16384, seed=50 + k, nsplit=8)
        d = B.device_inputs(wl)
        o_ref, lse_ref = plain.run(d, 2, wl["sm_scale"])
        B.mla_verify_run_noalloc(fused, d["q_nope"], d["q_rope"], d["kv_pool"], d["kv_indptr"], d["kv_indices"],
                                 d["out_cache_loc"], d["custom_mask"], d["mask_indptr"], 2, wl["sm_scale"], 8,
                                 o_na, lse_na)
        torch.cuda.synchronize()
        assert torch.equal(o_na.view(torch.int16), o_ref.view(torch.int16)) and torch.equal(lse_na, lse_ref)


def _noalloc(plan, d, batch, scale, nsplit, o, lse):
    B.mla_verify_run_noalloc(plan, d["q_nope"], d["q_rope"], d["kv_pool"], d["kv_indptr"], d["kv_indices"],
                             d["out_cache_loc"], d["custom_mask"], d["mask_indptr"], batch, scale, nsplit, o, lse)
    torch.cuda.synchronize()


def test_noalloc_matches_the_oracle():
    from oracle import ref
    for seed, P in ((61, [2500, 129]), (62, [40, 3000])):
        wl = W.tiny_workload(B=2, H=64, T=9, prefix_lens=P, pool_rows=16384, seed=seed, nsplit=8)
        d = B.device_inputs(wl)
        plan = B.mla_verify_plan(2, 64, 9, 3009, 16384, 8)
        o = torch.empty(18 * 64 * 512, dtype=torch.bfloat16, device="cuda")
        lse = torch.empty(18 * 64, dtype=torch.float32, device="cuda")
        _noalloc(plan, d, 2, wl["sm_scale"], 8, o, lse)
        o_ref, lse_ref = ref.verify(wl)
        a_o, a_l = _outputs(o.view(-1, 512), lse, 18 * 64)
        compare(a_o, a_l, o_ref, lse_ref, "noalloc vs oracle, prefix=%s" % P)


def test_noalloc_auto_split_eight_heads():
    """A plan that picked its own split count (nsplit = 0), 8 heads x 9 tokens."""
    from oracle import ref
    wl = W.tiny_workload(B=1, H=8, T=9, prefix_lens=[20000], pool_rows=32768, seed=63, nsplit=4)
    d = B.device_inputs(wl)
    plan = B.mla_verify_plan(1, 8, 9, 20009, 32768, 0)
    assert plan.workspace_bytes <= SCRATCH_BYTES
    o = torch.empty(9 * 8 * 512, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(9 * 8, dtype=torch.float32, device="cuda")
    for _ in range(2):
        _noalloc(plan, d, 1, wl["sm_scale"], 0, o, lse)
        o_ref, lse_ref = ref.verify(wl)
        a_o, a_l = _outputs(o.view(-1, 512), lse, 72)
        compare(a_o, a_l, o_ref, lse_ref, "noalloc nsplit=0, 8 heads")


def test_noalloc_after_a_call_with_an_out_of_range_row():
    """A call whose indices point outside the pool sets status bits in the
    shared array's header; the next, valid call still matches the workspace
    path (each call starts from a zeroed header)."""
    good = W.tiny_workload(B=2, H=64, T=9, prefix_lens=[2000, 700], pool_rows=16384, seed=64, nsplit=8)
    bad_idx = good["kv_indices"].copy()
    bad_idx[5] = 1 << 30
    bad = dict(good, kv_indices=bad_idx)
    v = B.Verifier(2, 64, 9, 3009, 16384, 8)
    o_na = torch.empty_like(v.o)
    lse_na = torch.empty_like(v.lse)
    _noalloc(v.plan, B.device_inputs(bad), 2, good["sm_scale"], 8, o_na, lse_na)
    d = B.device_inputs(good)
    o_ref, lse_ref = v.run(d, 2, good["sm_scale"])
    _noalloc(v.plan, d, 2, good["sm_scale"], 8, o_na, lse_na)
    a_o, a_l = _outputs(o_na, lse_na, 18)
    r_o, r_l = _outputs(o_ref, lse_ref, 18)
    compare(a_o, a_l, r_o, r_l, "noalloc after an out-of-range row")


def test_noalloc_rejects_bad_arguments_like_run():
    plan = B.mla_verify_plan(2, 64, 9, 3009, 16384, 8)
    t = torch.zeros(1 << 12, dtype=torch.uint8, device="cuda")
    for batch, nsplit, q, code in ((3, 8, t, B.MLA_VERIFY_EINVAL),       # batch above max_batch
                                   (1, 4, t, B.MLA_VERIFY_EINVAL),       # nsplit differs from the plan's
                                   (1, 8, t[2:], B.MLA_VERIFY_EINVAL)):  # misaligned query
        with pytest.raises(B.MlaVerifyError) as e:
            B.mla_verify_run_noalloc(plan, q, t, t, t, t, t, t, t, batch, 0.07, nsplit, t, t)
        assert e.value.code == code
    B.mla_verify_run_noalloc(plan, t, t, t, t, t, t, t, t, 0, 0.07, 8, t, t)  # batch 0: nothing to do


def test_noalloc_rejects_plans_beyond_the_scratch_size():
    p = B.mla_verify_plan(1, 64, 9, 100000, 1 << 20, 64)  # 64 splits x 576 rows of partials > 32 MiB
    assert p.workspace_bytes > SCRATCH_BYTES
    dummy = torch.zeros(1 << 10, dtype=torch.uint8, device="cuda")
    with pytest.raises(B.MlaVerifyError) as e:
        B.mla_verify_run_noalloc(p, dummy, dummy, dummy, dummy, dummy, dummy, dummy, dummy, 1, 0.07, 64,
                                 dummy, dummy)
    assert e.value.code == B.MLA_VERIFY_EWORKSPACE
    # batch 0 enqueues nothing and succeeds, as mla_verify_run does, whatever the plan's size
    B.mla_verify_run_noalloc(p, dummy, dummy, dummy, dummy, dummy, dummy, dummy, dummy, 0, 0.07, 64, dummy, dummy)
