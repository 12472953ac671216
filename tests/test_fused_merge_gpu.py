"""Merge fused into the tensor-core split kernel (MLA_VERIFY_FUSED_MERGE):
bit-identical to the separate merge kernel on the same inputs, across row-group
sizes, ragged batches, empty splits, varlen calls, repeated calls (the arrival
counters reset themselves) and CUDA-graph replay; and against the oracle."""

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


def _pair(wl, nsplit=None, mode=0):
    plain = B.verifier_for(wl, nsplit=nsplit, flags=mode)
    fused = B.verifier_for(wl, nsplit=nsplit, flags=B.MLA_VERIFY_FUSED_MERGE | mode)
    assert fused.plan.describe().merge_blocks == 0 and fused.plan.describe().kernel == 1
    return plain, fused


def _same(a, b):
    return torch.equal(a.o.view(torch.int16), b.o.view(torch.int16)) and torch.equal(a.lse, b.lse)


CASES = [
    # (B, H, T, prefixes, nsplit)
    (1, 64, 9, [4096], 16),
    (1, 64, 9, [300], 16),               # most splits empty
    (3, 64, 9, [2000, 0, 777], 8),       # an empty prefix in the batch
    (2, 16, 4, [5000, 129], 4),
    (4, 32, 3, [64, 1, 900, 4000], 32),
    (1, 8, 9, [20000], 64),              # few rows: 48-row groups
    (1, 64, 9, [6000], 48),              # 576 rows, 48 splits: partials past 48 MB, loaded after their LSEs
]


def test_every_merge_layout_is_compared():
    """The cases cover the merge kernel's three forms: two warps per row (many
    rows), four warps per row with the partials loaded ahead (partials <= 48 MB)
    and four warps per row without (describe().merge_blocks: rows/4 or rows/2)."""
    forms = set()
    for Bn, H, T, P, nsplit in CASES:
        info = B.mla_verify_plan(Bn, H, T, max(P) + T, 32768, nsplit, 0).describe()
        rows = Bn * H * T
        quarter = info.merge_blocks == (rows + 1) // 2
        assert quarter or info.merge_blocks == (rows + 3) // 4
        forms.add((quarter, quarter and nsplit * rows * 2048 <= 48 << 20))
    assert forms == {(False, False), (True, True), (True, False)}, forms


@pytest.mark.parametrize("mode", [0, B.MLA_VERIFY_REFETCH_VALUES], ids=["resident", "refetch"])
@pytest.mark.parametrize("case", CASES, ids=[str(i) for i in range(len(CASES))])
def test_fused_equals_separate_merge(case, mode):
    Bn, H, T, P, nsplit = case
    wl = W.tiny_workload(B=Bn, H=H, T=T, prefix_lens=P, pool_rows=32768, seed=Bn * 7 + H + T, nsplit=nsplit)
    d = B.device_inputs(wl)
    plain, fused = _pair(wl, mode=mode)
    fused.o.fill_(float("nan"))
    plain.run(d, wl["B"], wl["sm_scale"])
    fused.run(d, wl["B"], wl["sm_scale"])
    torch.cuda.synchronize()
    assert plain.status() == 0 and fused.status() == 0
    assert _same(plain, fused), "fused merge differs from the merge kernel (case %s)" % (case,)


def test_fused_matches_oracle():
    from oracle import ref
    wl = W.tiny_workload(B=2, H=64, T=9, prefix_lens=[1500, 333], pool_rows=8192, seed=77, nsplit=8)
    d = B.device_inputs(wl)
    v = B.verifier_for(wl, flags=B.MLA_VERIFY_FUSED_MERGE)
    o, lse = v.run(d, wl["B"], wl["sm_scale"])
    torch.cuda.synchronize()
    o_ref, lse_ref = ref.verify(wl, nthreads=os.cpu_count() or 4)
    compare(bf16_to_f64(o).reshape(-1, 512), lse.cpu().numpy().reshape(-1), o_ref, lse_ref, "fused merge vs oracle")


def test_fused_varlen_equals_separate():
    wl = W.varlen_workload(B=4, H=64, T_list=[9, 0, 3, 1], prefix_lens=[800, 50, 2100, 0], pool_rows=8192, seed=5,
                           nsplit=8)
    d = B.device_inputs(wl)
    plain, fused = _pair(wl)
    for v in (plain, fused):
        v.o.fill_(float("nan"))
        v.lse.fill_(float("nan"))
        v.run(d, wl["B"], wl["sm_scale"])
    torch.cuda.synchronize()
    n = int(wl["qo_indptr"][-1]) * wl["H"]
    assert torch.equal(plain.o.reshape(-1, 512)[:n].view(torch.int16), fused.o.reshape(-1, 512)[:n].view(torch.int16))
    assert torch.equal(plain.lse.reshape(-1)[:n], fused.lse.reshape(-1)[:n])
    # rows past the call's tokens are not written by either
    assert torch.isnan(fused.lse.reshape(-1)[n:]).all()


def test_repeated_calls_and_graph_replay():
    """The counters return to zero after every call: many calls in a row, with
    different prefix lengths, each equal the separate merge; then the same
    inside one captured graph."""
    H, T, nsplit, cap = 64, 9, 16, 6000
    wls = [W.tiny_workload(B=2, H=H, T=T, prefix_lens=p, pool_rows=16384, seed=90 + k, nsplit=nsplit)
           for k, p in enumerate([[5000, 100], [64, 5900], [3000, 3000]])]
    plain = B.Verifier(2, H, T, cap + T, 16384, nsplit)
    fused = B.Verifier(2, H, T, cap + T, 16384, nsplit, flags=B.MLA_VERIFY_FUSED_MERGE)
    for rep in range(2):
        for wl in wls:
            d = B.device_inputs(wl)
            plain.run(d, wl["B"], wl["sm_scale"])
            fused.run(d, wl["B"], wl["sm_scale"])
            torch.cuda.synchronize()
            assert _same(plain, fused)
    counters = fused.workspace[256:256 + 4 * 2 * fused.plan.describe().grid_x].view(torch.int32)
    assert int(counters.abs().sum()) == 0
    # graph: buffers of fixed size, contents replaced between replays
    d0 = B.device_inputs(wls[0])
    bufs = {k: t.clone() for k, t in d0.items()}
    big = max(int(np.sum(w["prefix_lens"])) for w in wls)
    bufs["kv_indices"] = torch.zeros(big, dtype=torch.int32, device="cuda")
    mask_bytes = max(w["custom_mask"].size for w in wls)
    bufs["custom_mask"] = torch.zeros(mask_bytes, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.Stream()

    def call():
        B.mla_verify_run(fused.plan, bufs["q_nope"], bufs["q_rope"], bufs["kv_pool"], bufs["kv_indptr"],
                         bufs["kv_indices"], bufs["out_cache_loc"], bufs["custom_mask"], bufs["mask_indptr"], 2,
                         wls[0]["sm_scale"], nsplit, fused.workspace, fused.o, fused.lse, stream=stream)

    def load(wl):
        fresh = B.device_inputs(wl)
        for k, t in bufs.items():
            src = fresh[k].reshape(-1)
            t.view(-1)[: src.numel()].copy_(src)
        torch.cuda.synchronize()
        return fresh

    load(wls[0])
    with torch.cuda.stream(stream):
        call()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        call()
    for wl in wls[1:] + wls[:1]:
        fresh = load(wl)
        with torch.cuda.stream(stream):
            g.replay()
        torch.cuda.synchronize()
        plain.run(fresh, wl["B"], wl["sm_scale"])
        torch.cuda.synchronize()
        assert _same(plain, fused)
