"""Per-request draft-token counts (mla_verify_run_varlen) and T = 1 decode on
the same kernels, against the oracle."""

import os

import numpy as np
import pytest

from mla_speculative_decode_tree_gb300 import binding as B
from mla_speculative_decode_tree_gb300 import workloads as W
from parity_util import bf16_to_f64, compare, sample_rows

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_speculative_decode_tree_gb300 import build
    build.build()


def _run(wl, flags=0, nsplit=None):
    d = B.device_inputs(wl)
    v = B.verifier_for(wl, flags=flags, nsplit=nsplit)
    v.o.fill_(float("nan"))
    v.lse.fill_(float("nan"))
    v.run(d, wl["B"], wl["sm_scale"])
    torch.cuda.synchronize()
    return v, v.status()


def _check(wl, v, what):
    from oracle import ref
    n = ref.n_token_rows(wl) * wl["H"]
    o = bf16_to_f64(v.o.reshape(-1, 512)[:n])
    lse = v.lse.reshape(-1)[:n].cpu().numpy().astype(np.float64)
    o_ref, lse_ref = ref.verify(wl, nthreads=os.cpu_count() or 4)
    compare(o, lse, o_ref, lse_ref, what)
    # rows past the call's tokens are never written
    rest_o = v.o.reshape(-1, 512)[n:]
    rest_l = v.lse.reshape(-1)[n:]
    assert torch.isnan(rest_o.float()).all() and torch.isnan(rest_l).all(), what + ": rows past the tokens written"


VARLEN = [
    # (H, T_list, prefixes, nsplit)
    (64, [3, 0, 9, 1], [500, 40, 0, 1300], 4),
    (64, [16, 1, 7], [257, 2000, 3], 8),
    (16, [1, 1, 1, 1, 1], [100, 0, 3000, 64, 129], 4),
    (8, [9, 2, 0, 5], [700, 130, 64, 1], 4),
    (3, [4, 9], [200, 50], 2),
]


@pytest.mark.parametrize("flags", [0, B.MLA_VERIFY_REFETCH_VALUES, B.MLA_VERIFY_FORCE_SIMT],
                         ids=["resident", "refetch", "simt"])
@pytest.mark.parametrize("case", VARLEN, ids=[str(i) for i in range(len(VARLEN))])
def test_varlen_parity(case, flags):
    H, T_list, prefixes, nsplit = case
    wl = W.varlen_workload(B=len(T_list), H=H, T_list=T_list, prefix_lens=prefixes, pool_rows=16384,
                           seed=sum(T_list) + H, nsplit=nsplit)
    v, st = _run(wl, flags=flags)
    assert st == 0
    _check(wl, v, "varlen H=%d T=%s flags=%d kernel=%d" % (H, T_list, flags, v.plan.describe().kernel))


@pytest.mark.parametrize("H", [64, 16, 8])
def test_decode_t1_uniform(H):
    """T = 1 through the plain entry point: the same kernels at N = H rows."""
    wl = W.tiny_workload(B=4, H=H, T=1, prefix_lens=[4096, 129, 1, 2500], pool_rows=16384, seed=H, nsplit=8)
    d = B.device_inputs(wl)
    v = B.verifier_for(wl)
    o, lse = v.run(d, wl["B"], wl["sm_scale"])
    torch.cuda.synchronize()
    from oracle import ref
    o_ref, lse_ref = ref.verify(wl, nthreads=os.cpu_count() or 4)
    compare(bf16_to_f64(o).reshape(-1, 512), lse.cpu().numpy().reshape(-1), o_ref, lse_ref,
            "decode H=%d kernel=%d rows/cta=%d" % (H, v.plan.describe().kernel, v.plan.describe().rows_per_cta))


def test_varlen_with_uniform_counts_matches_run():
    """All T_b equal: the varlen call and the uniform call give identical bits."""
    wl = W.varlen_workload(B=3, H=64, T_list=[9, 9, 9], prefix_lens=[1000, 77, 400], pool_rows=8192, seed=5,
                           nsplit=4)
    v, _ = _run(wl)
    o1, l1 = v.o.clone(), v.lse.clone()
    uni = dict(wl)
    del uni["qo_indptr"]
    d = B.device_inputs(uni)
    v.run(d, 3, wl["sm_scale"])
    torch.cuda.synchronize()
    assert torch.equal(v.o.view(torch.int16), o1.view(torch.int16)) and torch.equal(v.lse, l1)


@pytest.mark.slow
def test_decode_b16_full_size_sampled():
    """B = 16 decode (T = 1), H = 64, prefixes U[1024, 32768], pool 1M rows, NSPLIT = 16."""
    cfg = W.CONFIGS["decode_b16"]
    wl = W.make_workload(cfg)
    d = B.device_inputs(wl)
    v = B.verifier_for(wl)
    o, lse = v.run(d, wl["B"], wl["sm_scale"])
    torch.cuda.synchronize()
    from oracle import ref
    rows = sample_rows(wl, per_request=8)
    o_ref, lse_ref = ref.verify(wl, rows=rows, nthreads=os.cpu_count() or 4)
    compare(bf16_to_f64(o).reshape(-1, 512)[rows], lse.cpu().numpy().reshape(-1)[rows], o_ref, lse_ref,
            "decode_b16 sampled")


@pytest.mark.slow
def test_varlen_b16_full_size_sampled():
    wl = W.make_workload(W.CONFIGS["varlen_b16"])
    v, st = _run(wl)
    assert st == 0
    from oracle import ref
    qo = wl["qo_indptr"]
    rng = np.random.default_rng(3)
    rows = []
    for b in range(wl["B"]):
        for i in range(int(qo[b + 1] - qo[b])):
            rows.append((int(qo[b]) + i) * wl["H"] + int(rng.integers(0, wl["H"])))
    rows = np.array(rows, dtype=np.int64)
    o_ref, lse_ref = ref.verify(wl, rows=rows, nthreads=os.cpu_count() or 4)
    compare(bf16_to_f64(v.o.reshape(-1, 512)[rows]), v.lse.reshape(-1)[rows].cpu().numpy(), o_ref, lse_ref,
            "varlen_b16 sampled")


def test_varlen_capture_with_new_counts():
    """One captured varlen call replayed with new per-request counts (fixed-size buffers)."""
    from oracle import ref
    H, Tmax, pool_rows, cap_prefix = 64, 9, 8192, 1200
    cases = [([9, 1, 4], [900, 50, 1100]), ([2, 9, 0], [300, 1200, 17]), ([1, 1, 1], [5, 600, 1000])]
    wls = [W.varlen_workload(B=3, H=H, T_list=t, prefix_lens=p, pool_rows=pool_rows, seed=40 + k, nsplit=4)
           for k, (t, p) in enumerate(cases)]
    v = B.Verifier(3, H, Tmax, cap_prefix + Tmax, pool_rows, 4)
    dev = "cuda"
    bufs = dict(
        q_nope=torch.zeros((3 * Tmax, H, 512), dtype=torch.bfloat16, device=dev),
        q_rope=torch.zeros((3 * Tmax, H, 64), dtype=torch.bfloat16, device=dev),
        kv_pool=torch.zeros((pool_rows, 576), dtype=torch.bfloat16, device=dev),
        kv_indptr=torch.zeros(4, dtype=torch.int32, device=dev),
        kv_indices=torch.zeros(3 * cap_prefix, dtype=torch.int32, device=dev),
        qo_indptr=torch.zeros(4, dtype=torch.int32, device=dev),
        out_cache_loc=torch.zeros(3 * Tmax, dtype=torch.int32, device=dev),
        custom_mask=torch.zeros((3 * Tmax * (cap_prefix + Tmax) + 7) // 8, dtype=torch.uint8, device=dev),
        mask_indptr=torch.zeros(3, dtype=torch.int32, device=dev),
    )

    def load(wl):
        fresh = B.device_inputs(wl)
        for k, t in bufs.items():
            t.zero_()
            src = fresh[k].reshape(-1)
            t.view(-1)[: src.numel()].copy_(src)
        torch.cuda.synchronize()

    stream = torch.cuda.Stream()

    def call():
        B.mla_verify_run_varlen(v.plan, bufs["q_nope"], bufs["q_rope"], bufs["kv_pool"], bufs["kv_indptr"],
                                bufs["kv_indices"], bufs["qo_indptr"], bufs["out_cache_loc"], bufs["custom_mask"],
                                bufs["mask_indptr"], 3, wls[0]["sm_scale"], 4, v.workspace, v.o, v.lse,
                                stream=stream)

    load(wls[0])
    with torch.cuda.stream(stream):
        call()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        call()
    for wl in wls[1:] + wls[:1]:
        load(wl)
        with torch.cuda.stream(stream):
            g.replay()
        torch.cuda.synchronize()
        n = ref.n_token_rows(wl) * H
        o_ref, lse_ref = ref.verify(wl, nthreads=os.cpu_count() or 4)
        compare(bf16_to_f64(v.o.reshape(-1, 512)[:n]), v.lse.reshape(-1)[:n].cpu().numpy(), o_ref, lse_ref,
                "varlen replay T=%s" % list(wl["T_list"]))
