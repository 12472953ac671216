"""GPU parity: the CUDA path (through the C ABI) against the fp64 CPU oracle.

Small configurations are compared element by element on every output row;
full-size configurations on sampled rows, in the launch configuration the
benchmark times.  Row selection and mask decoding are checked bit-exactly
with rows that encode their own index and a single visible key per token.
"""

import os

import numpy as np
import pytest

from mla_speculative_decode_tree_gb300 import binding as B
from mla_speculative_decode_tree_gb300 import workloads as W
from parity_util import bf16_to_f64, compare, sample_rows

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

NTHREADS = os.cpu_count() or 4
# Tensor-core kernel in resident-tile mode (the default), in value-refetch
# mode, and the CUDA-core kernel.
MODES = [0, B.MLA_VERIFY_REFETCH_VALUES, B.MLA_VERIFY_FORCE_SIMT]
MODE_IDS = ["resident", "refetch", "simt"]


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_speculative_decode_tree_gb300 import build
    build.build()
    from oracle import ref
    ref.build()


def gpu_run(wl, flags=0, nsplit=None, d=None):
    d = d or B.device_inputs(wl)
    v = B.verifier_for(wl, flags=flags, nsplit=nsplit)
    o, lse = v.run(d, wl["B"], wl["sm_scale"])
    torch.cuda.synchronize()
    st = v.status()
    return bf16_to_f64(o).reshape(-1, 512), lse.cpu().numpy().astype(np.float64).reshape(-1), st, v


def check_full(wl, flags=0, nsplit=None, what=""):
    from oracle import ref
    o, lse, st, v = gpu_run(wl, flags, nsplit)
    assert st == 0, "device status %#x" % st
    o_ref, lse_ref = ref.verify(wl, nthreads=NTHREADS)
    return compare(o, lse, o_ref, lse_ref, what), v


SMALL = [
    ("tiny", {}),
    ("reg_p21", {}),
    ("reg_b2", {}),
]


@pytest.mark.parametrize("flags", MODES, ids=MODE_IDS)
@pytest.mark.parametrize("name", [s[0] for s in SMALL])
def test_parity_small_configs(name, flags):
    wl = W.make_workload(W.CONFIGS[name])
    check_full(wl, flags, what=name)


ADHOC = [
    # B, H, T, prefixes, pool, nsplit, tree
    (3, 64, 9, [0, 127, 1000], 4096, 4, "random"),   # empty prefix, ragged tail, multi-tile
    (2, 8, 9, [128, 385], 2048, 3, "random"),        # H=8: 72 rows, small grid
    (2, 16, 4, [256, 255], 2048, 2, "chain"),        # 64 rows
    (1, 64, 1, [700], 2048, 2, "random"),            # decode (T=1) on the tensor cores
    (2, 8, 1, [300, 5], 2048, 2, "random"),          # decode with 8 rows: half-empty 16-row tile
    (2, 5, 7, [200, 333], 2048, 3, "random"),        # 35 rows -> 48-row group, tokens straddle groups
    (1, 1, 16, [90], 1024, 1, "random"),             # 16 rows, one head
    (1, 32, 3, [5000], 8192, 64, "random"),          # more splits than needed: empty splits
    (2, 96, 2, [130, 129], 2048, 2, "random"),       # 192 rows = 3 x 64 or 2 x 96
    # one case per row-group size the planner can pick in each mode (the
    # fill-aware choice moves small grids to 48 rows, so the others need grids
    # of >= 152 CTAs)
    (2, 8, 4, [300, 77], 2048, 2, "random"),          # 32 rows -> 32-row groups
    (3, 16, 4, [2000, 300, 4000], 8192, 64, "random"),  # 64 rows, 192 CTAs -> 64-row groups
    (4, 8, 9, [3000, 100, 5000, 64], 16384, 64, "random"),  # 72 rows, 256 CTAs -> 48 rows, or one 96-row group
    (2, 64, 9, [5000, 3000], 16384, 64, "random"),    # 576 rows -> 64-row groups, or 96
    (1, 2, 64, [500], 4096, 2, "random"),             # q_len 64 (the maximum): 24 tokens per group
    (1, 16, 9, [1400], 4096, 8, "random"),            # one request: chunks of 192 keys end in a half tile
]


@pytest.mark.parametrize("flags", MODES, ids=MODE_IDS)
@pytest.mark.parametrize("case", ADHOC, ids=[str(i) for i in range(len(ADHOC))])
def test_parity_adhoc(case, flags):
    Bn, H, T, prefixes, pool, nsplit, tree = case
    wl = W.tiny_workload(B=Bn, H=H, T=T, prefix_lens=prefixes, pool_rows=pool, seed=sum(prefixes) + H,
                         tree=tree, nsplit=nsplit)
    check_full(wl, flags, what=str(case))


def test_a_half_tile_chunk_is_exercised():
    """One ad-hoc case plans chunks that end in a half tile (64-key granule)."""
    info = B.mla_verify_plan(1, 16, 9, 1409, 4096, 8, 0).describe()
    assert info.chunk_granule == 64 and info.resident_tile == 1  # ceil(1409 / 8) = 177 -> 192 keys


def test_every_mode_and_row_group_size_is_exercised():
    """The ad-hoc cases, planned with and without MLA_VERIFY_REFETCH_VALUES,
    cover every (mode, rows per CTA) pair the planner can pick."""
    pairs = set()
    for flags in MODES[:2]:
        for B_, H, T, prefixes, pool, nsplit, tree in ADHOC:
            info = B.mla_verify_plan(B_, H, T, max(prefixes) + T, pool, nsplit, flags).describe()
            assert info.kernel == 1 and not (flags and info.resident_tile)
            pairs.add((info.resident_tile, info.rows_per_cta))
    want = {(1, n) for n in (16, 32, 48, 64)} | {(0, n) for n in (16, 32, 48, 64, 96)}
    assert want <= pairs, want - pairs


FULL = ["short4k", "mid64k", "long185k_h8", "batch16_ragged", "needle64k"]
_wl_cache = {}


def full_workload(name):
    if name not in _wl_cache:
        _wl_cache.clear()
        _wl_cache[name] = W.make_workload(W.CONFIGS[name])
    return _wl_cache[name]


@pytest.mark.slow
@pytest.mark.parametrize("flags", MODES[:2], ids=MODE_IDS[:2])
@pytest.mark.parametrize("name", FULL)
def test_parity_full_configs_sampled(name, flags):
    from oracle import ref
    wl = full_workload(name)
    rows = sample_rows(wl, per_request=36 if wl["B"] == 1 else 6)
    o, lse, st, v = gpu_run(wl, flags=flags)
    assert st == 0
    o_ref, lse_ref = ref.verify(wl, rows=rows, nthreads=NTHREADS)
    err = compare(o[rows], lse[rows], o_ref, lse_ref, name)
    if name == "needle64k":
        assert np.abs(o_ref).max() > 1.0  # the planted keys really dominate
    print(name, v.plan.describe().kernel, err)


@pytest.mark.slow
def test_short4k_simt_cross_check():
    from oracle import ref
    wl = full_workload("short4k")
    rows = sample_rows(wl, per_request=18)
    o, lse, st, _ = gpu_run(wl, flags=B.MLA_VERIFY_FORCE_SIMT)
    o_ref, lse_ref = ref.verify(wl, rows=rows, nthreads=NTHREADS)
    compare(o[rows], lse[rows], o_ref, lse_ref, "short4k simt")


@pytest.mark.slow
@pytest.mark.parametrize("flags", MODES[:2], ids=MODE_IDS[:2])
def test_locality_pair_bit_identical(flags):
    """Scattered rows vs a sorted free list holding the same logical rows: identical bits."""
    from oracle import ref
    wl = W.make_workload(W.CONFIGS["mid64k"])
    wl_sorted = W.relayout(wl, "sorted", seed=1234)
    o1, lse1, st1, _ = gpu_run(wl, flags=flags)
    o2, lse2, st2, _ = gpu_run(wl_sorted, flags=flags)
    assert st1 == 0 and st2 == 0
    assert np.array_equal(o1, o2) and np.array_equal(lse1, lse2)
    rows = sample_rows(wl, per_request=12)
    o_ref, lse_ref = ref.verify(wl_sorted, rows=rows, nthreads=NTHREADS)
    compare(o2[rows], lse2[rows], o_ref, lse_ref, "sorted layout")


@pytest.mark.parametrize("flags", MODES[:2], ids=MODE_IDS[:2])
@pytest.mark.parametrize("nsplit", [1, 2, 5, 16, 64])
def test_nsplit_invariance(nsplit, flags):
    from oracle import ref
    wl = W.tiny_workload(B=2, H=64, T=9, prefix_lens=[3000, 1200], pool_rows=8192, seed=21, nsplit=nsplit)
    o, lse, st, _ = gpu_run(wl, flags=flags)
    o_ref, lse_ref = ref.verify(wl, nthreads=NTHREADS)
    compare(o, lse, o_ref, lse_ref, "nsplit=%d" % nsplit)


@pytest.mark.parametrize("flags", MODES[:2], ids=MODE_IDS[:2])
@pytest.mark.parametrize("nsplit", [1, 3, 7, 16, 40])
def test_nsplit_invariance_one_request(nsplit, flags):
    """One request (64 rows): in resident mode the chunks are multiples of 64 keys, so most
    of these end in a half tile (3004 keys: 1024, 448, 192 and 128-key chunks)."""
    from oracle import ref
    wl = W.tiny_workload(B=1, H=16, T=4, prefix_lens=[3000], pool_rows=8192, seed=22, nsplit=nsplit)
    info = B.mla_verify_plan(1, 16, 4, 3004, 8192, nsplit, flags).describe()
    assert info.chunk_granule == (128 if flags else 64)
    o, lse, st, _ = gpu_run(wl, flags=flags)
    assert st == 0
    o_ref, lse_ref = ref.verify(wl, nthreads=NTHREADS)
    compare(o, lse, o_ref, lse_ref, "one request, nsplit=%d" % nsplit)


def encoded_pool(pool_rows, rng):
    """Rows whose first three latent values spell their own index (exact in bf16)."""
    pool = np.zeros((pool_rows, 576), dtype=np.float32)
    r = np.arange(pool_rows)
    pool[:, 0] = r % 256
    pool[:, 1] = (r // 256) % 256
    pool[:, 2] = r // 65536
    pool[:, 3:512] = rng.standard_normal((pool_rows, 509)).astype(np.float32)
    pool[:, 512:] = rng.standard_normal((pool_rows, 64)).astype(np.float32)
    return W.f32_to_bf16_bits(pool)


@pytest.mark.parametrize("flags", MODES, ids=MODE_IDS)
@pytest.mark.parametrize("H,T,prefixes", [(64, 9, [300, 1001, 7]), (8, 9, [129, 0, 640]), (3, 5, [40, 9, 300]),
                                         (16, 4, [2900])])  # one request: 1472-key chunks end in a half tile
def test_row_selection_and_mask_decoding_exact(H, T, prefixes, flags):
    """One visible key per draft token at a chosen position: O must be that row, bit for bit."""
    rng = np.random.default_rng(H * 100 + T)
    wl = W.tiny_workload(B=len(prefixes), H=H, T=T, prefix_lens=prefixes, pool_rows=4096, seed=H + T)
    wl["pool"] = encoded_pool(4096, rng)
    dense, expect_rows = [], []
    for b, P in enumerate(prefixes):
        L = P + T
        m = np.zeros((T, L), dtype=bool)
        js = rng.integers(0, L, size=T)
        js[0] = L - 1
        if P > 0:
            js[min(1, T - 1)] = P - 1
        if T > 2 and L > 1472:
            js[2] = 1471  # the last key of the first chunk when chunks are 1472 keys (one request, nsplit 2)
        m[np.arange(T), js] = True
        dense.append(m)
        for i in range(T):
            j = int(js[i])
            row = (wl["kv_indices"][int(wl["kv_indptr"][b]) + j] if j < P else wl["out_cache_loc"][b * T + j - P])
            expect_rows.append(int(row))
    wl["custom_mask"] = W.pack_bits_lsb(np.concatenate([d.reshape(-1) for d in dense]))
    o, lse, st, _ = gpu_run(wl, flags=flags)
    assert st == 0
    o = o.reshape(len(prefixes) * T, H, 512)
    pool = W.bf16_bits_to_f32(wl["pool"]).astype(np.float64)
    for q in range(len(prefixes) * T):
        want = pool[expect_rows[q], :512]
        for h in range(H):
            got = o[q, h]
            decoded = int(got[0]) + 256 * int(got[1]) + 65536 * int(got[2])
            assert decoded == expect_rows[q], (q, h, decoded, expect_rows[q])
            assert np.array_equal(got, want), (q, h)


def test_bad_row_sets_status_and_is_excluded():
    """A key whose pool row is outside the pool is left out (as if masked) and flagged."""
    from oracle import ref
    wl = W.tiny_workload(B=2, H=16, T=4, prefix_lens=[200, 150], pool_rows=1024, seed=5)
    bad = wl["kv_indices"].copy()
    bad[17] = 5000  # request 0, prefix key 17
    for flags in MODES:
        o, lse, st, _ = gpu_run(dict(wl, kv_indices=bad), flags=flags)
        assert st & B.MLA_VERIFY_DEV_BAD_ROW
        # reference: the same call with key 17 of request 0 masked for every token
        L = 204
        bits = np.unpackbits(wl["custom_mask"], bitorder="little").astype(bool)
        for i in range(4):
            bits[i * L + 17] = False
        o_ref, lse_ref = ref.verify(dict(wl, custom_mask=W.pack_bits_lsb(bits)), nthreads=NTHREADS)
        compare(o, lse, o_ref, lse_ref, "bad row, flags=%d" % flags)
    # the status word is cleared by the read
    o2, lse2, st2, _ = gpu_run(wl)
    assert st2 == 0


def test_nothing_visible_gives_zero_and_neg_inf():
    wl = W.tiny_workload(B=1, H=16, T=4, prefix_lens=[300], pool_rows=1024, seed=6)
    mask = wl["custom_mask"].copy()
    # token 2 sees nothing at all
    L = 304
    bits = np.unpackbits(mask, bitorder="little")[: 4 * L].reshape(4, L)
    bits[2] = 0
    wl["custom_mask"] = W.pack_bits_lsb(bits.reshape(-1))
    check_full(wl, what="empty row")


def test_batch_below_max_and_zero():
    from oracle import ref
    wl = W.tiny_workload(B=2, H=64, T=9, prefix_lens=[500, 900], pool_rows=4096, seed=7)
    d = B.device_inputs(wl)
    L = 909
    v = B.Verifier(4, 64, 9, L, 4096, 8)
    o, lse = v.run(d, 2, wl["sm_scale"])
    o_ref, lse_ref = ref.verify(wl, nthreads=NTHREADS)
    compare(bf16_to_f64(o).reshape(-1, 512), lse.cpu().numpy().reshape(-1), o_ref, lse_ref, "batch 2 of 4")
    v.run(d, 0, wl["sm_scale"])  # nothing enqueued, no error
    torch.cuda.synchronize()


def test_split_and_merge_entry_points_match_run():
    wl = W.tiny_workload(B=1, H=64, T=9, prefix_lens=[2000], pool_rows=4096, seed=8)
    d = B.device_inputs(wl)
    v = B.verifier_for(wl, nsplit=4)
    o1, l1 = v.run(d, 1, wl["sm_scale"])
    o1, l1 = o1.clone(), l1.clone()
    o2 = torch.empty_like(v.o)
    l2 = torch.empty_like(v.lse)
    B.mla_verify_split(v.plan, d["q_nope"], d["q_rope"], d["kv_pool"], d["kv_indptr"], d["kv_indices"],
                       d["out_cache_loc"], d["custom_mask"], d["mask_indptr"], 1, wl["sm_scale"], 4, v.workspace)
    B.mla_verify_merge(v.plan, 1, 4, v.workspace, o2, l2)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2[:9]) and torch.equal(l1, l2[:9])


# ---- nsplit = 0: the number of chunks chosen by the plan --------------------
AUTO_SPLIT = [
    # B, H, T, prefixes, pool
    (1, 64, 9, [4096], 16384),
    (3, 64, 9, [0, 127, 3000], 8192),      # ragged, an empty prefix
    (1, 8, 9, [20000], 32768),             # few rows: long chunks, one row group
    (2, 16, 1, [5000, 77], 8192),          # decode
    (1, 2, 64, [900], 4096),               # q_len 64
]


@pytest.mark.parametrize("flags", MODES, ids=MODE_IDS)
@pytest.mark.parametrize("case", AUTO_SPLIT, ids=[str(i) for i in range(len(AUTO_SPLIT))])
def test_parity_auto_split(case, flags):
    Bn, H, T, prefixes, pool = case
    wl = W.tiny_workload(B=Bn, H=H, T=T, prefix_lens=prefixes, pool_rows=pool, seed=sum(prefixes) + 3 * H, nsplit=4)
    _, v = check_full(wl, flags, nsplit=0, what="nsplit=0 " + str(case))
    assert v.plan.nsplit == 0 and v.plan.describe().grid_y >= 1


@pytest.mark.slow
@pytest.mark.parametrize("name", ["short4k", "long185k_h8"])
def test_auto_split_full_size_sampled(name):
    from oracle import ref
    wl = W.make_workload(W.CONFIGS[name])
    o, lse, st, v = gpu_run(wl, nsplit=0)
    assert st == 0
    rows = sample_rows(wl, per_request=8)
    o_ref, lse_ref = ref.verify(wl, rows=rows, nthreads=NTHREADS)
    compare(o[rows], lse[rows], o_ref, lse_ref, name + " nsplit=0")
