"""C-ABI checks that need no GPU: the library loads, exports every symbol the
header declares, and its host-side validation and plan choices behave as
documented in include/mla_verify.h."""

import ctypes
import os
import re

import pytest

from mla_speculative_decode_tree_gb300 import binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mla_verify.h")


@pytest.fixture(scope="module")
def lib():
    from mla_speculative_decode_tree_gb300 import build
    build.build()
    return B.load()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:int|const char\*)\s+(mla_verify_\w+)\s*\(", text, re.M)))


def test_header_declares_the_binding_surface():
    assert declared_functions() == sorted(B.EXPORTED)


def test_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_strerror_codes(lib):
    for code in range(5):
        assert isinstance(B.strerror(code), str) and B.strerror(code)
    assert B.strerror(B.MLA_VERIFY_OK) == "ok"
    assert "unknown" in B.strerror(99)


def plan(**kw):
    args = dict(max_batch=1, num_heads=64, q_len=9, max_kv_len=4105, pool_rows=262144, nsplit=16)
    args.update(kw)
    return B.mla_verify_plan(**args)


def test_plan_workspace_formula(lib):
    p = plan(max_batch=2, nsplit=16)
    rows = 2 * 9 * 64
    off_o = (256 + 4 * 16 * rows + 255) // 256 * 256
    assert p.workspace_bytes == off_o + 4 * 16 * rows * 512
    assert p.describe().workspace_bytes == p.workspace_bytes


def test_fused_merge_plan(lib):
    """The counters sit between the header and the partials; no merge grid; the
    flag is ignored by the CUDA-core kernel; no split-only call."""
    p = plan(max_batch=2, nsplit=16, flags=B.MLA_VERIFY_FUSED_MERGE)
    info = p.describe()
    assert info.kernel == 1 and info.merge_blocks == 0
    rows = 2 * 9 * 64
    off_lse = (256 + 4 * 2 * info.grid_x + 255) // 256 * 256
    off_o = (off_lse + 4 * 16 * rows + 255) // 256 * 256
    assert p.workspace_bytes == off_o + 4 * 16 * rows * 512
    simt = plan(num_heads=2, q_len=4, flags=B.MLA_VERIFY_FUSED_MERGE | B.MLA_VERIFY_FORCE_SIMT)
    assert simt.describe().kernel == 0 and simt.describe().merge_blocks > 0
    assert simt.workspace_bytes == plan(num_heads=2, q_len=4, flags=B.MLA_VERIFY_FORCE_SIMT).workspace_bytes
    ptr = FAKE
    rc = lib.mla_verify_split(ctypes.c_void_p(p.handle), ptr, ptr, ptr, ptr, ptr, ptr, ptr, ptr, 1, 0.072, 16, FAKE,
                              p.workspace_bytes, None)
    assert rc == B.MLA_VERIFY_EINVAL


def test_plan_accepts_the_test_stall_flag(lib):
    assert plan(flags=B.MLA_VERIFY_TEST_STALL_GATHER).describe().kernel == 1


@pytest.mark.parametrize("kw,code", [
    (dict(d_latent=256), B.MLA_VERIFY_EUNSUPPORTED),
    (dict(d_rope=32), B.MLA_VERIFY_EUNSUPPORTED),
    (dict(q_len=0), B.MLA_VERIFY_EINVAL),
    (dict(q_len=65), B.MLA_VERIFY_EINVAL),
    (dict(num_heads=0), B.MLA_VERIFY_EINVAL),
    (dict(max_batch=0), B.MLA_VERIFY_EINVAL),
    (dict(nsplit=-1), B.MLA_VERIFY_EINVAL),
    (dict(pool_rows=0), B.MLA_VERIFY_EINVAL),
    (dict(max_kv_len=3), B.MLA_VERIFY_EINVAL),
    (dict(flags=0x200), B.MLA_VERIFY_EINVAL),
    (dict(flags=0x8), B.MLA_VERIFY_EINVAL),
])
def test_plan_rejects(lib, kw, code):
    with pytest.raises(B.MlaVerifyError) as e:
        plan(**kw)
    assert e.value.code == code


def test_plan_null_pointers(lib):
    ws = ctypes.c_size_t(0)
    h = ctypes.c_void_p(0)
    assert lib.mla_verify_plan(None, ctypes.byref(ws), ctypes.byref(h)) == B.MLA_VERIFY_EINVAL
    p = B.MlaVerifyParams(1, 8, 9, 100, 1000, 4, 512, 64, 0)
    assert lib.mla_verify_plan(ctypes.byref(p), None, ctypes.byref(h)) == B.MLA_VERIFY_EINVAL
    assert lib.mla_verify_plan_describe(None, None) == B.MLA_VERIFY_EINVAL
    assert lib.mla_verify_destroy(None) == B.MLA_VERIFY_OK


R = B.MLA_VERIFY_REFETCH_VALUES


@pytest.mark.parametrize("H,T,kv,ns,flags,kernel,res,nq", [
    # 576 rows, 64 splits: 342 CTAs at 96 rows (3 waves) beat 513 resident 64-row CTAs (4 waves)
    (64, 9, 65545, 64, 0, 1, 0, 96),
    (64, 9, 65545, 16, 0, 1, 1, 64),   # 16 splits of 33 tiles: 144 resident CTAs fill one wave
    (64, 9, 5009, 16, 0, 1, 1, 64),    # 14 splits: 9 x 14 = 126 CTAs (48 rows: 168, two waves)
    (64, 9, 4105, 16, 0, 1, 1, 64),    # 11 splits: 99 CTAs; 48 rows (132) would land each key 12 times
    (8, 9, 5009, 16, 0, 1, 1, 48),     # 72 rows: 2 resident groups of 48
    (16, 4, 5004, 16, 0, 1, 1, 64),    # 64 rows: one resident group
    (8, 1, 5001, 16, 0, 1, 1, 16),     # decode with 8 heads: 16-row tile, half padding, still tensor cores
    (64, 9, 4105, 16, R, 1, 0, 48),    # value-refetch mode: one wave at 48 rows (more ring slots)
    (8, 9, 185009, 64, R, 1, 0, 48),   # 72 rows, 63 splits: 2 x 63 = 126 CTAs in one wave
    (64, 9, 5009, 16, B.MLA_VERIFY_FORCE_SIMT, 0, 0, 8),
])
def test_plan_kernel_choice(lib, H, T, kv, ns, flags, kernel, res, nq):
    info = plan(num_heads=H, q_len=T, max_kv_len=kv, nsplit=ns, flags=flags).describe()
    assert info.kernel == kernel
    assert info.resident_tile == res
    assert info.rows_per_cta == nq
    assert info.grid_x == -(-(H * T) // nq)
    assert info.grid_y == ns and info.grid_z == 1
    if kernel:
        assert 116 * 1024 < info.smem_bytes <= 227 * 1024  # one CTA per SM


FAKE = 0x10000  # never dereferenced: every check below fails before device work


def run_raw(lib, p, batch=1, nsplit=None, ws=FAKE, ws_bytes=None, ptr=FAKE, o=FAKE):
    nsplit = p.nsplit if nsplit is None else nsplit
    ws_bytes = p.workspace_bytes if ws_bytes is None else ws_bytes
    return lib.mla_verify_run(ctypes.c_void_p(p.handle), ptr, ptr, ptr, ptr, ptr, ptr, ptr, ptr, batch, 0.072, nsplit,
                              ws, ws_bytes, o, o, None)


def test_run_host_validation(lib):
    p = plan(max_batch=2)
    assert run_raw(lib, p, batch=3) == B.MLA_VERIFY_EINVAL
    assert run_raw(lib, p, batch=-1) == B.MLA_VERIFY_EINVAL
    assert run_raw(lib, p, nsplit=8) == B.MLA_VERIFY_EINVAL
    assert run_raw(lib, p, ws_bytes=p.workspace_bytes - 1) == B.MLA_VERIFY_EWORKSPACE
    assert run_raw(lib, p, ws=None) == B.MLA_VERIFY_EWORKSPACE
    assert run_raw(lib, p, ws=FAKE + 16) == B.MLA_VERIFY_EINVAL          # workspace not 256-byte aligned
    assert run_raw(lib, p, ptr=FAKE + 2) == B.MLA_VERIFY_EINVAL          # q/kv not 16-byte aligned
    assert run_raw(lib, p, o=FAKE + 8) == B.MLA_VERIFY_EINVAL            # o not 16-byte aligned
    assert run_raw(lib, p, o=None) == B.MLA_VERIFY_EINVAL
    assert run_raw(lib, p, batch=0) == B.MLA_VERIFY_OK                   # nothing to enqueue
    assert lib.mla_verify_merge(ctypes.c_void_p(p.handle), 3, p.nsplit, FAKE, p.workspace_bytes, FAKE, FAKE,
                                None) == B.MLA_VERIFY_EINVAL
    assert lib.mla_verify_workspace_init(ctypes.c_void_p(p.handle), FAKE, 16, None) == B.MLA_VERIFY_EINVAL


def test_relocate_host_validation(lib):
    p = plan(max_batch=2)
    h = ctypes.c_void_p(p.handle)

    def call(pool=FAKE, indptr=FAKE, idx=FAKE, dst=FAKE, batch=1, ws=FAKE, ws_bytes=None):
        return lib.mla_verify_relocate_kv(h, pool, indptr, idx, dst, batch, ws,
                                          p.workspace_bytes if ws_bytes is None else ws_bytes, None)

    assert call(batch=0) == B.MLA_VERIFY_OK
    assert call(batch=3) == B.MLA_VERIFY_EINVAL
    assert call(batch=-1) == B.MLA_VERIFY_EINVAL
    assert call(pool=None) == B.MLA_VERIFY_EINVAL
    assert call(dst=None) == B.MLA_VERIFY_EINVAL
    assert call(pool=FAKE + 8) == B.MLA_VERIFY_EINVAL       # pool not 16-byte aligned
    assert call(idx=FAKE + 2) == B.MLA_VERIFY_EINVAL        # indices not 4-byte aligned
    assert call(ws=None) == B.MLA_VERIFY_EWORKSPACE
    assert call(ws_bytes=p.workspace_bytes - 1) == B.MLA_VERIFY_EWORKSPACE
    assert call(ws=FAKE + 16) == B.MLA_VERIFY_EINVAL        # workspace not 256-byte aligned
    assert lib.mla_verify_relocate_kv(None, FAKE, FAKE, FAKE, FAKE, 1, FAKE, 1 << 30, None) == B.MLA_VERIFY_EINVAL


@pytest.mark.parametrize("B_,kv,ns,flags,granule,min_chunk", [
    (1, 4105, 16, 0, 64, 128),         # one request, resident tiles: chunks of 320 keys (2.5 tiles)
    (1, 185009, 64, 0, 64, 1472),      # chunk 2944 keys; the shortest is half of it, in 64-key steps
    (1, 4105, 16, R, 128, 128),        # value refetch: whole tiles
    (16, 32777, 16, 0, 128, 1024),     # several requests: whole tiles
    (1, 4105, 16, B.MLA_VERIFY_FORCE_SIMT, 128, 128),
])
def test_chunk_granule(lib, B_, kv, ns, flags, granule, min_chunk):
    """Chunk lengths are multiples of the plan's granule: half a tile only
    for one request in resident mode."""
    H = 8 if kv > 100000 else 64
    info = plan(max_batch=B_, num_heads=H, q_len=9, max_kv_len=kv, pool_rows=1 << 20, nsplit=ns,
                flags=flags).describe()
    assert (info.chunk_granule, info.min_chunk) == (granule, min_chunk)
    assert info.min_chunk % info.chunk_granule == 0


def test_auto_split_plan(lib):
    """nsplit = 0: the plan picks the number of chunks per request (the grid's
    split dimension) and sizes the workspace by it."""
    p = plan(max_batch=1, max_kv_len=65545, pool_rows=1 << 20, nsplit=0)
    info = p.describe()
    assert info.kernel == 1 and 1 <= info.grid_y <= 513  # at most one chunk per 128-key tile
    rows = 9 * 64
    off_o = (256 + 4 * info.grid_y * rows + 255) // 256 * 256
    assert p.workspace_bytes == off_o + 4 * info.grid_y * rows * 512
    assert plan(nsplit=16).describe().grid_y == 16
    # the run's nsplit must be the plan's (0)
    assert run_raw(lib, p, nsplit=16) == B.MLA_VERIFY_EINVAL
    assert run_raw(lib, p, nsplit=0, batch=0) == B.MLA_VERIFY_OK


@pytest.mark.parametrize("B_,H,T,kv,res,nq,splits", [
    (1, 64, 9, 4105, 0, 96, 17),     # short4k: one wave of 102 CTAs, 2 tiles each
    (1, 64, 9, 65545, 0, 96, 25),    # mid64k: one wave of 150 CTAs
    (1, 8, 9, 185009, 0, 96, 145),   # long185k_h8: one row group, 145 CTAs of 10 tiles
    (16, 64, 1, 32769, 1, 64, 26),   # decode, 16 requests: one resident 64-row group each
])
def test_auto_split_choices_on_152_sms(lib, B_, H, T, kv, res, nq, splits):
    """The cost model's picks on a 152-SM GB300 (the host fallback count when
    no device answers)."""
    info = plan(max_batch=B_, num_heads=H, q_len=T, max_kv_len=kv, pool_rows=1 << 20, nsplit=0).describe()
    assert (info.resident_tile, info.rows_per_cta, info.grid_y) == (res, nq, splits)
    if B_ == 1:
        assert -(-H * T // nq) * splits <= 152
