"""Python binding of libmlaverify.so (argument marshalling only).

The functions carry the names of the C ABI in ``include/mla_verify.h`` and
take torch tensors (device memory) or raw integers.  Every step of the verify
path runs in the library's CUDA kernels; there is no Python or CPU fallback:
if the library is missing or the device is unsupported, the call raises.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmlaverify.so")

MLA_VERIFY_OK = 0
MLA_VERIFY_EINVAL = 1
MLA_VERIFY_EUNSUPPORTED = 2
MLA_VERIFY_EWORKSPACE = 3
MLA_VERIFY_ECUDA = 4
MLA_VERIFY_DEV_BAD_ROW = 0x1
MLA_VERIFY_DEV_TIMEOUT = 0x2
MLA_VERIFY_FORCE_SIMT = 0x1
MLA_VERIFY_FUSED_MERGE = 0x2
MLA_VERIFY_REFETCH_VALUES = 0x4
MLA_VERIFY_TEST_STALL_GATHER = 0x100

EXPORTED = ("mla_verify_plan", "mla_verify_plan_describe", "mla_verify_run", "mla_verify_split",
            "mla_verify_merge", "mla_verify_workspace_init", "mla_verify_read_status", "mla_verify_destroy",
            "mla_verify_strerror", "mla_verify_run_noalloc", "mla_verify_build_tree_mask",
            "mla_verify_run_varlen", "mla_verify_relocate_kv", "mla_verify_build_tree_mask_varlen")


class MlaVerifyParams(ctypes.Structure):
    _fields_ = [("max_batch", ctypes.c_int32), ("num_heads", ctypes.c_int32), ("q_len", ctypes.c_int32),
                ("max_kv_len", ctypes.c_int32), ("pool_rows", ctypes.c_int64), ("nsplit", ctypes.c_int32),
                ("d_latent", ctypes.c_int32), ("d_rope", ctypes.c_int32), ("flags", ctypes.c_int32)]


class MlaVerifyPlanInfo(ctypes.Structure):
    _fields_ = [("kernel", ctypes.c_int32), ("rows_per_cta", ctypes.c_int32), ("keys_per_tile", ctypes.c_int32),
                ("grid_x", ctypes.c_int32), ("grid_y", ctypes.c_int32), ("grid_z", ctypes.c_int32),
                ("merge_blocks", ctypes.c_int32), ("smem_bytes", ctypes.c_int32),
                ("workspace_bytes", ctypes.c_size_t), ("resident_tile", ctypes.c_int32),
                ("min_chunk", ctypes.c_int32), ("chunk_granule", ctypes.c_int32)]


class MlaVerifyError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__("%s failed with code %d: %s" % (what, code, strerror(code)))
        self.code = code


_lib = None


def load(path: str = LIB_PATH):
    """Load the shared library; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError("libmlaverify.so not built (run `python -c \"import __graft_entry__ as g; g.build()\"` "
                          "or `python mla_speculative_decode_tree_gb300/build.py`)")
    lib = ctypes.CDLL(path)
    P, i32, i64, f32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    lib.mla_verify_plan.argtypes = [ctypes.POINTER(MlaVerifyParams), ctypes.POINTER(sz), ctypes.POINTER(P)]
    lib.mla_verify_plan_describe.argtypes = [P, ctypes.POINTER(MlaVerifyPlanInfo)]
    run_args = [P, P, P, P, P, P, P, P, P, i32, f32, i32, P, sz]
    lib.mla_verify_run.argtypes = run_args + [P, P, P]
    lib.mla_verify_split.argtypes = run_args + [P]
    lib.mla_verify_run_varlen.argtypes = run_args[:6] + [P] + run_args[6:] + [P, P, P]
    lib.mla_verify_merge.argtypes = [P, i32, i32, P, sz, P, P, P]
    lib.mla_verify_run_noalloc.argtypes = [P, P, P, P, P, P, P, P, P, i32, f32, i32, P, P, P]
    lib.mla_verify_workspace_init.argtypes = [P, P, sz, P]
    lib.mla_verify_build_tree_mask.argtypes = [P, P, P, i32, P, sz, P, P]
    lib.mla_verify_relocate_kv.argtypes = [P, P, P, P, P, i32, P, sz, P]
    lib.mla_verify_build_tree_mask_varlen.argtypes = [P, P, P, P, i32, P, sz, P, P]
    lib.mla_verify_read_status.argtypes = [P, P, P, ctypes.POINTER(ctypes.c_uint32)]
    lib.mla_verify_destroy.argtypes = [P]
    lib.mla_verify_strerror.argtypes = [ctypes.c_int]
    lib.mla_verify_strerror.restype = ctypes.c_char_p
    for name in EXPORTED:
        if name != "mla_verify_strerror":
            getattr(lib, name).restype = ctypes.c_int
    _lib = lib
    return lib


def strerror(code: int) -> str:
    return load().mla_verify_strerror(int(code)).decode()


def _check(rc: int, what: str):
    if rc != MLA_VERIFY_OK:
        raise MlaVerifyError(rc, what)


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


class Plan:
    """Owns a host-side plan handle (mla_verify_destroy on close / GC)."""

    def __init__(self, handle: int, params: MlaVerifyParams, workspace_bytes: int):
        self.handle = handle
        self.params = params
        self.workspace_bytes = workspace_bytes

    @property
    def nsplit(self) -> int:
        return self.params.nsplit

    def describe(self) -> MlaVerifyPlanInfo:
        return mla_verify_plan_describe(self)

    def close(self):
        if self.handle:
            load().mla_verify_destroy(ctypes.c_void_p(self.handle))
            self.handle = 0

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def mla_verify_plan(max_batch: int, num_heads: int, q_len: int, max_kv_len: int, pool_rows: int, nsplit: int,
                    flags: int = 0, d_latent: int = 512, d_rope: int = 64) -> Plan:
    p = MlaVerifyParams(max_batch, num_heads, q_len, max_kv_len, pool_rows, nsplit, d_latent, d_rope, flags)
    ws = ctypes.c_size_t(0)
    h = ctypes.c_void_p(0)
    _check(load().mla_verify_plan(ctypes.byref(p), ctypes.byref(ws), ctypes.byref(h)), "mla_verify_plan")
    return Plan(h.value, p, ws.value)


def mla_verify_plan_describe(plan: Plan) -> MlaVerifyPlanInfo:
    info = MlaVerifyPlanInfo()
    _check(load().mla_verify_plan_describe(ctypes.c_void_p(plan.handle), ctypes.byref(info)),
           "mla_verify_plan_describe")
    return info


def mla_verify_run_varlen(plan: Plan, q_nope_absorbed, q_rope, kv_pool, kv_indptr, kv_indices, qo_indptr,
                          out_cache_loc, custom_mask, mask_indptr, batch: int, sm_scale: float, nsplit: int,
                          workspace, o, lse, stream=None, workspace_bytes: Optional[int] = None):
    ws_bytes = plan.workspace_bytes if workspace_bytes is None else workspace_bytes
    rc = load().mla_verify_run_varlen(ctypes.c_void_p(plan.handle), _ptr(q_nope_absorbed), _ptr(q_rope),
                                      _ptr(kv_pool), _ptr(kv_indptr), _ptr(kv_indices), _ptr(qo_indptr),
                                      _ptr(out_cache_loc), _ptr(custom_mask), _ptr(mask_indptr), int(batch),
                                      float(sm_scale), int(nsplit), _ptr(workspace), int(ws_bytes), _ptr(o),
                                      _ptr(lse), _stream(stream))
    _check(rc, "mla_verify_run_varlen")


def mla_verify_run(plan: Plan, q_nope_absorbed, q_rope, kv_pool, kv_indptr, kv_indices, out_cache_loc,
                   custom_mask, mask_indptr, batch: int, sm_scale: float, nsplit: int, workspace, o, lse,
                   stream=None, workspace_bytes: Optional[int] = None):
    ws_bytes = plan.workspace_bytes if workspace_bytes is None else workspace_bytes
    rc = load().mla_verify_run(ctypes.c_void_p(plan.handle), _ptr(q_nope_absorbed), _ptr(q_rope), _ptr(kv_pool),
                               _ptr(kv_indptr), _ptr(kv_indices), _ptr(out_cache_loc), _ptr(custom_mask),
                               _ptr(mask_indptr), int(batch), float(sm_scale), int(nsplit), _ptr(workspace),
                               int(ws_bytes), _ptr(o), _ptr(lse), _stream(stream))
    _check(rc, "mla_verify_run")


def mla_verify_split(plan: Plan, q_nope_absorbed, q_rope, kv_pool, kv_indptr, kv_indices, out_cache_loc,
                     custom_mask, mask_indptr, batch: int, sm_scale: float, nsplit: int, workspace, stream=None,
                     workspace_bytes: Optional[int] = None):
    ws_bytes = plan.workspace_bytes if workspace_bytes is None else workspace_bytes
    rc = load().mla_verify_split(ctypes.c_void_p(plan.handle), _ptr(q_nope_absorbed), _ptr(q_rope), _ptr(kv_pool),
                                 _ptr(kv_indptr), _ptr(kv_indices), _ptr(out_cache_loc), _ptr(custom_mask),
                                 _ptr(mask_indptr), int(batch), float(sm_scale), int(nsplit), _ptr(workspace),
                                 int(ws_bytes), _stream(stream))
    _check(rc, "mla_verify_split")


def mla_verify_run_noalloc(plan: Plan, q_nope_absorbed, q_rope, kv_pool, kv_indptr, kv_indices, out_cache_loc,
                           custom_mask, mask_indptr, batch: int, sm_scale: float, nsplit: int, o, lse, stream=None):
    """mla_verify_run on the library's built-in scratch array (no workspace, no allocation)."""
    rc = load().mla_verify_run_noalloc(ctypes.c_void_p(plan.handle), _ptr(q_nope_absorbed), _ptr(q_rope),
                                       _ptr(kv_pool), _ptr(kv_indptr), _ptr(kv_indices), _ptr(out_cache_loc),
                                       _ptr(custom_mask), _ptr(mask_indptr), int(batch), float(sm_scale), int(nsplit),
                                       _ptr(o), _ptr(lse), _stream(stream))
    _check(rc, "mla_verify_run_noalloc")


def mla_verify_merge(plan: Plan, batch: int, nsplit: int, workspace, o, lse, stream=None,
                     workspace_bytes: Optional[int] = None):
    ws_bytes = plan.workspace_bytes if workspace_bytes is None else workspace_bytes
    rc = load().mla_verify_merge(ctypes.c_void_p(plan.handle), int(batch), int(nsplit), _ptr(workspace),
                                 int(ws_bytes), _ptr(o), _ptr(lse), _stream(stream))
    _check(rc, "mla_verify_merge")


def mla_verify_build_tree_mask(plan: Plan, parents, kv_indptr, batch: int, custom_mask, mask_indptr, stream=None,
                               mask_bytes: Optional[int] = None):
    """Device tree-mask build: parents int32 [batch*q_len] -> packed custom_mask, mask_indptr int32 [batch]."""
    nbytes = custom_mask.numel() * custom_mask.element_size() if mask_bytes is None else mask_bytes
    rc = load().mla_verify_build_tree_mask(ctypes.c_void_p(plan.handle), _ptr(parents), _ptr(kv_indptr), int(batch),
                                           _ptr(custom_mask), int(nbytes), _ptr(mask_indptr), _stream(stream))
    _check(rc, "mla_verify_build_tree_mask")


def mla_verify_relocate_kv(plan: Plan, kv_pool, kv_indptr, kv_indices, dst_start, batch: int, workspace,
                           stream=None):
    """KV relocation: request b's prefix rows move to rows dst_start[b].. and kv_indices is rewritten in place."""
    rc = load().mla_verify_relocate_kv(ctypes.c_void_p(plan.handle), _ptr(kv_pool), _ptr(kv_indptr), _ptr(kv_indices),
                                       _ptr(dst_start), int(batch), _ptr(workspace),
                                       workspace.numel() * workspace.element_size(), _stream(stream))
    _check(rc, "mla_verify_relocate_kv")


def mla_verify_build_tree_mask_varlen(plan: Plan, parents, kv_indptr, qo_indptr, batch: int, custom_mask,
                                      mask_indptr, stream=None, mask_bytes: Optional[int] = None):
    """Device tree-mask build for a varlen call: parents int32 [qo_indptr[batch]] (request b's at
    qo_indptr[b]..), blocks [T_b, P_b + T_b]."""
    nbytes = custom_mask.numel() * custom_mask.element_size() if mask_bytes is None else mask_bytes
    rc = load().mla_verify_build_tree_mask_varlen(ctypes.c_void_p(plan.handle), _ptr(parents), _ptr(kv_indptr),
                                                  _ptr(qo_indptr), int(batch), _ptr(custom_mask), int(nbytes),
                                                  _ptr(mask_indptr), _stream(stream))
    _check(rc, "mla_verify_build_tree_mask_varlen")


def mla_verify_workspace_init(plan: Plan, workspace, stream=None):
    _check(load().mla_verify_workspace_init(ctypes.c_void_p(plan.handle), _ptr(workspace), plan.workspace_bytes,
                                            _stream(stream)), "mla_verify_workspace_init")


def mla_verify_read_status(plan: Plan, workspace, stream=None) -> int:
    st = ctypes.c_uint32(0)
    _check(load().mla_verify_read_status(ctypes.c_void_p(plan.handle), _ptr(workspace), _stream(stream),
                                         ctypes.byref(st)), "mla_verify_read_status")
    return int(st.value)


def mla_verify_destroy(plan: Plan):
    plan.close()


# ---------------------------------------------------------------------------
# Convenience layer over the C calls: device buffers for a host workload and a
# one-shot call that allocates outputs and workspace with torch.

def device_inputs(wl: dict, device="cuda"):
    """Copy a host workload (numpy arrays from ``workloads.make_workload``) to the device."""
    import numpy as np
    import torch

    def t(a, dtype):
        return torch.from_numpy(np.ascontiguousarray(a)).to(device=device).view(dtype)

    kv_idx = wl["kv_indices"] if wl["kv_indices"].size else np.zeros(1, np.int32)
    return dict(
        q_nope=t(wl["q_nope"].view(np.int16), torch.bfloat16),
        q_rope=t(wl["q_rope"].view(np.int16), torch.bfloat16),
        kv_pool=t(wl["pool"].view(np.int16), torch.bfloat16),
        kv_indptr=t(wl["kv_indptr"].astype(np.int32), torch.int32),
        kv_indices=t(kv_idx.astype(np.int32), torch.int32),
        out_cache_loc=t(wl["out_cache_loc"].astype(np.int32), torch.int32),
        custom_mask=t(wl["custom_mask"].astype(np.uint8), torch.uint8),
        mask_indptr=t(wl["mask_indptr"].astype(np.int32), torch.int32),
        **({"qo_indptr": t(wl["qo_indptr"].astype(np.int32), torch.int32)} if wl.get("qo_indptr") is not None
           else {}),
    )


class Verifier:
    """A plan plus its workspace and output buffers on one device."""

    def __init__(self, max_batch: int, num_heads: int, q_len: int, max_kv_len: int, pool_rows: int, nsplit: int,
                 flags: int = 0, device="cuda"):
        import torch
        self.plan = mla_verify_plan(max_batch, num_heads, q_len, max_kv_len, pool_rows, nsplit, flags)
        self.workspace = torch.zeros(self.plan.workspace_bytes, dtype=torch.uint8, device=device)
        rows = max_batch * q_len * num_heads
        self.o = torch.empty((max_batch * q_len, num_heads, 512), dtype=torch.bfloat16, device=device)
        self.lse = torch.empty((max_batch * q_len, num_heads), dtype=torch.float32, device=device)
        self.rows_max = rows

    def run(self, d: dict, batch: int, sm_scale: float, stream=None):
        """One call; with d["qo_indptr"] present, the varlen entry point.  Returns the
        output buffers' first batch*q_len token rows (varlen: the call's rows come first)."""
        if "qo_indptr" in d:
            mla_verify_run_varlen(self.plan, d["q_nope"], d["q_rope"], d["kv_pool"], d["kv_indptr"],
                                  d["kv_indices"], d["qo_indptr"], d["out_cache_loc"], d["custom_mask"],
                                  d["mask_indptr"], batch, sm_scale, self.plan.nsplit, self.workspace, self.o,
                                  self.lse, stream=stream)
        else:
            mla_verify_run(self.plan, d["q_nope"], d["q_rope"], d["kv_pool"], d["kv_indptr"], d["kv_indices"],
                           d["out_cache_loc"], d["custom_mask"], d["mask_indptr"], batch, sm_scale,
                           self.plan.nsplit, self.workspace, self.o, self.lse, stream=stream)
        n = batch * self.plan.params.q_len
        return self.o[:n], self.lse[:n]

    def status(self, stream=None) -> int:
        return mla_verify_read_status(self.plan, self.workspace, stream)


def verifier_for(wl: dict, flags: int = 0, nsplit: Optional[int] = None, device="cuda") -> Verifier:
    L = int(max(wl["prefix_lens"])) + wl["T"] if len(wl["prefix_lens"]) else wl["T"]  # bounds P_b + T_b too
    return Verifier(wl["B"], wl["H"], wl["T"], L, wl["pool"].shape[0], wl["nsplit"] if nsplit is None else nsplit,
                    flags, device)
