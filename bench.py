#!/usr/bin/env python3
"""Benchmark of the MLA tree-verify call on GB300.

One step = one verify call (split kernel + merge kernel) over one batch of
synthetic input already resident in HBM.  The headline workload is the
short-context tree verify (B=1, H=64, 9-token random draft tree, prefix 4096,
262,144-row pool, NSPLIT=16); the longer-context workloads are reported in
``sweep``.  L2 is flushed (a 512 MiB device write) before every timed step,
outside the timed events.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]
                    [--workload NAME] [--no-sweep]

For N > 1 it runs under torchrun as N independent replicas (the verify path
has no exchange step); value = total calls / max-over-ranks time.
``--impl reference`` times the fp64 CPU oracle on the host cores instead.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = ("verify-attn µs/call, gathered KV GB/s and % roofline at prefix 4k–185k (1 GB300)")
UNIT = "us/call"
FLUSH_BYTES = 512 << 20
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ----------------------------------------------------------------- helpers --
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def workload_desc(cfg) -> str:
    pre = ("U[%d,%d]" % cfg.prefix) if isinstance(cfg.prefix, tuple) else str(cfg.prefix)
    return ("%s: B=%d H=%d q_len=%d (%s tree) prefix=%s pool_rows=%d NSPLIT=%d layout=%s"
            % (cfg.name, cfg.B, cfg.H, cfg.T, cfg.tree, pre, cfg.pool_rows, cfg.nsplit, cfg.layout))


def gpu_config(cfg, nsplit, chunks, world) -> dict:
    """The GPU arm's ``config``: the workload and how it is timed."""
    return {"workload": workload_desc(cfg) + ("" if nsplit is None else
                                              " (run with nsplit=%d: %d chunks)" % (nsplit, chunks)),
            "l2": "flushed (512 MiB write) before every step",
            "parallelism": "replicas" if world > 1 else "single GPU", "graph": "split+merge in one CUDA graph"}


def reference_config(cfg, cores) -> dict:
    """The reference arm's ``config``: the GPU arm's keys, the same workload."""
    return {"workload": workload_desc(cfg), "l2": "not applicable (fp64 CPU oracle on the host)",
            "parallelism": "%d host threads" % cores, "graph": "none (no reference code exists to install)"}


def algorithmic(wl):
    """Algorithmic bytes and FLOPs of one verify call (and of its split kernel)."""
    H = wl["H"]
    P = np.asarray(wl["prefix_lens"], dtype=np.int64)
    Tb = np.asarray(wl["T_list"], dtype=np.int64) if wl.get("T_list") is not None else np.full(len(P), wl["T"])
    Lb = P + Tb
    N = int(Lb.sum())
    R = int(Tb.sum() * H)
    mask_bytes = int((Tb * Lb).sum() // 8)
    split_bytes = N * 1152 + 4 * int(P.sum()) + 4 * int(Tb.sum()) + mask_bytes + R * 1152
    call_bytes = split_bytes + R * 1028
    flops = 2 * int((Tb * H * Lb).sum()) * (576 + 512)
    return dict(rows=N, kv_bytes=N * 1152, split_bytes=split_bytes, call_bytes=call_bytes, flops=flops)


def _strip_comments(src: str) -> str:
    """C/C++ source without // and /* */ comments or blank space (string literals kept)."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if src.startswith("//", i):
            i = src.find("\n", i)
            i = n if i < 0 else i
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
        elif c == '"':
            j = i + 1
            while j < n and src[j] != '"':
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


# The split kernel's sources: its instantiations and the headers they include.
SPLIT_KERNEL_SOURCES = ("split_tc", "common.cuh", "tc_ptx.cuh", "merge_row.cuh")


def kernel_source_hash(cdir: str = None) -> str:
    """Hash of the split kernel's code (comments and layout ignored): the ncu
    counters in profiles/ stay valid across comment-only edits and across
    changes to the library's other kernels."""
    h = hashlib.sha256()
    cdir = cdir or os.path.join(ROOT, "mla_speculative_decode_tree_gb300", "csrc")
    for name in sorted(os.listdir(cdir)):
        if name.endswith((".cu", ".cuh")) and name.startswith(SPLIT_KERNEL_SOURCES):
            with open(os.path.join(cdir, name), encoding="utf-8") as f:
                h.update(name.encode() + _strip_comments(f.read()).encode())
    return h.hexdigest()[:16]


def traffic_key(workload: str, nsplit=None) -> str:
    """Key of a stored traffic record: the workload, with the nsplit override if any."""
    return workload if nsplit is None else "%s@nsplit%d" % (workload, nsplit)


def ncu_record(workload: str):
    """The committed ncu record of a workload's split kernel, if it matches this source."""
    path = os.path.join(ROOT, "profiles", "split_kernel_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    ent = rec.get(workload)
    if not ent or ent.get("source_hash") != kernel_source_hash():
        return None
    return ent


def ncu_traffic(workload: str):
    """DRAM bytes per split-kernel launch from the committed ncu summary, if it matches this source."""
    path = os.path.join(ROOT, "profiles", "split_kernel_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    ent = rec.get(workload)
    if not ent or ent.get("source_hash") != kernel_source_hash():
        return None
    return ent.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks/throttle sampling in the background."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,clocks.mem")

    def __init__(self, gpu_index: int, log_path=None):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.log_path = log_path
        self.marks = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "--query-gpu=" + self.Q, "--format=csv,noheader,nounits",
                                          "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, what):
        self.marks.append((what, time.time()))

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.log_path:
            try:
                with open(self.log_path, "w") as f:
                    for t, l in self.lines:
                        f.write("%.3f,%s\n" % (t, l))
            except OSError:
                pass
        t0 = dict(self.marks).get("timed_start")
        t1 = dict(self.marks).get("timed_end")
        rows = []
        for t, l in self.lines:
            parts = [p.strip() for p in l.split(",")]
            if len(parts) < 9 or parts[0] != str(self.gpu):
                continue
            rows.append((t, parts))
        if not rows:
            return None
        during = [r for r in rows if t0 is not None and t0 - 0.05 <= r[0] <= (t1 or r[0]) + 0.05]
        use = during if during else rows
        sm = [float(p[1]) for _, p in use if p[1].replace(".", "").isdigit()]
        mx = [float(p[2]) for _, p in use if p[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for _, p in use for k in range(4) if p[5 + k].lower().startswith("active")})
        mem = [float(p[9]) for _, p in use if len(p) > 9 and p[9].replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "mem_mhz": statistics.median(mem) if mem else None,
                "samples": len(use), "samples_in_timed_region": len(during)}


# ------------------------------------------------------- replica harness ----
def max_over_ranks(x: float, dist=None, device="cpu") -> float:
    """Max of a per-rank scalar over all ranks (identity on one rank)."""
    if dist is None or not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_us_per_call(max_total_ms: float, steps: int, world: int) -> float:
    """Replicas each run `steps` calls; the job processed steps*world calls in max_total_ms."""
    return max_total_ms * 1e3 / (steps * world)


# --------------------------------------------------------------- GPU arm ----
def time_graph(torch, graph_fn, steps, warmup, flush, stream):
    """Per-step device time (ms) of graph_fn() with an L2 flush before each step."""
    times = []
    with torch.cuda.stream(stream):
        for it in range(warmup + steps):
            flush.zero_()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            graph_fn()
            e1.record(stream)
            if it >= warmup:
                times.append((e0, e1))
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in times]


def capture(torch, fn, stream):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        fn()  # warm the allocator / first-call set-up outside capture
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=stream):
            fn()
    torch.cuda.synchronize()
    return g


def measure_workload(torch, name, steps, warmup, flush, stream, with_e2e=False, flags=0, nsplit=None):
    from mla_speculative_decode_tree_gb300 import binding as B
    from mla_speculative_decode_tree_gb300 import workloads as W

    cfg = W.CONFIGS[name]
    wl = W.make_workload(cfg)
    d = B.device_inputs(wl)
    v = B.verifier_for(wl, flags=flags, nsplit=nsplit)
    info = v.plan.describe()
    scale = wl["sm_scale"]

    def call():
        v.run(d, wl["B"], scale, stream=stream)  # the varlen entry point when the workload has qo_indptr

    def split_only():
        B.mla_verify_split(v.plan, d["q_nope"], d["q_rope"], d["kv_pool"], d["kv_indptr"], d["kv_indices"],
                           d["out_cache_loc"], d["custom_mask"], d["mask_indptr"], wl["B"], scale, v.plan.nsplit,
                           v.workspace, stream=stream)

    g_call = capture(torch, call, stream)
    t_call = time_graph(torch, g_call.replay, steps, warmup, flush, stream)
    if "qo_indptr" in d or info.merge_blocks == 0:  # varlen or fused merge: no split-only call
        g_split, t_split = None, t_call
    else:
        g_split = capture(torch, split_only, stream)
        t_split = time_graph(torch, g_split.replay, steps, warmup, flush, stream)
    status = v.status(stream)
    alg = algorithmic(wl)
    res = dict(wl=wl, info=info, t_call=t_call, t_split=t_split, alg=alg, status=status,
               tree_mask=measure_tree_mask(torch, wl, v.plan, stream, steps, warmup, flush))
    if with_e2e:
        res["e2e"] = measure_e2e(torch, wl, v, stream, steps, warmup, flush)
    del g_call, g_split, d
    return res


def measure_tree_mask(torch, wl, plan, stream, steps, warmup, flush):
    """Device tree-mask build (parents -> packed mask) timed alone, graph-replayed,
    L2 flushed before each launch; checked bit for bit against the call's mask."""
    from mla_speculative_decode_tree_gb300 import binding as B

    dev = B.device_inputs(wl)
    parents = torch.from_numpy(np.concatenate([np.asarray(p, np.int32) for p in wl["parents"]])).cuda()
    mask = torch.zeros_like(dev["custom_mask"])
    mip = torch.zeros_like(dev["mask_indptr"])

    def build():
        if "qo_indptr" in dev:
            B.mla_verify_build_tree_mask_varlen(plan, parents, dev["kv_indptr"], dev["qo_indptr"], wl["B"], mask, mip,
                                                stream=stream)
        else:
            B.mla_verify_build_tree_mask(plan, parents, dev["kv_indptr"], wl["B"], mask, mip, stream=stream)

    g = capture(torch, build, stream)
    t = time_graph(torch, g.replay, steps, warmup, flush, stream)
    torch.cuda.synchronize()
    counts = wl["T_list"] if wl.get("T_list") is not None else [wl["T"]] * wl["B"]
    n = (int(sum(int(t_b) * (int(p) + int(t_b)) for p, t_b in zip(wl["prefix_lens"], counts))) + 7) // 8
    same = bool(torch.equal(mask[:n], dev["custom_mask"][:n]) and torch.equal(mip, dev["mask_indptr"]))
    del g
    return {"us": round(statistics.mean(t) * 1e3, 3), "mask_bytes": n, "matches_input_mask": same,
            "launches_per_call": 1}


def measure_relocation(torch, name, stream, steps, warmup, flush, peaks):
    """KV relocation (mla_verify_relocate_kv) on a verify workload whose rows sit
    clear of a free block: µs per launch (graph-replayed, L2 flushed and the
    original indices restored before each launch, outside the timed events),
    GB/s of algorithmic traffic against the HBM peak, and the verify call timed
    on the scattered rows and again on the relocated, contiguous rows (their
    outputs must be bit-identical)."""
    from mla_speculative_decode_tree_gb300 import binding as B
    from mla_speculative_decode_tree_gb300 import workloads as W

    wl = W.with_free_block(W.make_workload(W.CONFIGS[name]), seed=1234)
    d = B.device_inputs(wl)
    v = B.verifier_for(wl)
    dst = torch.from_numpy(wl["dst_start"].astype(np.int32)).cuda()
    idx0 = d["kv_indices"].clone()

    def relocate():
        B.mla_verify_relocate_kv(v.plan, d["kv_pool"], d["kv_indptr"], d["kv_indices"], dst, wl["B"], v.workspace,
                                 stream=stream)

    def call():
        v.run(d, wl["B"], wl["sm_scale"], stream=stream)

    g_call = capture(torch, call, stream)
    t_before = time_graph(torch, g_call.replay, steps, warmup, flush, stream)
    o0, l0 = v.o.clone(), v.lse.clone()
    d["kv_indices"].copy_(idx0)
    g_rel = capture(torch, relocate, stream)
    times = []
    with torch.cuda.stream(stream):
        for it in range(warmup + steps):
            d["kv_indices"].copy_(idx0)
            flush.zero_()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            g_rel.replay()
            e1.record(stream)
            if it >= warmup:
                times.append((e0, e1))
    torch.cuda.synchronize()
    t_rel = [a.elapsed_time(b) for a, b in times]
    t_after = time_graph(torch, g_call.replay, steps, warmup, flush, stream)
    same = bool(torch.equal(o0.view(torch.int16), v.o.view(torch.int16)) and torch.equal(l0, v.lse))
    status = v.status(stream)
    rows = int(wl["kv_indptr"][-1] - wl["kv_indptr"][0])
    nbytes = rows * (2 * 1152 + 2 * 4) + 4 * (wl["B"] + 1) + 4 * wl["B"]
    us = statistics.mean(t_rel) * 1e3
    gbs = nbytes / (us * 1e-6) / 1e9
    del g_call, g_rel, d
    return {"workload": name + " rows moved into a free contiguous block", "rows": rows,
            "us": round(us, 3), "algorithmic_bytes": nbytes, "gbs": round(gbs, 1),
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": round(gbs / peaks["hbm_gbs"], 4)},
            "verify_us_scattered": round(statistics.mean(t_before) * 1e3, 3),
            "verify_us_relocated": round(statistics.mean(t_after) * 1e3, 3),
            "verify_bits_equal": same, "status": status}


def measure_e2e(torch, wl, v, stream, steps, warmup, flush):
    """Whole call through the C ABI from pinned host memory back to pinned host memory.

    The per-call inputs sit in one pinned staging buffer (each at a 256-byte
    aligned offset) and go to the device in one copy; O and LSE come back in
    one copy from one device buffer.  The pool stays resident on the device."""
    from mla_speculative_decode_tree_gb300 import binding as B

    dev = B.device_inputs(wl)
    per_call = ("q_nope", "q_rope", "kv_indptr", "kv_indices", "out_cache_loc", "custom_mask", "mask_indptr")
    offs, total = {}, 0
    for k in per_call:
        offs[k] = total
        total += (dev[k].numel() * dev[k].element_size() + 255) // 256 * 256
    stage_h = torch.empty(total, dtype=torch.uint8).pin_memory()
    stage_d = torch.empty(total, dtype=torch.uint8, device="cuda")
    views = {}
    for k in per_call:
        nbytes = dev[k].numel() * dev[k].element_size()
        stage_h[offs[k]:offs[k] + nbytes].copy_(dev[k].reshape(-1).view(torch.uint8).cpu())
        views[k] = stage_d[offs[k]:offs[k] + nbytes].view(dev[k].dtype).view(dev[k].shape)
    n_out = wl["B"] * wl["T"]
    H = wl["H"]
    o_bytes = n_out * H * 512 * 2
    l_off = (o_bytes + 255) // 256 * 256
    out_d = torch.empty(l_off + n_out * H * 4, dtype=torch.uint8, device="cuda")
    out_h = torch.empty(out_d.numel(), dtype=torch.uint8).pin_memory()
    o_d = out_d[:o_bytes].view(torch.bfloat16).view(n_out, H, 512)
    l_d = out_d[l_off:].view(torch.float32).view(n_out, H)
    times = []
    for it in range(warmup + steps):
        flush.zero_()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        with torch.cuda.stream(stream):
            stage_d.copy_(stage_h, non_blocking=True)
            B.mla_verify_run(v.plan, views["q_nope"], views["q_rope"], dev["kv_pool"], views["kv_indptr"],
                             views["kv_indices"], views["out_cache_loc"], views["custom_mask"],
                             views["mask_indptr"], wl["B"], wl["sm_scale"], v.plan.nsplit, v.workspace, o_d, l_d,
                             stream=stream)
            out_h.copy_(out_d, non_blocking=True)
        stream.synchronize()
        t1 = time.perf_counter()
        if it >= warmup:
            times.append((t1 - t0) * 1e3)
    # the staged call must give the device-resident call's result
    v.run(dev, wl["B"], wl["sm_scale"], stream=stream)
    torch.cuda.synchronize()
    got = out_h[:o_bytes].view(torch.bfloat16).view(n_out, H, 512)
    same = bool(torch.equal(got.view(torch.int16), v.o[:n_out].cpu().view(torch.int16)))
    return dict(times_ms=times, h2d=int(total), d2h=int(out_d.numel()), matches_device_call=same)


def summarize(res, peaks):
    alg = res["alg"]
    t_call_us = statistics.mean(res["t_call"]) * 1e3
    t_split_us = statistics.mean(res["t_split"]) * 1e3
    hbm = peaks["hbm_gbs"] * 1e9
    mma = peaks["bf16_tflops"] * 1e12
    t_hbm = alg["call_bytes"] / hbm * 1e6
    t_mma = alg["flops"] / mma * 1e6
    return dict(
        us_per_call=t_call_us, us_median=float(np.median(res["t_call"]) * 1e3),
        us_p10=float(np.percentile(res["t_call"], 10) * 1e3),
        us_p90=float(np.percentile(res["t_call"], 90) * 1e3), split_us=t_split_us,
        gathered_kv_gbs=alg["kv_bytes"] / (t_call_us * 1e-6) / 1e9,
        tflops=alg["flops"] / (t_call_us * 1e-6) / 1e12,
        roofline_frac=max(t_hbm, t_mma) / t_call_us, bound="tensor" if t_mma >= t_hbm else "hbm",
        kernel="tcgen05" if res["info"].kernel == 1 else "cuda-core", rows_per_cta=res["info"].rows_per_cta,
        status=res["status"], tree_mask=res.get("tree_mask"))


def run_profile_target(args):
    """A clean target for ncu: NAME's verify call (the varlen entry point when
    the workload has per-request token counts), warmup + steps launches of the
    split kernel in a row, each after an L2 flush, and nothing else on the
    device; prints the plan."""
    import torch
    from __graft_entry__ import build
    from mla_speculative_decode_tree_gb300 import binding as B
    from mla_speculative_decode_tree_gb300 import workloads as W
    build()
    wl = W.make_workload(W.CONFIGS[args.ncu_workload])
    d = B.device_inputs(wl)
    v = B.verifier_for(wl, nsplit=args.nsplit)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    for _ in range(args.warmup + args.steps):
        flush.zero_()
        v.run(d, wl["B"], wl["sm_scale"])
    torch.cuda.synchronize()
    info = v.plan.describe()
    print(json.dumps({"workload": args.ncu_workload, "status": v.status(), "rows_per_cta": info.rows_per_cta,
                      "resident_tile": info.resident_tile, "grid": [info.grid_x, info.grid_y, info.grid_z]}))


def run_gpu(args):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device (the GPU arm has no CPU fallback)")
    torch.cuda.set_device(local)
    if world > 1:
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    from __graft_entry__ import build
    if rank == 0 or world == 1:
        build()
    if world > 1:
        dist.barrier()
        build()

    peaks, peak_src = load_peaks()
    stream = torch.cuda.Stream()
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    phys = torch.cuda.get_device_properties(local)
    gpu_index = local
    sampler = ClockSampler(gpu_index, log_path=args.clock_log)
    sampler.start()
    time.sleep(0.3)

    # ---- headline workload: warm-up + exactly K timed steps, barrier + sync both sides
    from mla_speculative_decode_tree_gb300 import binding as B
    from mla_speculative_decode_tree_gb300 import workloads as W
    cfg = W.CONFIGS[args.workload]
    if cfg.T_range is not None:
        raise SystemExit("bench.py: %s has per-request token counts; it is timed in the sweep, not as the headline"
                         % args.workload)
    wl = W.make_workload(cfg)
    d = B.device_inputs(wl)
    v = B.verifier_for(wl, nsplit=args.nsplit)
    info = v.plan.describe()

    def call():
        B.mla_verify_run(v.plan, d["q_nope"], d["q_rope"], d["kv_pool"], d["kv_indptr"], d["kv_indices"],
                         d["out_cache_loc"], d["custom_mask"], d["mask_indptr"], wl["B"], wl["sm_scale"],
                         v.plan.nsplit, v.workspace, v.o, v.lse, stream=stream)

    def split_only():
        B.mla_verify_split(v.plan, d["q_nope"], d["q_rope"], d["kv_pool"], d["kv_indptr"], d["kv_indices"],
                           d["out_cache_loc"], d["custom_mask"], d["mask_indptr"], wl["B"], wl["sm_scale"],
                           v.plan.nsplit, v.workspace, stream=stream)

    g_call = capture(torch, call, stream)
    g_split = capture(torch, split_only, stream)
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            flush.zero_()
            g_call.replay()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    sampler.mark("timed_start")
    ev = []
    with torch.cuda.stream(stream):
        for _ in range(args.steps):
            flush.zero_()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            g_call.replay()
            e1.record(stream)
            ev.append((e0, e1))
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    sampler.mark("timed_end")
    step_ms = [a.elapsed_time(b) for a, b in ev]
    total_ms = max_over_ranks(sum(step_ms), dist if world > 1 else None, device="cuda")
    # live split-kernel timing (dominant kernel) on the same stream
    t_split = time_graph(torch, g_split.replay, args.steps, 3, flush, stream)
    status = v.status(stream)
    e2e = measure_e2e(torch, wl, v, stream, args.steps, args.warmup, flush)
    tree_mask = measure_tree_mask(torch, wl, v.plan, stream, min(args.steps, 50), 3, flush)
    clocks = sampler.stop()

    alg = algorithmic(wl)
    us_call = whole_job_us_per_call(total_ms, args.steps, world)
    split_us = statistics.mean(t_split) * 1e3
    t_hbm_us = alg["call_bytes"] / (peaks["hbm_gbs"] * 1e9) * 1e6
    t_mma_us = alg["flops"] / (peaks["bf16_tflops"] * 1e12) * 1e6
    bound = "tensor" if t_mma_us >= t_hbm_us else "hbm"
    if bound == "tensor":
        achieved = alg["flops"] / (split_us * 1e-6) / 1e12
        peak, unit = peaks["bf16_tflops"], "TFLOP/s"
    else:
        achieved = alg["split_bytes"] / (split_us * 1e-6) / 1e9
        peak, unit = peaks["hbm_gbs"], "GB/s"
    roofline = {"bound": bound, "achieved": round(achieved, 3), "peak": peak, "unit": unit,
                "frac": round(achieved / peak, 4), "traffic": ncu_traffic(traffic_key(args.workload, args.nsplit)),
                "kernel": "split (%s, %d query rows/CTA)" % ("tcgen05" if info.kernel else "cuda-core",
                                                              info.rows_per_cta),
                "peak_source": "%s (burst: kernel timed alone)" % peak_src,
                "split_us": round(split_us, 3)}
    e2e_us = statistics.mean(e2e["times_ms"]) * 1e3 / 1.0
    line = {
        "metric": METRIC, "value": round(us_call, 3), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(total_ms / args.steps, 6), "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": gpu_config(cfg, args.nsplit, info.grid_y, world),
        "us_per_call_median": round(float(np.median(step_ms)) * 1e3, 3),
        "us_per_call_p10_p90": [round(float(np.percentile(step_ms, 10)) * 1e3, 3),
                                round(float(np.percentile(step_ms, 90)) * 1e3, 3)],
        "gathered_kv_gbs": round(alg["kv_bytes"] / (us_call * world * 1e-6) / 1e9, 2),
        "roofline_frac_call": round(max(t_hbm_us, t_mma_us) / (us_call * world), 4),
        "roofline": roofline,
        "e2e": {"value": round(e2e_us, 3), "unit": UNIT, "h2d_bytes_per_step": e2e["h2d"],
                "d2h_bytes_per_step": e2e["d2h"], "copies_per_step": 2,
                "matches_device_call": e2e["matches_device_call"]},
        "gpu_launches": 2 * args.steps,
        "tree_mask_build": tree_mask,
        "clocks": clocks,
        "device_status": status,
        "gpu": phys.name,
        "plan": {"kernel": "tcgen05" if info.kernel == 1 else "cuda-core", "rows_per_cta": info.rows_per_cta,
                 "grid": [info.grid_x, info.grid_y, info.grid_z], "sm_count": phys.multi_processor_count},
    }
    if rank == 0 and not args.no_sweep:
        sweep = {}
        for name in ("mid64k", "mid64k_sorted", "long185k_h8", "batch16_ragged", "decode_b16", "decode_h8_b16",
                     "varlen_b16"):
            try:
                res = measure_workload(torch, name, min(args.steps, 30), 3, flush, stream)
                s = summarize(res, peaks)
                rec = ncu_record(name) or {}
                s["traffic"] = rec.get("dram_bytes_per_launch")
                s["tensor_pipe_pct"] = rec.get("tensor_pipe_pct")
                s["dram_throughput_pct"] = rec.get("dram_throughput_pct")
                sweep[name] = {k: (round(x, 4) if isinstance(x, float) else x) for k, x in s.items()}
                del res
            except Exception as exc:  # keep the headline line even if one sweep entry fails
                sweep[name] = {"error": repr(exc)[:200]}
            torch.cuda.empty_cache()
        line["sweep"] = sweep
        auto = {}
        for name in ("short4k", "mid64k", "long185k_h8", "batch16_ragged", "decode_b16"):
            try:
                res = measure_workload(torch, name, min(args.steps, 30), 3, flush, stream, nsplit=0)
                s = summarize(res, peaks)
                auto[name] = {"us_per_call": round(s["us_per_call"], 3), "split_us": round(s["split_us"], 3),
                              "roofline_frac": round(s["roofline_frac"], 4), "rows_per_cta": s["rows_per_cta"],
                              "chunks_per_request": res["info"].grid_y,
                              "nsplit_given_us_per_call": (round(us_call, 3) if name == args.workload else
                                                           sweep.get(name, {}).get("us_per_call")),
                              "status": res["status"]}
                del res
            except Exception as exc:
                auto[name] = {"error": repr(exc)[:200]}
            torch.cuda.empty_cache()
        line["auto_split"] = auto
        fused = {}
        for name in ("short4k", "mid64k", "decode_b16"):
            try:
                res = measure_workload(torch, name, min(args.steps, 30), 3, flush, stream,
                                       flags=B.MLA_VERIFY_FUSED_MERGE)
                fused[name] = {"us_per_call": round(statistics.mean(res["t_call"]) * 1e3, 3),
                               "separate_merge_us_per_call": round(us_call, 3) if name == args.workload else
                               sweep.get(name, {}).get("us_per_call"),
                               "status": res["status"]}
                del res
            except Exception as exc:
                fused[name] = {"error": repr(exc)[:200]}
            torch.cuda.empty_cache()
        line["fused_merge"] = fused
        try:
            line["kv_relocation"] = measure_relocation(torch, "mid64k", stream, min(args.steps, 30), 3, flush, peaks)
        except Exception as exc:
            line["kv_relocation"] = {"error": repr(exc)[:200]}
        torch.cuda.empty_cache()
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, budget_s=args.cpu_budget)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


# ---------------------------------------------------------- oracle (CPU) ----
def cpu_baseline(wl, budget_s=15.0, rows=None):
    """Time the fp64 oracle on a bounded sample of output rows; scale to one call."""
    from oracle import ref
    ref.build()
    n_all = wl["B"] * wl["T"] * wl["H"]
    cores = ref.max_threads()
    rng = np.random.default_rng(1)
    if rows is None:
        probe = np.sort(rng.choice(n_all, size=min(n_all, max(cores, 8)), replace=False))
        t0 = time.perf_counter()
        ref.verify(wl, rows=probe, nthreads=cores)
        per_row = (time.perf_counter() - t0) / probe.size
        k = int(min(n_all, max(cores, budget_s / max(per_row, 1e-9))))
        rows = np.sort(rng.choice(n_all, size=k, replace=False))
    t0 = time.perf_counter()
    ref.verify(wl, rows=rows, nthreads=cores)
    dt = time.perf_counter() - t0
    reps = 1
    if rows.size == n_all and dt < 0.5 * budget_s:
        # a whole call is cheap: repeat it to fill the budget
        more = int(min(1000, budget_s / max(dt, 1e-6))) - 1
        for _ in range(more):
            ref.verify(wl, rows=rows, nthreads=cores)
        reps += more
        dt = time.perf_counter() - t0
    us_call = dt / reps / rows.size * n_all * 1e6
    # the same oracle on one core, on a few rows, scaled to a whole call
    few = np.sort(rng.choice(n_all, size=min(n_all, 16), replace=False))
    t1 = time.perf_counter()
    ref.verify(wl, rows=few, nthreads=1)
    us_call_1 = (time.perf_counter() - t1) / few.size * n_all * 1e6
    if reps > 1:
        sample = "%d whole calls (all %d output rows each), fp64, %.1f s wall" % (reps, n_all, dt)
    else:
        sample = "%d of %d output rows (token x head) of the workload, fp64, %.1f s wall" % (rows.size, n_all, dt)
    return {"value": round(us_call, 1), "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample,
            "value_1core": round(us_call_1, 1), "sample_1core": "%d rows on 1 thread, scaled" % few.size}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return  # rank 0 alone runs the CPU oracle
    from mla_speculative_decode_tree_gb300 import workloads as W
    from oracle import ref
    ref.build()
    cfg = W.CONFIGS[args.workload]
    wl = W.make_workload(cfg)
    n_all = wl["B"] * wl["T"] * wl["H"]
    cores = ref.max_threads()
    sample = int(min(n_all, max(cores, 2 * cores)))
    rng = np.random.default_rng(2)
    times = []
    for it in range(args.warmup + args.steps):
        rows = np.sort(rng.choice(n_all, size=sample, replace=False))
        t0 = time.perf_counter()
        ref.verify(wl, rows=rows, nthreads=cores)
        dt = time.perf_counter() - t0
        if it >= args.warmup:
            times.append(dt / sample * n_all * 1e6)
    us = statistics.mean(times)
    line = {
        "impl": "reference", "metric": METRIC, "value": round(us, 1), "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(us / 1e3, 3), "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": reference_config(cfg, cores),
        "cpu_baseline": {"value": round(us, 1), "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": "%d of %d output rows per step, scaled to a whole call" % (sample, n_all)},
        "e2e": {"value": round(us, 1), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


PCT_METRICS = {"sm__pipe_tensor_cycles_active.avg.pct_of_peak_sustained_elapsed": "tensor_pipe_pct",
               "gpu__dram_throughput.avg.pct_of_peak_sustained_elapsed": "dram_throughput_pct"}


def record_traffic(csv_path: str, workload: str) -> dict:
    """Store the split kernel's DRAM bytes per launch from an ncu CSV capture
    (metrics dram__bytes_read.sum and dram__bytes_write.sum, and when present
    the tensor-pipe and DRAM-throughput percentages of PCT_METRICS) under the
    current kernel source hash, for the `traffic` fields of later runs."""
    import csv
    scale = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9, "KB": 1e3, "MB": 1e6, "GB": 1e9}
    per_launch = {}
    with open(csv_path) as f:
        rows = csv.DictReader(line for line in f if line.startswith('"'))
        for r in rows:
            if "split_tc_kernel" not in r.get("Kernel Name", "") and "split_simt_kernel" not in r.get("Kernel Name", ""):
                continue
            name = r.get("Metric Name", "")
            if name in PCT_METRICS:
                per_launch.setdefault(r["ID"], {})[name] = float(r["Metric Value"].replace(",", ""))
                continue
            if name not in ("dram__bytes_read.sum", "dram__bytes_write.sum"):
                continue
            v = float(r["Metric Value"].replace(",", "")) * scale.get(r.get("Metric Unit", "byte"), 1)
            per_launch.setdefault(r["ID"], {})[name] = v
    launches = [d for d in per_launch.values() if "dram__bytes_read.sum" in d and "dram__bytes_write.sum" in d]
    if not launches:
        raise SystemExit("no split-kernel launch with both DRAM metrics in %s" % csv_path)
    bytes_avg = sum(d["dram__bytes_read.sum"] + d["dram__bytes_write.sum"] for d in launches) / len(launches)
    path = os.path.join(ROOT, "profiles", "split_kernel_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        rec = {}
    rec[workload] = {"source_hash": kernel_source_hash(), "dram_bytes_per_launch": int(round(bytes_avg)),
                     "launches": len(launches),
                     "read_bytes": int(round(sum(d["dram__bytes_read.sum"] for d in launches) / len(launches))),
                     "write_bytes": int(round(sum(d["dram__bytes_write.sum"] for d in launches) / len(launches)))}
    for metric, key in PCT_METRICS.items():
        vals = [d[metric] for d in launches if metric in d]
        if vals:
            rec[workload][key] = round(sum(vals) / len(vals), 2)
    os.makedirs(os.path.dirname(path), exist_ok=True)
    with open(path, "w") as f:
        json.dump(rec, f, indent=1, sort_keys=True)
        f.write("\n")
    return rec[workload]


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("gb300", "reference"), default="gb300")
    ap.add_argument("--workload", default="short4k")
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--clock-log", metavar="CSV", default=None,
                    help="also write every nvidia-smi clock sample to this file")
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--ncu-workload", metavar="NAME", default=None,
                    help="profiling target: run only NAME's verify call (its own entry point), warmup+steps times")
    ap.add_argument("--record-traffic", metavar="NCU_CSV",
                    help="store the split kernel's DRAM bytes per launch from an ncu CSV for --workload, then exit")
    ap.add_argument("--nsplit", type=int, default=None,
                    help="run the headline workload with this nsplit instead of its own (0: the plan picks)")
    ap.add_argument("--relocation-only", action="store_true",
                    help="time only the KV relocation call on --workload's rows (steps/warmup as given)")
    args = ap.parse_args(argv)
    if args.record_traffic:
        print(json.dumps(record_traffic(args.record_traffic, traffic_key(args.workload, args.nsplit))))
        return
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    elif args.ncu_workload:
        run_profile_target(args)
    elif args.relocation_only:
        import torch
        from __graft_entry__ import build
        build()
        peaks, _ = load_peaks()
        stream = torch.cuda.Stream()
        flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device="cuda")
        print(json.dumps(measure_relocation(torch, args.workload, stream, args.steps, args.warmup, flush, peaks)))
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
