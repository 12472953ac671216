"""Host-side pieces of the benchmark (CPU only): the roofline arithmetic
against hand-computed figures for the headline workload, the source hash
that keys stored ncu counters, and the traffic-record keys."""

import bench
from mla_speculative_decode_tree_gb300 import workloads as W


def test_algorithmic_bytes_and_flops_short4k():
    # the headline shape (prefix 4096, 9 tokens, 64 heads); the pool size does not enter
    wl = W.tiny_workload(B=1, H=64, T=9, prefix_lens=[4096], pool_rows=8192, seed=0)
    a = bench.algorithmic(wl)
    N = 4096 + 9                      # gathered rows: prefix + draft
    R = 9 * 64                        # query rows
    assert a["rows"] == N and a["kv_bytes"] == N * 1152
    mask = 9 * N // 8
    assert a["split_bytes"] == N * 1152 + 4 * 4096 + 4 * 9 + mask + R * 1152
    assert a["call_bytes"] == a["split_bytes"] + R * (1024 + 4)   # bf16 O row + fp32 LSE
    assert a["flops"] == 2 * 9 * 64 * N * (576 + 512)
    assert abs(a["flops"] / 1e9 - 5.15) < 0.01


def test_algorithmic_varlen_counts_each_request():
    wl = W.varlen_workload(B=3, H=8, T_list=[2, 0, 5], prefix_lens=[10, 7, 0], pool_rows=256, seed=1)
    a = bench.algorithmic(wl)
    L = [12, 7, 5]
    assert a["rows"] == sum(L)
    assert a["flops"] == 2 * 8 * (2 * 12 + 0 * 7 + 5 * 5) * 1088


def test_source_hash_ignores_comments_and_other_kernels(tmp_path):
    d = tmp_path / "csrc"
    d.mkdir()
    (d / "split_tc.cuh").write_text("int a; // note\n/* block */ int b;\n")
    (d / "tree_mask.cu").write_text("int c;\n")
    h0 = bench.kernel_source_hash(str(d))
    (d / "split_tc.cuh").write_text("int a; // another note\nint b;\n")
    (d / "tree_mask.cu").write_text("int c; int d;\n")
    assert bench.kernel_source_hash(str(d)) == h0
    (d / "split_tc.cuh").write_text("int a; int b2;\n")
    assert bench.kernel_source_hash(str(d)) != h0


def test_traffic_keys():
    assert bench.traffic_key("mid64k") == "mid64k"
    assert bench.traffic_key("mid64k", 0) == "mid64k@nsplit0"


def test_reference_arm_config_has_the_gpu_arms_keys():
    from mla_speculative_decode_tree_gb300 import workloads as W
    cfg = W.CONFIGS["short4k"]
    g = bench.gpu_config(cfg, None, 16, 1)
    r = bench.reference_config(cfg, 16)
    assert set(g) == set(r) and g["workload"] == r["workload"]
