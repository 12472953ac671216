"""Helpers shared by the GPU parity tests: tolerances and comparisons.

Tolerances (fp32 accumulation, bf16 output): on O max-abs 1e-2, mean-abs
1e-3 and relative L2 1e-2; on LSE max-abs 1e-3.  Relative L2 guards long
prefixes, where |O| ~ N^-1/2 is itself below 1e-2.

O is bf16, so even the exact result rounded to bf16 misses the oracle by up
to half a bf16 spacing -- 0.0156 where |O| >= 4, which a row over one or two
visible keys reaches -- and by ~1e-3 on average where |O| ~ 1.  The O
tolerances therefore bound the error beyond that rounding: per element
|O_gpu - O| - |bf16(O) - O|, which is at most twice the computation's own
error whichever way the last bit goes.
"""

import numpy as np

from mla_speculative_decode_tree_gb300 import workloads as W

O_MAX_ABS = 1e-2
O_MEAN_ABS = 1e-3
O_REL_L2 = 1e-2
LSE_MAX_ABS = 1e-3


def bf16_to_f64(t):
    """torch bf16 tensor (any device) -> float64 numpy array, exactly."""
    import torch
    return t.detach().to("cpu").to(torch.float32).numpy().astype(np.float64)


def compare(o_gpu, lse_gpu, o_ref, lse_ref, what=""):
    """Assert the tolerances; returns a dict of the measured errors."""
    o_gpu = np.asarray(o_gpu, np.float64).reshape(o_ref.shape)
    lse_gpu = np.asarray(lse_gpu, np.float64).reshape(lse_ref.shape)
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isfinite(lse_gpu), fin), what + ": -inf pattern of LSE differs"
    assert np.all(lse_gpu[~fin] == -np.inf), what
    assert np.all(o_gpu[~fin] == 0), what + ": rows with nothing visible must be 0"
    d = np.abs(o_gpu - o_ref)
    ref_bf16 = W.bf16_bits_to_f32(W.f32_to_bf16_bits(o_ref.astype(np.float32))).astype(np.float64)
    excess = d - np.abs(ref_bf16 - o_ref)  # beyond the output format's own rounding
    err = dict(o_max=float(excess.max()) if d.size else 0.0, o_mean=float(excess.mean()) if d.size else 0.0,
               o_max_raw=float(d.max()) if d.size else 0.0,
               lse_max=float(np.abs(lse_gpu[fin] - lse_ref[fin]).max()) if fin.any() else 0.0)
    ref_norm = float(np.linalg.norm(o_ref[fin]))
    err["o_rel_l2"] = float(np.linalg.norm((o_gpu - o_ref)[fin]) / ref_norm) if ref_norm > 0 else 0.0
    assert err["o_max"] <= O_MAX_ABS, (what, err)
    assert err["o_mean"] <= O_MEAN_ABS, (what, err)
    assert err["lse_max"] <= LSE_MAX_ABS, (what, err)
    assert err["o_rel_l2"] <= O_REL_L2, (what, err)
    return err


def sample_rows(wl, per_request=36, seed=0):
    """Rows (b*T+i)*H+h covering every draft token of every request, spread over heads."""
    rng = np.random.default_rng(seed)
    B, T, H = wl["B"], wl["T"], wl["H"]
    rows = []
    for b in range(B):
        k = max(T, min(per_request, T * H))
        for n in range(k):
            i = n % T
            h = int(rng.integers(0, H)) if n >= T else (n * 7) % H
            rows.append((b * T + i) * H + h)
    return np.array(sorted(set(rows)), dtype=np.int64)
