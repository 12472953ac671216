"""Randomised parity: seeded random shapes (batch, heads, draft tokens,
prefix lengths at and around tile boundaries, split counts including the
planner's, every mode and flag, uniform and per-request draft counts), each
checked against the fp64 oracle with the shared tolerances."""

import os
import random

import numpy as np
import pytest

from mla_speculative_decode_tree_gb300 import binding as B
from mla_speculative_decode_tree_gb300 import workloads as W
from parity_util import bf16_to_f64, compare

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

FLAGS = [0, B.MLA_VERIFY_REFETCH_VALUES, B.MLA_VERIFY_FUSED_MERGE,
         B.MLA_VERIFY_FUSED_MERGE | B.MLA_VERIFY_REFETCH_VALUES, B.MLA_VERIFY_FORCE_SIMT]


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_speculative_decode_tree_gb300 import build
    build.build()
    from oracle import ref
    ref.build()


def _case(seed):
    rng = random.Random(seed)
    Bn = rng.choice([1, 1, 2, 3, 5])
    H = rng.choice([1, 2, 5, 8, 16, 24, 32, 64])
    T = rng.choice([1, 2, 4, 9, 13, 16, 33, 64])
    while H * T > 2048:
        T = max(1, T // 2)
    P = [rng.choice([0, 1, 63, 64, 65, 127, 128, 129, 300, 1000, 2047, 3000, 5000]) for _ in range(Bn)]
    ns = rng.choice([0, 1, 2, 3, 5, 7, 16, 33, 64])
    fl = rng.choice(FLAGS)
    varlen = Bn > 1 and rng.random() < 0.25
    Ts = [rng.randint(0, T) for _ in range(Bn)] if varlen else None
    return Bn, H, T, P, ns, fl, Ts


@pytest.mark.parametrize("seed", range(48))
def test_random_shape(seed):
    from oracle import ref
    Bn, H, T, P, ns, fl, Ts = _case(seed)
    pool = max(4096, sum(P) + Bn * T + 64)
    if Ts is not None:
        wl = W.varlen_workload(B=Bn, H=H, T_list=Ts, prefix_lens=P, pool_rows=pool, seed=seed + 500, nsplit=ns)
    else:
        wl = W.tiny_workload(B=Bn, H=H, T=T, prefix_lens=P, pool_rows=pool, seed=seed + 500, nsplit=ns,
                             tree="chain" if seed % 3 == 0 else "random")
    d = B.device_inputs(wl)
    v = B.verifier_for(wl, flags=fl)
    o, lse = v.run(d, wl["B"], wl["sm_scale"])
    torch.cuda.synchronize()
    assert v.status() == 0
    nrow = (int(wl["qo_indptr"][-1]) if Ts is not None else Bn * T) * H
    o = bf16_to_f64(o).reshape(-1, 512)[:nrow]
    lse = lse.cpu().numpy().astype(np.float64).reshape(-1)[:nrow]
    o_ref, lse_ref = ref.verify(wl, nthreads=os.cpu_count() or 4)
    compare(o, lse, o_ref, lse_ref, "random shape %d: %s" % (seed, (Bn, H, T, P, ns, fl, Ts)))
