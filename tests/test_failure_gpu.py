"""Failure detection without a GPU fault: a test-only plan flag makes the
tensor-core kernel's gather withhold its first block, so the pipeline's
bounded waits run out; the call must come back (no hang), report
MLA_VERIFY_DEV_TIMEOUT in the workspace status word, and leave the context
usable for the next, normal call."""

import os
import time

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


@pytest.mark.parametrize("mode", [0, B.MLA_VERIFY_REFETCH_VALUES], ids=["resident", "refetch"])
def test_stalled_pipeline_times_out_and_the_context_stays_usable(mode):
    from oracle import ref
    wl = W.tiny_workload(B=1, H=16, T=4, prefix_lens=[600], pool_rows=4096, seed=3, nsplit=2)
    d = B.device_inputs(wl)
    v = B.verifier_for(wl, flags=B.MLA_VERIFY_TEST_STALL_GATHER | mode)
    assert v.plan.describe().kernel == 1
    torch.cuda.synchronize()
    t0 = time.time()
    v.run(d, wl["B"], wl["sm_scale"])
    torch.cuda.synchronize()
    dt = time.time() - t0
    st = v.status()
    assert st & B.MLA_VERIFY_DEV_TIMEOUT, st
    assert 0.5 < dt < 60, dt  # the waits are bounded at about 2 s

    good = B.verifier_for(wl, flags=mode)
    o, lse = good.run(d, wl["B"], wl["sm_scale"])
    torch.cuda.synchronize()
    assert good.status() == 0
    o_ref, lse_ref = ref.verify(wl, nthreads=os.cpu_count() or 4)
    compare(bf16_to_f64(o).reshape(-1, 512), lse.cpu().numpy().astype(np.float64).reshape(-1), o_ref, lse_ref,
            "call after a timed-out call")
