"""The bounded waits' timeout path, on the GPU, without a fault.

rra_test_hold_append makes the fused step's append warp skip its arrival on the barrier that
the TMA producer of the appending CTA waits on before loading the tile with the new token. That
wait, and the consumer warps' wait for the tile that is then never loaded, run out after about
a second; the kernel sets RRA_ERR_TIMEOUT and finishes (nothing was in flight: the producer
issued no copy after the barrier and drained the ones before). The test checks the error bit,
that the launch ended within a few seconds, and that the same context then runs the step
correctly again.
"""

import time

import numpy as np
import pytest
import torch

from tests import gpu_harness as H
from workloads import CONFIGS, make_inputs, reduced

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["batched_paged", "llama3_8b_layer"])
def test_held_append_barrier_times_out_and_context_recovers(name):
    from rope_gqa_paged_gb300 import RRA_ERR_TIMEOUT, rra

    inp = make_inputs(reduced(CONFIGS[name], 16, 2))
    rra.rra_test_hold_append(True)
    try:
        t0 = time.perf_counter()
        held = H.run_gpu(inp, fused=True, fetch_cache=False)
        elapsed = time.perf_counter() - t0
    finally:
        rra.rra_test_hold_append(False)
    assert held.err & RRA_ERR_TIMEOUT, f"expected the timeout bit, got {held.err}"
    assert elapsed < 30.0

    ok = H.run_gpu(inp, fused=True)
    assert ok.err == 0
    q_ref, _, _, out_ref = H.run_oracle(inp)
    H.assert_close_stored(ok.q_rot, q_ref, "bf16", "q_rot")
    assert H.out_error(ok.out, out_ref, "bf16") <= H.OUT_ATOL["bf16"]
    assert torch.cuda.is_available() and np.isfinite(H.stored_to_f64(ok.out, "bf16")).all()
