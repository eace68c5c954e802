"""The RoPE angle routine on the GPU: the device evaluation (the code every fused kernel and
rope_append run) against the same routine on the host and against 200-bit cos / sin of
m * theta_i, for the head dims and bases of the workloads and positions up to 2^31 - 1."""

import numpy as np
import pytest
import torch

from tests.test_rope_angles import BOUND, CASES, _positions, _theta

mpmath = pytest.importorskip("mpmath")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rra():
    from rope_gqa_paged_gb300 import rra as binding
    return binding


@pytest.mark.parametrize("D,base", CASES)
def test_device_matches_host_and_mathematics(rra, D, base):
    mpmath.mp.prec = 200
    dev = torch.device("cuda", 0)
    pos = _positions(D + 1)
    out = rra.rra_rope_cos_sin(torch.tensor(pos, dtype=torch.int32, device=dev), D, base)
    torch.cuda.synchronize()
    out = out.cpu()
    phi = rra.rra_rope_phi(D, base)
    for p, m in enumerate(pos):
        for i in range(D // 2):
            d = [float(x) for x in out[p, :, i]]
            h = rra.rra_rope_cos_sin_host(m, phi[i])
            assert abs((d[0] + d[1]) - (h[0] + h[1])) < 2.0 ** -46 and abs((d[2] + d[3]) - (h[2] + h[3])) < 2.0 ** -46
            if i % 7 == 0:
                ang = mpmath.mpf(m) * mpmath.mpf(_theta(D, base, i))
                assert abs(mpmath.mpf(d[0]) + mpmath.mpf(d[1]) - mpmath.cos(ang)) < BOUND, (m, i)
                assert abs(mpmath.mpf(d[2]) + mpmath.mpf(d[3]) - mpmath.sin(ang)) < BOUND, (m, i)


def test_negative_position_and_empty(rra):
    dev = torch.device("cuda", 0)
    out = rra.rra_rope_cos_sin(torch.tensor([5, -3], dtype=torch.int32, device=dev), 64)
    torch.cuda.synchronize()
    assert torch.isfinite(out[0]).all() and torch.isnan(out[1]).all()
    assert rra.rra_rope_cos_sin(torch.empty(0, dtype=torch.int32, device=dev), 64).numel() == 0


# ------------------------------------------------------------------ one angle routine for every path
@pytest.mark.parametrize("name,factor,batch,rope_style",
                         [("llama3_8b_layer", 16, None, 0), ("batched_paged", 16, 8, 0), ("batched_paged", 16, 8, 1)],
                         ids=["contiguous", "paged", "paged_interleaved"])
def test_fused_step_and_two_calls_agree_bitwise(name, factor, batch, rope_style):
    """The fused decode step rotates inside the attention kernel, the two-call path in rope_append;
    both take the angles from the same routine and round once, so q_rot and the appended K (and V)
    must be the same bits, and the attention, reading the same bf16 q_rot, the same output."""
    from tests import gpu_harness as H
    from workloads import CONFIGS, make_inputs, reduced
    inp = make_inputs(reduced(CONFIGS[name], factor, batch), seed=11)
    a = H.run_gpu(inp, num_splits=3, rope_style=rope_style, fused=True)
    b = H.run_gpu(inp, num_splits=3, rope_style=rope_style, fused=False)
    assert a.err == 0 and b.err == 0
    assert np.array_equal(a.q_rot, b.q_rot)  # bf16 bit patterns
    assert np.array_equal(a.k_cache, b.k_cache)
    assert np.array_equal(a.v_cache, b.v_cache)
    assert np.abs(H.stored_to_f64(a.out, "bf16") - H.stored_to_f64(b.out, "bf16")).max() <= 1e-3


def test_verify_fused_and_two_calls_agree_bitwise():
    """The one-launch verify step against rope_append_verify + verify_attn: same q_rot and cache bits."""
    from tests import gpu_harness as H
    from workloads import CONFIGS, make_inputs, reduced
    inp = make_inputs(reduced(CONFIGS["batched_paged_verify4"], 16, 4), seed=5)
    a = H.run_gpu_verify(inp, num_splits=3, fused=True)
    b = H.run_gpu_verify(inp, num_splits=3, fused=False)
    assert a.err == 0 and b.err == 0
    assert np.array_equal(a.q_rot, b.q_rot)  # bf16 bit patterns
    assert np.array_equal(a.k_cache, b.k_cache)
    assert np.array_equal(a.v_cache, b.v_cache)
    assert np.abs(H.stored_to_f64(a.out, "bf16") - H.stored_to_f64(b.out, "bf16")).max() <= 1e-3


@pytest.mark.parametrize("name", ["batched_paged_int8", "batched_paged_int4"])
def test_quantised_fused_and_two_calls_agree_bitwise(name):
    """INT8 / INT4 caches: the fused step's append (inside the attention kernel) and rope_append_q8 /
    _q4 write the same codes and window values, and publish the same q_rot."""
    from tests import gpu_harness as H
    from workloads import CONFIGS, make_inputs, reduced
    inp = make_inputs(reduced(CONFIGS[name], 16, 4), seed=7)
    a = H.run_gpu_q8(inp, num_splits=3, fused=True)
    b = H.run_gpu_q8(inp, num_splits=3, fused=False)
    assert a.err == 0 and b.err == 0
    assert np.array_equal(a.q_rot, b.q_rot)
    assert np.array_equal(a.k_codes, b.k_codes) and np.array_equal(a.v_codes, b.v_codes)
    if a.k_win is not None:
        assert np.array_equal(a.k_win, b.k_win) and np.array_equal(a.v_win, b.v_win)
    assert np.abs(H.stored_to_f64(a.out, "bf16") - H.stored_to_f64(b.out, "bf16")).max() <= 1e-3
