"""The RoPE angle routine on the GPU: the device evaluation (the code every fused kernel and
rope_append run) against the same routine on the host and against 200-bit cos / sin of
m * theta_i, for the head dims and bases of the workloads and positions up to 2^31 - 1."""

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
