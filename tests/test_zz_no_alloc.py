"""rra_decode_attn_paged_noalloc: the paged decode for callers that cannot allocate.

Callers that may not allocate device memory when they run a step (a host framework owns
all device memory, or allocation is forbidden after start-up) use this entry point; its
split-K scratch is a fixed array inside the library. These tests call it through the C ABI
and check it against rra_decode_attn_paged with a torch-allocated, zeroed workspace at the
same split count -- the same kernel on the same inputs, so the outputs must be identical
bit for bit -- twice in a row, and across calls of different shapes (a later call's
counters may sit where an earlier call wrote partials). One case is also checked against
the float64 oracle. Collected last so a failure here never hides another test's result.
"""

import ctypes

import numpy as np
import pytest
import torch

from oracle import decode as odecode
from tests import gpu_harness as H
from workloads import CONFIGS, make_inputs, reduced

pytestmark = pytest.mark.gpu

RRA_EWORKSPACE = -4


def _noalloc_fn():
    from rope_gqa_paged_gb300 import _build, rra
    _build.build()
    fn = rra.lib().rra_decode_attn_paged_noalloc
    vp, ci = ctypes.c_void_p, ctypes.c_int
    fn.restype = ci
    fn.argtypes = [vp, vp, vp, vp, ci, vp, ci, ci, vp, ci, ci, ci, ci, ctypes.c_float, ci, ci, vp, vp]
    return fn


def _call_noalloc(fn, q, kp, vp_, table, lens, out, num_splits, err):
    B, Hq, D = q.shape
    nblk, bs, Hkv = kp.shape[0], kp.shape[1], kp.shape[2]
    return fn(q.data_ptr(), kp.data_ptr(), vp_.data_ptr(), table.data_ptr(), table.shape[1], lens.data_ptr(), bs,
              nblk, out.data_ptr(), B, Hq, Hkv, D, 0.0, num_splits, 1, err.data_ptr(),
              torch.cuda.current_stream().cuda_stream)


class _Case:
    """A paged workload on the device, attending the L_b - 1 cached tokens (no append: slot
    L_b - 1 is still NaN-poisoned), with the workspace entry point's output as reference."""

    def __init__(self, cfg, splits):
        from rope_gqa_paged_gb300 import rra
        self.inp = make_inputs(cfg)
        dev = torch.device("cuda", 0)
        self.q = H.to_torch(self.inp.q, "bf16", dev)
        self.kp, self.vp = H.to_torch(self.inp.k_cache, "bf16", dev), H.to_torch(self.inp.v_cache, "bf16", dev)
        self.table = H.to_torch(self.inp.block_table, "i32", dev)
        self.lens_np = (self.inp.lengths - 1).astype(np.int32)
        self.lens = H.to_torch(self.lens_np, "i32", dev)
        self.splits = splits
        self.eff = rra.rra_decode_num_splits(cfg.batch, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim, cfg.capacity,
                                             cfg.block_size, splits, rra.RRA_BF16)
        ws_bytes = rra.rra_decode_workspace_bytes(cfg.batch, cfg.n_q_heads, cfg.head_dim, self.eff)
        ws = torch.zeros(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
        err = torch.zeros(1, dtype=torch.int32, device=dev)
        self.ref = torch.full_like(self.q, float("nan"))
        rra.rra_decode_attn_paged(self.q, self.kp, self.vp, self.table, self.lens, self.ref, num_splits=splits,
                                  workspace=ws, err_flag=err)
        torch.cuda.synchronize()
        assert err.item() == 0
        assert torch.isfinite(self.ref.float()).all()

    def run_noalloc(self, fn):
        err = torch.zeros(1, dtype=torch.int32, device=self.q.device)
        out = torch.full_like(self.q, float("nan"))
        assert _call_noalloc(fn, self.q, self.kp, self.vp, self.table, self.lens, out, self.splits, err) == 0
        torch.cuda.synchronize()
        return out, int(err.item())

    def check_identical(self, out, err, what):
        assert err == 0, f"{what}: device error bits {err}"
        same = torch.equal(out.view(torch.int16), self.ref.view(torch.int16))
        if not same:
            diff = (out.float() - self.ref.float()).abs()
            pytest.fail(f"{what}: not bit-identical to the workspace entry point "
                        f"(max abs diff {diff.nan_to_num(float('inf')).max().item()})")


@pytest.mark.parametrize("name,factor,batch,splits", [("batched_paged", 16, 8, 3), ("long_context", 64, 1, 0),
                                                       ("prefix_sweep_kv1", 16, 4, 5)])
def test_noalloc_matches_workspace_entry_point_twice(name, factor, batch, splits):
    fn = _noalloc_fn()
    case = _Case(reduced(CONFIGS[name], factor, batch), splits)
    assert case.eff > 1
    for call in range(2):
        out, err = case.run_noalloc(fn)
        case.check_identical(out, err, f"{name} call {call}")


def test_noalloc_shapes_back_to_back():
    """Calls of different shapes in a row share the scratch: 8 sequences at 3 splits, then one
    32-head sequence at 2 splits (whose counters would sit among the first call's partials if
    the counters' place depended on the shape), then the first again."""
    fn = _noalloc_fn()
    first = _Case(reduced(CONFIGS["batched_paged"], 16, 8), 3)
    second = _Case(reduced(CONFIGS["long_context"], 64, 1), 2)
    assert first.eff == 3 and second.eff == 2
    assert second.inp.cfg.n_q_heads == 32 and second.inp.cfg.head_dim == 128
    for what, case in (("8 sequences, 3 splits", first), ("1 sequence, 2 splits", second),
                       ("8 sequences, 3 splits again", first)):
        out, err = case.run_noalloc(fn)
        case.check_identical(out, err, what)


def test_noalloc_against_the_oracle():
    """The no-workspace output against the float64 oracle over the same stored inputs."""
    fn = _noalloc_fn()
    case = _Case(reduced(CONFIGS["batched_paged"], 16, 4), 3)
    out, err = case.run_noalloc(fn)
    assert err == 0
    inp, cfg = case.inp, case.inp.cfg
    want = odecode.decode_attention(inp.q, inp.k_cache, inp.v_cache, case.lens_np, cfg.dtype, inp.block_table,
                                    cfg.block_size)
    got = H.to_numpy(out)
    assert H.out_error(got, want, "bf16") <= H.OUT_ATOL["bf16"]
    assert H.rel_rms_error(got, want, "bf16") <= H.REL_RMS_BAR


def test_noalloc_rejects_steps_larger_than_its_scratch():
    from rope_gqa_paged_gb300 import rra
    fn = _noalloc_fn()
    limit = rra.lib().rra_noalloc_scratch_bytes
    limit.restype = ctypes.c_size_t
    cap = int(limit())
    assert cap == 16 << 20
    # 512 sequences x 32 heads x 64 splits x (128 + 2) floats is far beyond 16 MiB
    B, Hq, Hkv, D, bs, mbps = 512, 32, 8, 128, 16, 512
    assert rra.rra_decode_workspace_bytes(B, Hq, D, 64) > cap
    dev = torch.device("cuda", 0)
    dummy = torch.zeros(16, dtype=torch.bfloat16, device=dev)      # never read: the size check comes first
    status = fn(dummy.data_ptr(), dummy.data_ptr(), dummy.data_ptr(), dummy.data_ptr(), mbps, dummy.data_ptr(),
                bs, 64, dummy.data_ptr(), B, Hq, Hkv, D, 0.0, 64, 1, None, None)
    assert status == RRA_EWORKSPACE
