"""rra_decode_attn_paged_noalloc: the paged decode for callers that cannot allocate.

Callers that may not allocate device memory when they run a step (a host framework owns
all device memory, or allocation is forbidden after start-up) use this entry point; its
split-K scratch is a fixed array inside the library. These tests call it through the C ABI
and check it against rra_decode_attn_paged with a torch-allocated workspace, twice in a
row (the second call reuses the scratch the first call left behind). Collected last so a
failure here never hides another test's result.
"""

import ctypes

import pytest
import torch

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


@pytest.mark.parametrize("name,factor,batch,splits", [("batched_paged", 16, 8, 3), ("long_context", 64, 1, 0),
                                                       ("prefix_sweep_kv1", 16, 4, 5)])
def test_noalloc_matches_workspace_entry_point_twice(name, factor, batch, splits):
    from rope_gqa_paged_gb300 import rra
    fn = _noalloc_fn()
    inp = make_inputs(reduced(CONFIGS[name], factor, batch))
    dev = torch.device("cuda", 0)
    q = H.to_torch(inp.q, "bf16", dev)
    kp, vp_ = H.to_torch(inp.k_cache, "bf16", dev), H.to_torch(inp.v_cache, "bf16", dev)
    table = H.to_torch(inp.block_table, "i32", dev)
    # no rope_append here: attend only the L_b - 1 cached tokens (slot L_b - 1 is still NaN-poisoned)
    lens = H.to_torch(inp.lengths - 1, "i32", dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)

    cfg = inp.cfg
    eff = rra.rra_decode_num_splits(cfg.batch, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim, cfg.capacity,
                                    cfg.block_size, splits, rra.RRA_BF16)
    ws_bytes = rra.rra_decode_workspace_bytes(cfg.batch, cfg.n_q_heads, cfg.head_dim, eff)
    ws = torch.zeros(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    ref = torch.empty_like(q)
    rra.rra_decode_attn_paged(q, kp, vp_, table, lens, ref, num_splits=splits, workspace=ws, err_flag=err)
    torch.cuda.synchronize()
    assert torch.isfinite(ref.float()).all()
    for call in range(2):
        out = torch.full_like(q, float("nan"))
        assert _call_noalloc(fn, q, kp, vp_, table, lens, out, splits, err) == 0
        torch.cuda.synchronize()
        diff = (out.float() - ref.float()).abs().max().item()
        assert diff <= H.OUT_ATOL["bf16"], f"call {call}: max abs diff {diff}"
    assert err.item() == 0


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
