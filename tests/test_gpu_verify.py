"""Multi-query decode (speculative verify, gamma new tokens per sequence) against the float64 oracle.

Bars: q_rot and the appended K rows within 1 bf16 ulp, appended V rows and every other cache
byte bit-exact, attention output (every new token, causal inside the chunk) max abs error
<= 1e-2 against the oracle's float64 result on the same stored inputs.
"""

import dataclasses

import numpy as np
import pytest

from tests import gpu_harness as H
from workloads import CONFIGS, WorkloadConfig, make_inputs, reduced
from workloads.gen import poison_unread

pytestmark = pytest.mark.gpu


def _slot(inp, b, pos):
    cfg = inp.cfg
    if inp.block_table is None:
        return (b, slice(None), pos)
    return (inp.block_table[b, pos // cfg.block_size], pos % cfg.block_size)


def _check(inp, gpu, ref):
    cfg = inp.cfg
    q_ref, k_ref, v_ref, out_ref = ref
    assert gpu.err == 0
    H.assert_close_stored(gpu.q_rot, q_ref, "bf16", "q_rot")
    err = H.out_error(gpu.out, out_ref, "bf16")
    assert err <= H.OUT_ATOL["bf16"], f"{cfg.name}: out max abs err {err:.3e}"
    rel = H.rel_rms_error(gpu.out, out_ref, "bf16")
    assert rel <= H.REL_RMS_BAR, f"{cfg.name}: out error {rel:.3e} of the row RMS"
    kc, vc = gpu.k_cache.copy(), gpu.v_cache.copy()
    for b in range(cfg.batch):
        for j in range(cfg.gamma):
            idx = _slot(inp, b, int(inp.positions[b]) + j)
            H.assert_close_stored(kc[idx], k_ref[idx], "bf16", f"appended K {b}/{j}")
            assert vc[idx].tobytes() == inp.v_new[b, j].tobytes(), f"appended V {b}/{j}"
            kc[idx], vc[idx] = inp.k_cache[idx], inp.v_cache[idx]
    assert kc.tobytes() == inp.k_cache.tobytes() and vc.tobytes() == inp.v_cache.tobytes(), "cache changed elsewhere"
    return err


REDUCED = [("batched_paged_verify4", 16, 8), ("long_context_verify4", 64, 1)]


@pytest.mark.parametrize("name,factor,batch", REDUCED, ids=[r[0] for r in REDUCED])
@pytest.mark.parametrize("splits", [0, 3])
@pytest.mark.parametrize("fused", [False, True], ids=["two_calls", "verify_step"])
def test_verify_reduced_workload(name, factor, batch, splits, fused):
    inp = make_inputs(reduced(CONFIGS[name], factor, batch))
    _check(inp, H.run_gpu_verify(inp, num_splits=splits, fused=fused), H.run_oracle_verify(inp))


def _cfg(layout, lengths, gamma, block_size=16, head_dim=128, hq=32, hkv=8):
    longest = max(lengths)
    kw = dict(name=f"verify_{layout}", batch=len(lengths), n_q_heads=hq, n_kv_heads=hkv, head_dim=head_dim,
              dtype="bf16", layout=layout, len_range=(longest, longest), gamma=gamma)
    if layout == "contiguous":
        kw["max_len"] = max(longest + 5, 16384 // (2 * head_dim))
    else:
        kw.update(block_size=block_size, max_blocks_per_seq=-(-longest // block_size))
        kw["num_blocks"] = len(lengths) * kw["max_blocks_per_seq"] + 5
    return WorkloadConfig(**kw)


def _inputs(cfg, lengths, seed=5):
    inp = make_inputs(cfg, seed=seed, poison=False)
    if cfg.gamma == 1:                       # the generator keeps decode shapes for one new token
        inp.q, inp.k_new, inp.v_new = inp.q[:, None], inp.k_new[:, None], inp.v_new[:, None]
    inp.lengths = np.asarray(lengths, dtype=np.int32)
    inp.positions = (inp.lengths - cfg.gamma).astype(np.int32)
    if inp.block_table is not None:
        for b, L in enumerate(lengths):
            inp.block_table[b, -(-L // cfg.block_size):] = -1
    poison_unread(inp)
    return inp


@pytest.mark.parametrize("layout,block_size", [("contiguous", 0), ("paged", 8), ("paged", 16), ("paged", 256)])
@pytest.mark.parametrize("gamma", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("fused", [True, False], ids=["verify_step", "two_calls"])
def test_verify_edge_lengths(layout, block_size, gamma, fused):
    """The verify step is one launch up to gamma 8 (RoPE and append inside the attention kernel),
    two launches above; the two calls (append, then attention) are checked alike. Lengths put the
    new tokens at the start of the cache, across tile edges and, with 2 splits, across chunks."""
    lengths = [gamma, gamma + 1, 63 + gamma, 64, 65 + gamma, 300]
    lengths = [max(L, gamma) for L in lengths]
    cfg = _cfg(layout, lengths, gamma, block_size=block_size or 16)
    inp = _inputs(cfg, lengths)
    for splits in (0, 2):
        _check(inp, H.run_gpu_verify(inp, num_splits=splits, fused=fused), H.run_oracle_verify(inp))


@pytest.mark.parametrize("hq,hkv", [(8, 8), (32, 1), (12, 4), (64, 4)], ids=["mha", "mqa", "nrep3", "nrep16"])
@pytest.mark.parametrize("head_dim", [64, 128])
@pytest.mark.parametrize("style", [0, 1], ids=["half_split", "interleaved"])
def test_verify_heads_and_head_dim(hq, hkv, head_dim, style):
    lengths = [9, 200, 611]
    cfg = _cfg("paged", lengths, 4, head_dim=head_dim, hq=hq, hkv=hkv)
    inp = _inputs(cfg, lengths, seed=9)
    _check(inp, H.run_gpu_verify(inp, num_splits=3, rope_style=style), H.run_oracle_verify(inp, rope_style=style))


@pytest.mark.parametrize("splits", [17, 40])
def test_verify_many_splits_merge(splits):
    lengths = [4100, 2500]
    cfg = _cfg("paged", lengths, 4, block_size=32)
    inp = _inputs(cfg, lengths, seed=13)
    gpu = H.run_gpu_verify(inp, num_splits=splits)
    assert gpu.splits > 16
    _check(inp, gpu, H.run_oracle_verify(inp))


def test_verify_position_errors_are_flagged():
    from rope_gqa_paged_gb300 import RRA_ERR_POSITION
    lengths = [40, 60]
    cfg = _cfg("paged", lengths, 4)
    inp = _inputs(cfg, lengths)
    inp.positions = np.array([36, cfg.capacity - 2], dtype=np.int32)   # the second chunk runs past the cache
    gpu = H.run_gpu_verify(inp)
    assert gpu.err & RRA_ERR_POSITION
