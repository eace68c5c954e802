"""CUDA path (through the C ABI) against the float64 oracle on the same seeded inputs.

Bars: appended K and q_rot within 1 bf16 ulp (4 fp32 ulps for fp32), appended V and
every untouched cache slot bit-exact, attention output max abs error <= 1e-4 (fp32)
or <= 1e-2 (bf16) against the oracle's float64 result.
"""

import math

import numpy as np
import pytest

from tests import gpu_harness as H
from workloads import CONFIGS, make_inputs, reduced

pytestmark = pytest.mark.gpu


def _check_step(inp, gpu, q_ref, out_ref, batches=None):
    cfg = inp.cfg
    bs = range(cfg.batch) if batches is None else batches
    H.assert_close_stored(gpu.q_rot[list(bs)], q_ref, cfg.dtype, "q_rot")
    err = H.out_error(gpu.out[list(bs)], out_ref, cfg.dtype)
    assert err <= H.OUT_ATOL[cfg.dtype], f"{cfg.name}: out max abs err {err:.3e}"
    rel = H.rel_rms_error(gpu.out[list(bs)], out_ref, cfg.dtype)
    assert rel <= H.REL_RMS_BAR, f"{cfg.name}: out error {rel:.3e} of the row RMS"
    return err


def _check_cache(inp, gpu, k_ref_rows=None):
    """Appended rows: K within 1 ulp of the oracle, V bit-exact; every other slot untouched."""
    cfg = inp.cfg
    kc, vc = gpu.k_cache.copy(), gpu.v_cache.copy()
    for b in range(cfg.batch):
        pos = int(inp.positions[b])
        if inp.block_table is None:
            k_row, v_row = kc[b, :, pos].copy(), vc[b, :, pos].copy()
            kc[b, :, pos], vc[b, :, pos] = inp.k_cache[b, :, pos], inp.v_cache[b, :, pos]
        else:
            phys, off = inp.block_table[b, pos // cfg.block_size], pos % cfg.block_size
            k_row, v_row = kc[phys, off].copy(), vc[phys, off].copy()
            kc[phys, off], vc[phys, off] = inp.k_cache[phys, off], inp.v_cache[phys, off]
        assert v_row.tobytes() == inp.v_new[b].tobytes(), f"appended V of sequence {b} differs"
        if k_ref_rows is not None:
            H.assert_close_stored(k_row, k_ref_rows[b], cfg.dtype, f"appended K of sequence {b}")
    assert kc.tobytes() == inp.k_cache.tobytes(), "K cache changed outside the appended slots"
    assert vc.tobytes() == inp.v_cache.tobytes(), "V cache changed outside the appended slots"


def _oracle_k_rows(inp, ref_k_cache):
    cfg = inp.cfg
    rows = []
    for b in range(cfg.batch):
        pos = int(inp.positions[b])
        if inp.block_table is None:
            rows.append(ref_k_cache[b, :, pos])
        else:
            rows.append(ref_k_cache[inp.block_table[b, pos // cfg.block_size], pos % cfg.block_size])
    return rows


# ------------------------------------------------------------------ whole batches at reduced size
REDUCED = [("tiny_fp32", 1, None), ("llama3_8b_layer", 16, None), ("batched_paged", 16, 8),
           ("long_context", 64, None), ("prefix_sweep_kv32", 16, 3), ("prefix_sweep_kv8", 16, 4),
           ("prefix_sweep_kv1", 16, 4)]


@pytest.mark.parametrize("name,factor,batch", REDUCED, ids=[r[0] for r in REDUCED])
@pytest.mark.parametrize("splits", [0, 1, 3])
@pytest.mark.parametrize("fused", [False, True], ids=["two_calls", "fused_step"])
def test_reduced_workload(name, factor, batch, splits, fused):
    cfg = CONFIGS[name] if factor == 1 else reduced(CONFIGS[name], factor, batch)
    inp = make_inputs(cfg)
    gpu = H.run_gpu(inp, num_splits=splits, fused=fused)
    q_ref, k_ref, _, out_ref = H.run_oracle(inp)
    assert gpu.err == 0
    _check_step(inp, gpu, q_ref, out_ref)
    _check_cache(inp, gpu, _oracle_k_rows(inp, k_ref))


@pytest.mark.parametrize("layout", ["contiguous", "paged"])
@pytest.mark.parametrize("fused", [False, True], ids=["two_calls", "fused_step"])
def test_interleaved_rope_pairs(layout, fused):
    base = CONFIGS["llama3_8b_layer"] if layout == "contiguous" else CONFIGS["batched_paged"]
    inp = make_inputs(reduced(base, 16, 4), seed=3)
    gpu = H.run_gpu(inp, rope_style=1, fused=fused)
    q_ref, k_ref, _, out_ref = H.run_oracle(inp, rope_style=1)
    _check_step(inp, gpu, q_ref, out_ref)
    _check_cache(inp, gpu, _oracle_k_rows(inp, k_ref))


def test_tiny_fp32_matches_tightly():
    inp = make_inputs(CONFIGS["tiny_fp32"])
    gpu = H.run_gpu(inp)
    _, _, _, out_ref = H.run_oracle(inp)
    assert H.out_error(gpu.out, out_ref, "f32") <= 1e-4


# ------------------------------------------------------------------ edge lengths
@pytest.mark.parametrize("layout,bs", [("contiguous", 0), ("paged", 16), ("paged", 32), ("paged", 64), ("paged", 8)])
@pytest.mark.parametrize("hq,hkv", [(32, 8), (32, 1), (128, 1)], ids=["gqa4", "mqa32", "mqa128"])
def test_edge_lengths(layout, bs, hq, hkv):
    """L = 1 (the new token alone), around tile and block edges (64-token tiles of the mma.sync
    kernel, 128-token tiles of the tcgen05 kernel that serves the 128-head group), and a full cache."""
    import dataclasses
    base = CONFIGS["llama3_8b_layer"] if layout == "contiguous" else CONFIGS["batched_paged"]
    cap = 256
    lens = [1, 2, 15, 16, 17, 31, 32, 33, 63, 64, 65, 127, 129, 200, 255, 256]
    kw = dict(batch=len(lens), seq_len=None, len_range=(1, cap), num_splits=0, n_q_heads=hq, n_kv_heads=hkv)
    if layout == "contiguous":
        kw["max_len"] = cap
    else:
        kw.update(block_size=bs, max_blocks_per_seq=cap // bs, num_blocks=len(lens) * (cap // bs) + 3)
    cfg = dataclasses.replace(base, name=f"edge_{layout}_{bs}_{hq}_{hkv}", **kw)
    from workloads import gen
    inp = gen.make_inputs(cfg, poison=False)
    inp.lengths[:] = lens
    inp.positions[:] = np.array(lens) - 1
    if layout == "paged":
        rng = np.random.default_rng(5)
        perm = rng.permutation(cfg.num_blocks)
        inp.block_table[:] = -1
        k = 0
        for b, L in enumerate(lens):
            nb = math.ceil(L / bs)
            inp.block_table[b, :nb] = perm[k:k + nb]
            k += nb
    gen.poison_unread(inp)
    for splits, fused in ((0, False), (1, False), (2, False), (5, False), (0, True), (1, True), (5, True)):
        gpu = H.run_gpu(inp, num_splits=splits, fused=fused)
        q_ref, k_ref, _, out_ref = H.run_oracle(inp)
        assert gpu.err == 0
        _check_step(inp, gpu, q_ref, out_ref)
        _check_cache(inp, gpu, _oracle_k_rows(inp, k_ref))


def test_one_hot_attention():
    """One cached key aligned with the rotated query dominates: out == that V row."""
    import oracle
    cfg = reduced(CONFIGS["batched_paged"], 16, 6)
    inp = make_inputs(cfg, seed=7)
    rng = np.random.default_rng(7)
    targets = []
    for b in range(cfg.batch):
        L = int(inp.lengths[b])
        t = int(rng.integers(0, L - 1))
        targets.append(t)
        qf = oracle.storage_to_f64(inp.q[b], "bf16")
        q_rot = oracle.apply_rope(qf, L - 1)
        phys, off = inp.block_table[b, t // cfg.block_size], t % cfg.block_size
        for g in range(cfg.n_kv_heads):
            grp = q_rot[g * cfg.n_rep:(g + 1) * cfg.n_rep].sum(0)
            inp.k_cache[phys, off, g] = oracle.f64_to_bf16_bits(8.0 * grp / np.linalg.norm(grp) * np.sqrt(cfg.head_dim))
            inp.v_cache[phys, off, g] = oracle.f64_to_bf16_bits(rng.uniform(-1, 1, cfg.head_dim))
    gpu = H.run_gpu(inp, num_splits=3)
    _, _, _, out_ref = H.run_oracle(inp)
    err = H.out_error(gpu.out, out_ref, "bf16")
    assert err <= 1e-2
    for b, t in enumerate(targets):                      # the reference is near one-hot on row t
        phys, off = inp.block_table[b, t // cfg.block_size], t % cfg.block_size
        v = oracle.storage_to_f64(inp.v_cache[phys, off], "bf16")
        got = oracle.storage_to_f64(gpu.out[b], "bf16")
        for h in range(cfg.n_q_heads):
            assert np.corrcoef(got[h], v[h // cfg.n_rep])[0, 1] > 0.9


# ------------------------------------------------------------------ device-side errors (no faults)
def test_device_errors_are_flagged_not_faulted():
    cfg = reduced(CONFIGS["batched_paged"], 16, 4)
    inp = make_inputs(cfg, seed=11)
    bad = inp.block_table.copy()
    bad[1, 0] = cfg.num_blocks + 5                        # block id outside the pool
    inp.block_table = bad
    gpu = H.run_gpu(inp, num_splits=2)
    from rope_gqa_paged_gb300 import RRA_ERR_BLOCK_ID, RRA_ERR_POSITION, RRA_ERR_SEQ_LEN
    assert gpu.err & RRA_ERR_BLOCK_ID
    # a length beyond the cache's capacity is clamped and flagged
    inp2 = make_inputs(cfg, seed=12)
    lens = inp2.lengths.copy()
    lens[0] = cfg.capacity + 100
    gpu2 = H.run_gpu(inp2, seq_lens=lens)
    assert gpu2.err & RRA_ERR_SEQ_LEN
    # a position beyond the capacity is not written and is flagged
    inp3 = make_inputs(reduced(CONFIGS["llama3_8b_layer"], 16, 2), seed=13)
    inp3.positions[1] = inp3.cfg.max_len + 3
    gpu3 = H.run_gpu(inp3)
    assert gpu3.err & RRA_ERR_POSITION


# ------------------------------------------------------------------ full size, sampled sequences
FULL = ["llama3_8b_layer", "batched_paged", "long_context", "prefix_sweep_kv32", "prefix_sweep_kv8",
        "prefix_sweep_kv1"]


@pytest.mark.slow
@pytest.mark.parametrize("name", FULL)
def test_full_size_sampled(name):
    cfg = CONFIGS[name]
    inp = make_inputs(cfg)
    gpu = H.run_gpu(inp, fused=True)                      # the launch configuration the bench uses
    assert gpu.err == 0
    rng = np.random.default_rng(1)
    sample = sorted(set([0, cfg.batch - 1] + rng.choice(cfg.batch, size=min(cfg.batch, 3), replace=False).tolist()))
    if cfg.len_range is not None:                         # include the longest and the shortest sequence
        sample = sorted(set(sample + [int(np.argmax(inp.lengths)), int(np.argmin(inp.lengths))]))
    q_ref, out_ref = H.oracle_for_sequences(inp, sample)
    _check_step(inp, gpu, q_ref, out_ref, batches=sample)
    _check_cache(inp, gpu)                                # untouched slots bit-exact, V appended exactly


# ------------------------------------------------------------------ many splits: two-level merge
@pytest.mark.parametrize("name,factor", [("llama3_8b_layer", 2), ("long_context", 32)])
@pytest.mark.parametrize("splits", [17, 33, 40, 64, 100])
def test_many_splits_merge(name, factor, splits):
    """More than 32 splits are merged in two levels (groups of 32, then the groups).

    The effective split count is the request rounded to whole tiles (one level up to 32 splits,
    two above, with a partial last group)."""
    cfg = reduced(CONFIGS[name], factor, 2)
    inp = make_inputs(cfg, seed=21)
    gpu = H.run_gpu(inp, num_splits=splits, fused=True)
    assert gpu.splits > 1
    q_ref, _, _, out_ref = H.run_oracle(inp)
    assert gpu.err == 0
    _check_step(inp, gpu, q_ref, out_ref)


# ------------------------------------------------------------------ many splits, ragged lengths
@pytest.mark.parametrize("layout,block", [("contiguous", 0), ("paged", 16), ("paged", 256)],
                         ids=["contiguous", "paged16", "paged256"])
@pytest.mark.parametrize("head_dim", [64, 128])
@pytest.mark.parametrize("fused", [False, True], ids=["two_calls", "fused_step"])
def test_many_splits_ragged(layout, block, head_dim, fused):
    """64 requested splits of a 4096-token capacity (one tile each: 32 splits at D 64) over
    lengths 70, 1500 and 4000: a sequence whose second split is partial, CTAs past a sequence's
    end that only return, and a sequence merged in two levels; paged blocks smaller and larger
    than the tile."""
    import dataclasses
    from workloads import gen
    lens, cap = [70, 1500, 4000], 4096
    if layout == "contiguous":
        cfg = dataclasses.replace(CONFIGS["llama3_8b_layer"], name=f"ragged_c_{head_dim}", batch=len(lens),
                                  head_dim=head_dim, seq_len=max(lens), max_len=cap, num_splits=64)
    else:
        nb = cap // block
        cfg = dataclasses.replace(CONFIGS["batched_paged"], name=f"ragged_p{block}_{head_dim}", batch=len(lens),
                                  head_dim=head_dim, block_size=block, len_range=(max(lens), max(lens)),
                                  max_blocks_per_seq=nb, num_blocks=len(lens) * nb + 5, num_splits=64)
    inp = gen.make_inputs(cfg, seed=31, poison=False)
    inp.lengths[:] = lens
    inp.positions[:] = np.array(lens) - 1
    if inp.block_table is not None:
        for b, L in enumerate(lens):
            inp.block_table[b, -(-L // block):] = -1
    gen.poison_unread(inp)
    style = 1 if head_dim == 64 else 0
    gpu = H.run_gpu(inp, fused=fused, rope_style=style)
    assert gpu.splits == cap // (16384 // (2 * head_dim))
    q_ref, k_ref, _, out_ref = H.run_oracle(inp, rope_style=style)
    assert gpu.err == 0
    _check_step(inp, gpu, q_ref, out_ref)
    _check_cache(inp, gpu, _oracle_k_rows(inp, k_ref))


def test_fused_step_position_errors_are_flagged():
    """A position outside the cache: flagged, that sequence untouched, the others correct."""
    cfg = reduced(CONFIGS["batched_paged"], 16, 4)
    inp = make_inputs(cfg, seed=14)
    from rope_gqa_paged_gb300 import RRA_ERR_POSITION
    good = H.run_gpu(inp, fused=True)
    bad = inp.positions.copy()
    inp.positions[2] = cfg.capacity + 7
    gpu = H.run_gpu(inp, fused=True)
    assert gpu.err & RRA_ERR_POSITION
    keep = [0, 1, 3]
    assert gpu.out[keep].tobytes() == good.out[keep].tobytes()
    inp.positions[:] = bad


# ------------------------------------------------------------------ heads per KV group
@pytest.mark.parametrize("hq,hkv", [(8, 8), (32, 1), (12, 4), (32, 2), (64, 4), (64, 1), (128, 1)],
                         ids=["mha", "mqa", "nrep3", "nrep16", "nrep16b", "nrep64", "nrep128"])
@pytest.mark.parametrize("head_dim", [64, 128])
@pytest.mark.parametrize("fused", [False, True], ids=["two_calls", "fused_step"])
@pytest.mark.parametrize("style", [0, 1], ids=["half_split", "interleaved"])
def test_heads_and_head_dim(hq, hkv, head_dim, fused, style):
    """GQA groups of 1 to 128 query heads (16 heads per CTA from 16 on; at head dim 128 groups of
    96 or more on the tcgen05 kernel, one CTA per group), both head dims and RoPE pairings, paged
    blocks of 16, lengths across tiles; split counts 0 and 3."""
    import dataclasses
    lens = [5, 200, 611]
    cfg = dataclasses.replace(CONFIGS["batched_paged"], name=f"heads_{hq}_{hkv}_{head_dim}", batch=len(lens),
                              n_q_heads=hq, n_kv_heads=hkv, head_dim=head_dim, len_range=(min(lens), max(lens)),
                              max_blocks_per_seq=-(-max(lens) // 16), num_blocks=len(lens) * (-(-max(lens) // 16)) + 5,
                              num_splits=0)
    from workloads import gen
    inp = gen.make_inputs(dataclasses.replace(cfg, len_range=(max(lens), max(lens))), seed=9, poison=False)
    inp.lengths[:] = lens
    inp.positions[:] = np.array(lens) - 1
    for b, L in enumerate(lens):
        inp.block_table[b, -(-L // 16):] = -1
    gen.poison_unread(inp)
    for splits in (0, 3):
        gpu = H.run_gpu(inp, num_splits=splits, fused=fused, rope_style=style)
        q_ref, k_ref, _, out_ref = H.run_oracle(inp, rope_style=style)
        assert gpu.err == 0
        _check_step(inp, gpu, q_ref, out_ref)
        _check_cache(inp, gpu, _oracle_k_rows(inp, k_ref))
