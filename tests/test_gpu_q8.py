"""INT8 / INT4 KV cache with per-head scales and a bf16 window: CUDA path against the float64 oracle.

Bars (same inputs on both sides): q_rot and the ring's k within 1 bf16 ulp; the ring's v and
every V code bit-exact; a K code equal to the quantisation of the GPU's own bf16 k wherever
that value is visible (window > 0) and never more than one code from the oracle's; every cache
and ring slot the step does not write unchanged; attention output max abs error <= 1e-2
against the oracle's float64 result over the dequantised cache.
"""

import dataclasses

import numpy as np
import pytest

import oracle
from tests import gpu_harness as H
from workloads import CONFIGS, WorkloadConfig, make_inputs, reduced

pytestmark = pytest.mark.gpu


def _slot(inp, b, pos):
    """Index of token pos of sequence b in the code cache (contiguous or pool)."""
    cfg = inp.cfg
    if inp.block_table is None:
        return (b, slice(None), pos)
    return (inp.block_table[b, pos // cfg.block_size], pos % cfg.block_size)


def _check_q8(inp, gpu, ref, fused_or_append=True, out_batches=None):
    cfg = inp.cfg
    q_ref, kc_ref, vc_ref, kw_ref, vw_ref, out_ref = ref
    bits = cfg.code_bits
    H.assert_close_stored(gpu.q_rot, q_ref, "bf16", "q_rot")
    bs = range(cfg.batch) if out_batches is None else out_batches
    err = H.out_error(gpu.out[list(bs)], out_ref[list(bs)], "bf16")
    assert err <= H.OUT_ATOL["bf16"], f"{cfg.name}: out max abs err {err:.3e}"
    rel = H.rel_rms_error(gpu.out[list(bs)], out_ref[list(bs)], "bf16")
    assert rel <= H.REL_RMS_BAR, f"{cfg.name}: out error {rel:.3e} of the row RMS"
    kc, vc = gpu.k_codes.copy(), gpu.v_codes.copy()
    W = cfg.window
    kw = gpu.k_win.copy() if W else None
    vw = gpu.v_win.copy() if W else None
    for b in range(cfg.batch):
        pos = int(inp.positions[b])
        idx = _slot(inp, b, pos)
        # V codes: the quantisation of an input value, bit-exact
        assert vc[idx].tobytes() == vc_ref[idx].tobytes(), f"V codes of sequence {b}"
        kd = np.abs(oracle.quant.load_codes(kc[idx], bits).astype(int) -
                    oracle.quant.load_codes(kc_ref[idx], bits).astype(int))
        assert kd.max() <= 1, f"K codes of sequence {b} differ by {kd.max()}"
        if W:
            s = pos % W
            H.assert_close_stored(kw[b, :, s], kw_ref[b, :, s], "bf16", f"ring k of sequence {b}")
            assert vw[b, :, s].tobytes() == vw_ref[b, :, s].tobytes(), f"ring v of sequence {b}"
            # the code is the quantisation of the GPU's own bf16 k, decided in float32
            mine = oracle.quant.store_codes(
                oracle.quant.quantize(oracle.bf16_bits_to_f64(kw[b, :, s]), inp.k_scale[:, None], bits), bits)
            assert np.array_equal(kc[idx], mine), f"K codes of sequence {b} vs its ring value"
            kw[b, :, s], vw[b, :, s] = inp.k_win[b, :, s], inp.v_win[b, :, s]
        else:
            assert (kd > 0).mean() < 0.01
        kc[idx], vc[idx] = inp.k_cache[idx], inp.v_cache[idx]
    assert kc.tobytes() == inp.k_cache.tobytes(), "K codes changed outside the appended slots"
    assert vc.tobytes() == inp.v_cache.tobytes(), "V codes changed outside the appended slots"
    if W:
        assert kw.tobytes() == inp.k_win.tobytes() and vw.tobytes() == inp.v_win.tobytes(), "ring changed elsewhere"
    return err


REDUCED = [("batched_paged_int8", 16, 8), ("long_context_int8", 64, 1), ("batched_paged_int4", 16, 8),
           ("long_context_int4", 64, 1)]


@pytest.mark.parametrize("name,factor,batch", REDUCED, ids=[r[0] for r in REDUCED])
@pytest.mark.parametrize("window", [None, 0], ids=["window", "no_window"])
@pytest.mark.parametrize("splits", [0, 3])
@pytest.mark.parametrize("fused", [False, True], ids=["two_calls", "fused_step"])
def test_q8_reduced_workload(name, factor, batch, window, splits, fused):
    cfg = reduced(CONFIGS[name], factor, batch)
    if window is not None:
        cfg = dataclasses.replace(cfg, window=window)
    inp = make_inputs(cfg)
    gpu = H.run_gpu_q8(inp, num_splits=splits, fused=fused)
    assert gpu.err == 0
    _check_q8(inp, gpu, H.run_oracle_q8(inp))


def _edge_cfg(layout, lengths, window, block_size=16, head_dim=128, hq=8, hkv=2, max_len=None, bits=8):
    lengths = list(lengths)
    longest = max(lengths)
    kw = dict(name=f"q{bits}_edge_{layout}", batch=len(lengths), n_q_heads=hq, n_kv_heads=hkv, head_dim=head_dim,
              dtype="bf16", layout=layout, len_range=(min(lengths), longest), kv_dtype=f"int{bits}", window=window)
    if layout == "contiguous":
        kw["max_len"] = max_len or max(longest, 8192 // (head_dim * bits // 8))
    else:
        kw.update(block_size=block_size, max_blocks_per_seq=-(-longest // block_size))
        kw["num_blocks"] = len(lengths) * kw["max_blocks_per_seq"] + 5
    return WorkloadConfig(**kw)


def _with_lengths(cfg, lengths, seed=3):
    """make_inputs with the drawn lengths replaced by ``lengths`` (tables drawn for the maxima)."""
    inp = make_inputs(dataclasses.replace(cfg, len_range=(max(lengths), max(lengths))), seed=seed, poison=False)
    inp.lengths = np.asarray(lengths, dtype=np.int32)
    inp.positions = inp.lengths - 1
    if inp.block_table is not None:
        for b, L in enumerate(lengths):
            inp.block_table[b, -(-L // cfg.block_size):] = -1
    from workloads.gen import poison_unread
    poison_unread(inp)
    return inp


EDGE_LENGTHS = [1, 2, 15, 16, 17, 31, 32, 33, 127, 128, 129, 300]


@pytest.mark.parametrize("layout,block_size", [("contiguous", 0), ("paged", 8), ("paged", 16), ("paged", 32),
                                               ("paged", 256)])
@pytest.mark.parametrize("window", [0, 16, 32])
@pytest.mark.parametrize("fused", [False, True], ids=["two_calls", "fused_step"])
@pytest.mark.parametrize("bits", [8, 4], ids=["int8", "int4"])
def test_q8_edge_lengths(layout, block_size, window, fused, bits):
    cfg = _edge_cfg(layout, EDGE_LENGTHS, window, block_size=block_size or 16, bits=bits)
    inp = _with_lengths(cfg, EDGE_LENGTHS)
    for splits in (0, 2):
        gpu = H.run_gpu_q8(inp, num_splits=splits, fused=fused)
        assert gpu.err == 0
        _check_q8(inp, gpu, H.run_oracle_q8(inp))


@pytest.mark.parametrize("hq,hkv", [(8, 8), (32, 1), (12, 4), (64, 4)], ids=["mha", "mqa", "nrep3", "nrep16"])
@pytest.mark.parametrize("head_dim,bits", [(64, 8), (128, 8), (128, 4)], ids=["d64_int8", "d128_int8", "d128_int4"])
@pytest.mark.parametrize("fused", [False, True], ids=["two_calls", "fused_step"])
def test_q8_heads_and_head_dim(hq, hkv, head_dim, bits, fused):
    lengths = [5, 200, 611]
    cfg = _edge_cfg("paged", lengths, 16, block_size=16, head_dim=head_dim, hq=hq, hkv=hkv, bits=bits)
    inp = _with_lengths(cfg, lengths, seed=7)
    gpu = H.run_gpu_q8(inp, num_splits=3, fused=fused, rope_style=1 if head_dim == 64 else 0)
    assert gpu.err == 0
    _check_q8(inp, gpu, H.run_oracle_q8(inp, rope_style=1 if head_dim == 64 else 0))


@pytest.mark.parametrize("splits", [17, 40])
@pytest.mark.parametrize("fused", [False, True], ids=["two_calls", "fused_step"])
@pytest.mark.parametrize("bits", [8, 4], ids=["int8", "int4"])
def test_q8_many_splits_merge(splits, fused, bits):
    lengths = [4100, 2500]
    cfg = _edge_cfg("paged", lengths, 64, block_size=32, bits=bits)
    inp = _with_lengths(cfg, lengths, seed=11)
    gpu = H.run_gpu_q8(inp, num_splits=splits, fused=fused)
    assert gpu.err == 0 and gpu.splits > 16
    _check_q8(inp, gpu, H.run_oracle_q8(inp))


@pytest.mark.parametrize("bits", [8, 4], ids=["int8", "int4"])
def test_q8_position_errors_are_flagged(bits):
    from rope_gqa_paged_gb300 import RRA_ERR_POSITION
    lengths = [40, 60]
    cfg = _edge_cfg("paged", lengths, 16, bits=bits)
    inp = _with_lengths(cfg, lengths)
    inp.positions = np.array([39, cfg.capacity], dtype=np.int32)      # second one is past the cache
    gpu = H.run_gpu_q8(inp, fused=True)
    assert gpu.err & RRA_ERR_POSITION


@pytest.mark.slow
def test_q8_full_size_sampled():
    """The full batch-64 INT8 workload in the bench's configuration; a few sequences checked."""
    cfg = CONFIGS["batched_paged_int8"]
    inp = make_inputs(cfg)
    gpu = H.run_gpu_q8(inp, fused=True)
    assert gpu.err == 0
    batches = [0, 17, 40, 63]
    bs = cfg.block_size
    for b in batches:
        L = int(inp.lengths[b])
        kc = oracle.logical_kv_paged(inp.k_cache, inp.block_table[b], bs, L)[None].copy()   # [1, Hkv, L, D]
        vc = oracle.logical_kv_paged(inp.v_cache, inp.block_table[b], bs, L)[None].copy()
        kw = inp.k_win[b:b + 1].copy()
        vw = inp.v_win[b:b + 1].copy()
        q_rot = oracle.quant.rope_append_q8(inp.q[b:b + 1], inp.k_new[b:b + 1], inp.v_new[b:b + 1],
                                            inp.positions[b:b + 1], kc, vc, inp.k_scale, inp.v_scale, kw, vw,
                                            cfg.window)
        out = oracle.quant.decode_attention_q8(q_rot, kc, vc, inp.k_scale, inp.v_scale, kw, vw, np.array([L]),
                                               cfg.window)
        H.assert_close_stored(gpu.q_rot[b], q_rot[0], "bf16", f"q_rot {b}")
        e = H.out_error(gpu.out[b], out[0], "bf16")
        assert e <= H.OUT_ATOL["bf16"], (b, e)
