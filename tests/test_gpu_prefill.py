"""Prefill (causal attention of a prompt, or of a chunk after a cached prefix) against the float64 oracle.

The oracle is the speculative-verify definition with gamma = T new tokens (each prompt token
rotated at its position, appended, and attending tokens [0, p_b + t]). Bars as for the decode
step: q_rot and appended K within 1 bf16 ulp, appended V and every other cache byte bit-exact,
output max abs error <= 1e-2.
"""

import numpy as np
import pytest

import oracle
from tests import gpu_harness as H
from workloads import CONFIGS, WorkloadConfig, make_inputs, reduced
from workloads.gen import poison_unread

pytestmark = pytest.mark.gpu


def _inputs(cfg, seed):
    inp = make_inputs(cfg, seed=seed)
    if cfg.gamma == 1:                       # the generator keeps decode shapes for one new token
        inp.q, inp.k_new, inp.v_new = inp.q[:, None], inp.k_new[:, None], inp.v_new[:, None]
    return inp


def _check(inp, gpu, rope_style=0):
    cfg = inp.cfg
    q_ref, k_ref, v_ref, out_ref = H.run_oracle_verify(inp, rope_style=rope_style)
    assert gpu.err == 0
    H.assert_close_stored(gpu.q_rot, q_ref, "bf16", "q_rot")
    err = H.out_error(gpu.out, out_ref, "bf16")
    assert err <= H.OUT_ATOL["bf16"], f"{cfg.name}: out max abs err {err:.3e}"
    rel = H.rel_rms_error(gpu.out, out_ref, "bf16")
    assert rel <= H.REL_RMS_BAR, f"{cfg.name}: out error {rel:.3e} of the row RMS"
    H.assert_close_stored(gpu.k_cache, k_ref, "bf16", "K cache")
    assert gpu.v_cache.tobytes() == v_ref.tobytes(), "V cache"
    return err


@pytest.mark.parametrize("fused", [False, True], ids=["two_calls", "prefill_step"])
def test_prefill_reduced_8k(fused):
    inp = make_inputs(reduced(CONFIGS["prefill_8k"], 16))
    _check(inp, H.run_gpu_prefill(inp, fused=fused))


def _cfg(layout, prefix, T, batch=2, block_size=16, head_dim=128, hq=32, hkv=8):
    L = prefix + T
    kw = dict(name=f"prefill_{layout}", batch=batch, n_q_heads=hq, n_kv_heads=hkv, head_dim=head_dim, dtype="bf16",
              layout=layout, seq_len=L, gamma=T)
    if layout == "contiguous":
        kw["max_len"] = max(L + 7, 16384 // (2 * head_dim))
    else:
        kw.update(block_size=block_size, max_blocks_per_seq=-(-L // block_size))
        kw["num_blocks"] = batch * kw["max_blocks_per_seq"] + 5
    return WorkloadConfig(**kw)


@pytest.mark.parametrize("layout,block_size", [("contiguous", 0), ("paged", 8), ("paged", 16), ("paged", 256)])
@pytest.mark.parametrize("prefix,T", [(0, 1), (0, 2), (0, 17), (0, 64), (0, 65), (0, 257), (0, 300), (37, 5),
                                      (100, 130), (200, 200), (1000, 64)])
def test_prefill_lengths_and_prefix(layout, block_size, prefix, T):
    inp = _inputs(_cfg(layout, prefix, T, block_size=block_size or 16), seed=prefix + T)
    _check(inp, H.run_gpu_prefill(inp))


@pytest.mark.parametrize("hq,hkv", [(8, 8), (32, 1), (12, 4), (64, 4)], ids=["mha", "mqa", "nrep3", "nrep16"])
@pytest.mark.parametrize("head_dim", [64, 128])
def test_prefill_heads_and_head_dim(hq, hkv, head_dim):
    style = 1 if head_dim == 64 else 0
    inp = _inputs(_cfg("paged", 20, 150, head_dim=head_dim, hq=hq, hkv=hkv), seed=3)
    _check(inp, H.run_gpu_prefill(inp, rope_style=style), rope_style=style)


def test_prefill_position_errors_are_flagged():
    from rope_gqa_paged_gb300 import RRA_ERR_POSITION
    inp = _inputs(_cfg("paged", 0, 40), seed=1)
    inp.positions = np.array([0, 10], dtype=np.int32)                  # the second prompt runs past the cache
    gpu = H.run_gpu_prefill(inp)
    assert gpu.err & RRA_ERR_POSITION


def _check_sampled_rows(inp, gpu, rows):
    """Every output value written (the harness starts from NaN), and the given prompt rows (one
    sequence, prompt from position 0) checked one by one against the oracle's definition."""
    assert gpu.err == 0
    bits = np.asarray(gpu.out).view(np.uint16)
    nan = ((bits & 0x7F80) == 0x7F80) & ((bits & 0x007F) != 0)
    assert not nan.any(), f"{int(nan.sum())} output values never written"
    T = inp.cfg.gamma
    pos = np.arange(T)
    k_rot = oracle.f64_to_bf16_bits(oracle.apply_rope(oracle.bf16_bits_to_f64(inp.k_new[0]), pos[:, None]))
    kf = oracle.bf16_bits_to_f64(k_rot)                           # [T, Hkv, D]
    vf = oracle.bf16_bits_to_f64(inp.v_new[0])
    for t in rows:
        q_rot = oracle.f64_to_bf16_bits(oracle.apply_rope(oracle.bf16_bits_to_f64(inp.q[0, t]), np.array([t])))
        H.assert_close_stored(gpu.q_rot[0, t], q_rot, "bf16", f"q_rot {t}")
        want = oracle.gqa_decode_attention(oracle.bf16_bits_to_f64(q_rot), np.transpose(kf[: t + 1], (1, 0, 2)),
                                           np.transpose(vf[: t + 1], (1, 0, 2)))
        e = H.out_error(gpu.out[0, t], want, "bf16")
        assert e <= H.OUT_ATOL["bf16"], (t, e)
        rel = H.rel_rms_error(gpu.out[0, t], want, "bf16")
        assert rel <= H.REL_RMS_BAR, (t, rel)


@pytest.mark.slow
def test_prefill_128k_sampled_rows():
    """The full 128K prompt (its CTAs run in bands of one KV head: 64 MB of K and V each)."""
    cfg = CONFIGS["prefill_128k"]
    inp = make_inputs(cfg)
    _check_sampled_rows(inp, H.run_gpu_prefill(inp), (0, 1, 63, 4095, 70001, cfg.gamma - 1))


@pytest.mark.parametrize("head_dim", [64, 128])
def test_prefill_40k_bands_sampled_rows(head_dim):
    """A 40000-token prompt: its CTAs run in bands of 4 (D 64) or 2 (D 128) of the 8 KV heads,
    the bands whose K and V fit in 64 MB; rows of the first and last query blocks and between."""
    T = 40000
    inp = _inputs(_cfg("paged", 0, T, batch=1, block_size=32, head_dim=head_dim), seed=40)
    rows = (0, 5, 127, 128, 20011, 39871, T - 1)
    _check_sampled_rows(inp, H.run_gpu_prefill(inp), rows)
