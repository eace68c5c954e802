"""Plant plausible mistakes in the oracle (on the CPU) and check that a pin catches each one."""

import math
import sys

import numpy as np
import pytest

import oracle
from tests import oracle_pins


def _patch_everywhere(monkeypatch, name, new):
    """Replace ``name`` in the oracle package and every oracle submodule that holds it."""
    old = getattr(sys.modules["oracle"], name, None)
    hit = False
    for modname, mod in list(sys.modules.items()):
        if (modname == "oracle" or modname.startswith("oracle.")) and mod is not None:
            if hasattr(mod, name) and (old is None or getattr(mod, name) is old):
                monkeypatch.setattr(mod, name, new)
                hit = True
    assert hit, name


def _rope_sign_flip(x, positions, base=10000.0, style=0):
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    ang = oracle.rope_angles(positions, d, base)
    c, s = np.cos(ang), np.sin(ang)
    out = np.empty_like(x)
    a, b = (x[..., : d // 2], x[..., d // 2:]) if style == 0 else (x[..., 0::2], x[..., 1::2])
    lo, hi = (a * c + b * s), (b * c - a * s)          # rotates the wrong way
    if style == 0:
        out[..., : d // 2], out[..., d // 2:] = lo, hi
    else:
        out[..., 0::2], out[..., 1::2] = lo, hi
    return out


def _rope_swapped_pairing(x, positions, base=10000.0, style=0):
    return _ORIG["apply_rope"](x, positions, base, 1 - style)


def _inv_freq_wrong_exponent(head_dim, base=10000.0):
    return 1.0 / (float(base) ** (np.arange(0, head_dim // 2, dtype=np.float64) / head_dim))


def _repeat_tile(kv, n_rep, axis=0):
    return np.concatenate([kv] * n_rep, axis=axis)


def _attention_no_scale(q, k, v, scale=None, mask=None, return_weights=False):
    return _ORIG["attention"](q, k, v, 1.0, mask, return_weights)


def _softmax_no_max(x, axis=-1):
    e = np.exp(x)
    return e / np.sum(e, axis=axis, keepdims=True)


def _append_contiguous_off_by_one(k_cache, v_cache, k, v, positions):
    return _ORIG["append_contiguous"](k_cache, v_cache, k, v, np.asarray(positions) + 1)


def _logical_kv_paged_reversed(pool, table_row, block_size, length):
    n = math.ceil(length / block_size)
    blocks = [pool[int(table_row[j])] for j in reversed(range(n))]
    return np.transpose(np.concatenate(blocks, axis=0)[:length], (1, 0, 2))


def _kv_bytes_no_factor_two(n_layers, n_kv_heads, head_dim, seq_len, batch, dtype_bytes):
    return n_layers * n_kv_heads * head_dim * seq_len * batch * dtype_bytes


def _bf16_double_rounding(x):
    u = np.asarray(x, dtype=np.float64).astype(np.float32).view(np.uint32)
    return ((u + (np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1)))) >> np.uint32(16)).astype(np.uint16)


def _logical_kv_contiguous_short(cache, b, length):
    return cache[b, :, : max(length - 1, 1), :]


def _q8_half_away_from_zero(x, scale, bits=8):
    r = np.asarray(x, dtype=np.float32) / np.asarray(scale, dtype=np.float32)
    m = (1 << (bits - 1)) - 1
    return np.clip(np.sign(r) * np.floor(np.abs(r) + 0.5), -m, m).astype(np.int8)


def _q8_range_to_minus_128(x, scale, bits=8):
    r = np.asarray(x, dtype=np.float32) / np.asarray(scale, dtype=np.float32)
    m = (1 << (bits - 1)) - 1
    return np.clip(np.rint(r), -m - 1, m).astype(np.int8)


def _q8_quotient_in_float64(x, scale, bits=8):
    r = np.asarray(x, dtype=np.float64) / np.asarray(scale, dtype=np.float32).astype(np.float64)
    m = (1 << (bits - 1)) - 1
    return np.clip(np.rint(r), -m, m).astype(np.int8)


def _q8_ring_slot_shifted(codes, scale, win, b, length, window, block_table=None, block_size=0, bits=8):
    n_old = max(0, length - window) if window > 0 else length
    out = _ORIG_Q["logical_kv_q8"](codes, scale, win, b, n_old, 0, block_table, block_size, bits)
    if n_old == length:
        return out
    recent = np.stack([oracle.bf16_bits_to_f64(win[b, :, (t + 1) % window, :]) for t in range(n_old, length)], axis=1)
    return np.concatenate([out, recent], axis=1)


def _q8_window_one_short(codes, scale, win, b, length, window, block_table=None, block_size=0, bits=8):
    w = max(window - 1, 0) if window > 1 else window
    return _ORIG_Q["logical_kv_q8"](codes, scale, win, b, length, w, block_table, block_size, bits)


def _q4_nibbles_swapped(codes):
    c = np.asarray(codes, dtype=np.int8).astype(np.uint8) & np.uint8(0x0F)
    return (c[..., 1::2] | (c[..., 0::2] << np.uint8(4))).astype(np.uint8)


def _q4_unpack_unsigned(packed):
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (2 * p.shape[-1],), dtype=np.int8)
    out[..., 0::2] = (p & np.uint8(0x0F)).astype(np.int8)
    out[..., 1::2] = (p >> np.uint8(4)).astype(np.int8)
    return out


def _q8_dequantize_without_scale(codes, scale):
    return np.asarray(codes, dtype=np.float64)


def _q8_v_with_k_scale(q, k_new, v_new, positions, k_codes, v_codes, k_scale, v_scale, *args, **kw):
    return _ORIG_Q["rope_append_q8"](q, k_new, v_new, positions, k_codes, v_codes, k_scale, k_scale, *args, **kw)


def _verify_without_chunk_mask(q_rot, k_cache, v_cache, positions, dtype, block_table=None, block_size=0,
                               scale=None, batches=None):
    gamma = q_rot.shape[1]
    outs = []
    for b in range(len(positions)):
        L = int(positions[b]) + gamma
        k = oracle.storage_to_f64(oracle.decode.logical_kv(k_cache, b, L, block_table, block_size), dtype)
        v = oracle.storage_to_f64(oracle.decode.logical_kv(v_cache, b, L, block_table, block_size), dtype)
        outs.append(np.stack([oracle.gqa_decode_attention(oracle.storage_to_f64(q_rot[b, j], dtype), k, v, scale)
                              for j in range(gamma)]))
    return np.stack(outs)


def _verify_rope_at_first_position(q, k_new, v_new, positions, k_cache, v_cache, dtype, block_table=None,
                                   block_size=0, rope_base=10000.0, rope_style=0):
    gamma = q.shape[1]
    pos = np.repeat(np.asarray(positions)[:, None], gamma, axis=1)
    q_rot = oracle.f64_to_storage(oracle.apply_rope(oracle.storage_to_f64(q, dtype), pos[:, :, None], rope_base,
                                                    rope_style), dtype)
    k_rot = oracle.f64_to_storage(oracle.apply_rope(oracle.storage_to_f64(k_new, dtype), pos[:, :, None],
                                                    rope_base, rope_style), dtype)
    for j in range(gamma):
        slot = np.asarray(positions) + j
        if block_table is None:
            oracle.append_contiguous(k_cache, v_cache, k_rot[:, j], v_new[:, j], slot)
        else:
            oracle.append_paged(k_cache, v_cache, block_table, block_size, k_rot[:, j], v_new[:, j], slot)
    return q_rot


_ORIG = {n: getattr(oracle, n) for n in ("apply_rope", "attention", "append_contiguous")}
_ORIG_Q = {n: getattr(oracle.quant, n) for n in ("logical_kv_q8", "rope_append_q8")}

MUTATIONS = {
    "rope rotates the wrong way": ("apply_rope", _rope_sign_flip),
    "rope pairs the wrong dims": ("apply_rope", _rope_swapped_pairing),
    "rope frequency exponent i/d": ("inv_freq", _inv_freq_wrong_exponent),
    "gqa uses tile instead of repeat_interleave": ("repeat_kv", _repeat_tile),
    "attention without 1/sqrt(d)": ("attention", _attention_no_scale),
    "softmax without max subtraction": ("softmax", _softmax_no_max),
    "append one slot late": ("append_contiguous", _append_contiguous_off_by_one),
    "paged gather in reverse block order": ("logical_kv_paged", _logical_kv_paged_reversed),
    "kv bytes without the K+V factor 2": ("kv_cache_bytes", _kv_bytes_no_factor_two),
    "bf16 rounded through fp32": ("f64_to_bf16_bits", _bf16_double_rounding),
    "attention drops the newest token": ("logical_kv_contiguous", _logical_kv_contiguous_short),
    "int8 rounds half away from zero": ("quantize", _q8_half_away_from_zero),
    "int8 codes reach -128": ("quantize", _q8_range_to_minus_128),
    "int8 quotient taken in float64": ("quantize", _q8_quotient_in_float64),
    "int4 nibbles packed in the wrong order": ("pack_int4", _q4_nibbles_swapped),
    "int4 nibbles read as unsigned": ("unpack_int4", _q4_unpack_unsigned),
    "window ring read one slot off": ("logical_kv_q8", _q8_ring_slot_shifted),
    "window one token short": ("logical_kv_q8", _q8_window_one_short),
    "dequantisation drops the scale": ("dequantize_int8", _q8_dequantize_without_scale),
    "v quantised with the k scales": ("rope_append_q8", _q8_v_with_k_scale),
    "verify without the causal mask inside the chunk": ("verify_attention", _verify_without_chunk_mask),
    "verify rotates every new token at the first position": ("rope_append_verify", _verify_rope_at_first_position),
}


@pytest.mark.parametrize("label", list(MUTATIONS))
def test_planted_mistake_is_caught(monkeypatch, label):
    name, bad = MUTATIONS[label]
    _patch_everywhere(monkeypatch, name, bad)
    assert oracle_pins.failing_pins(), f"no pin caught: {label}"


def test_unmutated_oracle_passes_every_pin():
    assert oracle_pins.failing_pins() == []
