"""INT8 KV cache with per-head scales and a bf16 window of recent tokens (test infrastructure).

[KVC-GQA-RoPE] §4.3 (KV-cache quantisation and compression): for very long contexts the
cached K and V are converted from FP16/BF16 to INT8 (or INT4), halving (quartering) the
cache; the conservative choice is INT8 with quantisation parameters calibrated finely, per
layer or even per attention head; some frameworks keep a mixed-precision cache in which the
most recent tokens stay at high precision and older tokens are quantised.

The page gives no formula, so this module takes the plainest reading that fits it:

* symmetric quantisation with one calibrated scale per KV head, separately for K and V
  (``k_scale[Hkv]``, ``v_scale[Hkv]``, positive finite float32): the code of a value x is
  ``clamp(round_half_even(x / s_h), -127, 127)`` and its value is ``code * s_h``; -128 is
  never produced;
* x is the value the bf16 cache would hold (the rotated k rounded to bf16, or v as given),
  and the quotient x / s_h is taken in float32 (IEEE division, nearest even) because it
  decides an integer: both sides of a comparison take that decision in the same precision;
* the high-precision window: W >= 0 recent tokens per sequence are also kept in bf16, in a
  ring of W slots per (sequence, KV head), ``win[B, Hkv, W, D]``, token t in slot t mod W.
  Every appended token is quantised at once (its code goes to cache slot t like a bf16
  cache's value would) AND written to its ring slot. Attention over L tokens reads tokens
  [0, L - W) from the INT8 cache and tokens [max(0, L - W), L) from the ring, so a token is
  read at high precision while it is among the W most recent and quantised afterwards.

INT4, which the passage names as the alternative to INT8, takes the same reading with 4-bit codes: ``clamp(round_half_even(x / s_h), -7, 7)``
(-8 is never produced), two codes per byte, the even dimension in the low nibble and the odd one
in the high nibble, each as a 4-bit two's complement; the caches hold D/2 bytes per token and
head.

Everything else (RoPE, the slot of the new token, paging, GQA, softmax) is the plain
decode step of ``oracle.decode``; attention runs in float64 on the dequantised values.
"""

from __future__ import annotations

import numpy as np

from .attention import gqa_decode_attention
from .bf16 import bf16_bits_to_f64, f64_to_bf16_bits
from .kvcache import append_contiguous, append_paged, logical_kv_contiguous, logical_kv_paged
from .rope import apply_rope

CODE_MAX = 127


def code_max(bits: int) -> int:
    return (1 << (bits - 1)) - 1


def quantize(x, scale, bits: int = 8) -> np.ndarray:
    """Codes of float values x (exactly representable in float32) at per-element scales.

    ``scale`` broadcasts against x. The quotient is formed in float32 (numpy float32
    division is IEEE, nearest even), rounded half to even and clamped to [-(2^(bits-1) - 1),
    2^(bits-1) - 1]. Returns int8 codes (one per element, not packed).
    """
    x32 = np.asarray(x, dtype=np.float32)
    s32 = np.asarray(scale, dtype=np.float32)
    r = x32 / s32
    m = code_max(bits)
    return np.clip(np.rint(r), -m, m).astype(np.int8)


def quantize_int8(x, scale) -> np.ndarray:
    return quantize(x, scale, 8)


def quantize_int4(x, scale) -> np.ndarray:
    return quantize(x, scale, 4)


def pack_int4(codes) -> np.ndarray:
    """int8 codes in [-8, 7], last axis even -> uint8 bytes: code 2i in the low nibble, 2i+1 high."""
    c = np.asarray(codes, dtype=np.int8).astype(np.uint8) & np.uint8(0x0F)
    return (c[..., 0::2] | (c[..., 1::2] << np.uint8(4))).astype(np.uint8)


def unpack_int4(packed) -> np.ndarray:
    """uint8 bytes -> int8 codes (4-bit two's complement nibbles), last axis doubled."""
    p = np.asarray(packed, dtype=np.uint8)
    lo = (p & np.uint8(0x0F)).astype(np.int16)
    hi = (p >> np.uint8(4)).astype(np.int16)
    lo = np.where(lo >= 8, lo - 16, lo)
    hi = np.where(hi >= 8, hi - 16, hi)
    out = np.empty(p.shape[:-1] + (2 * p.shape[-1],), dtype=np.int8)
    out[..., 0::2] = lo
    out[..., 1::2] = hi
    return out


def store_codes(codes, bits: int) -> np.ndarray:
    """The cache representation of codes: int8 as is, INT4 packed two per byte."""
    return np.asarray(codes, dtype=np.int8) if bits == 8 else pack_int4(codes)


def load_codes(stored, bits: int) -> np.ndarray:
    return np.asarray(stored, dtype=np.int8) if bits == 8 else unpack_int4(stored)


def dequantize_int8(codes, scale) -> np.ndarray:
    """code * s in float64 (exact: an 8-bit integer times a float32)."""
    return np.asarray(codes, dtype=np.float64) * np.asarray(scale, dtype=np.float32).astype(np.float64)


def rope_append_q8(q, k_new, v_new, positions, k_codes, v_codes, k_scale, v_scale, k_win, v_win,
                   window: int, block_table=None, block_size: int = 0, rope_base: float = 10000.0,
                   rope_style: int = 0, bits: int = 8):
    """RoPE on bf16 q and k_new at ``positions``; quantise rotated k and raw v into the INT8
    cache slot of the new token and, with a window, write their bf16 values to ring slot
    pos mod W. Caches and rings are updated in place; returns q_rot (bf16 bits).

    q [B, Hq, D], k_new / v_new [B, Hkv, D] are bf16 bit patterns (uint16); the INT8 caches
    are contiguous [B, Hkv, max_len, D] (block_table None) or pools [num_blocks, bs, Hkv, D].
    """
    pos = np.asarray(positions, dtype=np.int64)
    q_rot = f64_to_bf16_bits(apply_rope(bf16_bits_to_f64(q), pos[:, None], rope_base, rope_style))
    k_rot = f64_to_bf16_bits(apply_rope(bf16_bits_to_f64(k_new), pos[:, None], rope_base, rope_style))
    ks = np.asarray(k_scale, dtype=np.float32)[None, :, None]
    vs = np.asarray(v_scale, dtype=np.float32)[None, :, None]
    k_q = store_codes(quantize(bf16_bits_to_f64(k_rot), ks, bits), bits)
    v_q = store_codes(quantize(bf16_bits_to_f64(v_new), vs, bits), bits)
    if block_table is None:
        append_contiguous(k_codes, v_codes, k_q, v_q, pos)
    else:
        append_paged(k_codes, v_codes, block_table, block_size, k_q, v_q, pos)
    if window > 0:
        for b, p in enumerate(pos):
            k_win[b, :, int(p) % window, :] = k_rot[b]
            v_win[b, :, int(p) % window, :] = v_new[b]
    return q_rot


def logical_kv_q8(codes, scale, win, b: int, length: int, window: int, block_table=None,
                  block_size: int = 0, bits: int = 8) -> np.ndarray:
    """Sequence b's first ``length`` tokens of one of K or V as float64 [Hkv, length, D]:
    tokens [0, length - W) dequantised from the INT8 cache, the rest from the bf16 ring."""
    n_old = max(0, length - window) if window > 0 else length
    if block_table is None:
        old_codes = logical_kv_contiguous(codes, b, n_old)
    else:
        old_codes = logical_kv_paged(codes, block_table[b], block_size, n_old) if n_old else \
            np.zeros((codes.shape[2], 0, codes.shape[3]), dtype=codes.dtype)
    old = dequantize_int8(load_codes(old_codes, bits), np.asarray(scale, dtype=np.float32)[:, None, None])
    if n_old == length:
        return old
    recent = np.stack([bf16_bits_to_f64(win[b, :, t % window, :]) for t in range(n_old, length)], axis=1)
    return np.concatenate([old, recent], axis=1)


def decode_attention_q8(q_rot, k_codes, v_codes, k_scale, v_scale, k_win, v_win, seq_lens, window: int,
                        block_table=None, block_size: int = 0, scale=None, batches=None, bits: int = 8) -> np.ndarray:
    """GQA softmax attention of q_rot (bf16 bits) over the mixed-precision cache, float64."""
    seq_lens = np.asarray(seq_lens)
    batches = range(len(seq_lens)) if batches is None else batches
    outs = []
    for b in batches:
        L = int(seq_lens[b])
        k = logical_kv_q8(k_codes, k_scale, k_win, b, L, window, block_table, block_size, bits)
        v = logical_kv_q8(v_codes, v_scale, v_win, b, L, window, block_table, block_size, bits)
        outs.append(gqa_decode_attention(bf16_bits_to_f64(q_rot[b]), k, v, scale))
    return np.stack(outs)


def decode_step_q8(q, k_new, v_new, positions, k_codes, v_codes, k_scale, v_scale, k_win, v_win,
                   window: int, block_table=None, block_size: int = 0, seq_lens=None,
                   rope_base: float = 10000.0, rope_style: int = 0, scale=None, bits: int = 8):
    """RoPE + quantised append + attention on copies of the caches and rings.

    Returns ``(q_rot, k_codes_after, v_codes_after, k_win_after, v_win_after, out)``.
    """
    kc, vc = np.array(k_codes, copy=True), np.array(v_codes, copy=True)
    kw = np.array(k_win, copy=True) if window > 0 else k_win
    vw = np.array(v_win, copy=True) if window > 0 else v_win
    q_rot = rope_append_q8(q, k_new, v_new, positions, kc, vc, k_scale, v_scale, kw, vw, window,
                           block_table, block_size, rope_base, rope_style, bits)
    if seq_lens is None:
        seq_lens = np.asarray(positions) + 1
    out = decode_attention_q8(q_rot, kc, vc, k_scale, v_scale, kw, vw, seq_lens, window, block_table,
                              block_size, scale, bits=bits)
    return q_rot, kc, vc, kw, vw, out
