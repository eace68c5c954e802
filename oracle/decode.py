"""The whole decode step on stored (bf16 or fp32) tensors.

[KVC-GQA-RoPE] §5.1 b.ii-vi gives the per-layer order: rotate q and k at the
token's absolute position, write the new k and v at the end of the cache, expand
the KV heads to the query heads, scale the scores by 1/sqrt(d_k), softmax, weight V.
[SelfAttn-Step] §4.5 gives the same step on a preallocated cache: write slot
``step``, attend over slots [0, step]. [KVC-GQA-RoPE] §3: the cache holds the
*rotated* K of past tokens, so only the new token is rotated; V is never rotated.

Storage: q_rot, the cached k and v and the output live in the storage type
(``dtype``: 'bf16' as uint16 bits, or 'f32'); the oracle rounds each stored value
from float64 directly (nearest even) and computes attention in float64 on the
stored values. The attention output is returned unrounded, in float64.
"""

from __future__ import annotations

import numpy as np

from .attention import gqa_decode_attention
from .bf16 import f64_to_storage, storage_to_f64
from .kvcache import append_contiguous, append_paged, logical_kv_contiguous, logical_kv_paged
from .rope import apply_rope


def rope_append(q, k_new, v_new, positions, k_cache, v_cache, dtype, block_table=None, block_size=0,
                rope_base: float = 10000.0, rope_style: int = 0):
    """Rotate q and k_new at ``positions``, append rotated k and raw v in place; return q_rot (stored)."""
    pos = np.asarray(positions, dtype=np.int64)[:, None]
    q_rot = f64_to_storage(apply_rope(storage_to_f64(q, dtype), pos, rope_base, rope_style), dtype)
    k_rot = f64_to_storage(apply_rope(storage_to_f64(k_new, dtype), pos, rope_base, rope_style), dtype)
    if block_table is None:
        append_contiguous(k_cache, v_cache, k_rot, v_new, positions)
    else:
        append_paged(k_cache, v_cache, block_table, block_size, k_rot, v_new, positions)
    return q_rot


def logical_kv(cache, b, length, block_table=None, block_size=0):
    if block_table is None:
        return logical_kv_contiguous(cache, b, length)
    return logical_kv_paged(cache, block_table[b], block_size, length)


def decode_attention(q_rot, k_cache, v_cache, seq_lens, dtype, block_table=None, block_size=0,
                     scale=None, batches=None) -> np.ndarray:
    """out[b] = GQA softmax attention of q_rot[b] over the first L_b logical tokens, float64.

    ``batches`` limits the work to some sequences (rows of the result follow it).
    """
    seq_lens = np.asarray(seq_lens)
    batches = range(len(seq_lens)) if batches is None else batches
    outs = []
    for b in batches:
        L = int(seq_lens[b])
        k = storage_to_f64(logical_kv(k_cache, b, L, block_table, block_size), dtype)
        v = storage_to_f64(logical_kv(v_cache, b, L, block_table, block_size), dtype)
        outs.append(gqa_decode_attention(storage_to_f64(q_rot[b], dtype), k, v, scale))
    return np.stack(outs)


def decode_step(q, k_new, v_new, positions, k_cache, v_cache, dtype, block_table=None, block_size=0,
                seq_lens=None, rope_base: float = 10000.0, rope_style: int = 0, scale=None):
    """RoPE + append + attention on copies of the caches.

    Returns ``(q_rot, k_cache_after, v_cache_after, out)``; ``seq_lens`` defaults
    to positions + 1 (the new token attends to itself).
    """
    kc, vc = np.array(k_cache, copy=True), np.array(v_cache, copy=True)
    q_rot = rope_append(q, k_new, v_new, positions, kc, vc, dtype, block_table, block_size,
                        rope_base, rope_style)
    if seq_lens is None:
        seq_lens = np.asarray(positions) + 1
    out = decode_attention(q_rot, kc, vc, seq_lens, dtype, block_table, block_size, scale)
    return q_rot, kc, vc, out
