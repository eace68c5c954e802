"""Multi-query decode: the speculative-verify step (test infrastructure).

[Opt-2026] §五 (speculative decoding): a draft model proposes gamma tokens (gamma = 4 in the
page's class), and the target model checks all of them in one forward pass. For the
attention of that pass on a KV cache, this module takes the plainest reading: the gamma new
tokens of sequence b sit at positions p_b .. p_b + gamma - 1 (their cache slots); each is
rotated at its own position and appended like a decode step's token ([KVC-GQA-RoPE] §3,
§5.1), and query j attends the cached tokens and the new tokens 0..j -- the causal mask
inside the chunk -- i.e. L = p_b + j + 1 tokens, exactly what decoding the tokens one at a
time would give.

q [B, gamma, Hq, D], k_new / v_new [B, gamma, Hkv, D] (storage arrays); positions [B] = p_b.
"""

from __future__ import annotations

import numpy as np

from .attention import gqa_decode_attention
from .bf16 import f64_to_storage, storage_to_f64
from .decode import logical_kv
from .kvcache import append_contiguous, append_paged
from .rope import apply_rope


def rope_append_verify(q, k_new, v_new, positions, k_cache, v_cache, dtype, block_table=None, block_size=0,
                       rope_base: float = 10000.0, rope_style: int = 0):
    """Rotate q[b, j] and k_new[b, j] at p_b + j, append rotated k and raw v at slot p_b + j, in
    place; returns q_rot [B, gamma, Hq, D] (stored)."""
    gamma = q.shape[1]
    pos = np.asarray(positions, dtype=np.int64)[:, None] + np.arange(gamma)[None, :]     # [B, gamma]
    q_rot = f64_to_storage(apply_rope(storage_to_f64(q, dtype), pos[:, :, None], rope_base, rope_style), dtype)
    k_rot = f64_to_storage(apply_rope(storage_to_f64(k_new, dtype), pos[:, :, None], rope_base, rope_style), dtype)
    for j in range(gamma):
        if block_table is None:
            append_contiguous(k_cache, v_cache, k_rot[:, j], v_new[:, j], pos[:, j])
        else:
            append_paged(k_cache, v_cache, block_table, block_size, k_rot[:, j], v_new[:, j], pos[:, j])
    return q_rot


def verify_attention(q_rot, k_cache, v_cache, positions, dtype, block_table=None, block_size=0, scale=None,
                     batches=None) -> np.ndarray:
    """out[b, j] = GQA softmax attention of q_rot[b, j] over tokens [0, p_b + j], float64."""
    gamma = q_rot.shape[1]
    positions = np.asarray(positions)
    batches = range(len(positions)) if batches is None else batches
    outs = []
    for b in batches:
        L = int(positions[b]) + gamma
        k = storage_to_f64(logical_kv(k_cache, b, L, block_table, block_size), dtype)
        v = storage_to_f64(logical_kv(v_cache, b, L, block_table, block_size), dtype)
        rows = []
        for j in range(gamma):
            n = int(positions[b]) + j + 1                    # the causal mask inside the chunk
            rows.append(gqa_decode_attention(storage_to_f64(q_rot[b, j], dtype), k[:, :n], v[:, :n], scale))
        outs.append(np.stack(rows))
    return np.stack(outs)


def verify_step(q, k_new, v_new, positions, k_cache, v_cache, dtype, block_table=None, block_size=0,
                rope_base: float = 10000.0, rope_style: int = 0, scale=None):
    """RoPE + append of the gamma tokens + causal attention, on copies of the caches.

    Returns ``(q_rot, k_cache_after, v_cache_after, out [B, gamma, Hq, D] float64)``.
    """
    kc, vc = np.array(k_cache, copy=True), np.array(v_cache, copy=True)
    q_rot = rope_append_verify(q, k_new, v_new, positions, kc, vc, dtype, block_table, block_size, rope_base,
                               rope_style)
    out = verify_attention(q_rot, kc, vc, positions, dtype, block_table, block_size, scale)
    return q_rot, kc, vc, out
