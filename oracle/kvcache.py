"""KV-cache append and gather, plus the cache-size formula.

Contiguous cache ([SelfAttn-Step] §4.5, [KVC-GQA-RoPE] §2.2): one preallocated
tensor per K and V of shape [batch, kv_heads, max_len, head_dim]; the new token is
written by index at slot ``step`` (= its position) and attention reads slots
[0, step] (``K_cache[:, :, :step+1]``).

Paged cache ([Opt-2026] §四 PagedKVCache, [KVC-GQA-RoPE] §4.1): a pool of
fixed-size blocks of ``block_size`` tokens; each sequence owns a block table listing
physical block ids in logical order, and the logical K/V is the table-ordered
concatenation of those blocks truncated to the sequence length
(``get_kv_for_attention``). The page elides the pool's trailing dims; the reading
used here is one pool per K and V of shape [num_blocks, block_size, kv_heads,
head_dim], i.e. the token-major order of the page's contiguous ``KVCache``
([batch, seq, heads, head_dim]) applied inside each block.

All functions work on whatever array type they are given (the cache keeps its
storage type; callers pass already-rounded values).
"""

from __future__ import annotations

import math

import numpy as np


def append_contiguous(k_cache: np.ndarray, v_cache: np.ndarray, k: np.ndarray, v: np.ndarray,
                      positions) -> None:
    """cache[b, :, pos_b, :] = k[b] / v[b] in place. k, v: [B, Hkv, D]."""
    for b, pos in enumerate(np.asarray(positions)):
        k_cache[b, :, int(pos), :] = k[b]
        v_cache[b, :, int(pos), :] = v[b]


def append_paged(k_pool: np.ndarray, v_pool: np.ndarray, block_table: np.ndarray, block_size: int,
                 k: np.ndarray, v: np.ndarray, positions) -> None:
    """Write token pos_b of sequence b: block = table[b][pos_b // bs], slot = pos_b % bs."""
    for b, pos in enumerate(np.asarray(positions)):
        pos = int(pos)
        phys = int(block_table[b, pos // block_size])
        k_pool[phys, pos % block_size] = k[b]
        v_pool[phys, pos % block_size] = v[b]


def logical_kv_contiguous(cache: np.ndarray, b: int, length: int) -> np.ndarray:
    """[Hkv, length, D] view of sequence b's first ``length`` slots."""
    return cache[b, :, :length, :]


def logical_kv_paged(pool: np.ndarray, table_row: np.ndarray, block_size: int, length: int) -> np.ndarray:
    """Concatenate the sequence's blocks in table order, keep ``length`` tokens -> [Hkv, length, D]."""
    n_blocks = math.ceil(length / block_size)
    blocks = [pool[int(table_row[j])] for j in range(n_blocks)]      # each [bs, Hkv, D]
    tokens = np.concatenate(blocks, axis=0)[:length]                  # [length, Hkv, D]
    return np.transpose(tokens, (1, 0, 2))


def kv_cache_bytes(n_layers: int, n_kv_heads: int, head_dim: int, seq_len: int, batch: int,
                   dtype_bytes: int) -> int:
    """Bytes of a K+V cache: 2 x layers x kv_heads x head_dim x seq_len x batch x bytes.

    [Opt-2026] §四 (memory formula, with n_heads read as the KV heads, which is
    what §六's MHA/GQA/MQA comparison varies) and [KVC-GQA-RoPE] §5.3.
    """
    return 2 * int(n_layers) * int(n_kv_heads) * int(head_dim) * int(seq_len) * int(batch) * int(dtype_bytes)
