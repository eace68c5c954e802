"""Scaled dot-product attention with GQA head sharing, float64.

[KVC-GQA-RoPE] §2.1 and [SelfAttn-Step] §4.1: Attention(Q, K, V) =
softmax(Q K^T / sqrt(d_k)) V, one softmax per query row; in decode the query is
the single new token. [Opt-2026] §三 fixes the default scale at 1/sqrt(d_k).

GQA ([KVC-GQA-RoPE] §2.2, [Opt-2026] §六): n_q query heads share n_kv key/value
heads, n_rep = n_q / n_kv (n_q must be a multiple of n_kv); the KV heads are
expanded with ``repeat_interleave(n_rep)`` along the head axis, so query head h
reads KV head floor(h / n_rep). n_kv = n_q is MHA, n_kv = 1 is MQA.

Causal masking ([KVC-GQA-RoPE] §5.1 b.v, [Opt-2026] §二 masked_fill): query t
sees keys 0..t. In decode this is simply "the L_b tokens in the cache".
"""

from __future__ import annotations

import math

import numpy as np


def repeat_kv(kv: np.ndarray, n_rep: int, axis: int = 0) -> np.ndarray:
    """repeat_interleave along ``axis``: [.., Hkv, ..] -> [.., Hkv * n_rep, ..]."""
    return np.repeat(kv, n_rep, axis=axis)


def softmax(x: np.ndarray, axis: int = -1) -> np.ndarray:
    """Two-pass softmax: subtract the row max, exponentiate, divide by the row sum."""
    m = np.max(x, axis=axis, keepdims=True)
    e = np.exp(x - m)
    return e / np.sum(e, axis=axis, keepdims=True)


def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float | None = None,
              mask: np.ndarray | None = None, return_weights: bool = False):
    """One head: q [Tq, D], k [Tk, D], v [Tk, Dv] -> [Tq, Dv].

    ``mask`` [Tq, Tk] is True where a query may see a key; hidden scores get -inf.
    """
    d = q.shape[-1]
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    scores = (q @ k.T) * scale
    if mask is not None:
        scores = np.where(mask, scores, -np.inf)
    w = softmax(scores, axis=-1)
    out = w @ v
    return (out, w) if return_weights else out


def gqa_decode_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float | None = None) -> np.ndarray:
    """One sequence's decode attention.

    q [Hq, D] (rotated), k and v [Hkv, L, D] (the L cached tokens incl. the new one)
    -> out [Hq, D]. An empty cache (L = 0) gives zeros.
    """
    hq, hkv = q.shape[0], k.shape[0]
    if hq % hkv:
        raise ValueError("n_q_heads must be a multiple of n_kv_heads")
    if k.shape[1] == 0:
        return np.zeros((hq, v.shape[-1]), dtype=np.float64)
    k_all = repeat_kv(k, hq // hkv)
    v_all = repeat_kv(v, hq // hkv)
    out = np.empty((hq, v.shape[-1]), dtype=np.float64)
    for h in range(hq):
        out[h] = attention(q[h][None, :], k_all[h], v_all[h], scale)[0]
    return out


def causal_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float | None = None,
                     return_weights: bool = False):
    """Full-sequence causal GQA attention without any cache.

    q [T, Hq, D], k and v [T, Hkv, D] -> out [T, Hq, D] (and weights [Hq, T, T]).
    """
    t, hq, _ = q.shape
    hkv = k.shape[1]
    k_all = repeat_kv(k, hq // hkv, axis=1)
    v_all = repeat_kv(v, hq // hkv, axis=1)
    mask = np.tril(np.ones((t, t), dtype=bool))
    out = np.empty(q.shape[:2] + (v.shape[-1],), dtype=np.float64)
    weights = np.empty((hq, t, t), dtype=np.float64)
    for h in range(hq):
        o, w = attention(q[:, h], k_all[:, h], v_all[:, h], scale, mask=mask, return_weights=True)
        out[:, h] = o
        weights[h] = w
    return (out, weights) if return_weights else out
