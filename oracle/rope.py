"""Rotary position embedding, float64.

[KVC-GQA-RoPE] §3: the frequencies are theta_i = base^(-2(i-1)/d) for
i = 1..d/2 (base 10000), i.e. ``1 / base ** (arange(0, d, 2) / d)``; the angle of
pair i at position m is m * theta_i; q and k are rotated pairwise by those angles,
so (R_m q)^T (R_n k) depends only on the offset n - m.

Pairing. The page names the rotation ``_rotate_half`` and also speaks of
interleaving real and imaginary parts; both pairings are provided:

* style 0, half-split (the default): pair i couples dims (i, i + d/2);
* style 1, interleaved: pair i couples dims (2i, 2i + 1).

Within a pair (a, b) the rotation by angle phi is the complex product
(a + i b) * e^{i phi}: a' = a cos(phi) - b sin(phi), b' = b cos(phi) + a sin(phi).
"""

from __future__ import annotations

import numpy as np


def inv_freq(head_dim: int, base: float = 10000.0) -> np.ndarray:
    """theta_i for the d/2 pairs, float64 [d/2]."""
    if head_dim % 2:
        raise ValueError("head_dim must be even")
    return 1.0 / (float(base) ** (np.arange(0, head_dim, 2, dtype=np.float64) / head_dim))


def rope_angles(positions, head_dim: int, base: float = 10000.0) -> np.ndarray:
    """positions [...] -> angles m * theta_i, float64 [..., d/2]."""
    pos = np.asarray(positions, dtype=np.float64)
    return pos[..., None] * inv_freq(head_dim, base)


def apply_rope(x: np.ndarray, positions, base: float = 10000.0, style: int = 0) -> np.ndarray:
    """Rotate the last axis of ``x`` (length d) at ``positions``.

    ``positions`` broadcasts against ``x.shape[:-1]`` (e.g. [B, 1] for x [B, H, d]).
    Returns a new float64 array.
    """
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    ang = rope_angles(positions, d, base)
    c, s = np.cos(ang), np.sin(ang)
    out = np.empty_like(x)
    if style == 0:
        a, b = x[..., : d // 2], x[..., d // 2:]
        out[..., : d // 2] = a * c - b * s
        out[..., d // 2:] = b * c + a * s
    elif style == 1:
        a, b = x[..., 0::2], x[..., 1::2]
        out[..., 0::2] = a * c - b * s
        out[..., 1::2] = b * c + a * s
    else:
        raise ValueError("rope style must be 0 (half-split) or 1 (interleaved)")
    return out
