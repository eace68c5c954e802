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


_ORIG = {n: getattr(oracle, n) for n in ("apply_rope", "attention", "append_contiguous")}

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
}


@pytest.mark.parametrize("label", list(MUTATIONS))
def test_planted_mistake_is_caught(monkeypatch, label):
    name, bad = MUTATIONS[label]
    _patch_everywhere(monkeypatch, name, bad)
    assert oracle_pins.failing_pins(), f"no pin caught: {label}"


def test_unmutated_oracle_passes_every_pin():
    assert oracle_pins.failing_pins() == []
