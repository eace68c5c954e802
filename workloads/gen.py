"""Seeded synthetic decode-step inputs.

Recipe (one numpy ``Generator(PCG64(seed))`` per workload, draws in this order):

1. attended lengths L_b: the fixed ``seq_len``, else ``integers(lo, hi, endpoint=True, size=B)``;
2. paged only: ``permutation(num_blocks)`` is the free list; shared-prefix blocks are
   popped from its end first, then sequences b = 0..B-1 pop ``ceil(L_b / bs)`` ids each
   (prefix blocks excluded) in logical order; unused table entries are -1;
3. q [B, Hq, D], then k_new [B, Hkv, D], then v_new [B, Hkv, D];
4. the whole K cache, then the whole V cache (contiguous [B, Hkv, max_len, D] or
   pool [num_blocks, bs, Hkv, D]), drawn in chunks of 2**24 values.

Values are ``standard_normal(dtype=float32)`` rounded to the storage type (bf16 by
round-to-nearest-even on the float32 bits; fp32 unchanged). The cache is read as
already-rotated K (a rotation keeps iid N(0,1) vectors iid N(0,1)).

Poisoning: every cache slot the step must not read before the append is NaN: in
the contiguous cache the slots t >= L_b - 1 of sequence b; in the pools every block
no table references, and in each sequence's last block the slots at positions
>= L_b - 1. Position L_b - 1 is where the new token goes, so a missing append or an
out-of-range read shows up as NaN in the output.

bf16 arrays are carried as ``uint16`` bit patterns, fp32 as ``float32``.

Speculative verify (``gamma > 1``): q, k_new, v_new are drawn as [B, gamma, H, D]; the gamma new
tokens of sequence b sit at positions L_b - gamma .. L_b - 1 (``positions`` holds the first),
and every slot from L_b - gamma on is poisoned.

INT4 caches (``kv_dtype == "int4"``): as INT8 with codes ``clip(rint(1.75 * N(0,1)), -7, 7)``
packed two per byte (even dimension in the low nibble), scales (1 + (h mod 4)/8)/1.75 and
(1 + ((h+2) mod 4)/8)/1.75, and the poison byte 0x88 (two -8 codes, which quantisation never
produces).

INT8 caches (``kv_dtype == "int8"``): steps 1-3 are unchanged; step 4 draws the K then the V
cache as integer codes ``clip(rint(32 * standard_normal(float32)), -127, 127)`` (N(0,1)
values at a resolution of 1/32), then, with a window of W slots, the K then the V ring
[B, Hkv, W, D] as bf16 N(0,1). The per-head scales are fixed, not drawn:
k_scale[h] = (1 + (h % 4) / 8) / 32 and v_scale[h] = (1 + ((h + 2) % 4) / 8) / 32 (float32).
Poisoning: -128 (a code quantisation never produces) in every cache slot the step must not
read -- slots t >= max(0, L_b - max(W, 1)), i.e. the new token's slot and every slot the
window covers -- and in every unreferenced block; NaN in the ring slot the new token will
overwrite ((L_b - 1) mod W) and, while L_b - 1 < W, in the ring slots not yet filled.
"""

from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

from .configs import WorkloadConfig

_CHUNK = 1 << 24
BF16_NAN = np.uint16(0x7FC0)


def bf16_bits_from_f32(x: np.ndarray) -> np.ndarray:
    """Round finite float32 values to bf16 (nearest, ties to even); returns uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = (u + (np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1)))) >> np.uint32(16)
    return r.astype(np.uint16)


def _normal_storage(rng: np.random.Generator, shape, dtype: str) -> np.ndarray:
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16 if dtype == "bf16" else np.float32)
    for s in range(0, n, _CHUNK):
        e = min(n, s + _CHUNK)
        x = rng.standard_normal(e - s, dtype=np.float32)
        out[s:e] = bf16_bits_from_f32(x) if dtype == "bf16" else x
    return out.reshape(shape)


@dataclasses.dataclass
class DecodeInputs:
    cfg: WorkloadConfig
    lengths: np.ndarray            # int32 [B], attended lengths incl. the new token
    positions: np.ndarray          # int32 [B], = lengths - gamma (position and slot of the (first) new token)
    q: np.ndarray                  # [B, Hq, D]  ([B, gamma, Hq, D] when gamma > 1)
    k_new: np.ndarray              # [B, Hkv, D] ([B, gamma, Hkv, D] when gamma > 1)
    v_new: np.ndarray              # [B, Hkv, D] ([B, gamma, Hkv, D] when gamma > 1)
    k_cache: np.ndarray            # contiguous [B, Hkv, max_len, D] or pool [num_blocks, bs, Hkv, D]
    v_cache: np.ndarray
    block_table: Optional[np.ndarray] = None   # int32 [B, max_blocks_per_seq], paged only
    k_scale: Optional[np.ndarray] = None       # int8 only: float32 [Hkv]
    v_scale: Optional[np.ndarray] = None
    k_win: Optional[np.ndarray] = None         # int8 with a window: bf16 ring [B, Hkv, W, D]
    v_win: Optional[np.ndarray] = None

    @property
    def nan_value(self):
        if self.cfg.kv_dtype == "int4":
            return np.uint8(0x88)
        if self.cfg.int8:
            return np.int8(-128)
        return BF16_NAN if self.cfg.dtype == "bf16" else np.float32(np.nan)


def draw_lengths(cfg: WorkloadConfig, rng: np.random.Generator) -> np.ndarray:
    if cfg.seq_len is not None:
        lengths = np.full(cfg.batch, cfg.seq_len, dtype=np.int64)
    else:
        lo, hi = cfg.len_range
        lengths = rng.integers(lo, hi, endpoint=True, size=cfg.batch)
    if np.any(lengths > cfg.capacity) or np.any(lengths < cfg.gamma):
        raise ValueError(f"{cfg.name}: lengths outside [{cfg.gamma}, {cfg.capacity}]")
    return lengths.astype(np.int32)


def draw_block_table(cfg: WorkloadConfig, lengths: np.ndarray, rng: np.random.Generator) -> np.ndarray:
    bs = cfg.block_size
    free = list(rng.permutation(cfg.num_blocks))
    n_shared = cfg.shared_prefix_tokens // bs
    if cfg.shared_prefix_tokens % bs:
        raise ValueError("shared prefix must be a whole number of blocks")
    if n_shared and int(lengths.min()) - 1 < cfg.shared_prefix_tokens:
        raise ValueError("the new token's slot must lie past the shared prefix")
    shared = [free.pop() for _ in range(n_shared)]
    table = np.full((cfg.batch, cfg.max_blocks_per_seq), -1, dtype=np.int32)
    for b in range(cfg.batch):
        nb = math.ceil(int(lengths[b]) / bs)
        table[b, :n_shared] = shared
        for j in range(n_shared, nb):
            if not free:
                raise ValueError(f"{cfg.name}: pool of {cfg.num_blocks} blocks exhausted")
            table[b, j] = free.pop()
    return table


def make_inputs(cfg: WorkloadConfig, seed: Optional[int] = None, poison: bool = True) -> DecodeInputs:
    rng = np.random.Generator(np.random.PCG64(cfg.seed if seed is None else seed))
    B, Hq, Hkv, D = cfg.batch, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim
    lengths = draw_lengths(cfg, rng)
    table = draw_block_table(cfg, lengths, rng) if cfg.layout == "paged" else None
    lead = (B,) if cfg.gamma == 1 else (B, cfg.gamma)
    q = _normal_storage(rng, lead + (Hq, D), cfg.dtype)
    k_new = _normal_storage(rng, lead + (Hkv, D), cfg.dtype)
    v_new = _normal_storage(rng, lead + (Hkv, D), cfg.dtype)
    if cfg.layout == "contiguous":
        shape = (B, Hkv, cfg.max_len, D)
    else:
        shape = (cfg.num_blocks, cfg.block_size, Hkv, D)
    extra = {}
    if cfg.int8:
        per_unit = 32.0 if cfg.code_bits == 8 else 1.75      # codes per unit of N(0,1)
        k_cache = _codes(rng, shape, cfg.code_bits, per_unit)
        v_cache = _codes(rng, shape, cfg.code_bits, per_unit)
        h = np.arange(Hkv)
        extra["k_scale"] = ((1.0 + (h % 4) / 8.0) / per_unit).astype(np.float32)
        extra["v_scale"] = ((1.0 + ((h + 2) % 4) / 8.0) / per_unit).astype(np.float32)
        if cfg.window:
            extra["k_win"] = _normal_storage(rng, (B, Hkv, cfg.window, D), "bf16")
            extra["v_win"] = _normal_storage(rng, (B, Hkv, cfg.window, D), "bf16")
    else:
        k_cache = _normal_storage(rng, shape, cfg.dtype)
        v_cache = _normal_storage(rng, shape, cfg.dtype)
    inp = DecodeInputs(cfg=cfg, lengths=lengths, positions=(lengths - cfg.gamma).astype(np.int32),
                       q=q, k_new=k_new, v_new=v_new, k_cache=k_cache, v_cache=v_cache,
                       block_table=table, **extra)
    if poison:
        poison_unread(inp)
    return inp


def _codes(rng: np.random.Generator, shape, bits: int, per_unit: float) -> np.ndarray:
    """Integer codes clip(rint(per_unit * N(0,1)), -(2^(bits-1) - 1), ...): int8, or for 4 bits
    packed two per byte (even index in the low nibble) along the last axis."""
    m = (1 << (bits - 1)) - 1
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.int8)
    for s in range(0, n, _CHUNK):
        e = min(n, s + _CHUNK)
        x = rng.standard_normal(e - s, dtype=np.float32)
        out[s:e] = np.clip(np.rint(x * per_unit), -m, m)
    out = out.reshape(shape)
    if bits == 8:
        return out
    u = out.astype(np.uint8) & np.uint8(0x0F)
    return (u[..., 0::2] | (u[..., 1::2] << np.uint8(4))).astype(np.uint8)


def make_structure(cfg: WorkloadConfig, seed: Optional[int] = None):
    """Only the first two draws of the recipe: (lengths, block_table or None).

    Same values as ``make_inputs`` gives for the same seed; used where the large cache
    arrays are filled elsewhere (the benchmark fills them on the device).
    """
    rng = np.random.Generator(np.random.PCG64(cfg.seed if seed is None else seed))
    lengths = draw_lengths(cfg, rng)
    table = draw_block_table(cfg, lengths, rng) if cfg.layout == "paged" else None
    return lengths, table


def poison_unread(inp: DecodeInputs) -> None:
    """Write NaN (INT8: -128) into every cache slot the step must not read before its append."""
    cfg, nan = inp.cfg, inp.nan_value
    # first slot not read from the main cache: the new token's, or the window's first
    first = [max(0, int(L) - max(cfg.window, 1)) if cfg.int8 else int(L) - cfg.gamma for L in inp.lengths]
    if cfg.int8 and cfg.window:
        W = cfg.window
        for b, L in enumerate(inp.lengths):
            for ring in (inp.k_win, inp.v_win):
                ring[b, :, (int(L) - 1) % W, :] = BF16_NAN
                if int(L) - 1 < W:
                    ring[b, :, int(L) - 1:, :] = BF16_NAN
    if cfg.layout == "contiguous":
        for b, L in enumerate(inp.lengths):
            inp.k_cache[b, :, first[b]:, :] = nan
            inp.v_cache[b, :, first[b]:, :] = nan
        return
    bs = cfg.block_size
    used = np.zeros(cfg.num_blocks, dtype=bool)
    for b, L in enumerate(inp.lengths):
        nb = math.ceil(int(L) / bs)
        used[inp.block_table[b, :nb]] = True
        n_shared = cfg.shared_prefix_tokens // bs
        for t0 in range(first[b] - first[b] % bs, int(L), bs):   # blocks from the first unread slot on
            blk, off = inp.block_table[b, t0 // bs], max(first[b] - t0, 0)
            if t0 // bs >= n_shared:
                inp.k_cache[blk, off:] = nan
                inp.v_cache[blk, off:] = nan
    inp.k_cache[~used] = nan
    inp.v_cache[~used] = nan
