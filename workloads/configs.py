"""The decode-step workloads: sizes, layouts and the seeded recipe's knobs.

Every length here is an *attended* length L_b: L_b - 1 tokens already sit in
the cache and the new token is written at position (and slot) L_b - 1, then
attends to all L_b tokens including itself.
"""

from __future__ import annotations

import dataclasses
import math
from typing import Optional, Tuple


@dataclasses.dataclass(frozen=True)
class WorkloadConfig:
    name: str
    batch: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    dtype: str                      # "f32" or "bf16": storage type of q, k, v, caches, out
    layout: str                     # "contiguous" [B, Hkv, max_len, D] or "paged" [blocks, bs, Hkv, D]
    seq_len: Optional[int] = None   # fixed attended length for every sequence
    len_range: Optional[Tuple[int, int]] = None  # inclusive uniform integer range of L_b
    max_len: int = 0                # contiguous capacity per sequence
    block_size: int = 0             # paged: tokens per block
    num_blocks: int = 0             # paged: physical blocks in each of the K and V pools
    max_blocks_per_seq: int = 0     # paged: columns of the block table
    shared_prefix_tokens: int = 0   # paged: leading tokens of every sequence mapped to the same blocks
    num_splits: int = 0             # split-K chunks per sequence; 0 lets the library choose
    kv_dtype: str = ""              # "" = the caches hold ``dtype``; "int8" / "int4" = codes + per-head scales
    window: int = 0                 # int8 only: recent tokens also kept in a bf16 ring of this many slots
    gamma: int = 1                  # new tokens per sequence (> 1: a speculative-verify step)
    rope_base: float = 10000.0
    seed: int = 0
    description: str = ""

    @property
    def n_rep(self) -> int:
        return self.n_q_heads // self.n_kv_heads

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2

    @property
    def capacity(self) -> int:
        """Largest attended length the cache can hold per sequence."""
        if self.layout == "contiguous":
            return self.max_len
        return self.max_blocks_per_seq * self.block_size

    @property
    def int8(self) -> bool:
        """A quantised cache (INT8 or INT4 codes with per-head scales)."""
        return self.kv_dtype in ("int8", "int4")

    @property
    def code_bits(self) -> int:
        return 4 if self.kv_dtype == "int4" else 8

    def kv_bytes(self, lengths) -> int:
        """Algorithmic K+V bytes one decode step streams: 2 * sum_b L_b * Hkv * D * elem.

        INT8 caches: the tokens older than the window cost 1 byte per element, the (at most
        ``window``) most recent ones 2 bytes (bf16 ring); the per-head scales are not counted.
        """
        row = 2 * self.n_kv_heads * self.head_dim
        if self.int8:
            total = 0
            for x in lengths:
                recent = min(int(x), self.window)
                total += (int(x) - recent) * row * self.code_bits // 8 + recent * row * 2
            return total
        return int(sum(int(x) for x in lengths)) * row * self.elem_bytes

    def unique_kv_bytes(self, lengths) -> int:
        """K+V bytes with the shared prefix counted once (equals kv_bytes without sharing)."""
        if not self.shared_prefix_tokens or self.int8:
            return self.kv_bytes(lengths)
        p = self.shared_prefix_tokens
        toks = p + sum(int(x) - p for x in lengths)
        return 2 * toks * self.n_kv_heads * self.head_dim * self.elem_bytes


def _paged(name, **kw) -> WorkloadConfig:
    kw.setdefault("layout", "paged")
    return WorkloadConfig(name=name, **kw)


# The five workloads of the decode step, at full size.
CONFIGS = {
    "tiny_fp32": WorkloadConfig(
        name="tiny_fp32", batch=1, n_q_heads=4, n_kv_heads=2, head_dim=64, dtype="f32",
        layout="contiguous", seq_len=128, max_len=128,
        description="tiny fp32 decode step: batch 1, 4 q / 2 kv heads, D 64, 127 cached + 1 new at position 127"),
    "llama3_8b_layer": WorkloadConfig(
        name="llama3_8b_layer", batch=1, n_q_heads=32, n_kv_heads=8, head_dim=128, dtype="bf16",
        layout="contiguous", seq_len=4096, max_len=8192,
        description="Llama-3-8B-shaped single-layer decode: batch 1, 32q/8kv, D 128, context 4096, cache [1,8,8192,128]"),
    "batched_paged": _paged(
        "batched_paged", batch=64, n_q_heads=32, n_kv_heads=8, head_dim=128, dtype="bf16",
        len_range=(512, 8192), block_size=16, num_blocks=40000, max_blocks_per_seq=512,
        description="batched paged decode: batch 64, 32q/8kv, D 128, L_b ~ U[512,8192], block 16, pool 40000"),
    "long_context": _paged(
        "long_context", batch=1, n_q_heads=32, n_kv_heads=8, head_dim=128, dtype="bf16",
        seq_len=131072, block_size=32, num_blocks=8192, max_blocks_per_seq=4096, num_splits=128,
        description="long-context decode: batch 1, 32q/8kv, D 128, context 131072, block 32, split-K 128"),
}
for _hkv in (32, 8, 1):
    CONFIGS[f"prefix_sweep_kv{_hkv}"] = _paged(
        f"prefix_sweep_kv{_hkv}", batch=16, n_q_heads=32, n_kv_heads=_hkv, head_dim=128, dtype="bf16",
        seq_len=8192, block_size=16, num_blocks=128 + 16 * 384, max_blocks_per_seq=512,
        shared_prefix_tokens=2048,
        description=f"MHA/GQA/MQA sweep, n_kv {_hkv}: batch 16, 32 q heads, D 128, context 8192, "
                    "first 2048 tokens on 128 shared blocks, block 16")

# The INT8 cache ([KVC-GQA-RoPE] §4.3): the batch-64 paged and 128K workloads with INT8 codes,
# per-head scales and the 128 most recent tokens kept in bf16.
CONFIGS["batched_paged_int8"] = dataclasses.replace(
    CONFIGS["batched_paged"], name="batched_paged_int8", kv_dtype="int8", window=128,
    description="batched paged decode, INT8 KV cache (per-head scales) + 128-token bf16 window: batch 64, "
                "32q/8kv, D 128, L_b ~ U[512,8192], block 16, pool 40000")
CONFIGS["batched_paged_int4"] = dataclasses.replace(
    CONFIGS["batched_paged_int8"], name="batched_paged_int4", kv_dtype="int4",
    description="batched paged decode, INT4 KV cache (per-head scales) + 128-token bf16 window: batch 64, "
                "32q/8kv, D 128, L_b ~ U[512,8192], block 16, pool 40000")
CONFIGS["long_context_int8"] = dataclasses.replace(
    CONFIGS["long_context"], name="long_context_int8", kv_dtype="int8", window=128, num_splits=0,
    description="long-context decode, INT8 KV cache (per-head scales) + 128-token bf16 window: batch 1, "
                "32q/8kv, D 128, context 131072, block 32")
CONFIGS["long_context_int4"] = dataclasses.replace(
    CONFIGS["long_context_int8"], name="long_context_int4", kv_dtype="int4",
    description="long-context decode, INT4 KV cache (per-head scales) + 128-token bf16 window: batch 1, "
                "32q/8kv, D 128, context 131072, block 32")

# The speculative-verify step ([Opt-2026] §五, gamma = 4): the batch-64 paged and 128K workloads
# with 4 new tokens per sequence, causal inside the chunk; L_b counts all 4.
CONFIGS["batched_paged_verify4"] = dataclasses.replace(
    CONFIGS["batched_paged"], name="batched_paged_verify4", gamma=4,
    description="speculative verify, 4 new tokens per sequence: batch 64, 32q/8kv, D 128, L_b ~ U[512,8192], "
                "block 16, pool 40000")
CONFIGS["long_context_verify4"] = dataclasses.replace(
    CONFIGS["long_context"], name="long_context_verify4", gamma=4, num_splits=0,
    description="speculative verify, 4 new tokens: batch 1, 32q/8kv, D 128, context 131072, block 32")

# Prefill ([Opt-2026] §三, FlashAttention and its 128K figure): the whole prompt as new tokens at
# positions 0 .. T-1, causal attention; gamma = T.
CONFIGS["prefill_8k"] = _paged(
    "prefill_8k", batch=1, n_q_heads=32, n_kv_heads=8, head_dim=128, dtype="bf16", seq_len=8192, gamma=8192,
    block_size=32, num_blocks=256, max_blocks_per_seq=256,
    description="prefill of an 8K prompt: batch 1, 32q/8kv, D 128, causal, paged block 32")
CONFIGS["prefill_128k"] = _paged(
    "prefill_128k", batch=1, n_q_heads=32, n_kv_heads=8, head_dim=128, dtype="bf16", seq_len=131072, gamma=131072,
    block_size=32, num_blocks=4096, max_blocks_per_seq=4096,
    description="prefill of a 128K prompt: batch 1, 32q/8kv, D 128, causal, paged block 32")


def get_config(name: str) -> WorkloadConfig:
    return CONFIGS[name]


def reduced(cfg: WorkloadConfig, factor: int = 16, batch: Optional[int] = None) -> WorkloadConfig:
    """A smaller twin of ``cfg`` with the same heads, D, dtype, layout and block size.

    Lengths, capacities and pools shrink by ``factor`` (kept >= a few blocks),
    so the float64 oracle finishes in seconds while the kernels still see
    several tiles, several splits and a ragged last block.
    """
    def shrink(x: int, lo: int) -> int:
        return max(lo, x // factor)

    kw = dataclasses.asdict(cfg)
    kw["name"] = cfg.name + f"_div{factor}"
    if batch is not None:
        kw["batch"] = batch
    B = kw["batch"]
    if cfg.seq_len is not None:
        kw["seq_len"] = shrink(cfg.seq_len, 40) + 3       # +3: ragged tail in the last block
    if cfg.len_range is not None:
        lo, hi = cfg.len_range
        kw["len_range"] = (shrink(lo, 17), shrink(hi, 80))
    longest = kw["seq_len"] if kw["seq_len"] is not None else kw["len_range"][1]
    if cfg.layout == "contiguous":
        kw["max_len"] = max(longest, shrink(cfg.max_len, longest))
    else:
        bs = cfg.block_size
        kw["shared_prefix_tokens"] = (shrink(cfg.shared_prefix_tokens, bs) // bs) * bs if cfg.shared_prefix_tokens else 0
        kw["max_blocks_per_seq"] = math.ceil(longest / bs)
        need = B * kw["max_blocks_per_seq"]
        kw["num_blocks"] = max(need + 7, shrink(cfg.num_blocks, need + 7))
    if cfg.num_splits:
        kw["num_splits"] = max(2, cfg.num_splits // factor)
    if cfg.window:
        kw["window"] = max(16, (cfg.window // factor) // 8 * 8)
    if cfg.gamma > 16:                     # a prefill: the prompt is the whole sequence
        kw["gamma"] = kw["seq_len"]
    return WorkloadConfig(**kw)
