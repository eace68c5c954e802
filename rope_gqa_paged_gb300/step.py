"""DecodeStep: one layer's decode step (RoPE + append + GQA attention) on caller-owned caches.

It owns the per-step buffers (rotated q, output, split-K workspace, device error word),
allocated once through torch, and issues the library's kernels on the current stream:
``rra_rope_append`` then ``rra_decode_attn_contig`` / ``rra_decode_attn_paged``.
"""

from __future__ import annotations

from typing import Optional

import torch

from . import rra


class DecodeStep:
    def __init__(self, batch: int, n_q_heads: int, n_kv_heads: int, head_dim: int, k_cache: torch.Tensor,
                 v_cache: torch.Tensor, block_table: Optional[torch.Tensor] = None, num_splits: int = 0,
                 rope_base: float = 10000.0, rope_style: int = 0, scale: float = 0.0):
        self.B, self.Hq, self.Hkv, self.D = batch, n_q_heads, n_kv_heads, head_dim
        self.k_cache, self.v_cache, self.block_table = k_cache, v_cache, block_table
        self.rope_base, self.rope_style, self.scale = rope_base, rope_style, scale
        self.dtype, dev = k_cache.dtype, k_cache.device
        code = rra.RRA_BF16 if self.dtype == torch.bfloat16 else rra.RRA_F32
        if block_table is not None:
            bs = k_cache.shape[1]
            max_tokens = block_table.shape[1] * bs
        else:
            bs, max_tokens = 0, k_cache.shape[2]
        self.splits = rra.rra_decode_num_splits(batch, n_q_heads, n_kv_heads, head_dim, max_tokens, bs,
                                                num_splits, code)
        self.num_splits = self.splits
        ws = rra.rra_decode_workspace_bytes(batch, n_q_heads, head_dim, self.splits)
        self.workspace = torch.zeros(ws, dtype=torch.uint8, device=dev) if ws else None  # zeroed once
        self.q_rot = torch.empty(batch, n_q_heads, head_dim, dtype=self.dtype, device=dev)
        self.out = torch.empty(batch, n_q_heads, head_dim, dtype=self.dtype, device=dev)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        self.graph = None

    def rope_append(self, q, k_new, v_new, positions, stream=None) -> None:
        rra.rra_rope_append(q, k_new, v_new, positions, self.q_rot, self.k_cache, self.v_cache, self.block_table,
                            self.rope_base, self.rope_style, self.err, stream)

    def attend(self, seq_lens, stream=None) -> torch.Tensor:
        if self.block_table is None:
            rra.rra_decode_attn_contig(self.q_rot, self.k_cache, self.v_cache, seq_lens, self.out, self.scale,
                                       self.num_splits, self.workspace, self.err, stream)
        else:
            rra.rra_decode_attn_paged(self.q_rot, self.k_cache, self.v_cache, self.block_table, seq_lens, self.out,
                                      self.scale, self.num_splits, self.workspace, self.err, stream)
        return self.out

    def fused(self, q, k_new, v_new, positions, stream=None) -> torch.Tensor:
        """The whole step in one library call (one kernel for bf16 caches); attends positions + 1."""
        if self.block_table is None:
            rra.rra_decode_step_contig(q, k_new, v_new, positions, self.q_rot, self.k_cache, self.v_cache, self.out,
                                       self.rope_base, self.rope_style, self.scale, self.num_splits, self.workspace,
                                       self.err, stream)
        else:
            rra.rra_decode_step_paged(q, k_new, v_new, positions, self.q_rot, self.k_cache, self.v_cache,
                                      self.block_table, self.out, self.rope_base, self.rope_style, self.scale,
                                      self.num_splits, self.workspace, self.err, stream)
        return self.out

    def __call__(self, q, k_new, v_new, positions, seq_lens=None, stream=None) -> torch.Tensor:
        """Rotate, append, attend. Without ``seq_lens`` this is the fused step (attending
        positions + 1 tokens); with it, the two calls rra_rope_append + rra_decode_attn_*."""
        if seq_lens is None:
            return self.fused(q, k_new, v_new, positions, stream)
        self.rope_append(q, k_new, v_new, positions, stream)
        return self.attend(seq_lens, stream)

    def capture(self, q, k_new, v_new, positions, seq_lens=None, repeat: int = 1, between=None, before=None,
                after=None):
        """Record the step (``repeat`` times back to back, calling ``between()`` before each
        repetition after the first) into a CUDA graph; returns it and keeps it for ``replay()``.

        The graph is bound to these input tensors and to this object's output, workspace
        and error buffers: refill the inputs in place, then ``replay()``. Replaying saves
        the host-side launch cost of every kernel of the step, and inside one graph each
        decode kernel overlaps its launch with the end of the kernel before it.
        ``before()`` / ``after()`` record work around every repetition into the same graph,
        e.g. the copy of the step's inputs from pinned host memory and of its output back.
        """
        def one():
            if before is not None:
                before()
            self(q, k_new, v_new, positions, seq_lens)
            if after is not None:
                after()

        side = torch.cuda.Stream(device=q.device)
        side.wait_stream(torch.cuda.current_stream(q.device))
        with torch.cuda.stream(side):
            one()
        torch.cuda.current_stream(q.device).wait_stream(side)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for i in range(repeat):
                if i and between is not None:
                    between()
                one()
        self.graph = graph
        return graph

    def replay(self) -> torch.Tensor:
        """Run the captured step on the current stream; returns the output buffer."""
        self.graph.replay()
        return self.out

    def error_bits(self) -> int:
        """Device error word (RRA_ERR_* bits) accumulated since the last reset; synchronises."""
        return int(self.err.item())

    def reset_errors(self) -> None:
        self.err.zero_()


class DecodeStepQ8(DecodeStep):
    """The decode step on an INT8 (bits 8) or INT4 (bits 4, two codes per byte) KV cache with
    per-head scales and a bf16 window of recent tokens.

    k_codes / v_codes: int8 [B, Hkv, max_len, D] or pools [num_blocks, block_size, Hkv, D] (with
    ``block_table``); k_scale / v_scale: float32 [Hkv]; k_win / v_win: bf16 rings [B, Hkv, W, D]
    or None (no window). q, k_new, v_new and the output are bf16.
    """

    def __init__(self, batch: int, n_q_heads: int, n_kv_heads: int, head_dim: int, k_codes: torch.Tensor,
                 v_codes: torch.Tensor, k_scale: torch.Tensor, v_scale: torch.Tensor,
                 k_win: Optional[torch.Tensor] = None, v_win: Optional[torch.Tensor] = None,
                 block_table: Optional[torch.Tensor] = None, num_splits: int = 0, rope_base: float = 10000.0,
                 rope_style: int = 0, scale: float = 0.0, bits: int = 8):
        self.B, self.Hq, self.Hkv, self.D = batch, n_q_heads, n_kv_heads, head_dim
        self.bits = bits
        self.k_cache, self.v_cache, self.block_table = k_codes, v_codes, block_table
        self.k_scale, self.v_scale, self.k_win, self.v_win = k_scale, v_scale, k_win, v_win
        self.window = k_win.shape[2] if k_win is not None else 0
        self.rope_base, self.rope_style, self.scale = rope_base, rope_style, scale
        self.dtype, dev = torch.bfloat16, k_codes.device
        if block_table is not None:
            bs = k_codes.shape[1]
            max_tokens = block_table.shape[1] * bs
        else:
            bs, max_tokens = 0, k_codes.shape[2]
        self.splits = rra.rra_decode_q8_num_splits(batch, n_q_heads, n_kv_heads, head_dim, max_tokens, bs,
                                                   num_splits, self.window, bits)
        self.num_splits = num_splits
        ws = rra.rra_decode_workspace_bytes(batch, n_q_heads, head_dim, self.splits)
        self.workspace = torch.zeros(ws, dtype=torch.uint8, device=dev) if ws else None  # zeroed once
        self.q_rot = torch.empty(batch, n_q_heads, head_dim, dtype=self.dtype, device=dev)
        self.out = torch.empty(batch, n_q_heads, head_dim, dtype=self.dtype, device=dev)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        self.graph = None

    def rope_append(self, q, k_new, v_new, positions, stream=None) -> None:
        rra.rra_rope_append_q8(q, k_new, v_new, positions, self.q_rot, self.k_cache, self.v_cache, self.k_scale,
                               self.v_scale, self.k_win, self.v_win, self.block_table, self.rope_base,
                               self.rope_style, self.err, stream, bits=self.bits)

    def attend(self, seq_lens, stream=None) -> torch.Tensor:
        rra.rra_decode_attn_q8(self.q_rot, self.k_cache, self.v_cache, self.k_scale, self.v_scale, seq_lens,
                               self.out, self.k_win, self.v_win, self.block_table, self.scale, self.num_splits,
                               self.workspace, self.err, stream, bits=self.bits)
        return self.out

    def fused(self, q, k_new, v_new, positions, stream=None) -> torch.Tensor:
        rra.rra_decode_step_q8(q, k_new, v_new, positions, self.q_rot, self.k_cache, self.v_cache, self.k_scale,
                               self.v_scale, self.out, self.k_win, self.v_win, self.block_table, self.rope_base,
                               self.rope_style, self.scale, self.num_splits, self.workspace, self.err, stream,
                               bits=self.bits)
        return self.out


class VerifyStep(DecodeStep):
    """The speculative-verify step: gamma new tokens per sequence, causal inside the chunk.

    q / k_new / v_new are [B, gamma, H, D]; ``positions[b]`` is the first new token's position,
    and the output is [B, gamma, Hq, D]. Caches as for DecodeStep (bf16).
    """

    def __init__(self, batch: int, gamma: int, n_q_heads: int, n_kv_heads: int, head_dim: int,
                 k_cache: torch.Tensor, v_cache: torch.Tensor, block_table: Optional[torch.Tensor] = None,
                 num_splits: int = 0, rope_base: float = 10000.0, rope_style: int = 0, scale: float = 0.0):
        self.B, self.gamma, self.Hq, self.Hkv, self.D = batch, gamma, n_q_heads, n_kv_heads, head_dim
        self.k_cache, self.v_cache, self.block_table = k_cache, v_cache, block_table
        self.rope_base, self.rope_style, self.scale = rope_base, rope_style, scale
        self.dtype, dev = k_cache.dtype, k_cache.device
        if block_table is not None:
            bs = k_cache.shape[1]
            max_tokens = block_table.shape[1] * bs
        else:
            bs, max_tokens = 0, k_cache.shape[2]
        self.splits = rra.rra_verify_num_splits(batch, gamma, n_q_heads, n_kv_heads, head_dim, max_tokens, bs,
                                                num_splits)
        self.num_splits = num_splits
        ws = rra.rra_verify_workspace_bytes(batch, gamma, n_q_heads, n_kv_heads, head_dim, self.splits)
        self.workspace = torch.zeros(ws, dtype=torch.uint8, device=dev) if ws else None  # zeroed once
        self.q_rot = torch.empty(batch, gamma, n_q_heads, head_dim, dtype=self.dtype, device=dev)
        self.out = torch.empty(batch, gamma, n_q_heads, head_dim, dtype=self.dtype, device=dev)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        self.graph = None

    def rope_append(self, q, k_new, v_new, positions, stream=None) -> None:
        rra.rra_rope_append_verify(q, k_new, v_new, positions, self.q_rot, self.k_cache, self.v_cache,
                                   self.block_table, self.rope_base, self.rope_style, self.err, stream)

    def attend(self, positions, stream=None) -> torch.Tensor:
        """Attention of the already-appended gamma tokens (``positions``: the first one's)."""
        rra.rra_verify_attn(self.q_rot, self.k_cache, self.v_cache, positions, self.out, self.block_table, self.scale,
                            self.num_splits, self.workspace, self.err, stream)
        return self.out

    def fused(self, q, k_new, v_new, positions, stream=None) -> torch.Tensor:
        rra.rra_verify_step(q, k_new, v_new, positions, self.q_rot, self.k_cache, self.v_cache, self.out,
                            self.block_table, self.rope_base, self.rope_style, self.scale, self.num_splits,
                            self.workspace, self.err, stream)
        return self.out

    def __call__(self, q, k_new, v_new, positions, seq_lens=None, stream=None) -> torch.Tensor:
        """The step in one library call (seq_lens None), or the two calls (seq_lens ignored: the
        attended lengths follow from the positions)."""
        if seq_lens is None:
            return self.fused(q, k_new, v_new, positions, stream)
        self.rope_append(q, k_new, v_new, positions, stream)
        return self.attend(positions, stream)


class PrefillStep(VerifyStep):
    """Prefill of T prompt tokens per sequence (positions[b]: the first one's position, 0 for a
    fresh prompt): RoPE + append, then causal attention. No split-K workspace."""

    def __init__(self, batch: int, prompt_len: int, n_q_heads: int, n_kv_heads: int, head_dim: int,
                 k_cache: torch.Tensor, v_cache: torch.Tensor, block_table: Optional[torch.Tensor] = None,
                 rope_base: float = 10000.0, rope_style: int = 0, scale: float = 0.0):
        self.B, self.gamma, self.Hq, self.Hkv, self.D = batch, prompt_len, n_q_heads, n_kv_heads, head_dim
        self.k_cache, self.v_cache, self.block_table = k_cache, v_cache, block_table
        self.rope_base, self.rope_style, self.scale = rope_base, rope_style, scale
        self.dtype, dev = k_cache.dtype, k_cache.device
        self.splits = self.num_splits = 1
        self.workspace = None
        self.q_rot = torch.empty(batch, prompt_len, n_q_heads, head_dim, dtype=self.dtype, device=dev)
        self.out = torch.empty(batch, prompt_len, n_q_heads, head_dim, dtype=self.dtype, device=dev)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        self.graph = None

    def attend(self, positions, stream=None) -> torch.Tensor:
        rra.rra_prefill_attn(self.q_rot, self.k_cache, self.v_cache, positions, self.out, self.block_table, self.scale,
                             self.err, stream)
        return self.out

    def fused(self, q, k_new, v_new, positions, stream=None) -> torch.Tensor:
        rra.rra_prefill_step(q, k_new, v_new, positions, self.q_rot, self.k_cache, self.v_cache, self.out,
                             self.block_table, self.rope_base, self.rope_style, self.scale, self.err, stream)
        return self.out
