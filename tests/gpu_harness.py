"""Run one decode step through the C ABI and, separately, through the float64 oracle.

The two sides share only the seeded inputs from ``workloads``: the GPU side gets
torch device copies of the storage arrays; the oracle gets the same arrays on the host.
"""

from __future__ import annotations

import dataclasses
from typing import Optional, Sequence

import numpy as np
import torch

import oracle
from oracle import decode as odecode
from workloads import DecodeInputs

# Tolerances on the attention output (max abs error against the float64 oracle, computed on
# the same stored inputs, beyond half an ulp of the output's storage type -- see out_error):
# 1e-4 for fp32 storage, 1e-2 for bf16 storage.
OUT_ATOL = {"f32": 1e-4, "bf16": 1e-2}


def to_torch(arr: np.ndarray, dtype: str, device) -> torch.Tensor:
    if dtype == "bf16":
        t = torch.from_numpy(np.ascontiguousarray(arr).view(np.int16)).view(torch.bfloat16)
    elif dtype == "f32":
        t = torch.from_numpy(np.ascontiguousarray(arr, dtype=np.float32))
    else:
        t = torch.from_numpy(np.ascontiguousarray(arr))
    return t.to(device)


def to_numpy(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


@dataclasses.dataclass
class GpuResult:
    q_rot: np.ndarray
    out: np.ndarray
    k_cache: Optional[np.ndarray]
    v_cache: Optional[np.ndarray]
    err: int
    splits: int


def run_gpu(inp: DecodeInputs, num_splits: int = 0, rope_style: int = 0, device="cuda:0",
            fetch_cache: bool = True, seq_lens: Optional[np.ndarray] = None, fused: bool = False) -> GpuResult:
    """One decode step through the C ABI: the fused call (``fused``) or rra_rope_append +
    rra_decode_attn_* (attending ``seq_lens``, default positions + 1)."""
    from rope_gqa_paged_gb300 import DecodeStep

    cfg = inp.cfg
    dt = cfg.dtype
    kc, vc = to_torch(inp.k_cache, dt, device), to_torch(inp.v_cache, dt, device)
    table = to_torch(inp.block_table, "i32", device) if inp.block_table is not None else None
    step = DecodeStep(cfg.batch, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim, kc, vc, table,
                      num_splits=num_splits or cfg.num_splits, rope_base=cfg.rope_base, rope_style=rope_style)
    lens = inp.lengths if seq_lens is None else seq_lens
    args = (to_torch(inp.q, dt, device), to_torch(inp.k_new, dt, device), to_torch(inp.v_new, dt, device),
            to_torch(inp.positions, "i32", device))
    if fused:
        out = step(*args)
    else:
        out = step(*args, to_torch(np.asarray(lens, dtype=np.int32), "i32", device))
    torch.cuda.synchronize(device)
    res = GpuResult(q_rot=to_numpy(step.q_rot), out=to_numpy(out),
                    k_cache=to_numpy(kc) if fetch_cache else None, v_cache=to_numpy(vc) if fetch_cache else None,
                    err=step.error_bits(), splits=step.splits)
    del kc, vc, step
    return res


def run_oracle(inp: DecodeInputs, rope_style: int = 0, seq_lens=None):
    """Whole-batch oracle on copies of the caches: (q_rot, k_cache, v_cache, out float64)."""
    cfg = inp.cfg
    bs = cfg.block_size if inp.block_table is not None else 0
    return odecode.decode_step(inp.q, inp.k_new, inp.v_new, inp.positions, inp.k_cache, inp.v_cache, cfg.dtype,
                               inp.block_table, bs, seq_lens=seq_lens, rope_base=cfg.rope_base,
                               rope_style=rope_style)


def oracle_for_sequences(inp: DecodeInputs, batches: Sequence[int], rope_style: int = 0):
    """Oracle outputs for a few sequences of a (possibly huge) batch, one sequence at a time.

    For each sequence b the logical K/V (L_b - 1 cached tokens) is gathered from the
    input cache, the oracle appends the new token into a private one-sequence cache and
    attends. Returns (q_rot rows, out rows float64), each [len(batches), Hq, D].
    """
    cfg = inp.cfg
    bs = cfg.block_size if inp.block_table is not None else 0
    q_rows, outs = [], []
    for b in batches:
        L = int(inp.lengths[b])
        k = odecode.logical_kv(inp.k_cache, b, L, inp.block_table, bs)
        v = odecode.logical_kv(inp.v_cache, b, L, inp.block_table, bs)
        kc, vc = np.array(k)[None].copy(), np.array(v)[None].copy()       # [1, Hkv, L, D]
        q_rot = odecode.rope_append(inp.q[b:b + 1], inp.k_new[b:b + 1], inp.v_new[b:b + 1],
                                    inp.positions[b:b + 1], kc, vc, cfg.dtype, rope_base=cfg.rope_base,
                                    rope_style=rope_style)
        outs.append(odecode.decode_attention(q_rot, kc, vc, np.array([L]), cfg.dtype)[0])
        q_rows.append(q_rot[0])
    return np.stack(q_rows), np.stack(outs)


def bf16_ulp_distance(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Distance in bf16 ulps between two arrays of bf16 bit patterns (sign-magnitude aware)."""
    def ordered(x):
        x = x.astype(np.int32)
        return np.where(x & 0x8000, 0x8000 - x, x)  # negative values map below zero, -0 == +0
    return np.abs(ordered(a) - ordered(b))


def stored_to_f64(arr: np.ndarray, dtype: str) -> np.ndarray:
    return oracle.storage_to_f64(arr, dtype)


def assert_close_stored(got: np.ndarray, want: np.ndarray, dtype: str, what: str):
    """Stored values (q_rot, appended k) agree within 1 bf16 ulp, or 4 fp32 ulps."""
    if dtype == "bf16":
        d = bf16_ulp_distance(got, want)
        assert d.max() <= 1, f"{what}: {int(d.max())} bf16 ulps apart at {np.unravel_index(d.argmax(), d.shape)}"
    else:
        g, w = got.astype(np.float64), want.astype(np.float64)
        tol = 4 * np.spacing(np.abs(w).astype(np.float32)).astype(np.float64)
        assert np.all(np.abs(g - w) <= tol), f"{what}: max diff {np.abs(g - w).max()}"


def half_ulp(x: np.ndarray, dtype: str) -> np.ndarray:
    """Half a unit in the last place of the storage type at |x| (the rounding every stored
    output carries): bf16 keeps 8 significant bits, fp32 24."""
    bits = 8 if dtype == "bf16" else 24
    ax = np.abs(np.asarray(x, dtype=np.float64))
    _, e = np.frexp(ax)
    e = np.where(ax > 0, np.maximum(e, -125), -125)   # below the normal range the grid stops shrinking
    return np.ldexp(0.5, e - bits)


# Relative bar: long rows average many values, so their outputs are small (|out| ~ sqrt(1/L),
# about 0.005 at 128K) and an absolute 1e-2 says little there. The error beyond the storage
# rounding, over the RMS of the same output row of the float64 result, stays below 5 %: the bf16
# (f16 for quantised caches) probabilities perturb each weight by about 2^-9 relative, well under
# 1 % of the row's RMS, while a wrong token, head or block gives errors of order one.
REL_RMS_BAR = 0.05


def rel_rms_error(got_stored: np.ndarray, want_f64: np.ndarray, dtype: str) -> float:
    """Max over output rows (last axis) of the error beyond half an ulp over the row's RMS."""
    want = np.asarray(want_f64, dtype=np.float64)
    got = stored_to_f64(got_stored, dtype)
    excess = np.maximum(np.abs(got - want) - half_ulp(np.maximum(np.abs(want), np.abs(got)), dtype), 0.0).max(axis=-1)
    rms = np.sqrt(np.mean(want * want, axis=-1))
    return float((excess / np.maximum(rms, 1e-30)).max())


def out_error(got_stored: np.ndarray, want_f64: np.ndarray, dtype: str) -> float:
    """Attention-output error beyond the output's own storage rounding: max over elements of
    |stored - float64 result| - half an ulp of the storage type at the result. The tolerance
    (1e-2 bf16, 1e-4 fp32) bounds the computation; a value stored in bf16 cannot be closer than
    half an ulp to an arbitrary real (0.0156 for outputs of magnitude 4..8)."""
    g = stored_to_f64(got_stored, dtype)
    assert np.all(np.isfinite(g)), "non-finite attention output"
    want = np.asarray(want_f64, dtype=np.float64)
    return float((np.abs(g - want) - half_ulp(np.maximum(np.abs(want), np.abs(g)), dtype)).max())


# ---------------------------------------------------------------------------- INT8 cache
@dataclasses.dataclass
class GpuQ8Result:
    q_rot: np.ndarray
    out: np.ndarray
    k_codes: np.ndarray
    v_codes: np.ndarray
    k_win: Optional[np.ndarray]
    v_win: Optional[np.ndarray]
    err: int
    splits: int


def run_gpu_q8(inp: DecodeInputs, num_splits: int = 0, rope_style: int = 0, device="cuda:0",
               seq_lens: Optional[np.ndarray] = None, fused: bool = False) -> GpuQ8Result:
    """One INT8-cache step through the C ABI: the fused call or rra_rope_append_q8 + rra_decode_attn_q8."""
    from rope_gqa_paged_gb300 import DecodeStepQ8

    cfg = inp.cfg
    kc = torch.from_numpy(np.ascontiguousarray(inp.k_cache)).to(device)
    vc = torch.from_numpy(np.ascontiguousarray(inp.v_cache)).to(device)
    kw = to_torch(inp.k_win, "bf16", device) if inp.k_win is not None else None
    vw = to_torch(inp.v_win, "bf16", device) if inp.v_win is not None else None
    table = to_torch(inp.block_table, "i32", device) if inp.block_table is not None else None
    step = DecodeStepQ8(cfg.batch, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim, kc, vc,
                        torch.from_numpy(inp.k_scale).to(device), torch.from_numpy(inp.v_scale).to(device), kw, vw,
                        table, num_splits=num_splits or cfg.num_splits, rope_base=cfg.rope_base,
                        rope_style=rope_style, bits=cfg.code_bits)
    args = (to_torch(inp.q, "bf16", device), to_torch(inp.k_new, "bf16", device), to_torch(inp.v_new, "bf16", device),
            to_torch(inp.positions, "i32", device))
    if fused:
        out = step(*args)
    else:
        lens = inp.lengths if seq_lens is None else seq_lens
        out = step(*args, to_torch(np.asarray(lens, dtype=np.int32), "i32", device))
    torch.cuda.synchronize(device)
    res = GpuQ8Result(q_rot=to_numpy(step.q_rot), out=to_numpy(out), k_codes=kc.cpu().numpy(),
                      v_codes=vc.cpu().numpy(), k_win=to_numpy(kw) if kw is not None else None,
                      v_win=to_numpy(vw) if vw is not None else None, err=step.error_bits(), splits=step.splits)
    del kc, vc, kw, vw, step
    return res


def run_oracle_q8(inp: DecodeInputs, rope_style: int = 0, seq_lens=None):
    """(q_rot, k_codes, v_codes, k_win, v_win, out float64) of the oracle on copies of the caches."""
    cfg = inp.cfg
    bs = cfg.block_size if inp.block_table is not None else 0
    return oracle.quant.decode_step_q8(inp.q, inp.k_new, inp.v_new, inp.positions, inp.k_cache, inp.v_cache,
                                       inp.k_scale, inp.v_scale, inp.k_win, inp.v_win, cfg.window, inp.block_table,
                                       bs, seq_lens=seq_lens, rope_base=cfg.rope_base, rope_style=rope_style,
                                       bits=cfg.code_bits)


# ---------------------------------------------------------------------------- speculative verify
def run_gpu_verify(inp: DecodeInputs, num_splits: int = 0, rope_style: int = 0, device="cuda:0",
                   fused: bool = True) -> GpuResult:
    """One verify step (gamma new tokens per sequence) through the C ABI."""
    from rope_gqa_paged_gb300 import VerifyStep

    cfg = inp.cfg
    dt = cfg.dtype
    kc, vc = to_torch(inp.k_cache, dt, device), to_torch(inp.v_cache, dt, device)
    table = to_torch(inp.block_table, "i32", device) if inp.block_table is not None else None
    step = VerifyStep(cfg.batch, cfg.gamma, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim, kc, vc, table,
                      num_splits=num_splits or cfg.num_splits, rope_base=cfg.rope_base, rope_style=rope_style)
    args = (to_torch(inp.q, dt, device), to_torch(inp.k_new, dt, device), to_torch(inp.v_new, dt, device),
            to_torch(inp.positions, "i32", device))
    out = step(*args) if fused else step(*args, seq_lens=True)
    torch.cuda.synchronize(device)
    res = GpuResult(q_rot=to_numpy(step.q_rot), out=to_numpy(out), k_cache=to_numpy(kc), v_cache=to_numpy(vc),
                    err=step.error_bits(), splits=step.splits)
    del kc, vc, step
    return res


def run_oracle_verify(inp: DecodeInputs, rope_style: int = 0):
    cfg = inp.cfg
    bs = cfg.block_size if inp.block_table is not None else 0
    return oracle.verify.verify_step(inp.q, inp.k_new, inp.v_new, inp.positions, inp.k_cache, inp.v_cache, cfg.dtype,
                                     inp.block_table, bs, rope_base=cfg.rope_base, rope_style=rope_style)


def run_gpu_prefill(inp: DecodeInputs, rope_style: int = 0, device="cuda:0", fused: bool = True) -> GpuResult:
    """One prefill step (T = gamma prompt tokens per sequence) through the C ABI. The output is
    filled with NaN first, so a row that no CTA writes cannot pass for a result."""
    from rope_gqa_paged_gb300 import PrefillStep

    cfg = inp.cfg
    kc, vc = to_torch(inp.k_cache, "bf16", device), to_torch(inp.v_cache, "bf16", device)
    table = to_torch(inp.block_table, "i32", device) if inp.block_table is not None else None
    step = PrefillStep(cfg.batch, inp.q.shape[1], cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim, kc, vc, table,
                       rope_base=cfg.rope_base, rope_style=rope_style)
    args = (to_torch(inp.q, "bf16", device), to_torch(inp.k_new, "bf16", device), to_torch(inp.v_new, "bf16", device),
            to_torch(inp.positions, "i32", device))
    step.out.fill_(float("nan"))
    out = step(*args) if fused else step(*args, seq_lens=True)
    torch.cuda.synchronize(device)
    res = GpuResult(q_rot=to_numpy(step.q_rot), out=to_numpy(out), k_cache=to_numpy(kc), v_cache=to_numpy(vc),
                    err=step.error_bits(), splits=1)
    del kc, vc, step
    return res
