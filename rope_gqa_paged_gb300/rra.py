"""ctypes binding of librra_gb300.so: the C entry points under the same names.

Argument marshalling only: shapes are read from the torch tensors, pointers and the
current CUDA stream are passed through, and a non-zero status raises RraError. Every
step of the decode path runs in the library's CUDA kernels; there is no fallback.
"""

from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

from . import _build

RRA_F32, RRA_BF16 = 0, 1
RRA_ERR_POSITION, RRA_ERR_BLOCK_ID, RRA_ERR_SEQ_LEN, RRA_ERR_TIMEOUT, RRA_ERR_WORKSPACE = 1, 2, 4, 8, 16

_lib: Optional[ctypes.CDLL] = None

_c_int, _c_i64, _c_u64, _c_size, _c_f32, _c_f64, _vp = (ctypes.c_int, ctypes.c_int64, ctypes.c_uint64,
                                                         ctypes.c_size_t, ctypes.c_float, ctypes.c_double,
                                                         ctypes.c_void_p)
_SIGNATURES = {
    "rra_rope_append": (_c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int,
                                 _c_int, _c_int, _c_int, _c_int, _c_f64, _c_int, _c_int, _vp, _vp]),
    "rra_decode_attn_contig": (_c_int, [_vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int, _c_int, _c_f32,
                                        _c_int, _vp, _c_size, _c_int, _vp, _vp]),
    "rra_decode_attn_paged": (_c_int, [_vp, _vp, _vp, _vp, _c_int, _vp, _c_int, _c_int, _vp, _c_int, _c_int,
                                       _c_int, _c_int, _c_f32, _c_int, _vp, _c_size, _c_int, _vp, _vp]),
    "rra_kv_bytes": (_c_u64, [_c_int, _c_int, _c_int, _c_i64, _c_int, _c_int]),
    "rra_decode_num_splits": (_c_int, [_c_int, _c_int, _c_int, _c_int, _c_i64, _c_int, _c_int, _c_int]),
    "rra_decode_workspace_bytes": (_c_size, [_c_int, _c_int, _c_int, _c_int]),
    "rra_status_str": (ctypes.c_char_p, [_c_int]),
    "rra_last_cuda_error": (ctypes.c_char_p, []),
    "rra_use_device": (_c_int, [_c_int]),
    "rra_test_hold_append": (_c_int, [_c_int]),
    "rra_rope_phi": (_c_int, [_c_int, _c_f64, _vp]),
    "rra_rope_cos_sin_host": (_c_int, [_c_int, _vp, _vp]),
    "rra_rope_cos_sin": (_c_int, [_vp, _c_int, _c_int, _c_f64, _vp, _vp]),
    "rra_decode_step_contig": (_c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _c_int, _vp, _c_int, _c_int, _c_int,
                                        _c_int, _c_f64, _c_int, _c_f32, _c_int, _vp, _c_size, _c_int, _vp, _vp]),
    "rra_decode_step_paged": (_c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _vp, _c_int,
                                       _c_int, _c_int, _c_int, _c_f64, _c_int, _c_f32, _c_int, _vp, _c_size, _c_int,
                                       _vp, _vp]),
    "rra_rope_append_q8": (_c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _c_int, _vp, _c_int,
                                    _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_f64, _c_int, _vp,
                                    _vp]),
    "rra_decode_attn_q8": (_c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _c_int, _vp, _c_int, _vp, _c_int, _c_int,
                                    _c_int, _vp, _c_int, _c_int, _c_int, _c_int, _c_f32, _c_int, _vp, _c_size, _vp,
                                    _vp]),
    "rra_decode_step_q8": (_c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _c_int, _vp, _c_int,
                                    _c_int, _c_int, _c_int, _vp, _c_int, _c_int, _c_int, _c_int, _c_f64, _c_int,
                                    _c_f32, _c_int, _vp, _c_size, _vp, _vp]),
    "rra_decode_q8_num_splits": (_c_int, [_c_int, _c_int, _c_int, _c_int, _c_i64, _c_int, _c_int, _c_int]),
    "rra_rope_append_q4": None, "rra_decode_attn_q4": None, "rra_decode_step_q4": None,
    "rra_decode_q4_num_splits": None,
    "rra_rope_append_verify": (_c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int,
                                        _c_int, _c_int, _c_int, _c_int, _c_int, _c_f64, _c_int, _c_int, _vp, _vp]),
    "rra_verify_attn": (_c_int, [_vp, _vp, _vp, _vp, _c_int, _vp, _c_int, _c_int, _c_int, _vp, _c_int, _c_int,
                                 _c_int, _c_int, _c_int, _c_f32, _c_int, _vp, _c_size, _vp, _vp]),
    "rra_verify_step": (_c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int, _vp,
                                 _c_int, _c_int, _c_int, _c_int, _c_int, _c_f64, _c_int, _c_f32, _c_int, _vp, _c_size,
                                 _vp, _vp]),
    "rra_verify_num_splits": (_c_int, [_c_int, _c_int, _c_int, _c_int, _c_int, _c_i64, _c_int, _c_int]),
    "rra_verify_workspace_bytes": (_c_size, [_c_int, _c_int, _c_int, _c_int, _c_int, _c_int]),
    "rra_prefill_attn": (_c_int, [_vp, _vp, _vp, _vp, _c_int, _vp, _c_int, _c_int, _c_int, _vp, _c_int, _c_int,
                                  _c_int, _c_int, _c_int, _c_f32, _vp, _vp]),
    "rra_prefill_step": (_c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int, _vp,
                                  _c_int, _c_int, _c_int, _c_int, _c_int, _c_f64, _c_int, _c_f32, _vp, _vp]),
}


class RraError(RuntimeError):
    def __init__(self, fn: str, status: int):
        detail = lib().rra_status_str(status).decode()
        if status == -5:
            detail += ": " + lib().rra_last_cuda_error().decode()
        super().__init__(f"{fn} returned {status} ({detail})")
        self.status = status


def lib_path() -> str:
    return _build.LIB_PATH


def lib() -> ctypes.CDLL:
    """Load the library (it must have been built; see __graft_entry__.build())."""
    global _lib
    if _lib is None:
        if not os.path.exists(_build.LIB_PATH):
            raise RuntimeError(f"{_build.LIB_PATH} is missing: build the CUDA library first "
                               "(python -c 'import __graft_entry__ as g; g.build()')")
        handle = ctypes.CDLL(_build.LIB_PATH)
        for name in [n for n, sig in _SIGNATURES.items() if sig is None]:   # INT4 twins of the INT8 calls
            _SIGNATURES[name] = _SIGNATURES[name.replace("_q4", "_q8")]
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype, fn.argtypes = res, args
        _lib = handle
    return _lib


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return RRA_BF16
    if t.dtype == torch.float32:
        return RRA_F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensors passed to the decode kernels must be on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return t.data_ptr()


_device_of_thread = threading.local()


def _stream(stream, t: torch.Tensor) -> Optional[int]:
    """The stream handle for a call on tensor ``t``'s device (selecting that device in the
    library when the call runs on the default stream, which carries no device)."""
    dev = t.device.index if t.device.index is not None else torch.cuda.current_device()
    if getattr(_device_of_thread, "dev", None) != dev:
        _check("rra_use_device", lib().rra_use_device(dev))
        _device_of_thread.dev = dev
    if stream is None:
        return torch.cuda.current_stream(t.device).cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check(name: str, status: int) -> None:
    if status != 0:
        raise RraError(name, status)


# --------------------------------------------------------------------------- host-only helpers
def rra_kv_bytes(n_layers: int, n_kv_heads: int, head_dim: int, seq_len: int, batch: int, dtype_bytes: int) -> int:
    return int(lib().rra_kv_bytes(n_layers, n_kv_heads, head_dim, seq_len, batch, dtype_bytes))


def rra_decode_num_splits(B: int, Hq: int, Hkv: int, D: int, max_tokens: int, block_size: int,
                          num_splits: int, dtype: int) -> int:
    r = lib().rra_decode_num_splits(B, Hq, Hkv, D, max_tokens, block_size, num_splits, dtype)
    _check("rra_decode_num_splits", min(r, 0))
    return r


def rra_decode_workspace_bytes(B: int, Hq: int, D: int, splits: int) -> int:
    return int(lib().rra_decode_workspace_bytes(B, Hq, D, splits))


def rra_test_hold_append(hold: bool) -> None:
    """Test hook of the bounded-wait timeout path: while held, fused bf16 steps never release
    their append barrier, so their waits run out (~1 s) and set RRA_ERR_TIMEOUT."""
    _check("rra_test_hold_append", lib().rra_test_hold_append(1 if hold else 0))


def rra_rope_phi(head_dim: int, rope_base: float = 10000.0) -> list:
    """theta_i / 2pi (i < head_dim/2) as 96-bit fractions: [[w0, w1, w2], ...], w0 least significant."""
    buf = (ctypes.c_uint32 * (3 * (head_dim // 2) if head_dim > 0 else 1))()
    _check("rra_rope_phi", lib().rra_rope_phi(head_dim, rope_base, ctypes.cast(buf, _vp)))
    return [[int(buf[3 * i + w]) for w in range(3)] for i in range(head_dim // 2)]


def rra_rope_cos_sin_host(position: int, phi) -> tuple:
    """(cos hi, cos lo, sin hi, sin lo) of 2pi * (position * phi mod 1), by the kernels' float32 steps."""
    ph = (ctypes.c_uint32 * 3)(*[int(w) & 0xffffffff for w in phi])
    out = (ctypes.c_float * 4)()
    _check("rra_rope_cos_sin_host",
           lib().rra_rope_cos_sin_host(int(position), ctypes.cast(ph, _vp), ctypes.cast(out, _vp)))
    return tuple(float(x) for x in out)


def rra_status_str(status: int) -> str:
    return lib().rra_status_str(status).decode()


# --------------------------------------------------------------------------- device entry points
def rra_rope_cos_sin(positions: torch.Tensor, head_dim: int, rope_base: float = 10000.0, out=None,
                     stream=None) -> torch.Tensor:
    """cos hi, cos lo, sin hi, sin lo of positions[p] * theta_i on the device: float32 [n, 4, head_dim/2]."""
    if positions.dtype != torch.int32 or not positions.is_cuda or not positions.is_contiguous():
        raise ValueError("positions: a contiguous int32 CUDA tensor")
    n = positions.numel()
    if out is None:
        out = torch.empty(n, 4, head_dim // 2, dtype=torch.float32, device=positions.device)
    _check("rra_rope_cos_sin", lib().rra_rope_cos_sin(positions.data_ptr(), n, head_dim, rope_base, out.data_ptr(),
                                                      _stream(stream, positions)))
    return out


def rra_rope_append(q, k_new, v_new, positions, q_out, k_cache, v_cache, block_table=None,
                    rope_base: float = 10000.0, rope_style: int = 0, err_flag=None, stream=None) -> None:
    """RoPE on q / k_new at ``positions`` and append of rotated k and raw v into the cache.

    Contiguous cache: k_cache/v_cache [B, Hkv, max_len, D]. Paged: pools
    [num_blocks, block_size, Hkv, D] plus ``block_table`` [B, max_blocks_per_seq] int32.
    """
    B, Hq, D = q.shape
    Hkv = k_new.shape[1]
    if block_table is not None:
        num_blocks, block_size = k_cache.shape[0], k_cache.shape[1]
        mbps, max_len = block_table.shape[1], 0
    else:
        num_blocks = block_size = mbps = 0
        max_len = k_cache.shape[2]
    st = lib().rra_rope_append(_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(positions), _ptr(q_out), _ptr(k_cache),
                               _ptr(v_cache), _ptr(block_table), mbps, block_size, num_blocks, max_len, B, Hq, Hkv,
                               D, float(rope_base), int(rope_style), _dtype_code(q), _ptr(err_flag), _stream(stream, q))
    _check("rra_rope_append", st)


def rra_decode_attn_contig(q_rot, k_cache, v_cache, seq_lens, out, scale: float = 0.0, num_splits: int = 0,
                           workspace=None, err_flag=None, stream=None) -> None:
    """out = GQA softmax attention of q_rot over the first seq_lens[b] slots of a contiguous cache."""
    B, Hq, D = q_rot.shape
    Hkv, max_len = k_cache.shape[1], k_cache.shape[2]
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = lib().rra_decode_attn_contig(_ptr(q_rot), _ptr(k_cache), _ptr(v_cache), _ptr(seq_lens), _ptr(out), B, Hq,
                                      Hkv, D, max_len, float(scale), int(num_splits), _ptr(workspace), ws_bytes,
                                      _dtype_code(q_rot), _ptr(err_flag), _stream(stream, q_rot))
    _check("rra_decode_attn_contig", st)


def rra_decode_attn_paged(q_rot, k_pool, v_pool, block_table, seq_lens, out, scale: float = 0.0,
                          num_splits: int = 0, workspace=None, err_flag=None, stream=None) -> None:
    """out = GQA softmax attention of q_rot over each sequence's blocks of a paged pool."""
    B, Hq, D = q_rot.shape
    num_blocks, block_size, Hkv = k_pool.shape[0], k_pool.shape[1], k_pool.shape[2]
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = lib().rra_decode_attn_paged(_ptr(q_rot), _ptr(k_pool), _ptr(v_pool), _ptr(block_table),
                                     block_table.shape[1], _ptr(seq_lens), block_size, num_blocks, _ptr(out), B, Hq,
                                     Hkv, D, float(scale), int(num_splits), _ptr(workspace), ws_bytes,
                                     _dtype_code(q_rot), _ptr(err_flag), _stream(stream, q_rot))
    _check("rra_decode_attn_paged", st)


def rra_decode_step_contig(q, k_new, v_new, positions, q_out, k_cache, v_cache, out, rope_base: float = 10000.0,
                           rope_style: int = 0, scale: float = 0.0, num_splits: int = 0, workspace=None,
                           err_flag=None, stream=None) -> None:
    """The whole decode step on a contiguous cache: RoPE, append at positions, attention over positions+1."""
    B, Hq, D = q.shape
    Hkv, max_len = k_cache.shape[1], k_cache.shape[2]
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = lib().rra_decode_step_contig(_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(positions), _ptr(q_out), _ptr(k_cache),
                                      _ptr(v_cache), max_len, _ptr(out), B, Hq, Hkv, D, float(rope_base),
                                      int(rope_style), float(scale), int(num_splits), _ptr(workspace), ws_bytes,
                                      _dtype_code(q), _ptr(err_flag), _stream(stream, q))
    _check("rra_decode_step_contig", st)


def rra_decode_step_paged(q, k_new, v_new, positions, q_out, k_pool, v_pool, block_table, out,
                          rope_base: float = 10000.0, rope_style: int = 0, scale: float = 0.0, num_splits: int = 0,
                          workspace=None, err_flag=None, stream=None) -> None:
    """The whole decode step on a paged pool: RoPE, append at positions, attention over positions+1."""
    B, Hq, D = q.shape
    num_blocks, block_size, Hkv = k_pool.shape[0], k_pool.shape[1], k_pool.shape[2]
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = lib().rra_decode_step_paged(_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(positions), _ptr(q_out), _ptr(k_pool),
                                     _ptr(v_pool), _ptr(block_table), block_table.shape[1], block_size, num_blocks,
                                     _ptr(out), B, Hq, Hkv, D, float(rope_base), int(rope_style), float(scale),
                                     int(num_splits), _ptr(workspace), ws_bytes, _dtype_code(q), _ptr(err_flag),
                                     _stream(stream, q))
    _check("rra_decode_step_paged", st)


# --------------------------------------------------------------------------- INT8 KV cache
def _q8_layout(codes, block_table, D: int, bits: int):
    """(block_table columns, block_size, num_blocks, max_len) of an INT8 / INT4 code cache, whose
    rows must hold D * bits / 8 bytes (one code per byte, or two)."""
    if codes.shape[-1] * codes.element_size() != D * bits // 8:
        raise ValueError(f"a {bits}-bit code cache of head dim {D} has rows of {D * bits // 8} bytes, "
                         f"got {codes.shape[-1] * codes.element_size()}")
    if block_table is not None:
        return block_table.shape[1], codes.shape[1], codes.shape[0], 0
    return 0, 0, 0, codes.shape[2]


def _qfn(name: str, bits: int):
    """The INT8 (bits 8) or INT4 (bits 4) entry point of a quantised-cache call."""
    if bits not in (8, 4):
        raise ValueError("code width must be 8 or 4 bits")
    full = name if bits == 8 else name.replace("_q8", "_q4")
    return full, getattr(lib(), full)


def rra_decode_q8_num_splits(B: int, Hq: int, Hkv: int, D: int, max_tokens: int, block_size: int, num_splits: int,
                             window: int, bits: int = 8) -> int:
    name, fn = _qfn("rra_decode_q8_num_splits", bits)
    r = fn(B, Hq, Hkv, D, max_tokens, block_size, num_splits, window)
    _check(name, min(r, 0))
    return r


def rra_rope_append_q8(q, k_new, v_new, positions, q_out, k_codes, v_codes, k_scale, v_scale, k_win=None, v_win=None,
                       block_table=None, rope_base: float = 10000.0, rope_style: int = 0, err_flag=None,
                       stream=None, bits: int = 8) -> None:
    """RoPE on bf16 q / k_new, then quantised append into the INT8 (or INT4) caches and the bf16 rings."""
    B, Hq, D = q.shape
    Hkv = k_new.shape[1]
    window = k_win.shape[2] if k_win is not None else 0
    mbps, bs, nblk, max_len = _q8_layout(k_codes, block_table, D, bits)
    name, fn = _qfn("rra_rope_append_q8", bits)
    st = fn(_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(positions), _ptr(q_out), _ptr(k_codes),
                                  _ptr(v_codes), _ptr(k_scale), _ptr(v_scale), _ptr(k_win), _ptr(v_win), window,
                                  _ptr(block_table), mbps, bs, nblk, max_len, B, Hq, Hkv, D, float(rope_base),
                                  int(rope_style), _ptr(err_flag), _stream(stream, q))
    _check(name, st)


def rra_decode_attn_q8(q_rot, k_codes, v_codes, k_scale, v_scale, seq_lens, out, k_win=None, v_win=None,
                       block_table=None, scale: float = 0.0, num_splits: int = 0, workspace=None, err_flag=None,
                       stream=None, bits: int = 8) -> None:
    """Attention of q_rot over the INT8 cache (tokens older than the window) and the bf16 rings."""
    B, Hq, D = q_rot.shape
    Hkv = k_codes.shape[2] if block_table is not None else k_codes.shape[1]
    window = k_win.shape[2] if k_win is not None else 0
    mbps, bs, nblk, max_len = _q8_layout(k_codes, block_table, D, bits)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    name, fn = _qfn("rra_decode_attn_q8", bits)
    st = fn(_ptr(q_rot), _ptr(k_codes), _ptr(v_codes), _ptr(k_scale), _ptr(v_scale),
                                  _ptr(k_win), _ptr(v_win), window, _ptr(block_table), mbps, _ptr(seq_lens), bs, nblk,
                                  max_len, _ptr(out), B, Hq, Hkv, D, float(scale), int(num_splits), _ptr(workspace),
                                  ws_bytes, _ptr(err_flag), _stream(stream, q_rot))
    _check(name, st)


def rra_decode_step_q8(q, k_new, v_new, positions, q_out, k_codes, v_codes, k_scale, v_scale, out, k_win=None,
                       v_win=None, block_table=None, rope_base: float = 10000.0, rope_style: int = 0,
                       scale: float = 0.0, num_splits: int = 0, workspace=None, err_flag=None, stream=None,
                       bits: int = 8) -> None:
    """The whole step on an INT8 cache in one kernel: RoPE, quantised append, attention over positions + 1."""
    B, Hq, D = q.shape
    Hkv = k_new.shape[1]
    window = k_win.shape[2] if k_win is not None else 0
    mbps, bs, nblk, max_len = _q8_layout(k_codes, block_table, D, bits)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    name, fn = _qfn("rra_decode_step_q8", bits)
    st = fn(_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(positions), _ptr(q_out), _ptr(k_codes),
                                  _ptr(v_codes), _ptr(k_scale), _ptr(v_scale), _ptr(k_win), _ptr(v_win), window,
                                  _ptr(block_table), mbps, bs, nblk, max_len, _ptr(out), B, Hq, Hkv, D,
                                  float(rope_base), int(rope_style), float(scale), int(num_splits), _ptr(workspace),
                                  ws_bytes, _ptr(err_flag), _stream(stream, q))
    _check(name, st)


# --------------------------------------------------------------------------- speculative verify
def _cache_layout(k_cache, block_table):
    """(block_table columns, block_size, num_blocks, max_len, Hkv) of a bf16 / fp32 cache."""
    if block_table is not None:
        return block_table.shape[1], k_cache.shape[1], k_cache.shape[0], 0, k_cache.shape[2]
    return 0, 0, 0, k_cache.shape[2], k_cache.shape[1]


def rra_verify_num_splits(B: int, gamma: int, Hq: int, Hkv: int, D: int, max_tokens: int, block_size: int,
                          num_splits: int) -> int:
    r = lib().rra_verify_num_splits(B, gamma, Hq, Hkv, D, max_tokens, block_size, num_splits)
    _check("rra_verify_num_splits", min(r, 0))
    return r


def rra_verify_workspace_bytes(B: int, gamma: int, Hq: int, Hkv: int, D: int, splits: int) -> int:
    return int(lib().rra_verify_workspace_bytes(B, gamma, Hq, Hkv, D, splits))


def rra_rope_append_verify(q, k_new, v_new, positions, q_out, k_cache, v_cache, block_table=None,
                           rope_base: float = 10000.0, rope_style: int = 0, err_flag=None, stream=None) -> None:
    """RoPE on q / k_new [B, gamma, H, D] (token j at positions[b] + j) and append of the gamma tokens."""
    B, gamma, Hq, D = q.shape
    mbps, bs, nblk, max_len, Hkv = _cache_layout(k_cache, block_table)
    st = lib().rra_rope_append_verify(_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(positions), _ptr(q_out), _ptr(k_cache),
                                      _ptr(v_cache), _ptr(block_table), mbps, bs, nblk, max_len, B, gamma, Hq, Hkv, D,
                                      float(rope_base), int(rope_style), _dtype_code(q), _ptr(err_flag),
                                      _stream(stream, q))
    _check("rra_rope_append_verify", st)


def rra_verify_attn(q_rot, k_cache, v_cache, positions, out, block_table=None, scale: float = 0.0, num_splits: int = 0,
                    workspace=None, err_flag=None, stream=None) -> None:
    """out[b, j] = attention of q_rot[b, j] over tokens [0, positions[b] + j] (bf16 caches)."""
    B, gamma, Hq, D = q_rot.shape
    mbps, bs, nblk, max_len, Hkv = _cache_layout(k_cache, block_table)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = lib().rra_verify_attn(_ptr(q_rot), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), mbps, _ptr(positions), bs,
                               nblk, max_len, _ptr(out), B, gamma, Hq, Hkv, D, float(scale), int(num_splits),
                               _ptr(workspace), ws_bytes, _ptr(err_flag), _stream(stream, q_rot))
    _check("rra_verify_attn", st)


def rra_verify_step(q, k_new, v_new, positions, q_out, k_cache, v_cache, out, block_table=None,
                    rope_base: float = 10000.0, rope_style: int = 0, scale: float = 0.0, num_splits: int = 0,
                    workspace=None, err_flag=None, stream=None) -> None:
    """The whole speculative-verify step: RoPE + append of the gamma tokens, then their causal attention."""
    B, gamma, Hq, D = q.shape
    mbps, bs, nblk, max_len, Hkv = _cache_layout(k_cache, block_table)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = lib().rra_verify_step(_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(positions), _ptr(q_out), _ptr(k_cache),
                               _ptr(v_cache), _ptr(block_table), mbps, bs, nblk, max_len, _ptr(out), B, gamma, Hq, Hkv,
                               D, float(rope_base), int(rope_style), float(scale), int(num_splits), _ptr(workspace),
                               ws_bytes, _ptr(err_flag), _stream(stream, q))
    _check("rra_verify_step", st)


# --------------------------------------------------------------------------- prefill
def rra_prefill_attn(q_rot, k_cache, v_cache, positions, out, block_table=None, scale: float = 0.0, err_flag=None,
                     stream=None) -> None:
    """out[b, t] = causal attention of prompt token t (q_rot [B, T, Hq, D]) over tokens [0, positions[b] + t]."""
    B, T, Hq, D = q_rot.shape
    mbps, bs, nblk, max_len, Hkv = _cache_layout(k_cache, block_table)
    st = lib().rra_prefill_attn(_ptr(q_rot), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), mbps, _ptr(positions), bs,
                                nblk, max_len, _ptr(out), B, T, Hq, Hkv, D, float(scale), _ptr(err_flag),
                                _stream(stream, q_rot))
    _check("rra_prefill_attn", st)


def rra_prefill_step(q, k_new, v_new, positions, q_out, k_cache, v_cache, out, block_table=None,
                     rope_base: float = 10000.0, rope_style: int = 0, scale: float = 0.0, err_flag=None,
                     stream=None) -> None:
    """RoPE + append of the T prompt tokens, then their causal attention."""
    B, T, Hq, D = q.shape
    mbps, bs, nblk, max_len, Hkv = _cache_layout(k_cache, block_table)
    st = lib().rra_prefill_step(_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(positions), _ptr(q_out), _ptr(k_cache),
                                _ptr(v_cache), _ptr(block_table), mbps, bs, nblk, max_len, _ptr(out), B, T, Hq, Hkv, D,
                                float(rope_base), int(rope_style), float(scale), _ptr(err_flag), _stream(stream, q))
    _check("rra_prefill_step", st)
