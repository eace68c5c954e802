"""The C-ABI library on the host: it builds, loads, exports every declared symbol, and its
host-only functions and argument checks behave as documented (no GPU needed)."""

import ctypes
import os
import re

import numpy as np
import pytest
import torch

import oracle
from rope_gqa_paged_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
RRA_OK, RRA_EINVAL, RRA_EUNSUPPORTED, RRA_ERANGE, RRA_EWORKSPACE, RRA_ECUDA = 0, -1, -2, -3, -4, -5


@pytest.fixture(scope="module")
def rra():
    _build.build()
    from rope_gqa_paged_gb300 import rra as binding
    return binding


def _declared_symbols():
    text = open(os.path.join(ROOT, "include", "rra.h"), encoding="utf-8").read()
    return sorted(set(re.findall(r"RRA_API\s+[\w\s\*]+?\b(rra_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    syms = _declared_symbols()
    for name in ("rra_rope_append", "rra_decode_attn_contig", "rra_decode_attn_paged", "rra_kv_bytes"):
        assert name in syms


def test_library_exports_every_declared_symbol(rra):
    lib = ctypes.CDLL(_build.LIB_PATH)
    for name in _declared_symbols():
        assert hasattr(lib, name), name
    exported = set(re.findall(r" T (rra_\w+)", os.popen(f"nm -D --defined-only {_build.LIB_PATH}").read()))
    assert exported == set(_declared_symbols())


def test_kv_bytes_matches_oracle_and_pages(rra):
    rng = np.random.default_rng(0)
    for _ in range(200):
        args = [int(x) for x in rng.integers(0, 300, size=6)]
        args[3] = int(rng.integers(0, 1 << 20))
        assert rra.rra_kv_bytes(*args) == oracle.kv_cache_bytes(*args)
    assert rra.rra_kv_bytes(32, 32, 128, 1024, 1, 2) == 536870912            # 0.5 GB
    assert rra.rra_kv_bytes(32, 32, 128, 131072, 1, 2) == 64 * 2 ** 30       # 64 GB
    assert rra.rra_kv_bytes(-1, 8, 128, 10, 1, 2) == 0
    assert rra.rra_kv_bytes(1 << 30, 1 << 30, 1 << 30, 1 << 30, 1, 2) == 0  # overflow


def test_workspace_bytes(rra):
    assert rra.rra_decode_workspace_bytes(64, 32, 128, 1) == 0
    assert rra.rra_decode_workspace_bytes(0, 32, 128, 8) == 0
    b = rra.rra_decode_workspace_bytes(1, 32, 128, 128)
    assert b >= 32 * 128 * (128 + 2) * 4
    assert rra.rra_decode_workspace_bytes(2, 32, 128, 128) > b


def test_num_splits_planning(rra):
    S = rra.rra_decode_num_splits
    assert S(1, 32, 8, 128, 131072, 32, 128, rra.RRA_BF16) == 128              # explicit split count honoured
    assert S(1, 4, 2, 64, 128, 0, 0, rra.RRA_F32) == 1                         # tiny case: one split
    assert S(4, 32, 8, 128, 8192, 0, 1, rra.RRA_BF16) == 1
    # a paged split holds at most 2047 block ids: block size 1 forces more splits than asked
    assert S(1, 8, 8, 128, 65536, 1, 1, rra.RRA_BF16) > 1
    for bad, status in (((1, 6, 4, 128, 64, 0, 0, 1), RRA_EINVAL), ((1, 8, 8, 96, 64, 0, 0, 1), RRA_EUNSUPPORTED),
                        ((1, 8, 8, 128, 64, 12, 0, 1), RRA_EUNSUPPORTED), ((1, 8, 8, 128, 64, 0, 0, 7), RRA_EUNSUPPORTED),
                        ((70000, 8, 8, 128, 64, 0, 0, 1), RRA_ERANGE), ((1, 8, 8, 128, 64, 0, -1, 1), RRA_EINVAL)):
        assert rra.lib().rra_decode_num_splits(*bad) == status, bad


def test_status_strings(rra):
    for s in (RRA_OK, RRA_EINVAL, RRA_EUNSUPPORTED, RRA_ERANGE, RRA_EWORKSPACE, RRA_ECUDA):
        assert rra.rra_status_str(s) not in ("", "unknown status")
    assert rra.rra_status_str(42) == "unknown status"


@pytest.mark.skipif(torch.cuda.is_available(), reason="host-only argument checks; never given fake pointers on a GPU")
def test_argument_checks_reject_before_any_launch(rra):
    lib = rra.lib()
    P = 4096                                                                   # never dereferenced: checks fail first
    # decode contig: Hq % Hkv != 0, unsupported D, null pointer, misaligned pointer, missing workspace
    c = lib.rra_decode_attn_contig
    assert c(P, P, P, P, P, 1, 6, 4, 128, 64, 0.0, 0, None, 0, 1, None, None) == RRA_EINVAL
    assert c(P, P, P, P, P, 1, 8, 8, 96, 64, 0.0, 0, None, 0, 1, None, None) == RRA_EUNSUPPORTED
    assert c(P, None, P, P, P, 1, 8, 8, 128, 64, 0.0, 0, None, 0, 1, None, None) == RRA_EINVAL
    assert c(P + 8, P, P, P, P, 1, 8, 8, 128, 64, 0.0, 0, None, 0, 1, None, None) == RRA_EINVAL
    assert c(P, P, P, P, P, 1, 8, 8, 128, 4096, 0.0, 8, None, 0, 1, None, None) == RRA_EWORKSPACE
    assert c(P, P, P, P, P, 0, 8, 8, 128, 64, 0.0, 0, None, 0, 1, None, None) == RRA_OK   # empty batch: no-op
    # decode paged: block size not a power of two, missing table
    p = lib.rra_decode_attn_paged
    assert p(P, P, P, P, 4, P, 12, 10, P, 1, 8, 8, 128, 0.0, 0, None, 0, 1, None, None) == RRA_EUNSUPPORTED
    assert p(P, P, P, None, 4, P, 16, 10, P, 1, 8, 8, 128, 0.0, 0, None, 0, 1, None, None) == RRA_EINVAL
    # rope append: bad style, bad base, Hq % Hkv
    r = lib.rra_rope_append
    assert r(P, P, P, P, P, P, P, None, 0, 0, 0, 64, 1, 8, 8, 128, 10000.0, 2, 1, None, None) == RRA_EINVAL
    assert r(P, P, P, P, P, P, P, None, 0, 0, 0, 64, 1, 8, 8, 128, 0.5, 0, 1, None, None) == RRA_EINVAL
    assert r(P, P, P, P, P, P, P, None, 0, 0, 0, 64, 1, 6, 4, 128, 10000.0, 0, 1, None, None) == RRA_EINVAL
    assert r(P, P, P, P, P, P, P, None, 0, 0, 0, 64, 0, 8, 8, 128, 10000.0, 0, 1, None, None) == RRA_OK


def test_q8_planning(rra):
    S = rra.rra_decode_q8_num_splits
    assert S(1, 32, 8, 128, 131072, 32, 64, 128) == 64                          # the ring adds no split
    assert S(1, 32, 8, 128, 131072, 32, 64, 0) == 64
    # one split asked for, but a split spans at most 255 block ids of 16 tokens
    assert S(4, 32, 8, 128, 8192, 16, 1, 16) == 3
    lib = rra.lib()
    for bad, status in (((1, 8, 8, 128, 1024, 16, 0, 12), RRA_EUNSUPPORTED),   # window not a multiple of 8
                        ((1, 8, 8, 128, 1024, 16, 0, -8), RRA_EINVAL),
                        ((1, 8, 8, 128, 1024, 4, 0, 16), RRA_EUNSUPPORTED),    # blocks under 8 tokens
                        ((1, 8, 8, 128, 32, 0, 0, 16), RRA_EUNSUPPORTED),      # contiguous cache under one tile
                        ((1, 8, 8, 96, 1024, 16, 0, 16), RRA_EUNSUPPORTED),
                        ((1, 6, 4, 128, 1024, 16, 0, 16), RRA_EINVAL)):
        assert lib.rra_decode_q8_num_splits(*bad) == status, bad


@pytest.mark.skipif(torch.cuda.is_available(), reason="host-only argument checks; never given fake pointers on a GPU")
def test_q8_argument_checks_reject_before_any_launch(rra):
    lib = rra.lib()
    P = 4096
    a = lib.rra_decode_attn_q8
    # (q_rot, kc, vc, ks, vs, kw, vw, W, table, mbps, lens, bs, nblk, max_len, out, B, Hq, Hkv, D, scale, splits,
    #  ws, ws_bytes, err, stream)
    ok = [P, P, P, P, P, P, P, 16, P, 64, P, 16, 100, 0, P, 1, 8, 8, 128, 0.0, 1, None, 0, None, None]
    def call(**kw):
        args = list(ok)
        names = ["q", "kc", "vc", "ks", "vs", "kw", "vw", "W", "table", "mbps", "lens", "bs", "nblk", "max_len",
                 "out", "B", "Hq", "Hkv", "D", "scale", "splits", "ws", "ws_bytes", "err", "stream"]
        for k, v in kw.items():
            args[names.index(k)] = v
        return a(*args)
    assert call(B=0) == RRA_OK
    assert call(ks=None) == RRA_EINVAL                                          # scales are required
    assert call(kw=None) == RRA_EINVAL                                          # a window needs its rings
    assert call(W=12) == RRA_EUNSUPPORTED
    assert call(bs=4, nblk=100) == RRA_EUNSUPPORTED
    assert call(kc=P + 8) == RRA_EINVAL
    assert call(splits=8) == RRA_EWORKSPACE                                     # several splits need scratch
    assert call(table=None, max_len=32) == RRA_EUNSUPPORTED                    # contiguous shorter than a tile
    r = lib.rra_rope_append_q8
    assert r(P, P, P, P, P, P, P, None, P, P, P, 16, None, 0, 0, 0, 256, 1, 8, 8, 128, 10000.0, 0, None,
             None) == RRA_EINVAL                                                # missing K scale
    assert r(P, P, P, P, P, P, P, P, P, None, P, 16, None, 0, 0, 0, 256, 1, 8, 8, 128, 10000.0, 0, None,
             None) == RRA_EINVAL                                                # missing k ring


def test_verify_planning(rra):
    S = rra.rra_verify_num_splits
    assert S(64, 4, 32, 8, 128, 8192, 16, 4) == 4
    assert S(1, 4, 32, 8, 128, 131072, 32, 64) == 64
    lib = rra.lib()
    for bad, status in (((1, 0, 32, 8, 128, 1024, 16, 0), RRA_EINVAL),        # gamma 0
                        ((1, 17, 32, 8, 128, 1024, 16, 0), RRA_EUNSUPPORTED),  # gamma above 16
                        ((1, 4, 32, 8, 128, 1024, 4, 0), RRA_EUNSUPPORTED),   # blocks under 8 tokens
                        ((1, 4, 32, 8, 128, 32, 0, 0), RRA_EUNSUPPORTED),     # contiguous cache under one tile
                        ((1, 4, 6, 4, 128, 1024, 16, 0), RRA_EINVAL)):
        assert lib.rra_verify_num_splits(*bad) == status, bad
    # 16 partial rows per (sequence, KV head, head slice): MQA with gamma 4 takes 8 slices of 4 heads
    assert rra.rra_verify_workspace_bytes(2, 4, 32, 1, 128, 4) == rra.rra_verify_workspace_bytes(1, 4, 32, 8, 128, 4) * 2
    assert rra.rra_verify_workspace_bytes(2, 4, 32, 8, 128, 1) == 0


@pytest.mark.skipif(torch.cuda.is_available(), reason="host-only argument checks; never given fake pointers on a GPU")
def test_prefill_and_verify_argument_checks(rra):
    lib = rra.lib()
    P = 4096
    a = lib.rra_prefill_attn
    # (q, kc, vc, table, mbps, pos, bs, nblk, max_len, out, B, T, Hq, Hkv, D, scale, err, stream)
    assert a(P, P, P, P, 64, P, 16, 100, 0, P, 0, 8, 32, 8, 128, 0.0, None, None) == RRA_OK        # empty batch
    assert a(P, P, P, P, 64, P, 16, 100, 0, P, 1, 0, 32, 8, 128, 0.0, None, None) == RRA_EINVAL    # no prompt
    assert a(P, P, P, P, 64, P, 4, 100, 0, P, 1, 8, 32, 8, 128, 0.0, None, None) == RRA_EUNSUPPORTED  # block < 8
    assert a(P, P, P, None, 0, P, 0, 0, 32, P, 1, 8, 32, 8, 128, 0.0, None, None) == RRA_EUNSUPPORTED  # short cache
    assert a(P + 8, P, P, P, 64, P, 16, 100, 0, P, 1, 8, 32, 8, 128, 0.0, None, None) == RRA_EINVAL  # misaligned
    big_t = (1 << 30) - 1                                                                           # CTAs
    assert a(P, P, P, P, 1 << 20, P, 1024, 100, 0, P, 1, big_t, 256, 8, 128, 0.0, None, None) == RRA_ERANGE
    assert a(P, P, P, P, 1 << 20, P, 1024, 100, 0, P, 0, big_t, 64, 8, 128, 0.0, None, None) == RRA_OK
    v = lib.rra_verify_attn
    # (q, kc, vc, table, mbps, pos, bs, nblk, max_len, out, B, gamma, Hq, Hkv, D, scale, splits, ws, ws_bytes, err, st)
    assert v(P, P, P, P, 64, P, 16, 100, 0, P, 1, 4, 32, 8, 128, 0.0, 8, None, 0, None, None) == RRA_EWORKSPACE
    assert v(P, P, P, P, 64, P, 16, 100, 0, P, 1, 20, 32, 8, 128, 0.0, 0, None, 0, None, None) == RRA_EUNSUPPORTED


@pytest.mark.parametrize("bits,width,dtype,ok", [(8, 128, torch.int8, True), (4, 64, torch.uint8, True),
                                                 (4, 128, torch.int8, False), (8, 64, torch.uint8, False)])
def test_binding_checks_the_code_row_width(rra, bits, width, dtype, ok):
    """A code cache whose rows do not hold D * bits / 8 bytes is refused by the binding."""
    codes = torch.zeros(4, 16, 2, width, dtype=dtype)
    table = torch.zeros(1, 4, dtype=torch.int32)
    if ok:
        assert rra._q8_layout(codes, table, 128, bits) == (4, 16, 4, 0)
    else:
        with pytest.raises(ValueError):
            rra._q8_layout(codes, table, 128, bits)
