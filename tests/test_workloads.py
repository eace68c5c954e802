"""The seeded input generator: determinism, block tables, shared prefixes, NaN poisoning (CPU)."""

import math

import numpy as np
import pytest

from workloads import CONFIGS, make_inputs, reduced


def _finite(x, dtype):
    if x.dtype == np.int8:                                   # INT8 codes: -128 is the poison
        return x != -128
    if x.dtype == np.uint8:                                  # packed INT4 codes: 0x88 (two -8 codes)
        return x != 0x88
    if dtype == "bf16":
        return (x & 0x7F80) != 0x7F80
    return np.isfinite(x)


@pytest.mark.parametrize("name", list(CONFIGS))
def test_full_size_configs_are_consistent(name):
    cfg = CONFIGS[name]
    assert cfg.n_q_heads % cfg.n_kv_heads == 0
    longest = cfg.seq_len if cfg.seq_len is not None else cfg.len_range[1]
    assert longest <= cfg.capacity
    if cfg.layout == "paged":
        n_shared = cfg.shared_prefix_tokens // cfg.block_size
        need = n_shared + cfg.batch * (math.ceil(longest / cfg.block_size) - n_shared)
        assert need <= cfg.num_blocks


@pytest.mark.parametrize("name", list(CONFIGS))
def test_reduced_inputs_structure(name):
    cfg = reduced(CONFIGS[name], batch=min(CONFIGS[name].batch, 5))
    a = make_inputs(cfg)
    b = make_inputs(cfg)
    for f in ("q", "k_new", "v_new", "k_cache", "v_cache", "lengths"):
        assert getattr(a, f).tobytes() == getattr(b, f).tobytes()
    assert np.array_equal(a.positions, a.lengths - cfg.gamma)
    assert a.q.shape[:-2] == ((cfg.batch,) if cfg.gamma == 1 else (cfg.batch, cfg.gamma))
    L = a.lengths
    # slots read from the main cache: [0, first); the new tokens' slots and the window are poisoned
    first = [max(0, int(x) - max(cfg.window, 1)) if cfg.int8 else int(x) - cfg.gamma for x in L]
    if cfg.int8 and cfg.window:
        W = cfg.window
        for bb in range(cfg.batch):
            live = [t % W for t in range(max(0, int(L[bb]) - W), int(L[bb]) - 1)]   # older window tokens
            assert _finite(a.k_win[bb][:, live], "bf16").all()
            dead = sorted(set(range(W)) - set(live))
            assert (int(L[bb]) - 1) % W in dead and not _finite(a.v_win[bb][:, dead], "bf16").any()
    if cfg.layout == "contiguous":
        for bb in range(cfg.batch):
            assert _finite(a.k_cache[bb, :, : first[bb]], cfg.dtype).all()
            assert not _finite(a.k_cache[bb, :, first[bb]:], cfg.dtype).any()
        return
    bs, t = cfg.block_size, a.block_table
    n_shared = cfg.shared_prefix_tokens // bs
    owned = []
    for bb in range(cfg.batch):
        nb = math.ceil(int(L[bb]) / bs)
        assert np.all((t[bb, :nb] >= 0) & (t[bb, :nb] < cfg.num_blocks))
        assert np.all(t[bb, nb:] == -1)
        assert np.array_equal(t[bb, :n_shared], t[0, :n_shared])
        owned.extend(t[bb, n_shared:nb].tolist())
        for tok in range(first[bb]):                        # every token read from the cache is finite
            assert _finite(a.k_cache[t[bb, tok // bs], tok % bs], cfg.dtype).all()
        for tok in range(max(first[bb], n_shared * bs), int(L[bb])):   # the rest of the sequence is poisoned
            assert not _finite(a.v_cache[t[bb, tok // bs], tok % bs], cfg.dtype).any()
    owned.extend(t[0, :n_shared].tolist())
    assert len(owned) == len(set(owned))                     # private blocks are never shared
    unused = np.setdiff1d(np.arange(cfg.num_blocks), owned)
    if unused.size:
        assert not _finite(a.k_cache[unused], cfg.dtype).any()


@pytest.mark.parametrize("name", ["batched_paged_int8", "batched_paged_int4", "long_context_int4"])
def test_bench_device_workload_matches_the_code_width(name):
    """The bench's device-drawn caches have the storage of the numpy recipe: one INT8 code per
    byte, or two INT4 codes per byte with the even dimension in the low nibble, and the recipe's
    scales."""
    import torch

    import bench
    from oracle import quant
    cfg = reduced(CONFIGS[name], 64, batch=2)
    w, _ = bench.device_workload(cfg, 0, torch.device("cpu"))
    kc = w["k_cache"]
    assert kc.dtype == (torch.int8 if cfg.code_bits == 8 else torch.uint8)
    assert kc.shape[-1] == cfg.head_dim * cfg.code_bits // 8
    codes = quant.load_codes(kc.numpy(), cfg.code_bits)
    m = (1 << (cfg.code_bits - 1)) - 1
    assert codes.min() >= -m and codes.max() <= m and len(np.unique(codes)) > m
    ref = make_inputs(cfg)
    assert np.array_equal(w["k_scale"].numpy(), ref.k_scale) and np.array_equal(w["v_scale"].numpy(), ref.v_scale)
