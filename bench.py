#!/usr/bin/env python3
"""Decode-step benchmark: RoPE + KV append + split-K GQA decode attention on one GB300.

One step = one pass of the whole path over one batch: rra_rope_append, then the decode
kernel (and the split merge when there is more than one split). Prints ONE JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Under torchrun (N > 1) every rank runs an independent replica on its own GPU with its
own seeded batch (no collective on the data path); the time is the max over ranks and
the value counts the KV bytes of all ranks.
"""

from __future__ import annotations

import sys

if "--impl" in sys.argv and "reference" in sys.argv or "--cpu-worker" in sys.argv:
    import os as _os
    for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS"):
        _os.environ[_v] = "1"           # the oracle runs on exactly one host core

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from workloads import CONFIGS, make_inputs, make_structure  # noqa: E402

METRIC = "decode-attn KV GB/s & % of GB300 HBM peak; decode steps/s per layer"
PREFILL_METRIC = "prefill causal attention TFLOP/s & % of GB300 bf16 tensor peak"
UNIT = "GB/s"
DEFAULT_WORKLOAD = "batched_paged"
EXTRA_WORKLOAD = "long_context"
# keys of a workload record that the extra record does not repeat (they describe the whole line)
SHARED_KEYS = ("metric", "n_gpus", "steps", "warmup", "higher_is_better", "scaling", "vs_baseline", "data",
               "cpu_baseline")
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 2 ** 20
KERNEL_SOURCES = ["rope_gqa_paged_gb300/csrc/decode_mma.cuh", "rope_gqa_paged_gb300/csrc/decode_kernels.cuh",
                  "rope_gqa_paged_gb300/csrc/rra_device.cuh", "rope_gqa_paged_gb300/csrc/decode_paged.cu",
                  "rope_gqa_paged_gb300/csrc/decode_contig.cu", "rope_gqa_paged_gb300/csrc/rra_internal.h"]
KERNEL_SOURCES_INT8 = KERNEL_SOURCES + ["rope_gqa_paged_gb300/csrc/decode_q8.cuh",
                                        "rope_gqa_paged_gb300/csrc/decode_q8.cu"]
KERNEL_SOURCES_VERIFY = KERNEL_SOURCES + ["rope_gqa_paged_gb300/csrc/verify.cuh", "rope_gqa_paged_gb300/csrc/verify.cu",
                                          "rope_gqa_paged_gb300/csrc/rope_append.cu"]
KERNEL_SOURCES_PREFILL = KERNEL_SOURCES_VERIFY + ["rope_gqa_paged_gb300/csrc/prefill.cuh",
                                                  "rope_gqa_paged_gb300/csrc/prefill_tc.cuh",
                                                  "rope_gqa_paged_gb300/csrc/tcgen05.cuh",
                                                  "rope_gqa_paged_gb300/csrc/prefill.cu"]


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=50)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", choices=sorted(CONFIGS), default=None,
                   help=f"default: {DEFAULT_WORKLOAD}, with a {EXTRA_WORKLOAD} record in the same line")
    p.add_argument("--no-extra", action="store_true", help=f"default workload only (no {EXTRA_WORKLOAD} record)")
    p.add_argument("--num-splits", type=int, default=-1, help="-1: the workload's own setting (0 = library choice)")
    p.add_argument("--batch", type=int, default=0,
                   help="override the batch (a smaller case for profiling; the paged pool shrinks to fit)")
    p.add_argument("--cpu-seconds", type=float, default=12.0, help="bounded CPU oracle sample (seconds)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-graph", action="store_true", help="time eager launches instead of a captured step")
    p.add_argument("--cpu-worker", action="store_true", help=argparse.SUPPRESS)
    return p.parse_args(argv)


# ---------------------------------------------------------------------------- helpers
def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)), int(os.environ.get("WORLD_SIZE", 1))


def aggregate(ms_per_step: float, kv_bytes: int, world: int, device=None):
    """Max of the step time and sum of the KV bytes over ranks (a no-op for one rank)."""
    if world <= 1:
        return ms_per_step, kv_bytes
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms_per_step], dtype=torch.float64, device=device)
    b = torch.tensor([float(kv_bytes)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(b, op=dist.ReduceOp.SUM)
    return float(t.item()), int(b.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def tensor_peak():
    """Sustained bf16 dense TFLOP/s (the prefill kernel runs for tens to hundreds of ms)."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops_sustained"]), "measured (MEASURED_PEAKS.json bf16_tflops_sustained)"
    except (OSError, KeyError, ValueError):
        return 1700.0, "fallback (1.7 PFLOP/s sustained)"


def prefill_flops(cfg, lengths) -> int:
    """Causal attention FLOPs of a prefill step: 4 D Hq per (prompt token, attended key)."""
    T = cfg.gamma
    keys = sum(T * (int(L) - T) + T * (T + 1) // 2 for L in lengths)
    return 4 * cfg.head_dim * cfg.n_q_heads * keys


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def kernel_sources(cfg) -> list:
    """The sources of the kernels a workload's step runs (its recorded traffic is stale once one changes)."""
    if cfg.gamma > 16:
        return KERNEL_SOURCES_PREFILL
    if cfg.gamma > 1:
        return KERNEL_SOURCES_VERIFY
    return KERNEL_SOURCES_INT8 if cfg.int8 else KERNEL_SOURCES


def kernel_source_hash(cfg) -> str:
    h = hashlib.sha256()
    for rel in kernel_sources(cfg):
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


TRAFFIC_FILE = os.path.join("profiles", "traffic.json")


def recorded_traffic(workload: str):
    """DRAM bytes per launch of the workload's dominant kernel from the committed ncu capture
    (``profiles/traffic.json``, one record per workload), if its kernel sources are unchanged."""
    if workload not in CONFIGS:
        return None
    try:
        with open(os.path.join(ROOT, TRAFFIC_FILE), encoding="utf-8") as f:
            rec = json.load(f).get(workload)
    except (OSError, ValueError):
        return None
    if not isinstance(rec, dict) or rec.get("kernel_source_sha256") != kernel_source_hash(CONFIGS[workload]):
        return None
    t = rec.get("traffic_bytes_per_launch")
    return int(t) if isinstance(t, int) and t > 0 else None


class ClockSampler:
    """nvidia-smi clock / throttle samples every 200 ms while the timed region runs."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_uuid):
        self.path = os.path.join(tempfile.gettempdir(), f"rra_clocks_{os.getpid()}.csv")
        self.proc = None
        self.gpu = gpu_uuid

    def start(self):
        os.makedirs(os.path.dirname(self.path), exist_ok=True)
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200"]
        if self.gpu:
            cmd += ["-i", self.gpu]
        try:
            self.proc = subprocess.Popen(cmd, stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        try:
            with open(self.path) as f:
                lines = f.readlines()
        except OSError:
            lines = []
        try:
            os.remove(self.path)
        except OSError:
            pass
        return summarize_clock_samples(lines)


def summarize_clock_samples(lines):
    """nvidia-smi rows in ClockSampler.FIELDS order -> {sm_mhz (median), sm_max_mhz, reasons
    (throttle reasons seen active in any sample), samples}, or None without a usable row."""
    sm, mx, reasons = [], [], set()
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    for ln in lines:
        r = [x.strip() for x in ln.split(",")]
        if len(r) < 8:
            continue
        try:
            sm.append(float(r[0]))
            mx.append(float(r[1]))
        except ValueError:
            continue
        for n, v in zip(names, r[4:8]):
            if v.lower() == "active":
                reasons.add(n)
    if not sm:
        return None
    return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------- our arm
def capture_repeat(fn, times: int, device):
    """One CUDA graph of ``fn()`` recorded ``times`` times back to back."""
    import torch
    side = torch.cuda.Stream(device=device)
    side.wait_stream(torch.cuda.current_stream(device))
    with torch.cuda.stream(side):
        fn()
    torch.cuda.current_stream(device).wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(times):
            fn()
    return g


def workload_config(args):
    cfg = CONFIGS[args.workload or DEFAULT_WORKLOAD]
    if args.batch and args.batch != cfg.batch:
        import dataclasses
        import math
        kw = {"batch": args.batch, "name": cfg.name}
        if cfg.layout == "paged":
            longest = cfg.seq_len if cfg.seq_len is not None else cfg.len_range[1]
            need = args.batch * math.ceil(longest / cfg.block_size) + 8
            kw["num_blocks"] = min(cfg.num_blocks, need) if args.batch < cfg.batch else max(cfg.num_blocks, need)
        cfg = dataclasses.replace(cfg, **kw)
    return cfg


def device_workload(cfg, seed, device):
    """Seeded inputs at full size: lengths and block tables from the numpy recipe, cache
    values N(0,1) drawn on the device (torch Philox, seeded), stored in the workload dtype."""
    import torch
    dt = torch.bfloat16 if cfg.dtype == "bf16" else torch.float32
    lengths, table = make_structure(cfg, seed)
    g = torch.Generator(device=device)
    g.manual_seed(1000003 * seed + 17)
    B, Hq, Hkv, D = cfg.batch, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim
    shape = (B, Hkv, cfg.max_len, D) if cfg.layout == "contiguous" else (cfg.num_blocks, cfg.block_size, Hkv, D)
    lead = (B,) if cfg.gamma == 1 else (B, cfg.gamma)
    per_unit = 32.0 if cfg.code_bits == 8 else 1.75   # codes per unit of N(0,1), as in the numpy recipe
    if cfg.int8:  # codes: N(0,1) at a resolution of 1/per_unit, clipped; fixed per-head scales; bf16 rings
        m = (1 << (cfg.code_bits - 1)) - 1

        def codes():
            c = torch.randn(shape, generator=g, device=device).mul_(per_unit).round_().clamp_(-m, m).to(torch.int8)
            if cfg.code_bits == 8:
                return c
            n = c.to(torch.uint8) & 0x0F                   # INT4: two codes per byte, the even dim low
            return (n[..., 0::2] | (n[..., 1::2] << 4)).contiguous()

        kc, vc = codes(), codes()
    else:
        kc = torch.randn(shape, generator=g, device=device, dtype=dt)
        vc = torch.randn(shape, generator=g, device=device, dtype=dt)
    w = {
        "k_cache": kc,
        "v_cache": vc,
        "q": torch.randn(*lead, Hq, D, generator=g, device=device, dtype=dt),
        "k_new": torch.randn(*lead, Hkv, D, generator=g, device=device, dtype=dt),
        "v_new": torch.randn(*lead, Hkv, D, generator=g, device=device, dtype=dt),
        "positions": torch.from_numpy(lengths - cfg.gamma).to(device),
        "seq_lens": torch.from_numpy(lengths).to(device),
        "block_table": torch.from_numpy(table).to(device) if table is not None else None,
    }
    if cfg.int8:
        h = np.arange(Hkv)
        w["k_scale"] = torch.from_numpy(((1.0 + (h % 4) / 8.0) / per_unit).astype(np.float32)).to(device)
        w["v_scale"] = torch.from_numpy(((1.0 + ((h + 2) % 4) / 8.0) / per_unit).astype(np.float32)).to(device)
        w["k_win"] = w["v_win"] = None
        if cfg.window:
            w["k_win"] = torch.randn(B, Hkv, cfg.window, D, generator=g, device=device, dtype=torch.bfloat16)
            w["v_win"] = torch.randn(B, Hkv, cfg.window, D, generator=g, device=device, dtype=torch.bfloat16)
    return w, lengths


def run_ours(args):
    import torch

    from rope_gqa_paged_gb300 import _build

    rank, local_rank, world = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group(backend="nccl" if torch.cuda.is_available() else "gloo")
    if not torch.cuda.is_available():
        print(json.dumps({"metric": METRIC, "error": "no CUDA device"}))
        return 1
    torch.cuda.set_device(local_rank)
    device = torch.device("cuda", local_rank)
    _build.build()                                    # no-op when the library is current

    cfg = workload_config(args)
    line = measure(args, cfg, device, rank, world)
    # The default run also measures the 128K long-context step (the second configuration the
    # >= 70 %-of-HBM target names) in the same process, at its configured 128 splits.
    extra = None
    if args.workload is None and not args.no_extra:
        import gc
        gc.collect()
        torch.cuda.empty_cache()
        extra = measure(args, CONFIGS[EXTRA_WORKLOAD], device, rank, world, splits_override=-1)
    if rank != 0:
        return 0
    if extra is not None:
        line[EXTRA_WORKLOAD] = {k: v for k, v in extra.items() if k not in SHARED_KEYS}
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(cfg.name, args.cpu_seconds)
    print(json.dumps(line), flush=True)
    return 0


def measure(args, cfg, device, rank, world, splits_override=None):
    """Times one workload's step (per-kernel eager times, the captured step, clocks, e2e) and
    returns its JSON record (without the CPU baseline)."""
    import torch

    from rope_gqa_paged_gb300 import DecodeStep, DecodeStepQ8, PrefillStep, VerifyStep

    nsplit = args.num_splits if splits_override is None else splits_override
    splits_arg = cfg.num_splits if nsplit < 0 else nsplit
    w, lengths = device_workload(cfg, cfg.seed + rank, device)
    # The numerator is the unique KV bytes DRAM must deliver: a shared prefix is counted once.
    # Without prefix sharing this equals the logical bytes the attention consumes.
    kv_bytes = cfg.unique_kv_bytes(lengths)
    logical_bytes = cfg.kv_bytes(lengths)
    prefill = cfg.gamma > 16
    if prefill:   # the work is causal attention FLOPs, reported in TFLOP/s
        work, div, unit, metric = prefill_flops(cfg, lengths), 1e12, "TFLOP/s", PREFILL_METRIC
    else:         # the work is KV bytes, reported in GB/s
        work, div, unit, metric = kv_bytes, 1e9, UNIT, METRIC
    if prefill:
        step = PrefillStep(cfg.batch, cfg.gamma, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim, w["k_cache"],
                           w["v_cache"], w["block_table"], rope_base=cfg.rope_base)
    elif cfg.gamma > 1:
        step = VerifyStep(cfg.batch, cfg.gamma, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim, w["k_cache"],
                          w["v_cache"], w["block_table"], num_splits=splits_arg, rope_base=cfg.rope_base)
    elif cfg.int8:
        step = DecodeStepQ8(cfg.batch, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim, w["k_cache"], w["v_cache"],
                            w["k_scale"], w["v_scale"], w["k_win"], w["v_win"], w["block_table"],
                            num_splits=splits_arg, rope_base=cfg.rope_base, bits=cfg.code_bits)
    else:
        step = DecodeStep(cfg.batch, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim, w["k_cache"], w["v_cache"],
                          w["block_table"], num_splits=splits_arg, rope_base=cfg.rope_base)
    # the fused step is one kernel for INT8 caches and for bf16 with the tensor-core path, else rope + decode
    mma_path = cfg.int8 or (cfg.dtype == "bf16" and (
        (cfg.layout == "paged" and cfg.block_size >= 8) or
        (cfg.layout == "contiguous" and cfg.max_len >= 16384 // (2 * cfg.head_dim))))
    # one kernel: the fused decode step (tensor-core path) and the verify step up to 8 new tokens
    launches_per_step = 1 if (mma_path and cfg.gamma == 1) or 1 < cfg.gamma <= 8 else 2
    attend_arg = w["positions"] if cfg.gamma > 1 else w["seq_lens"]   # verify: lengths follow the positions
    flush = None
    if 2 * kv_bytes < 3 * L2_BYTES:                     # inputs not much larger than L2: flush between steps
        flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)

    for _ in range(max(args.warmup, 3)):
        step(w["q"], w["k_new"], w["v_new"], w["positions"], w["seq_lens"])
        step(w["q"], w["k_new"], w["v_new"], w["positions"])
    torch.cuda.synchronize(device)
    step.reset_errors()

    K = args.steps
    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(device).uuid)
    except Exception:
        pass

    # (1) per-kernel times: eager launches with events between the two library calls
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    barrier(world)
    torch.cuda.synchronize(device)
    for i in range(K):
        if flush is not None:
            flush.fill_(i & 0xFF)
        ev[i][0].record(stream)
        step.rope_append(w["q"], w["k_new"], w["v_new"], w["positions"])
        ev[i][1].record(stream)
        step.attend(attend_arg)
        ev[i][2].record(stream)
    torch.cuda.synchronize(device)
    rope_ms = [ev[i][0].elapsed_time(ev[i][1]) for i in range(K)]
    dec_ms = [ev[i][1].elapsed_time(ev[i][2]) for i in range(K)]
    eager_ms = sum(ev[i][0].elapsed_time(ev[i][2]) for i in range(K)) / K
    # the fused step (the dominant and, for bf16, only kernel of the step), eager
    fev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    torch.cuda.synchronize(device)
    for i in range(K):
        if flush is not None:
            flush.fill_(i & 0xFF)
        fev[i][0].record(stream)
        step(w["q"], w["k_new"], w["v_new"], w["positions"])
        fev[i][1].record(stream)
    torch.cuda.synchronize(device)
    fused_ms = sum(fev[i][0].elapsed_time(fev[i][1]) for i in range(K)) / K

    # (2) the step, K times back to back. Inputs larger than L2: all K steps captured in one CUDA
    # graph (a decode loop's shape: each decode kernel overlaps its launch and first loads with
    # the end of the kernel before it), timed by events around that one replay. Inputs that fit
    # in L2: one graph of K x (2xL2 flush, step) and one of the K flushes alone, each replayed once
    # between events; the step time is the difference over K (events around every replay of a
    # one-step graph add about 6 us that a trivial kernel measures too: reported beside it).
    graph_note = "eager launches"
    multi = fgraph = None
    if not args.no_graph:
        try:
            single = step.capture(w["q"], w["k_new"], w["v_new"], w["positions"])
            if flush is None:
                multi = step.capture(w["q"], w["k_new"], w["v_new"], w["positions"], repeat=K)
            else:
                multi = step.capture(w["q"], w["k_new"], w["v_new"], w["positions"], repeat=K,
                                     before=lambda: flush.fill_(1))
                fgraph = capture_repeat(lambda: flush.fill_(1), K, device)
            step.graph = single
            graph_note = (f"one CUDA graph of {K} fused steps, replayed once" if flush is None else
                          f"one CUDA graph of {K} x (2xL2 flush + fused step) minus one of the {K} flushes, "
                          "each replayed once")
        except Exception as e:  # capture is an optimisation; report how the step was timed
            step.graph, multi, fgraph = None, None, None
            graph_note = f"eager launches (graph capture failed: {type(e).__name__})"

    def one_step():
        if step.graph is not None:
            step.replay()
        else:
            step(w["q"], w["k_new"], w["v_new"], w["positions"])

    # per-step replays (the reported time when L2 is flushed; otherwise the single-step figure)
    sev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    barrier(world)
    torch.cuda.synchronize(device)
    for i in range(K):
        if flush is not None:
            flush.fill_(i & 0xFF)
        sev[i][0].record(stream)
        one_step()
        sev[i][1].record(stream)
    torch.cuda.synchronize(device)
    single_ms = sum(sev[i][0].elapsed_time(sev[i][1]) for i in range(K)) / K

    sampler = ClockSampler(uuid)
    sampler.start()
    t_warm = time.perf_counter()
    while time.perf_counter() - t_warm < 0.6:     # load the GPU so the clock samples see it busy
        (multi.replay() if multi is not None else one_step())
        torch.cuda.synchronize(device)
    flush_ms = None
    if multi is not None:
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world)
        torch.cuda.synchronize(device)
        ev0.record(stream)
        multi.replay()
        ev1.record(stream)
        torch.cuda.synchronize(device)
        ms_local = ev0.elapsed_time(ev1) / K
        if fgraph is not None:          # the flushes alone, timed the same way
            ev0.record(stream)
            fgraph.replay()
            ev1.record(stream)
            torch.cuda.synchronize(device)
            flush_ms = ev0.elapsed_time(ev1) / K
            ms_local -= flush_ms
        barrier(world)
    else:
        barrier(world)
        torch.cuda.synchronize(device)
        for i in range(K):
            if flush is not None:
                flush.fill_(i & 0xFF)
            sev[i][0].record(stream)
            one_step()
            sev[i][1].record(stream)
        torch.cuda.synchronize(device)
        barrier(world)
        ms_local = sum(sev[i][0].elapsed_time(sev[i][1]) for i in range(K)) / K
    clocks = sampler.stop()
    step.graph = single if step.graph is not None else None
    err_bits = step.error_bits()

    # (3) end to end through the public API: pinned host inputs in, host output back, every step
    e2e = None
    if not args.no_e2e:
        # The step's inputs (q, k_new, v_new, positions) live in one pinned host buffer and one
        # device buffer (16-byte aligned parts), so each step makes one host->device copy and one
        # device->host copy of the output, in the step's stream.
        names = ("q", "k_new", "v_new", "positions")
        offs, total = {}, 0
        for k in names:
            offs[k] = total
            total += (w[k].numel() * w[k].element_size() + 15) // 16 * 16
        hbuf = torch.empty(total, dtype=torch.uint8).pin_memory()
        dbuf = torch.empty(total, dtype=torch.uint8, device=device)

        def part(buf, k):
            n = w[k].numel() * w[k].element_size()
            return buf[offs[k]:offs[k] + n].view(w[k].dtype).view(w[k].shape)

        hv, dv = {k: part(hbuf, k) for k in names}, {k: part(dbuf, k) for k in names}
        for k in names:
            hv[k].copy_(w[k].cpu())
        dbuf.copy_(hbuf)
        out_host = torch.empty(step.out.shape, dtype=step.out.dtype).pin_memory()
        if step.graph is not None:   # one graph: input copy in, the step on the device buffer's parts, output out
            step.capture(dv["q"], dv["k_new"], dv["v_new"], dv["positions"],
                         before=lambda: dbuf.copy_(hbuf, non_blocking=True),
                         after=lambda: out_host.copy_(step.out, non_blocking=True))
        h2d = total
        d2h = out_host.numel() * out_host.element_size()
        e_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
        barrier(world)
        torch.cuda.synchronize(device)
        for i in range(K):
            if flush is not None:
                flush.fill_(i & 0xFF)
            e_ev[i][0].record(stream)
            if step.graph is not None:
                step.replay()
            else:
                dbuf.copy_(hbuf, non_blocking=True)
                out = step(dv["q"], dv["k_new"], dv["v_new"], dv["positions"])
                out_host.copy_(out, non_blocking=True)
            e_ev[i][1].record(stream)
        torch.cuda.synchronize(device)
        barrier(world)
        e2e_ms = sum(e_ev[i][0].elapsed_time(e_ev[i][1]) for i in range(K)) / K
        e2e_ms, e2e_work = aggregate(e2e_ms, work, world, device)
        e2e = {"value": round(e2e_work / (e2e_ms * 1e-3) / div, 2), "unit": unit, "ms_per_step": round(e2e_ms, 4),
               "h2d_bytes_per_step": h2d * world, "d2h_bytes_per_step": d2h * world}

    ms, total_work = aggregate(ms_local, work, world, device)
    dec_avg = sum(dec_ms) / K
    if prefill:   # the dominant kernel is the attention itself (the append is ~1 % of the step)
        peak, peak_src = tensor_peak()
        achieved = work / (dec_avg * 1e-3) / div
    else:
        peak, peak_src = hbm_peak()
        peak_src = f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)"
        # the fused step's kernel (decode, or verify up to 8 new tokens); above that the verify attention launch
        achieved = work / ((dec_avg if cfg.gamma > 8 else fused_ms) * 1e-3) / div
    value = total_work / (ms * 1e-3) / div
    line = {
        "metric": metric, "value": round(value, 2), "unit": unit, "n_gpus": world, "steps": K,
        "warmup": max(args.warmup, 3), "ms_per_step": round(ms, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": f"int{cfg.code_bits} K/V codes + bf16 window, f16 mma, f32 softmax" if cfg.int8 else cfg.dtype, "data": "synthetic (seeded N(0,1); lengths/tables from the recipe)",
        "config": {
            "workload": cfg.name, "description": cfg.description, "batch_per_gpu": cfg.batch,
            "n_q_heads": cfg.n_q_heads, "n_kv_heads": cfg.n_kv_heads, "head_dim": cfg.head_dim,
            "layout": cfg.layout, "block_size": cfg.block_size or None,
            "seq_lens": (f"U[{cfg.len_range[0]},{cfg.len_range[1]}] mean {float(np.mean(lengths)):.1f}"
                         if cfg.len_range else cfg.seq_len),
            "num_splits": step.splits, "kv_bytes_per_step_per_gpu": kv_bytes,
            "new_tokens_per_sequence": cfg.gamma,
            "work_per_step_per_gpu": work, "work_unit": "FLOP" if prefill else "byte",
            "logical_kv_bytes_per_step_per_gpu": logical_bytes,
            "logical_kv_gbs": round(logical_bytes * world / (ms * 1e-3) / 1e9, 2),
            "l2": ("flushed before every step (2x L2 write in the step graph; the flushes' own time, "
                   "flush_ms_per_step, is subtracted)" if flush is not None
                   else f"inputs larger than L2 ({kv_bytes / 2**20:.0f} MiB KV per step vs 129 MiB L2)"),
            "parallelism": f"replicas x{world}",
        },
        "decode_steps_per_s_per_layer": round(1e3 / ms, 2),
        "pct_of_nominal_8TBs": None if prefill else round(100 * value / world / NOMINAL_HBM_GBS, 2),
        "pct_of_measured_hbm": None if prefill else round(100 * value / world / peak, 2),
        "pct_of_measured_tensor": round(100 * value / world / peak, 2) if prefill else None,
        "kernel_ms": {"fused_step": round(fused_ms, 5), "two_calls": {"rope_append": round(sum(rope_ms) / K, 5),
                                                                       "decode_attn": round(dec_avg, 5),
                                                                       "both": round(eager_ms, 5)}},
        "step_timing": graph_note,
        "single_step_graph_ms": round(single_ms, 5),
        "flush_ms_per_step": None if flush_ms is None else round(flush_ms, 5),
        "roofline": {"kernel": (("prefill_tc_kernel (tcgen05: causal attention of the prompt, 128 tokens x 2 query heads per "
                                 "CTA, S and O in Tensor Memory)" if cfg.head_dim == 128 else
                                 "prefill_kernel (mma.sync: causal attention of the prompt, 64 query rows per CTA)") if prefill else
                                ("decode_verify_kernel, fused step (RoPE + append of "
                                 f"{cfg.gamma} new tokens per sequence + causal split-K attention + merge)"
                                 if cfg.gamma <= 8 else "decode_verify_kernel (causal split-K attention of "
                                 f"{cfg.gamma} new tokens per sequence + merge; the append is a separate launch)")
                                if cfg.gamma > 1 else
                                "decode_q8_kernel, fused step (RoPE + quantised append + split-K attention over "
                                f"INT{cfg.code_bits} codes and the bf16 window + merge)" if cfg.int8 else
                                "decode_mma_kernel, fused step (RoPE + append + split-K attention + merge)"
                                if mma_path else "rope_append + decode_split_kernel (fused-step call)"),
                     "bound": "tensor" if prefill else "hbm",
                     "achieved": round(achieved, 2), "peak": peak, "unit": unit,
                     "frac": round(achieved / peak, 4), "peak_source": peak_src,
                     "traffic": recorded_traffic(cfg.name)},
        "gpu_launches": K * launches_per_step,
        "device_error_bits": err_bits,
        "clocks": clocks,
        "e2e": e2e,
        "cpu_baseline": None,
    }
    del step, w
    return line


# ---------------------------------------------------------------------------- the oracle on host cores
def oracle_sample_config(cfg, batch):
    """The first ``batch`` sequences of a workload, with a pool just big enough for them."""
    import dataclasses
    import math
    kw = {"batch": batch, "name": cfg.name + f"_sample{batch}"}
    if cfg.gamma > 16:          # prefill: a 512-token prompt of the same shape
        kw.update(seq_len=512, gamma=512)
    if cfg.layout == "paged":
        longest = cfg.seq_len if cfg.seq_len is not None else cfg.len_range[1]
        kw["num_blocks"] = batch * math.ceil(longest / cfg.block_size) + 8
    return dataclasses.replace(cfg, **kw)


def sample_work(inp):
    """(work, divisor, unit, metric) of one oracle step on a sample: KV bytes in GB/s, or for a
    prefill the causal attention FLOPs in TFLOP/s."""
    cfg = inp.cfg
    if cfg.gamma > 16:
        return prefill_flops(cfg, inp.lengths), 1e12, "TFLOP/s", PREFILL_METRIC
    return cfg.unique_kv_bytes(inp.lengths), 1e9, UNIT, METRIC


def oracle_step_seconds(inp):
    """Time the oracle's whole decode step (RoPE, append, attention) on one sample."""
    from oracle import decode as odecode
    cfg = inp.cfg
    bs = cfg.block_size if inp.block_table is not None else 0
    t0 = time.perf_counter()
    if cfg.gamma > 1:
        from oracle import verify
        verify.verify_step(inp.q, inp.k_new, inp.v_new, inp.positions, inp.k_cache, inp.v_cache, cfg.dtype,
                           inp.block_table, bs, rope_base=cfg.rope_base)
    elif cfg.int8:
        from oracle import quant
        quant.decode_step_q8(inp.q, inp.k_new, inp.v_new, inp.positions, inp.k_cache, inp.v_cache, inp.k_scale,
                             inp.v_scale, inp.k_win, inp.v_win, cfg.window, inp.block_table, bs,
                             rope_base=cfg.rope_base, bits=cfg.code_bits)
    else:
        odecode.decode_step(inp.q, inp.k_new, inp.v_new, inp.positions, inp.k_cache, inp.v_cache, cfg.dtype,
                            inp.block_table, bs, rope_base=cfg.rope_base)
    return time.perf_counter() - t0


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def available_memory_bytes() -> int:
    """Memory the oracle processes may use: MemAvailable, capped by a cgroup limit if one is set."""
    avail = 8 << 30
    try:
        with open("/proc/meminfo") as f:
            for ln in f:
                if ln.startswith("MemAvailable:"):
                    avail = int(ln.split()[1]) * 1024
    except OSError:
        pass
    for path in ("/sys/fs/cgroup/memory.max", "/sys/fs/cgroup/memory/memory.limit_in_bytes"):
        try:
            with open(path) as f:
                v = f.read().strip()
            if v.isdigit():
                avail = min(avail, int(v))
        except OSError:
            pass
    return avail


def oracle_sample_bytes(cfg) -> int:
    """Rough peak memory of one oracle step on a batch-1 sample: the stored caches twice (input and
    the step's copy) and the float64 logical K and V."""
    s = oracle_sample_config(cfg, 1)
    longest = s.seq_len if s.seq_len is not None else s.len_range[1]
    per_tok = s.n_kv_heads * s.head_dim
    cache = (s.num_blocks * s.block_size if s.layout == "paged" else s.max_len) * per_tok * 4
    return 2 * cache + 2 * longest * per_tok * 8 + (256 << 20)


def _oracle_proc(workload, index, conn):
    """One host core's share: a batch-1 sample of the workload (seed + index), then commands:
    ("step",) runs one oracle step; ("run", seconds) repeats steps for that long; None stops."""
    cfg = CONFIGS[workload]
    inp = make_inputs(oracle_sample_config(cfg, 1), seed=cfg.seed + index)
    work = sample_work(inp)[0]
    conn.send(("ready", int(inp.lengths[0])))
    while True:
        cmd = conn.recv()
        if cmd is None:
            break
        if cmd[0] == "step":
            conn.send((work, oracle_step_seconds(inp)))
        else:
            elapsed, done = 0.0, 0
            while elapsed < cmd[1] or done == 0:
                elapsed += oracle_step_seconds(inp)
                done += 1
            conn.send((done * work, elapsed))
    conn.close()


class OracleCores:
    """The float64 oracle on every host core: one process per core (spawned, so safe to start after
    CUDA), each with its own batch-1 sample of the workload, driven in lock step."""

    def __init__(self, workload: str, cores: int):
        import multiprocessing as mp
        ctx = mp.get_context("spawn")
        self.conns, self.procs = [], []
        for i in range(cores):
            parent, child = ctx.Pipe()
            p = ctx.Process(target=_oracle_proc, args=(workload, i, child), daemon=True)
            p.start()
            self.conns.append(parent)
            self.procs.append(p)
        self.lengths = [c.recv()[1] for c in self.conns]

    def step(self):
        """One oracle step on every core's sample: (work summed over cores, wall seconds)."""
        t0 = time.perf_counter()
        for c in self.conns:
            c.send(("step",))
        work = sum(c.recv()[0] for c in self.conns)
        return work, time.perf_counter() - t0

    def run(self, seconds: float):
        """Every core repeats steps for ``seconds``: (work summed over cores, longest elapsed)."""
        for c in self.conns:
            c.send(("run", seconds))
        res = [c.recv() for c in self.conns]
        return sum(r[0] for r in res), max(r[1] for r in res)

    def close(self):
        for c in self.conns:
            try:
                c.send(None)
            except OSError:
                pass
        for p in self.procs:
            p.join(timeout=10)


def oracle_core_count(cfg) -> int:
    """Every host core, fewer if the batch-1 samples would not fit in half the available memory."""
    return max(1, min(host_cores(), available_memory_bytes() // 2 // oracle_sample_bytes(cfg)))


def cpu_worker(workload: str, seconds: float):
    cfg = CONFIGS[workload]
    # all host cores: one process per core, each its own batch-1 sample (seeds seed .. seed + n - 1)
    n = oracle_core_count(cfg)
    pool = OracleCores(workload, n)
    try:
        work_all, wall = pool.run(seconds)
        lengths = pool.lengths
    finally:
        pool.close()
    _, div, unit, _ = sample_work(make_inputs(oracle_sample_config(cfg, 1), seed=cfg.seed))
    # one host core: the first sequences of the workload
    sample_batch = 1 if cfg.batch == 1 or cfg.layout == "contiguous" else 2
    inp = make_inputs(oracle_sample_config(cfg, sample_batch), seed=cfg.seed)
    work = sample_work(inp)[0]
    elapsed, done = 0.0, 0
    while elapsed < seconds or done == 0:
        elapsed += oracle_step_seconds(inp)
        done += 1
    return {"value": round(work_all / wall / div, 6), "unit": unit, "cores": n, "kind": "oracle",
            "sample": (f"float64 numpy oracle (RoPE + append + attention), one process per host core ({n} of "
                       f"{host_cores()}), each on its own batch-1 sample of {workload} (seeds {cfg.seed}.."
                       f"{cfg.seed + n - 1}, lengths {lengths}) repeated for {seconds:.0f} s; BLAS limited to 1 "
                       "thread per process"),
            "one_core": {"value": round(done * work / elapsed / div, 6), "unit": unit, "cores": 1,
                         "sample": (f"the first {sample_batch} sequence(s) of {workload} (lengths "
                                    f"{inp.lengths.tolist()}), repeated {done}x in {elapsed:.1f} s on one core")}}


def cpu_baseline(workload: str, seconds: float):
    env = dict(os.environ)
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS"):
        env[v] = "1"
    for v in ("RANK", "LOCAL_RANK", "WORLD_SIZE"):
        env.pop(v, None)
    cmd = [sys.executable, os.path.abspath(__file__), "--cpu-worker", "--workload", workload,
           "--cpu-seconds", str(seconds)]
    try:
        r = subprocess.run(cmd, env=env, stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True,
                           timeout=max(180.0, 10 * seconds))
        return json.loads(r.stdout.strip().splitlines()[-1])
    except Exception as e:  # the baseline is reported, never required
        return {"value": None, "unit": UNIT, "cores": 0, "kind": "oracle", "sample": f"failed: {e}"}


def run_reference(args):
    """The reference arm: the float64 oracle on every host core (one process per core, each its own
    batch-1 sample of the workload); one step = one oracle step on every core's sample."""
    rank, _, world = dist_env()
    if rank != 0:
        return 0
    cfg = CONFIGS[args.workload or DEFAULT_WORKLOAD]
    n = oracle_core_count(cfg)
    pool = OracleCores(cfg.name, n)
    try:
        for _ in range(args.warmup):
            pool.step()
        steps = [pool.step() for _ in range(args.steps)]
    finally:
        pool.close()
    work = sum(w for w, _ in steps) / len(steps)
    ms = 1e3 * sum(t for _, t in steps) / len(steps)
    _, div, unit, metric = sample_work(make_inputs(oracle_sample_config(cfg, 1), seed=cfg.seed))
    value = work / (ms * 1e-3) / div
    sample = (f"float64 numpy oracle, one process per host core ({n} of {host_cores()}), each on its own batch-1 "
              f"sample of {cfg.name} (seeds {cfg.seed}..{cfg.seed + n - 1}, lengths {pool.lengths}); one step = one "
              "oracle step on every sample; BLAS limited to 1 thread per process")
    print(json.dumps({
        "impl": "reference", "metric": metric, "value": round(value, 6), "unit": unit, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": cfg.name, "description": cfg.description, "sample": f"{n} batch-1 samples"},
        "cpu_baseline": {"value": round(value, 6), "unit": unit, "cores": n, "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 6), "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)
    return 0


def main(argv=None):
    args = parse_args(argv)
    if args.cpu_worker:
        print(json.dumps(cpu_worker(args.workload or DEFAULT_WORKLOAD, args.cpu_seconds)), flush=True)
        return 0
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
