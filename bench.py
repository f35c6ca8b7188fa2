#!/usr/bin/env python
"""Benchmark of the GB300 attention library on the pages' workloads (synthetic, seeded).

One step is one attn_fwd call on the headline workload: causal GQA prefill,
bf16, batch 4, 32 query / 8 kv heads, 4096 tokens, head_dim 128.  The same run
also times the KV-cache decode workload (batch 64, 32/8 heads, 8192 cached
keys, head_dim 128), the attention prelude (split QKV + QK norm + RoPE for the
headline's 16384 tokens) and the two smaller prefill workloads, and reports each
against its roofline.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun each rank runs the same workload on its own GPU (replicas, weak
scaling); rank 0 prints one JSON line with the whole-job throughput.
`--impl reference` times the fp64 CPU oracle on bounded samples of the same
workload (rank 0 only).
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from head_attention_attn_gb300.inputs import WORKLOADS, make_inputs  # noqa: E402

METRIC = "attention TFLOP/s (prefill) and KV GB/s (decode) on 1 GB300, % of roofline"
HEADLINE = "causal_gqa_bf16_4x32q8kv_4096x128"
DECODE = "decode_bf16_64x32q8kv_8192x128"
EXTRA_PREFILL = ["causal_mha_f32_1x4x64x32", "bidir_keypad_bf16_8x12x512x64", "window128_bf16_4x12x8192x64"]
KEYPAD = "bidir_keypad_bf16_8x12x512x64"
PRELUDE = "qkv_prelude_bf16_16384x32q8kv_128_normrope"
PAGED_PREFILL = "paged_prefill_bf16_4x32q8kv_512of4096x128_page16"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

# DRAM bytes per launch measured by ncu (dram__bytes_read.sum + dram__bytes_write.sum) for a
# kernel's code state (its hash); the entry stops applying as soon as the kernel's code changes.
NCU_TRAFFIC = {
    # prefill_persist_kernel<bf16, positive scale>, causal GQA (one CTA per SM over the query
    # blocks, paired heads): 289.54 MB read + 84.92 MB written
    ("prefill", "20541aa39a87"): 374458112.0,
    # prefill_tc_kernel<128, 2, bf16, paged, paired heads>, chunked prefill with 16-row pages:
    # 113.00 MB read + 8.64 MB written
    ("prefill", "20541aa39a87", "paged16"): 121643264.0,
    # decode_tc_kernel<G4, bf16>: 537.11 MB read + 3.26 MB written at batch 16, scaled by the units
    # (items) to the bench's batch 64
    ("decode_tc", "b900f0549270"): 4 * 540366336.0,
    # prefill_narrow_kernel<bf16, head-major, positive scale>, per workload: window 151.07 MB read +
    # 28.00 MB written; key padding 15.78 MB read, 0 written (the output stays in L2)
    ("prefill_narrow", "3a6262fe1152", "window128_bf16_4x12x8192x64"): 179073280.0,
    ("prefill_narrow", "3a6262fe1152", "bidir_keypad_bf16_8x12x512x64"): 15775232.0,
}


# ----------------------------------------------------------------------------- distributed plumbing

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1 and not torch.distributed.is_initialized():
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        torch.distributed.init_process_group(backend=backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(x: float, world: int, device=None) -> float:
    if world == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, world: int, device=None) -> float:
    if world == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.SUM)
    return float(t.item())


# ----------------------------------------------------------------------------- algorithmic work

def visible_pairs(c, key_lens=None) -> int:
    """Number of (query row, visible key) pairs of one head, summed over the batch."""
    total = 0
    for b in range(c.B):
        klen = c.Lk if key_lens is None else int(max(0, min(c.Lk, int(key_lens[b]))))
        for_rows = np.arange(c.Lq, dtype=np.int64) + c.pos_offset
        lo = np.zeros_like(for_rows)
        hi = np.full_like(for_rows, klen)
        if c.mask_mode == 1:
            hi = np.minimum(hi, for_rows + 1)
        elif c.mask_mode == 2 and c.window > 0:
            lo = np.maximum(lo, for_rows - c.window // 2)
            hi = np.minimum(hi, for_rows + c.window // 2 + 1)
        elif c.mask_mode == 3:
            hi = np.minimum(hi, for_rows + 1)
            if c.window > 0:
                lo = np.maximum(lo, for_rows - c.window + 1)
        total += int(np.maximum(hi - lo, 0).sum())
    return total


def flops_of(c, key_lens=None) -> float:
    """4 * D flops per visible (row, key) pair (QK^T and PV), over every query head."""
    return 4.0 * c.D * c.Hq * visible_pairs(c, key_lens)


def bytes_of(c, key_lens=None) -> float:
    """Q and O once, plus the K and V rows the workload can see (each kv head read once)."""
    esz = 2 if c.dtype == "bf16" else 4
    qo = 2.0 * c.B * c.Hq * c.Lq * c.D * esz
    if key_lens is None:
        kv_rows = c.B * c.Lk
    else:
        kv_rows = int(sum(max(0, min(c.Lk, int(x))) for x in key_lens))
    return qo + 2.0 * c.Hkv * kv_rows * c.D * esz


# ----------------------------------------------------------------------------- measurement helpers

def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            with open(path) as f:
                d = json.load(f)
            out = {}
            for key in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained"):
                if key in d and isinstance(d[key], (int, float)):
                    out[key] = float(d[key])
            if "hbm_gbs" in out and "bf16_tflops" in out:
                out.setdefault("bf16_tflops_sustained", out["bf16_tflops"])
                return out, "measured"
        except Exception:
            pass
    return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 20 ms while running.

    Entering waits (up to 5 s) for the first sample, so the samples cover the timed
    region that follows rather than nvidia-smi's own start-up."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        import tempfile
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        if self.proc is not None:
            t0 = time.time()
            while time.time() - t0 < 5.0 and self.proc.poll() is None:
                try:
                    if os.path.getsize(self.path) > 0:
                        break
                except OSError:
                    pass
                time.sleep(0.01)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        rows = []
        try:
            with open(self.path) as f:
                for line in f:
                    parts = [p.strip() for p in line.split(",")]
                    if len(parts) >= 9:
                        rows.append(parts)
        except Exception:
            pass
        finally:
            try:
                os.remove(self.path)
            except Exception:
                pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "", 1).isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "", 1).isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def prelude_leg(args, world, dev, peaks, peak_src):
    """GB/s of attn_qkv_prelude on 16384 tokens of a 32q/8kv, head_dim 128 layer (qk_mode 1)."""
    import head_attention_attn_gb300 as attn
    T, Hq, Hkv, hd = 16384, 32, 8, 128
    g = torch.Generator().manual_seed(1005)
    qkv = torch.randn(T, (Hq + 2 * Hkv) * hd, generator=g).to(torch.bfloat16).to(dev)
    w = (torch.rand(hd, generator=g) + 0.5).to(dev)
    j = torch.arange(hd // 2, dtype=torch.float64)
    ang = torch.arange(T, dtype=torch.float64)[:, None] * 1.0e6 ** (-2.0 * j / hd)[None, :]
    cos, sin = torch.cos(ang).float().to(dev), torch.sin(ang).float().to(dev)
    q = torch.empty(Hq, T, hd, dtype=torch.bfloat16, device=dev)

    def call():
        attn.attn_qkv_prelude(qkv, Hq, Hkv, hd, qk_mode=attn.QK_NORM_ROPE, cos=cos, sin=sin, q_norm_w=w, k_norm_w=w,
                              q_out=q)
    steps = max(3, min(args.steps, 500))
    sec = time_device(call, steps, args.warmup, world, dev)
    if attn.sync_status() != attn.ATTN_OK:
        raise RuntimeError("device status after the prelude: " + attn.last_error())
    nbytes = 2.0 * qkv.numel() * 2 + cos.numel() * 4 * 2 + 2 * hd * 4  # qkv in, q/k/v out, tables, weights
    gbs = nbytes / sec / 1e9
    return {"workload": PRELUDE, "value": round(gbs * world, 1), "unit": "GB/s",
            "steps": steps, "ms_per_step": round(sec * 1e3, 4), "launch_ms": LAUNCH_STATS.get(call),
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": round(gbs / peaks["hbm_gbs"], 4), "peak_source": f"{peak_src} HBM copy",
                         "traffic": None, "kernel": "prelude_kernel<128, bf16>", "algorithmic_bytes_per_launch": nbytes},
            "l2": f"inputs {qkv.numel() * 2 / 1e6:.0f} MB > {L2_BYTES / 1e6:.0f} MB L2, no flush"}


KERNEL_SOURCES = {
    "prefill": ("head_attention_attn_gb300/csrc/prefill_tc.cu",),
    "prefill_narrow": ("head_attention_attn_gb300/csrc/prefill_narrow.cu",),
    "decode_tc": ("head_attention_attn_gb300/csrc/decode_tc.cu",),
}
SHARED_SOURCES = ("head_attention_attn_gb300/csrc/common.cuh", "head_attention_attn_gb300/csrc/kernels.h")


def decode_forms_leg(args, world, dev, peaks, peak_src, dec_bytes):
    """GB/s of attn_decode_caches and attn_decode_paged at the decode workload's shape: 64 items,
    8 kv heads, 8192 cached positions each, head_dim 128, bf16, device kv_lens, with 32 query heads
    (as the workload) and with 64.  Every launch reads the same 2.15 GB of K and V as the
    contiguous decode, plus its Q and O."""
    import head_attention_attn_gb300 as attn
    c = WORKLOADS[DECODE]
    m, Hkv, cap, D = c.B, c.Hkv, c.Lk, c.D
    kv_bytes = 2.0 * m * Hkv * cap * D * 2
    kv_lens = torch.full((m,), cap, dtype=torch.int32, device=dev)
    scale = float(torch.tensor(1.0 / math.sqrt(D), dtype=torch.float32))
    steps = max(3, min(args.steps, 300))
    legs = []
    torch.cuda.manual_seed(1006)

    def leg(name, call, kernel, Hq):
        nbytes = kv_bytes + 2.0 * m * Hq * D * 2
        sec = time_device(call, steps, args.warmup, world, dev)
        if attn.sync_status() != attn.ATTN_OK:
            raise RuntimeError(f"device status after {name}: " + attn.last_error())
        gbs = nbytes / sec / 1e9
        legs.append({"workload": name, "value": round(gbs * world, 1), "unit": "GB/s", "steps": steps,
                     "ms_per_step": round(sec * 1e3, 4), "launch_ms": LAUNCH_STATS.get(call),
                     "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                  "frac": round(gbs / peaks["hbm_gbs"], 4), "peak_source": f"{peak_src} HBM copy",
                                  "traffic": None, "kernel": kernel, "algorithmic_bytes_per_launch": nbytes},
                     "l2": f"inputs {nbytes / 1e6:.0f} MB > {L2_BYTES / 1e6:.0f} MB L2, no flush"})

    # per-item caches [Hkv, capacity, D], one allocation each, through device pointer arrays
    ks = [torch.empty(Hkv, cap, D, dtype=torch.bfloat16, device=dev).normal_() for _ in range(m)]
    vs = [torch.empty(Hkv, cap, D, dtype=torch.bfloat16, device=dev).normal_() for _ in range(m)]
    kp = torch.tensor([t.data_ptr() for t in ks], dtype=torch.int64, device=dev)
    vp = torch.tensor([t.data_ptr() for t in vs], dtype=torch.int64, device=dev)
    for Hq, kernel in ((32, "decode_tc_kernel<G4, bf16, per-item caches> (TMA, tensor maps built on the device)"),
                       (64, "decode_tc_kernel<G8, bf16, per-item caches> (TMA, tensor maps built on the device)")):
        q = torch.empty(m, Hq, D, dtype=torch.bfloat16, device=dev).normal_()
        out = torch.empty_like(q)
        leg(f"decode_caches_bf16_{m}x{Hq}q{Hkv}kv_{cap}x{D}",
            lambda q=q, out=out: attn.attn_decode_caches(q, kp, vp, kv_lens, out, scale=scale, kv_heads=Hkv,
                                                         capacity=cap),
            kernel, Hq)
    del ks, vs, kp, vp
    torch.cuda.empty_cache()

    # paged: pools [num_pages, Hkv, page_size, D] and a shuffled page table
    g = torch.Generator().manual_seed(1007)
    for ps, Hq, kernel in ((16, 32, "decode_splitkv_kernel<128, G4, bf16> (paged, bulk copy per page piece)"),
                           (16, 64, "decode_tc_kernel<G8, bf16, paged> (TMA per page)"),
                           (128, 32, "decode_tc_kernel<G4, bf16, paged> (TMA per page)"),
                           (1, 32, "decode_splitkv_kernel<128, G4, bf16> (paged, bulk copy per page piece)")):
        max_pages = cap // ps
        num_pages = m * max_pages
        k_pool = torch.empty(num_pages, Hkv, ps, D, dtype=torch.bfloat16, device=dev).normal_()
        v_pool = torch.empty_like(k_pool).normal_()
        table = torch.randperm(num_pages, generator=g).to(torch.int32).view(m, max_pages).to(dev)
        q = torch.empty(m, Hq, D, dtype=torch.bfloat16, device=dev).normal_()
        out = torch.empty_like(q)
        leg(f"decode_paged_bf16_{m}x{Hq}q{Hkv}kv_{cap}x{D}_page{ps}",
            lambda q=q, out=out, k_pool=k_pool, v_pool=v_pool, table=table:
                attn.attn_decode_paged(q, k_pool, v_pool, table, kv_lens, out, scale=scale),
            kernel, Hq)
        del k_pool, v_pool, table
        torch.cuda.empty_cache()
    return legs


# chunked prefill over paged caches: 4 sequences whose newest 512 positions (the queries) follow
# 3,584 older ones (4,096 cached positions each), 32 query / 8 kv heads, head_dim 128, bf16, causal
PAGED_SHAPE = dict(B=4, Hq=32, Hkv=8, D=128, chunk=512, kv=4096)


def paged_prefill_inputs(ps, dev, g):
    """Queries, output, cu_seqlens, kv_lens and shuffled pools with pages of ps rows."""
    B, Hq, Hkv, D, chunk, kv = (PAGED_SHAPE[k] for k in ("B", "Hq", "Hkv", "D", "chunk", "kv"))
    q = torch.empty(B * chunk, Hq, D, dtype=torch.bfloat16, device=dev).normal_()
    cu = torch.arange(0, (B + 1) * chunk, chunk, dtype=torch.int32, device=dev)
    kv_lens = torch.full((B,), kv, dtype=torch.int32, device=dev)
    max_pages = kv // ps
    num_pages = B * max_pages
    k_pool = torch.empty(num_pages, Hkv, ps, D, dtype=torch.bfloat16, device=dev).normal_()
    v_pool = torch.empty_like(k_pool).normal_()
    table = torch.randperm(num_pages, generator=g).to(torch.int32).view(B, max_pages).to(dev)
    return q, torch.empty_like(q), cu, kv_lens, k_pool, v_pool, table


def paged_prefill_leg(args, world, dev, peaks, peak_src):
    """TFLOP/s of attn_fwd_varlen_paged on the chunked prefill of PAGED_SHAPE, with pages of 16
    and of 128 rows.  Algorithmic FLOPs count the visible (query, key) pairs only."""
    import head_attention_attn_gb300 as attn
    B, Hq, Hkv, D, chunk, kv = (PAGED_SHAPE[k] for k in ("B", "Hq", "Hkv", "D", "chunk", "kv"))
    P = kv - chunk
    flops = 4.0 * D * Hq * B * sum(P + i + 1 for i in range(chunk))
    scale = float(torch.tensor(1.0 / math.sqrt(D), dtype=torch.float32))
    steps = max(3, min(args.steps, 200))
    g = torch.Generator().manual_seed(1008)
    legs = []
    for ps in (16, 128):
        q, out, cu, kv_lens, k_pool, v_pool, table = paged_prefill_inputs(ps, dev, g)

        def call(q=q, out=out, cu=cu, kv_lens=kv_lens, k_pool=k_pool, v_pool=v_pool, table=table):
            attn.attn_fwd_varlen_paged(q, k_pool, v_pool, table, cu, kv_lens, chunk, out, scale=scale)
        sec = time_device(call, steps, args.warmup, world, dev)
        if attn.sync_status() != attn.ATTN_OK:
            raise RuntimeError("device status after the paged prefill: " + attn.last_error())
        tflops = flops / sec / 1e12
        legs.append({"workload": f"paged_prefill_bf16_{B}x{Hq}q{Hkv}kv_{chunk}of{kv}x{D}_page{ps}",
                     "value": round(tflops * world, 1), "unit": "TFLOP/s", "steps": steps,
                     "ms_per_step": round(sec * 1e3, 4), "launch_ms": LAUNCH_STATS.get(call),
                     "roofline": {"bound": "tensor", "achieved": round(tflops, 1), "peak": peaks["bf16_tflops"],
                                  "unit": "TFLOP/s", "frac": round(tflops / peaks["bf16_tflops"], 4),
                                  "peak_source": f"{peak_src} bf16 dense (burst)",
                                  "traffic": NCU_TRAFFIC.get(("prefill", kernel_source_hash("prefill"), f"paged{ps}")),
                                  "kernel": "prefill_tc_kernel<128, 2, bf16, paged> (K/V copied by TMA a page piece at a time)",
                                  "algorithmic_flops_per_launch": flops}})
        del q, out, k_pool, v_pool, table
        torch.cuda.empty_cache()
    return legs


def kernel_source_hash(kernel: str = "prefill") -> str:
    """Identifies a kernel's code: its source, the shared device headers and the nvcc flags
    (comments and blank lines do not count), so a DRAM-traffic figure stays attached to the
    code it was measured on."""
    from head_attention_attn_gb300 import build as _build
    h = hashlib.sha1()
    for rel in KERNEL_SOURCES[kernel] + SHARED_SOURCES:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        h.update("\n".join(line.rstrip() for line in text.splitlines() if line.strip()).encode())
    h.update(" ".join(_build.ARCH_FLAGS + _build.NVCC_FLAGS).encode())
    return h.hexdigest()[:12]


LAUNCH_STATS = {}  # fn -> per-launch statistics of its last time_device run


def time_device(fn, steps: int, warmup: int, world: int, device) -> float:
    """Seconds per call: CUDA events on the launching stream, synced on both sides, max over ranks.

    The returned mean is the whole timed region over `steps`.  An event also sits between
    consecutive launches (recorded on the stream, no synchronisation), so LAUNCH_STATS[fn] holds
    the median, 10th and 90th percentile of the per-launch durations on this rank."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    barrier(world)
    stream = torch.cuda.current_stream()
    events = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    events[0].record(stream)
    for i in range(steps):
        fn()
        events[i + 1].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    sec = events[0].elapsed_time(events[-1]) / 1e3 / steps
    per = sorted(events[i].elapsed_time(events[i + 1]) for i in range(steps))
    LAUNCH_STATS[fn] = {"median_ms": round(per[len(per) // 2], 4), "p10_ms": round(per[len(per) // 10], 4),
                        "p90_ms": round(per[(9 * len(per)) // 10], 4), "launches": steps}
    return max_over_ranks(sec, world, device)


# ----------------------------------------------------------------------------- our arm

def run_ours(args, rank, world, local):
    import head_attention_attn_gb300 as attn
    from head_attention_attn_gb300 import build
    if rank == 0 or world == 1:
        build.build_library()
    barrier(world)
    attn.load()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    peaks, peak_src = read_peaks()

    def setup(name):
        c = WORKLOADS[name]
        q, k, v, kl = make_inputs(c)
        qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
        kld = None if kl is None else kl.to(dev)
        out = torch.empty_like(qd)
        scale = float(torch.tensor(1.0 / math.sqrt(c.D), dtype=torch.float32))

        def call(o=out, qq=qd, kk=kd, vv=vd):
            attn.attn_fwd(qq, kk, vv, o, pos_offset=c.pos_offset, mask_mode=c.mask_mode, window=c.window,
                          key_lens=kld, scale=scale)
        return c, (q, k, v, kl), (qd, kd, vd, kld, out), call

    # ---- headline: causal GQA prefill
    c, host, devt, call = setup(HEADLINE)
    flops = flops_of(c)
    with ClockSampler(local) as clk:
        sec = time_device(call, args.steps, args.warmup, world, dev)
    clocks = clk.summary()
    if attn.sync_status() != attn.ATTN_OK:
        raise RuntimeError("device status after prefill: " + attn.last_error())
    tflops = flops / sec / 1e12
    value = tflops * world  # replicas: every rank processes one full workload per step
    roof = {"bound": "tensor", "achieved": round(tflops, 2), "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
            "frac": round(tflops / peaks["bf16_tflops"], 4), "peak_source": f"{peak_src} bf16 dense (burst)",
            "traffic": NCU_TRAFFIC.get(("prefill", kernel_source_hash("prefill"))),
            "kernel": "prefill_persist_kernel<bf16> (one CTA per SM, two query heads of a kv group per block)",
            "algorithmic_flops_per_launch": flops}

    # ---- end to end through the public call with pinned host buffers: every step copies its
    # inputs host->device and its result device->host.  Steps are double-buffered over three
    # streams (inputs in, compute, result out), so step i's copies overlap step i-1's compute.
    q, k, v, kl = host
    qh, kh, vh = q.pin_memory(), k.pin_memory(), v.pin_memory()
    qd, kd, vd, kld, out = devt
    bufs = [(qd, kd, vd, out), tuple(torch.empty_like(x) for x in (qd, kd, vd, out))]
    outs_h = [torch.empty(out.shape, dtype=out.dtype, pin_memory=True) for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    s_comp = torch.cuda.current_stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    for e in ev_out:
        e.record(s_out)
    e2e_steps = max(1, min(args.steps, 200))
    scale = float(torch.tensor(1.0 / math.sqrt(c.D), dtype=torch.float32))
    state = {"i": 0}

    def e2e_step():
        i = state["i"] % 2
        bq, bk, bv, bo = bufs[i]
        with torch.cuda.stream(s_in):
            s_in.wait_event(ev_done[i])          # buffer i is free once its previous compute finished
            bq.copy_(qh, non_blocking=True)
            bk.copy_(kh, non_blocking=True)
            bv.copy_(vh, non_blocking=True)
            ev_in[i].record(s_in)
        s_comp.wait_event(ev_in[i])
        s_comp.wait_event(ev_out[i])             # the previous result in buffer i has been read out
        attn.attn_fwd(bq, bk, bv, bo, pos_offset=c.pos_offset, mask_mode=c.mask_mode, window=c.window,
                      key_lens=kld, scale=scale)
        ev_done[i].record(s_comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_done[i])
            outs_h[i].copy_(bo, non_blocking=True)
            ev_out[i].record(s_out)
        state["i"] += 1

    def e2e_timed(steps):
        for _ in range(min(args.warmup, 3)):
            e2e_step()
        torch.cuda.synchronize()
        barrier(world)
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(s_comp)
        for _ in range(steps):
            e2e_step()
        s_comp.wait_event(ev_out[(state["i"] - 1) % 2])  # the last result has reached the host
        t1.record(s_comp)
        torch.cuda.synchronize()
        barrier(world)
        return max_over_ranks(t0.elapsed_time(t1) / 1e3 / steps, world, dev)

    e2e_sec = e2e_timed(e2e_steps)
    h2d = (qh.numel() + kh.numel() + vh.numel()) * qh.element_size()
    d2h = out.numel() * out.element_size()
    e2e = {"value": round(flops / e2e_sec / 1e12 * world, 3), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": d2h, "steps": e2e_steps, "ms_per_step": round(e2e_sec * 1e3, 4),
           "pipeline": "inputs in / compute / result out on three streams, double-buffered"}
    del bufs, outs_h
    del host, devt, qh, kh, vh
    torch.cuda.empty_cache()

    # ---- decode leg
    c_d, host_d, devt_d, call_d = setup(DECODE)
    dec_bytes = bytes_of(c_d)
    dec_steps = max(3, min(args.steps, 500))
    dsec = time_device(call_d, dec_steps, args.warmup, world, dev)
    gbs = dec_bytes / dsec / 1e9
    decode = {"workload": DECODE, "value": round(gbs * world, 1), "unit": "GB/s", "steps": dec_steps,
              "ms_per_step": round(dsec * 1e3, 4), "launch_ms": LAUNCH_STATS.get(call_d),
              "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                           "frac": round(gbs / peaks["hbm_gbs"], 4), "peak_source": f"{peak_src} HBM copy",
                           "traffic": NCU_TRAFFIC.get(("decode_tc", kernel_source_hash("decode_tc"))),
                           "kernel": "decode_tc_kernel<G4, bf16>",
                           "algorithmic_bytes_per_launch": dec_bytes},
              "l2": f"inputs {dec_bytes / 1e6:.0f} MB > {L2_BYTES / 1e6:.0f} MB L2, no flush"}
    del host_d, devt_d
    torch.cuda.empty_cache()

    # ---- per-item and paged caches at the decode workload's shape (ferrum-kernels
    # flash_attention_batched_per_cache): the same K/V bytes, addressed by the device
    decode_forms = decode_forms_leg(args, world, dev, peaks, peak_src, dec_bytes)
    paged_prefill = paged_prefill_leg(args, world, dev, peaks, peak_src)

    # ---- attention prelude leg: split fused QKV + QK RMS norm + RoPE + head-major transpose for
    # the headline workload's 4 x 4096 tokens (32 q / 8 kv heads, head_dim 128, bf16)
    prelude = prelude_leg(args, world, dev, peaks, peak_src)

    # ---- the other workloads (smaller; context)
    def timed(call_x, nbytes):
        """Seconds per call; L2 is flushed between calls where the inputs fit in it (the flush time
        is measured alone and subtracted)."""
        if nbytes < 2 * L2_BYTES:
            flush = torch.empty(int(2 * L2_BYTES), dtype=torch.uint8, device=dev)

            def call_xf(cx=call_x):
                flush.zero_()
                cx()
            tsec_with = time_device(call_xf, min(args.steps, 200), args.warmup, world, dev)
            tsec_flush = time_device(lambda: flush.zero_(), min(args.steps, 200), args.warmup, world, dev)
            del flush
            return max(tsec_with - tsec_flush, 1e-9), "flushed (2x L2 write between calls)"
        return time_device(call_x, min(args.steps, 200), args.warmup, world, dev), "inputs > L2"

    per_config = []
    outputs = {}  # one output per workload, for the oracle comparison of the CPU leg
    for name in EXTRA_PREFILL:
        c_x, host_x, devt_x, call_x = setup(name)
        kl_x = host_x[3]
        f_x, b_x = flops_of(c_x, kl_x), bytes_of(c_x, kl_x)
        xs, l2 = timed(call_x, b_x)
        call_x()
        outputs[name] = devt_x[4].float().cpu()
        entry = {"workload": name, "ms_per_step": round(xs * 1e3, 4),
                 "launch_ms": LAUNCH_STATS.get(call_x) if l2 == "inputs > L2" else None,
                 "tflops": round(f_x / xs / 1e12, 3), "gbs": round(b_x / xs / 1e9, 1),
                 "frac_hbm": round(b_x / xs / 1e9 / peaks["hbm_gbs"], 4),
                 "frac_tensor": round(f_x / xs / 1e12 / peaks["bf16_tflops"], 4), "l2": l2}
        if c_x.dtype == "f32":
            entry["bound"] = "launch latency (1.06 MFLOP); TFLOP/s for the record only"
        else:
            entry["traffic"] = NCU_TRAFFIC.get(("prefill_narrow", kernel_source_hash("prefill_narrow"), name))
        per_config.append(entry)
        if name == KEYPAD:
            # the same valid rows through attn_fwd_varlen: the sequences packed, no padded query rows
            # (ripvec-core Driver::prepare_batch_unpadded), against the padded call above
            q, k, v, kl = host_x
            lens = [int(x) for x in kl]
            cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32, device=dev)
            qp = torch.cat([q[b, :, :lens[b]].transpose(0, 1) for b in range(c_x.B)]).contiguous().to(dev)
            kp = torch.cat([k[b, :, :lens[b]].transpose(0, 1) for b in range(c_x.B)]).contiguous().to(dev)
            vp = torch.cat([v[b, :, :lens[b]].transpose(0, 1) for b in range(c_x.B)]).contiguous().to(dev)
            op = torch.empty_like(qp)
            scale_x = float(torch.tensor(1.0 / math.sqrt(c_x.D), dtype=torch.float32))

            def call_p():
                attn.attn_fwd_varlen(qp, kp, vp, cu, max(lens), op, mask_mode=c_x.mask_mode, scale=scale_x)
            useful = 4.0 * c_x.D * c_x.Hq * sum(n * n for n in lens)  # valid query rows x valid keys
            bp = 2.0 * (qp.numel() + kp.numel()) * 2
            ps, l2p = timed(call_p, bp)
            call_p()
            outputs[name + ":packed"] = (op.float().cpu(), lens)
            entry["useful_tflops"] = round(useful / xs / 1e12, 3)
            per_config.append({"workload": name + " packed (attn_fwd_varlen)", "ms_per_step": round(ps * 1e3, 4),
                               "useful_tflops": round(useful / ps / 1e12, 3), "gbs": round(bp / ps / 1e9, 1),
                               "frac_hbm": round(bp / ps / 1e9 / peaks["hbm_gbs"], 4),
                               "speedup_vs_padded": round(xs / ps, 3), "l2": l2p})
            del qp, kp, vp, op, cu
        del host_x, devt_x
        torch.cuda.empty_cache()
    for name in (HEADLINE, DECODE):  # the outputs of the two legs above, for the comparison
        c_x, host_x, devt_x, call_x = setup(name)
        call_x()
        outputs[name] = devt_x[4].float().cpu()
        del host_x, devt_x
        torch.cuda.empty_cache()

    if attn.sync_status() != attn.ATTN_OK:
        raise RuntimeError("device status: " + attn.last_error())

    result = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(sec * 1e3, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": HEADLINE, "batch": c.B, "q_heads": c.Hq, "kv_heads": c.Hkv, "seq_len": c.Lq,
                   "head_dim": c.D, "mask": "causal", "pos_offset": c.pos_offset,
                   "l2": f"inputs {bytes_of(c) / 1e6:.0f} MB > {L2_BYTES / 1e6:.0f} MB L2, no flush",
                   "parallelism": f"replicas x{world}"},
        "launch_ms": LAUNCH_STATS.get(call),
        "roofline": roof, "e2e": e2e, "gpu_launches": args.steps, "clocks": clocks, "decode": decode,
        "decode_forms": decode_forms, "paged_prefill": paged_prefill, "prelude": prelude, "per_config": per_config,
    }
    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(args.cpu_seconds)
        result["cpu_baseline"]["per_config"] = oracle_per_config(outputs)
    return result


# ----------------------------------------------------------------------------- oracle (CPU) arms

def _oracle_sample_flops(c, rows):
    i = rows % c.Lq
    pos = i + c.pos_offset
    vis = np.minimum(pos + 1, c.Lk) if c.mask_mode == 1 else np.full_like(pos, c.Lk)
    return float(4.0 * c.D * vis.sum())


def cpu_baseline(target_seconds: float):
    """The oracle as it stands, on a bounded random sample of query rows of the headline workload."""
    import oracle
    c = WORKLOADS[HEADLINE]
    q, k, v, kl = make_inputs(c)
    qf, kf, vf = q.float().numpy(), k.float().numpy(), v.float().numpy()
    rng = np.random.default_rng(0)
    cores = len(os.sched_getaffinity(0))
    n = 256
    total_rows, total_flops, total_sec = 0, 0.0, 0.0
    while total_sec < target_seconds:
        rows = np.sort(rng.integers(0, c.B * c.Hq * c.Lq, size=n))
        t0 = time.perf_counter()
        oracle.attention(qf, kf, vf, mask_mode=c.mask_mode, pos_offset=c.pos_offset, rows=rows, nthreads=cores)
        dt = time.perf_counter() - t0
        total_rows += n
        total_flops += _oracle_sample_flops(c, rows)
        total_sec += dt
        n = int(min(65536, max(256, n * min(4.0, max(1.0, (target_seconds - total_sec) / max(dt, 1e-3))))))
    return {"value": round(total_flops / total_sec / 1e12, 6), "unit": "TFLOP/s", "cores": cores,
            "kind": "oracle",
            "sample": f"{total_rows} random query rows of {HEADLINE} (fp64 C oracle, {total_sec:.1f} s)"}


def oracle_per_config(outputs):
    """The oracle as it stands on every workload in full: its wall time on all host cores (and on
    one thread for the two smallest), and the max-abs and relative-L2 error of the GPU output
    measured above against it."""
    import oracle
    cores = len(os.sched_getaffinity(0))
    rows = []
    for name in [n for n in WORKLOADS if n in outputs]:
        c = WORKLOADS[name]
        q, k, v, kl = make_inputs(c)
        scale = float(torch.tensor(1.0 / math.sqrt(c.D), dtype=torch.float32))
        kw = dict(key_lens=kl, pos_offset=c.pos_offset, mask_mode=c.mask_mode, window=c.window, scale=scale)
        t0 = time.perf_counter()
        ref = oracle.attention(q, k, v, nthreads=cores, **kw)
        sec = time.perf_counter() - t0
        got = outputs[name].double().numpy()
        diff = got - ref
        entry = {"workload": name, "oracle_s": round(sec, 3), "cores": cores,
                 "max_abs": float(np.max(np.abs(diff))),
                 "rel_l2": float(np.linalg.norm(diff) / max(np.linalg.norm(ref), 1e-300))}
        if c.B * c.Hq * c.Lq * c.Lk <= 8 * 12 * 512 * 512:  # the fp32 and key-padding workloads
            t0 = time.perf_counter()
            oracle.attention(q, k, v, nthreads=1, **kw)
            entry["oracle_single_thread_s"] = round(time.perf_counter() - t0, 3)
        if name + ":packed" in outputs:  # the packed call: each sequence's valid rows
            got_p, lens = outputs[name + ":packed"]
            off, worst, num, den = 0, 0.0, 0.0, 0.0
            for b, n in enumerate(lens):
                r = ref[b, :, :n].transpose(1, 0, 2)
                d = got_p[off:off + n].double().numpy() - r
                worst = max(worst, float(np.max(np.abs(d))))
                num += float(np.sum(d * d))
                den += float(np.sum(r * r))
                off += n
            entry["packed_max_abs"] = worst
            entry["packed_rel_l2"] = float(np.sqrt(num / den))
        rows.append(entry)
        del ref, got, diff
    return rows


def run_reference(args, rank, world):
    import oracle
    if rank != 0:
        return None
    c = WORKLOADS[HEADLINE]
    q, k, v, kl = make_inputs(c)
    qf, kf, vf = q.float().numpy(), k.float().numpy(), v.float().numpy()
    cores = len(os.sched_getaffinity(0))
    rng = np.random.default_rng(1)
    rows_per_step = args.ref_rows

    def step():
        rows = np.sort(rng.integers(0, c.B * c.Hq * c.Lq, size=rows_per_step))
        oracle.attention(qf, kf, vf, mask_mode=c.mask_mode, pos_offset=c.pos_offset, rows=rows, nthreads=cores)
        return _oracle_sample_flops(c, rows)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    flops = sum(step() for _ in range(args.steps))
    sec = time.perf_counter() - t0
    value = flops / sec / 1e12
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(sec / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": HEADLINE, "batch": c.B, "q_heads": c.Hq, "kv_heads": c.Hkv, "seq_len": c.Lq,
                   "head_dim": c.D, "mask": "causal", "parallelism": "host cores"},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": f"{rows_per_step} random query rows per step of {HEADLINE}"},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def run_profile_case(args):
    """A few launches of one workload and nothing else: the command ncu captures."""
    import head_attention_attn_gb300 as attn
    from head_attention_attn_gb300.inputs import case
    from head_attention_attn_gb300 import build
    build.build_library()
    attn.load()
    if args.profile == PRELUDE:
        T, Hq, Hkv, hd = 16384, 32, 8, 128
        g = torch.Generator().manual_seed(1005)
        qkv = torch.randn(T, (Hq + 2 * Hkv) * hd, generator=g).to(torch.bfloat16).to("cuda:0")
        w = (torch.rand(hd, generator=g) + 0.5).to("cuda:0")
        ang = torch.arange(T, dtype=torch.float64)[:, None] * 1.0e6 ** (-2.0 * torch.arange(hd // 2) / hd)[None, :]
        cos, sin = torch.cos(ang).float().to("cuda:0"), torch.sin(ang).float().to("cuda:0")
        for _ in range(args.warmup + args.steps):
            attn.attn_qkv_prelude(qkv, Hq, Hkv, hd, qk_mode=attn.QK_NORM_ROPE, cos=cos, sin=sin, q_norm_w=w,
                                  k_norm_w=w)
        torch.cuda.synchronize()
        attn.check_device_status()
        print(json.dumps({"profile": args.profile, "launches": args.warmup + args.steps}))
        return
    if args.profile == PAGED_PREFILL:
        q, out, cu, kv_lens, k_pool, v_pool, table = paged_prefill_inputs(16, "cuda:0", torch.Generator().manual_seed(1008))
        for _ in range(args.warmup + args.steps):
            attn.attn_fwd_varlen_paged(q, k_pool, v_pool, table, cu, kv_lens, PAGED_SHAPE["chunk"], out)
        torch.cuda.synchronize()
        attn.check_device_status()
        print(json.dumps({"profile": args.profile, "launches": args.warmup + args.steps}))
        return
    c = WORKLOADS[args.profile] if args.batch is None else case(args.profile, B=args.batch)
    q, k, v, kl = make_inputs(c, device="cuda:0")
    out = torch.empty_like(q)
    for _ in range(args.warmup + args.steps):
        attn.attn_fwd(q, k, v, out, pos_offset=c.pos_offset, mask_mode=c.mask_mode, window=c.window, key_lens=kl)
    torch.cuda.synchronize()
    attn.check_device_status()
    print(json.dumps({"profile": args.profile, "batch": c.B, "launches": args.warmup + args.steps}))


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ref-rows", type=int, default=64)
    ap.add_argument("--profile", choices=sorted(WORKLOADS) + [PRELUDE, PAGED_PREFILL], default=None,
                    help="only run --warmup + --steps launches of one workload (for profilers)")
    ap.add_argument("--batch", type=int, default=None, help="batch size override for --profile")
    args = ap.parse_args(argv)
    if args.profile is None:
        args.warmup = max(3, args.warmup)  # at least 3 untimed warm-up steps
    if args.profile is not None:
        run_profile_case(args)
        return
    rank, world, local = dist_setup()
    if args.impl == "reference":
        res = run_reference(args, rank, world)
    else:
        res = run_ours(args, rank, world, local)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    if world > 1 and torch.distributed.is_initialized():
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
