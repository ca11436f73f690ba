#!/usr/bin/env python
"""Benchmark: paged FP8 decode attention on the Llama-3.1-8B-shaped layer.

One step = one decode step of one attention layer through the C ABI:
kv_append of the new token (B=32 x Hkv=8 rows quantised into e4m3 page slots)
then paged_decode_attn (tag validation, split-KV attention, combine) over
lengths ~ U[512, 8192] + 1, Hq=32, Hkv=8, head_dim 128, 16-token pages
scattered over a 65,536-page pool.  Steps rotate over R independent layer
replicas (each its own pool, tables and query) so that the live KV read by a
step (~286 MB; R x that in total) is never resident in the 129 MB L2.

Reported (one JSON line on rank 0):
  value        KV GB/s of the whole job: algorithmic bytes of the step (KV +
               tables + scales + tags + q + out + flags + appended rows) per
               second, summed over ranks
  tokens_per_s decode tokens/s of a 32-layer model whose every layer is this
               layer: ranks x B / (32 x step time)
  roofline     decode_split (the dominant kernel) timed live with CUDA events
               around its stage launch, against MEASURED_PEAKS.json hbm_gbs
  e2e          the same metric with the step's inputs copied from pinned host
               memory and its result read back inside the timed region
  cpu_baseline the oracle (test infrastructure) on a bounded sample, host cores

--impl reference times the oracle alone (CPU), as the reference arm.

--workload {tiny,long,sweep,evict} measures the other workloads instead, one
JSON line each: the long-context split (B=4, 128K..512K tokens, split 4096),
the 80 GB-pool sweep (--batch, --kv-dtype; every sequence 32,768 tokens) and
the eviction batch (per-head tables and lengths, stale tags) with tags on,
with every tag matching and with tags off.  These run one batch and flush L2
between steps (a write and then a read of buffers larger than L2) outside the
timed interval of each step.
"""
from __future__ import annotations

import argparse
import dataclasses
import ctypes
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged decode attention KV GB/s (Llama-3.1-8B-shaped FP8 layer, append + attend)"
UNIT = "GB/s"
WORKLOAD = "llama8b-fp8-decode-layer"
N_LAYERS = 32  # Llama-3.1-8B layer count, for tokens/s


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", default="pfkv", choices=["pfkv", "reference"])
    ap.add_argument("--replicas", type=int, default=8)
    ap.add_argument("--split", type=int, default=0, help="split-KV tokens (0 = library choice)")
    ap.add_argument("--no-tags", action="store_true", help="no-op tracker (no tag validation)")
    ap.add_argument("--fused-tags", action="store_true",
                    help="tag check inside the attention kernel instead of a separate pass")
    ap.add_argument("--e2e-steps", type=int, default=2000)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--clocks-csv", default=None,
                    help="keep the raw nvidia-smi clock samples at this path (the JSON line "
                         "carries their summary either way)")
    ap.add_argument("--workload", default="llama8b",
                    choices=["llama8b", "tiny", "long", "sweep", "evict"],
                    help="llama8b (default): the Llama-shaped layer; the others are the "
                         "tiny, long-context, 80 GB-pool sweep and eviction + tags workloads")
    ap.add_argument("--graph-layers", type=int, default=0,
                    help="time one decode step of this many Llama-shaped layers, each with its "
                         "own pool, captured as one CUDA graph (pfkv_step_graph_*)")
    ap.add_argument("--multi", type=int, default=0,
                    help="multi-query verify: append this many candidate tokens per request "
                         "and attend with all of them, causally (pfkv_paged_decode_attn_multi)")
    ap.add_argument("--batch", type=int, default=32, help="sweep: batch size")
    ap.add_argument("--kv-dtype", default="fp8", choices=["fp8", "bf16"], help="sweep: pool dtype")
    ap.add_argument("--head-dim", type=int, default=128, choices=[64, 128], help="sweep: head_dim")
    return ap.parse_args(argv)


# --------------------------------------------------------------------------
# multi-rank helpers (pure host logic; covered by a gloo test)
# --------------------------------------------------------------------------
def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def rank_seed(base: int, rank: int, replica: int) -> int:
    """Every (rank, replica) draws its own batch: same shapes, own data."""
    return base + 1000 * rank + replica


def reduce_max(value: float, world: int, device=None) -> float:
    """Max of a float over ranks (identity for one rank)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(bytes_per_step_per_rank: float, steps: int, seconds_max: float, world: int) -> float:
    """Whole-job GB/s: every rank moved bytes_per_step per step; the job took
    the slowest rank's time."""
    return bytes_per_step_per_rank * steps * world / seconds_max / 1e9


# --------------------------------------------------------------------------
# clocks
# --------------------------------------------------------------------------
def clocks_path(args) -> str:
    """Where the raw clock samples go: --clocks-csv, else a temporary file."""
    if args.clocks_csv:
        d = os.path.dirname(os.path.abspath(args.clocks_csv))
        os.makedirs(d, exist_ok=True)
        return args.clocks_csv
    import tempfile
    fd, path = tempfile.mkstemp(prefix="pfkv_clocks_", suffix=".csv")
    os.close(fd)
    return path


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, path: str):
        self.path, self.proc = path, None
        self.gpu = gpu_index

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.f,
                stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        return self.summary()

    def summary(self):
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), float(parts[3]), parts[5:9]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        load = [r for r in rows if r[2] > 200.0] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in load for i, v in enumerate(r[3]) if v == "Active"})
        return {"sm_mhz": statistics.median(r[0] for r in load),
                "sm_max_mhz": max(r[1] for r in rows), "reasons": reasons,
                "samples": len(load), "power_w_max": max(r[2] for r in rows)}


# --------------------------------------------------------------------------
# the GPU arm
# --------------------------------------------------------------------------
class PreparedStep:
    """The C-ABI calls of one step with their argument structs built once."""

    def __init__(self, db, B, stream_handle, cache=None, pages=None, fused_tags=False):
        self.db, self.B, self.s = db, B, stream_handle
        self.opt = B.PFKV_STAGE_FUSED_TAGS if fused_tags else 0
        L = B.lib()
        self.L = L
        self.c = (cache or db.cache).c_struct()
        self.p = (pages or db.pages).c_struct()
        ws = db.workspace
        self.args = (ctypes.byref(self.c), ctypes.byref(self.p), db.q.data_ptr(), db.spec.Hq,
                     ctypes.c_float(db.spec.sm_scale), db.split_tokens, db.max_seq_len,
                     ws.data_ptr(), ws.numel(), db.out.data_ptr(), db.flags.data_ptr())
        self.append_args = None
        if db.spec.append:
            self.append_args = (ctypes.byref(self.c), ctypes.byref(self.p), db.positions.data_ptr(),
                                None, 1, db.k_new.data_ptr(), db.v_new.data_ptr(),
                                db.append_flags.data_ptr(), stream_handle)

    def full_step(self):
        """The whole step through the public API: pfkv_decode_step (append and
        attention in one call) where the workload appends, else the attention
        call with every stage."""
        if self.append_args is None:
            self.stage(self.B.PFKV_STAGE_ALL)
            return
        a = self.append_args
        st = self.L.pfkv_decode_step(a[0], a[1], a[2], a[3], a[4], a[5], a[6], a[7], *self.args[2:],
                                     self.opt, self.s)
        if st:
            raise RuntimeError(f"pfkv_decode_step: status {st}")

    def append(self):
        if self.append_args is not None:
            st = self.L.pfkv_kv_append(*self.append_args)
            if st:
                raise RuntimeError(f"pfkv_kv_append: status {st}")

    def stage(self, mask):
        st = self.L.pfkv_paged_decode_attn_stages(*self.args, mask | self.opt, self.s)
        if st:
            raise RuntimeError(f"pfkv_paged_decode_attn_stages: status {st}")


class PreparedMassStep(PreparedStep):
    """A step whose attention also adds every live token's attention mass to a
    running total (pfkv_paged_decode_attn_mass); stage() runs the whole call."""

    def __init__(self, db, B, stream_handle, cache=None):
        import torch
        super().__init__(db, B, stream_handle, cache=cache)
        L = db.max_seq_len
        self.ws = torch.empty(B.pfkv_decode_mass_workspace_size(cache or db.cache, db.pages,
                                                                db.spec.Hq, db.split_tokens, L),
                              dtype=torch.uint8, device=db.q.device)
        self.mass = torch.zeros((db.spec.B, db.spec.Hkv, L), dtype=torch.float32,
                                device=db.q.device)
        self.margs = (ctypes.byref(self.c), ctypes.byref(self.p), db.q.data_ptr(), db.spec.Hq,
                      ctypes.c_float(db.spec.sm_scale), db.split_tokens, L, self.ws.data_ptr(),
                      self.ws.numel(), db.out.data_ptr(), db.flags.data_ptr(),
                      self.mass.data_ptr(), self.mass.stride(0), self.mass.stride(1), 0,
                      stream_handle)

    def stage(self, mask):
        st = self.L.pfkv_paged_decode_attn_mass(*self.margs)
        if st:
            raise RuntimeError(f"pfkv_paged_decode_attn_mass: status {st}")


# the arithmetic of the FP8 path (head_dim 128, query groups of up to 8 heads):
# e4m3 bytes converted exactly to f16, products on the tensor cores, fp32 sums
FP8_DTYPE = "fp8_e4m3 KV, f16 x f16 tensor-core MMA with fp32 accumulation, bf16 q/out"
# BF16 pools with head_dim 128 and groups of up to 8 heads: the same kernel
BF16_MMA_DTYPE = "bf16 KV, bf16 x bf16 tensor-core MMA with fp32 accumulation, bf16 q/out"


def path_dtype(spec) -> str:
    """The arithmetic a workload's split kernel computes in: the tensor-core
    kernel takes head_dim 128 or 64 with groups of up to 8 heads (every
    single-query workload), the CUDA-core kernel the rest."""
    mma = spec.D in (64, 128) and spec.Hq // spec.Hkv <= 8
    if spec.kv_dtype == "fp8":
        return FP8_DTYPE if mma else "fp8_e4m3 KV, fp32 FMA, bf16 q/out"
    return BF16_MMA_DTYPE if mma else "bf16 KV, fp32 FMA, bf16 q/out"


def profiled_traffic(bytes_per_launch: float, summary: str = "decode_split_pers_llama8b_fp8.md"):
    """DRAM bytes per launch of the split kernel from a committed ncu summary of
    the same workload, scaled to this run's algorithmic bytes; None if the
    kernel source changed since the capture (or there is no summary)."""
    import hashlib
    path = os.path.join(ROOT, "profiles", summary)
    if not os.path.exists(path):
        return None
    kv = {}
    for line in open(path):
        parts = line.strip().split(": ", 1)
        if len(parts) == 2:
            kv[parts[0]] = parts[1]
    try:
        src = os.path.join(ROOT, kv["kernel_source"])
        digest = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
        if digest != kv["kernel_source_sha256_16"]:
            return None
        return float(kv["dram_bytes_per_launch"]) * bytes_per_launch / float(
            kv["algorithmic_bytes_per_launch"])
    except (KeyError, OSError, ValueError):
        return None


# workloads with a committed ncu capture of their own split-kernel launch
WORKLOAD_PROFILES = {"long": "decode_split_pers_long_fp8.md"}


def workload_traffic(workload: str, bytes_per_launch: float):
    if workload not in WORKLOAD_PROFILES:
        return None
    t = profiled_traffic(bytes_per_launch, WORKLOAD_PROFILES[workload])
    return None if t is None else int(t)


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def gpu_hold(stream, us: float = 2000.0):
    """Keep the GPU busy on `stream` for about `us` microseconds (a spin
    kernel), so that work queued behind it starts without a host gap."""
    import torch
    with torch.cuda.stream(stream):
        torch.cuda._sleep(int(us * 2.0e3))  # cycles at about 2 GHz


def run_gpu(args):
    import torch
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import __graft_entry__
    __graft_entry__.build()
    from paged_fp8_kv_decode_gb300 import binding as B
    from paged_fp8_kv_decode_gb300 import workloads as W
    from paged_fp8_kv_decode_gb300.device_batch import DeviceBatch

    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    reps = []
    for r in range(args.replicas):
        spec = W.spec_llama8b("full", seed=rank_seed(W.BASE_SEED + 2, rank, r))
        spec.split_tokens = args.split
        if args.no_tags:
            spec.tags = False
        db = DeviceBatch(W.make_batch(spec), device=dev)
        db.pack_step_io()  # one host-to-device and one device-to-host copy per e2e step
        reps.append(PreparedStep(db, B, sh, fused_tags=args.fused_tags))
    torch.cuda.synchronize()
    spec0 = reps[0].db.spec
    # bytes per step (same shapes in every replica; lengths differ): mean over replicas
    attn_bytes = statistics.mean(p.db.algorithmic_bytes() for p in reps)
    kv_bytes = statistics.mean(p.db.kv_bytes() for p in reps)
    append_bytes = spec0.B * spec0.Hkv * spec0.D * (2 * 2 + 2 * 1) + spec0.B * spec0.Hkv * 8
    step_bytes = attn_bytes + append_bytes

    S_ALL = B.PFKV_STAGE_ALL
    S_V, S_S, S_C = B.PFKV_STAGE_VALIDATE, B.PFKV_STAGE_SPLIT, B.PFKV_STAGE_COMBINE

    def split_timed(p, ev):
        """The same work as one step, as separate calls, with events around the
        split kernel (events between kernels break their dependent-launch
        chain, so these steps are timed apart from the headline loop)."""
        p.append()
        p.stage(S_V)
        ev[0].record(stream)
        p.stage(S_S)
        ev[1].record(stream)
        p.stage(S_C)

    # Warm-up: every path the timed loops below take, on every replica, then
    # the requested number of steps.
    warm_ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
    for p in reps:
        p.full_step()
        split_timed(p, warm_ev)
    for i in range(args.warmup):
        reps[i % len(reps)].full_step()
    torch.cuda.synchronize()

    K = args.steps
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    sampler = None
    if rank == 0 and not args.no_clocks:
        sampler = ClockSampler(local, clocks_path(args))
        sampler.start()
        time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    # Hold the GPU for a moment so that the host queues the first steps before
    # the timed region starts: the region then times the GPU's work, not the
    # latency of the first launch.
    gpu_hold(stream)
    t0.record(stream)
    for i in range(K):
        reps[i % len(reps)].full_step()
    t1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop() if sampler else None
    elapsed = t0.elapsed_time(t1) / 1e3
    elapsed_max = reduce_max(elapsed, world, dev)

    # The split kernel alone, in a loop of its own after the headline loop.
    KS = max(2 * len(reps), min(K, 4000))
    ev_split = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                for _ in range(KS)]
    gpu_hold(stream)
    for i in range(KS):
        split_timed(reps[i % len(reps)], ev_split[i])
    torch.cuda.synchronize()
    split_ms = [a.elapsed_time(b) for a, b in ev_split]
    split_avg = sum(split_ms) / len(split_ms) / 1e3
    # the split kernel's algorithmic bytes: KV + table entries + scales of the
    # live pages (tags are read by the validation kernel)
    lens = [p.db.batch.lens_bh("seq").astype(np.int64) for p in reps]
    pages_live = statistics.mean(int(((l + 15) // 16).sum()) for l in lens)
    split_bytes = kv_bytes + pages_live * (4 + 8) + 2 * spec0.B * spec0.Hq * spec0.D
    split_gbs = split_bytes / split_avg / 1e9
    peak, peak_kind = peaks()

    # The same split stage on the per-chunk CUDA-core kernels, for comparison
    # with the tensor-core kernel (PFKV_STAGE_CUDA_CORES; a workspace of its own).
    cuda_core = None
    CC = B.PFKV_STAGE_CUDA_CORES
    for p in reps:
        p.args_tc = p.args

    def use(p, ws):
        a = list(p.args_tc)
        if ws is not None:
            a[7], a[8] = ws.data_ptr(), ws.numel()
        p.args = tuple(a)
    try:
        ws_cc = torch.empty(64 << 20, dtype=torch.uint8, device=dev)
        for p in reps:  # warm the CUDA-core kernels on every replica
            use(p, ws_cc)
            p.stage(S_V | CC), p.stage(S_S | CC), p.stage(S_C | CC)
        KC = max(len(reps), min(KS, 1000))
        ev_cc = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                 for _ in range(KC)]
        gpu_hold(stream)
        for i in range(KC):
            p = reps[i % len(reps)]
            p.append()
            p.stage(S_V | CC)
            ev_cc[i][0].record(stream)
            p.stage(S_S | CC)
            ev_cc[i][1].record(stream)
            p.stage(S_C | CC)
        torch.cuda.synchronize()
        cc_avg = sum(a.elapsed_time(b) for a, b in ev_cc) / KC / 1e3
        cuda_core = {"kernel": "decode_split_kernel (per-chunk CTAs, e4m3 dequantised to fp32 in "
                               "registers, fp32 FMAs, no tensor cores)",
                     "achieved": round(split_bytes / cc_avg / 1e9, 1), "unit": "GB/s",
                     "frac": round(split_bytes / cc_avg / 1e9 / peak, 4),
                     "avg_launch_us": round(cc_avg * 1e6, 3), "timed_launches": KC}
    except RuntimeError as e:  # a workspace too small for the per-chunk plan
        cuda_core = {"unavailable": str(e)}
    finally:
        for p in reps:
            use(p, None)

    # check the last step's flags (no request should be flagged in this workload)
    for p in reps:
        if int(p.db.flags[:spec0.B].sum()) or int(p.db.append_flags[:spec0.B].sum()):
            raise RuntimeError("benchmark workload flagged a request")

    value = aggregate(step_bytes, K, elapsed_max, world)
    ms_per_step = elapsed_max / K * 1e3
    tokens_per_s = world * spec0.B / (N_LAYERS * elapsed_max / K)

    e2e = run_e2e(args, reps, B, stream, step_bytes, world, dev)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(reps[0].db)

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
            "steps": K, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": FP8_DTYPE, "data": "synthetic",
            "config": {"workload": WORKLOAD, "batch": spec0.B, "num_q_heads": spec0.Hq,
                       "num_kv_heads": spec0.Hkv, "head_dim": spec0.D, "page_size": 16,
                       "seq_lens": "U[512,8192]+1 appended", "num_pages": spec0.num_pages,
                       "kv_dtype": spec0.kv_dtype, "tags": not args.no_tags,
                       "tag_check": ("none" if args.no_tags else
                                     "fused into attention" if args.fused_tags else "separate pass"),
                       "split_tokens": args.split, "replicas": args.replicas,
                       "step_call": "pfkv_decode_step (kv_append and validation share a launch); "
                                    "the split kernel is timed in a loop of its own after the "
                                    "timed steps, with events around its launch",
                       "l2": "inputs larger than L2: %d rotating replicas, %.0f MB live KV each"
                             % (args.replicas, kv_bytes / 1e6),
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
            "tokens_per_s": round(tokens_per_s, 1),
            "pct_of_hbm_peak": round(100 * value / world / peak, 2),
            "roofline": {"kernel": "decode_split", "bound": "hbm",
                         "achieved": round(split_gbs, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(split_gbs / peak, 4),
                         "traffic": (None if profiled_traffic(split_bytes) is None
                                     else int(profiled_traffic(split_bytes))),
                         "peak_kind": peak_kind, "avg_launch_us": round(split_avg * 1e6, 3),
                         "bytes_per_launch": int(split_bytes),
                         "timed_launches": len(split_ms)},
            "cuda_core_split": cuda_core,
            "e2e": e2e, "gpu_launches": 3 * K,
            "clocks": clocks, "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


class E2EStepGraph:
    """One end-to-end step through the library's public API with host buffers,
    as one CUDA graph of two calls: pfkv_stage_copy of the step's packed inputs
    (q, new K/V rows, positions, lengths, block table, expected tags) from
    pinned host memory into device memory (a copy kernel over the CPU-GPU
    link), then pfkv_decode_step (or the attention call where the workload does
    not append), whose kernels write out and flags straight into pinned host
    memory.  The object owns the pinned buffers the graph reads and writes:
    they live as long as the graph."""

    def __init__(self, db, B, fused_tags):
        import torch
        s = torch.cuda.Stream()
        self.h_in = db.io_in.detach().cpu().pin_memory()
        self.h_out = torch.zeros_like(db.io_out, device="cpu").pin_memory()
        hout = lambda t: self.h_out.data_ptr() + (t.data_ptr() - db.io_out.data_ptr())
        step = PreparedStep(db, B, s.cuda_stream, fused_tags=fused_tags)
        a = list(step.args)
        a[9], a[10] = hout(db.out), hout(db.flags)  # out and flags: host memory
        step.args = tuple(a)
        n = db.io_in.numel()
        with torch.cuda.stream(s):  # warm both calls on the capture stream
            B.pfkv_stage_copy(db.io_in, self.h_in, n, s)
            step.full_step()
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph, stream=s):
            B.pfkv_stage_copy(db.io_in, self.h_in, n, s)
            step.full_step()
        torch.cuda.synchronize()

    def replay(self):
        self.graph.replay()


def e2e_bytes(db):
    h2d = sum(t.numel() * t.element_size() for t in
              [db.q, db.positions, db.seq_lens, db.block_tables]
              + ([db.k_new, db.v_new] if db.spec.append else [])
              + ([db.expected_tags] if db.cache.page_tags is not None else []))
    d2h = db.out.numel() * db.out.element_size() + db.flags.numel()
    return int(h2d), int(d2h)


E2E_API = ("every step: one replay of a CUDA graph of two public calls, pfkv_stage_copy of the "
           "packed inputs (q, new K/V rows, positions, lengths, block table, expected tags) from "
           "pinned host memory into device memory (a copy kernel over NVLink-C2C), then "
           "pfkv_decode_step, whose kernels write out and flags straight into pinned host "
           "memory; then a stream synchronize")


def run_e2e(args, reps, B, stream, step_bytes, world, dev):
    """Same metric through the public API with host buffers: each step copies
    its inputs (q, new K/V rows, positions, lengths, block table, expected
    tags: packed in one buffer) from pinned host memory, runs append +
    attention, and reads the output and flags (one buffer) back, waiting for
    them before the next step."""
    import torch
    K = max(1, min(args.e2e_steps, args.steps))
    graphs = [E2EStepGraph(p.db, B, args.fused_tags) for p in reps]
    h2d, d2h = e2e_bytes(reps[0].db)
    for i in range(5):
        graphs[i % len(reps)].replay()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    t0 = time.perf_counter()
    for i in range(K):
        graphs[i % len(reps)].replay()
        stream.synchronize()
    el = time.perf_counter() - t0
    el = reduce_max(el, world, dev)
    return {"value": round(aggregate(step_bytes, K, el, world), 2), "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": K,
            "ms_per_step": round(el / K * 1e3, 4), "api": E2E_API}


# --------------------------------------------------------------------------
# the oracle (test infrastructure) as CPU baseline / reference arm
# --------------------------------------------------------------------------
def _oracle_sample(spec, n_requests: int, n_kv_heads: int, seed: int):
    """A bounded sample of the workload for the oracle: the first n requests
    with the workload's lengths, group size and head_dim but only n_kv_heads
    kv heads (and their G query heads each), quantised by the oracle itself,
    with every tag matching (attention only)."""
    import dataclasses
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import oracle
    from oracle_cases import cache_dict, fill_pool, pages_dict
    from paged_fp8_kv_decode_gb300 import workloads as W
    lens = np.asarray(spec.lens)
    lens = lens[:n_requests] if lens.ndim == 1 else lens[:n_requests, :n_kv_heads]
    need = (lens.astype(np.int64) + (1 if spec.append else 0) + 15) // 16
    num_pages = int(need.sum() if lens.ndim == 1 else need.sum(axis=0).max()) + 16
    sub = dataclasses.replace(spec, B=n_requests, lens=np.ascontiguousarray(lens),
                              Hkv=n_kv_heads, Hq=spec.G * n_kv_heads, seed=seed,
                              num_pages=num_pages, stale_per_mille=0.0)
    batch = W.make_batch(sub)
    T = int(batch.fill_lens.max())
    k_rows = W.draw_kv_rows(sub, T, "k")
    v_rows = W.draw_kv_rows(sub, T, "v")
    k, v, ks, vs = fill_pool(sub, batch, W.bf16_bits(k_rows), W.bf16_bits(v_rows))
    cache = cache_dict(sub, batch, k, v, ks, vs)
    pages = pages_dict(sub, batch, batch.seq_lens)
    if sub.append:
        oracle.kv_append(cache, pages, batch.positions,
                         W.bf16_bits(W.draw_new_token(sub, "k")),
                         W.bf16_bits(W.draw_new_token(sub, "v")))
    q = W.bf16_bits(W.draw_q(sub))
    el = 2 if sub.kv_dtype == "bf16" else 1
    kv = int(batch.lens_bh("seq").astype(np.int64).sum()) * sub.D * 2 * el
    return oracle, cache, pages, q, sub, batch, kv


def _time_oracle(oracle, cache, pages, q, sub, batch):
    t0 = time.perf_counter()
    oracle.paged_decode(cache, pages, q, sub.Hq, sub.sm_scale, int(batch.seq_lens.max()))
    return time.perf_counter() - t0


def _sample_shape(spec, head_tokens: int = 600_000):
    """Requests and kv heads of a bounded oracle sample: up to 4 requests, as
    many kv heads as keep (tokens x kv heads) under head_tokens."""
    lens = np.asarray(spec.lens).astype(np.int64)
    per_req = lens if lens.ndim == 1 else lens.max(axis=1)
    n = min(spec.B, 4)
    while n > 1 and int(per_req[:n].sum()) > head_tokens:
        n -= 1
    nh = max(1, min(spec.Hkv, head_tokens // max(1, int(per_req[:n].sum()))))
    return n, nh


def cpu_baseline_spec(spec, target_s: float = 15.0):
    """Oracle KV GB/s on the host cores over a bounded sample of the workload
    (and on one core, from a single call)."""
    n, nh = _sample_shape(spec)
    oracle, cache, pages, q, sub, batch, kv = _oracle_sample(spec, n, nh, spec.seed + 555)
    threads = oracle.num_threads()
    oracle.set_num_threads(1)
    t_one = _time_oracle(oracle, cache, pages, q, sub, batch)
    oracle.set_num_threads(threads)
    t = _time_oracle(oracle, cache, pages, q, sub, batch)
    reps = max(1, min(400, int(target_s / max(t, 1e-3))))
    total = t
    for _ in range(reps - 1):
        total += _time_oracle(oracle, cache, pages, q, sub, batch)
    return {"value": round(kv * reps / total / 1e9, 4), "unit": UNIT, "cores": threads,
            "kind": "oracle", "value_1_core": round(kv / t_one / 1e9, 4),
            "sample": f"{sub.B} of {spec.B} requests ({int(batch.lens_bh('seq')[:, 0].sum())} "
                      f"tokens per kv head), {sub.Hkv} of {spec.Hkv} kv heads ({sub.Hq} q heads), "
                      f"attention only, {reps} repetitions in {total:.1f} s; "
                      f"KV bytes read / oracle time"}


def cpu_baseline(db, target_s: float = 15.0):
    return cpu_baseline_spec(db.spec, target_s)


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    spec = workload_spec(args)
    # per step: one request of the workload, restricted to enough kv heads that
    # warmup + steps fit in about two minutes of oracle time
    oracle, cache, pages, q, sub, batch, kv = _oracle_sample(spec, 1, 1, spec.seed + 777)
    t1 = min(_time_oracle(oracle, cache, pages, q, sub, batch) for _ in range(2))
    budget = 120.0 / max(1, args.steps + args.warmup)
    nh = max(1, min(spec.Hkv, int(budget / max(t1, 1e-6))))
    if nh > 1:
        oracle, cache, pages, q, sub, batch, kv = _oracle_sample(spec, 1, nh, spec.seed + 777)
    for _ in range(args.warmup):
        _time_oracle(oracle, cache, pages, q, sub, batch)
    ts = [_time_oracle(oracle, cache, pages, q, sub, batch) for _ in range(args.steps)]
    total = sum(ts)
    value = kv * len(ts) / total / 1e9
    sample = (f"1 request ({int(batch.lens_bh('seq')[0, 0])} tokens), {sub.Hkv} of {spec.Hkv} kv heads "
              f"({sub.Hq} q heads) per step, attention only; KV bytes read / oracle time")
    metric = METRIC if args.workload == "llama8b" else \
        "paged decode attention KV GB/s (" + spec.name + ")"
    line = {"impl": "reference", "metric": metric, "value": round(value, 5), "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(total / len(ts) * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64 attention, f32 quantiser",
            "data": "synthetic",
            "config": {"workload": WORKLOAD if args.workload == "llama8b" else spec.name + "-full",
                       "batch": spec.B, "num_q_heads": spec.Hq,
                       "num_kv_heads": spec.Hkv, "head_dim": spec.D, "page_size": 16,
                       "kv_dtype": spec.kv_dtype},
            "cpu_baseline": {"value": round(value, 5), "unit": UNIT, "cores": oracle.num_threads(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 5), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def workload_spec(args, rank: int = 0):
    """The spec of --workload (each rank draws its own data)."""
    from paged_fp8_kv_decode_gb300 import workloads as W
    seed_of = {"tiny": W.BASE_SEED + 1, "long": W.BASE_SEED + 3, "sweep": W.BASE_SEED + 4,
               "evict": W.BASE_SEED + 5, "llama8b": W.BASE_SEED + 2}
    seed = rank_seed(seed_of[args.workload], rank, 0)
    if args.workload == "tiny":
        return W.spec_tiny(seed=seed)
    if args.workload == "long":
        return W.spec_long("full", seed=seed)
    if args.workload == "sweep":
        spec = W.spec_sweep(args.batch, args.kv_dtype, seed=seed)
        return dataclasses.replace(spec, D=args.head_dim) if args.head_dim != spec.D else spec
    if args.workload == "evict":
        return W.spec_evict("full", seed=seed)
    return W.spec_llama8b("full", seed=seed)


def sweep_admissible(spec, pool_bytes: float = 80e9, layers: int = N_LAYERS) -> int:
    """Largest batch whose KV for every layer of a 32-layer model fits an 80 GB
    pool, with every sequence at this workload's length."""
    el = 2 if spec.kv_dtype == "bf16" else 1
    per_token = 2 * spec.Hkv * spec.D * el + (2 * spec.Hkv * 4 / 16 if spec.kv_dtype == "fp8" else 0)
    return int(pool_bytes // (int(spec.lens[0]) * layers * per_token))


class L2Flush:
    """Evicts L2 between timed steps: writes one buffer larger than L2, then
    reads another so that the written lines are clean (their write-back
    happens here, not inside the next step)."""

    def __init__(self, dev, mb: int = 512):
        import torch
        self.w = torch.empty(mb << 20, dtype=torch.uint8, device=dev)
        self.r = torch.ones((mb << 20) // 4, dtype=torch.int32, device=dev)

    def __call__(self):
        self.w.fill_(1)
        self.r.max()


def _median_times(ms):
    ms = sorted(ms)
    q = lambda f: ms[min(len(ms) - 1, int(f * (len(ms) - 1) + 0.5))]
    return q(0.5), q(0.1), q(0.9)


def run_workload(args):
    """One JSON line for --workload tiny/long/sweep/evict (see module docstring)."""
    import torch
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import __graft_entry__
    __graft_entry__.build()
    from paged_fp8_kv_decode_gb300 import binding as B
    from paged_fp8_kv_decode_gb300 import workloads as W
    from paged_fp8_kv_decode_gb300.device_batch import DeviceBatch

    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    spec = workload_spec(args, rank)
    if args.split:  # a caller's fixed split size instead of the workload's
        spec.split_tokens = args.split
    db = DeviceBatch(W.make_batch(spec), device=dev)
    db.pack_step_io()  # one host-to-device and one device-to-host copy per e2e step
    variants = [("tags" if spec.tags else "no_tags", PreparedStep(db, B, sh), spec.tags)]
    if args.workload == "evict":
        # every live unit carrying the tag its request expects (no request aborted)
        batch = db.batch
        match = batch.page_tags.copy()
        bt, ex = batch.block_tables, batch.expected_tags
        lens = batch.lens_bh("seq")
        for b in range(spec.B):
            for h in range(spec.Hkv):
                k = (int(lens[b, h]) + 15) // 16
                match[bt[b, h, :k], h] = ex[b, h, :k]
        match_t = torch.from_numpy(match.view(np.int32)).to(dev)
        c_match = B.Cache(db.cache.k_pages, db.cache.v_pages, db.cache.k_scale, db.cache.v_scale,
                          match_t)
        p_off = B.Pages(db.pages.batch, db.pages.max_pages, db.pages.block_tables,
                        db.pages.bt_stride_b, db.pages.bt_stride_h, db.pages.seq_lens,
                        db.pages.len_stride_b, db.pages.len_stride_h, None)
        variants.append(("tags_all_match", PreparedStep(db, B, sh, cache=c_match), True))
        variants.append(("fused_tags_all_match",
                         PreparedStep(db, B, sh, cache=c_match, fused_tags=True), True))
        variants.append(("fused_tags", PreparedStep(db, B, sh, fused_tags=True), True))
        variants.append(("tags_all_match_attn_mass", PreparedMassStep(db, B, sh, cache=c_match),
                         True))
        variants.append(("no_tags", PreparedStep(db, B, sh, cache=db.cache_untracked,
                                                 pages=p_off), False))
    flush = L2Flush(dev)
    S_ALL = B.PFKV_STAGE_ALL
    S_V, S_S, S_C = B.PFKV_STAGE_VALIDATE, B.PFKV_STAGE_SPLIT, B.PFKV_STAGE_COMBINE
    K = args.steps

    def timed(p, split_only=False):
        for _ in range(args.warmup):
            flush()
            p.append()
            p.stage(S_ALL)
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(K)]
        for i in range(K):
            flush()
            if split_only:
                p.append()
                p.stage(S_V)
                evs[i][0].record(stream)
                p.stage(S_S)
                evs[i][1].record(stream)
                p.stage(S_C)
            else:
                evs[i][0].record(stream)
                p.append()
                p.stage(S_ALL)
                evs[i][1].record(stream)
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in evs]

    append_bytes = (spec.B * spec.Hkv * spec.D * (2 * 2 + 2 * (2 if spec.kv_dtype == "bf16" else 1))
                    + (spec.B * spec.Hkv * 8 if spec.kv_dtype == "fp8" else 0)) if spec.append else 0
    sampler = None
    if rank == 0 and not args.no_clocks:
        sampler = ClockSampler(local, clocks_path(args))
        sampler.start()
        time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    results = {}
    for name, p, tags in variants:
        ms = timed(p)
        flags = db.flags[:spec.B].cpu().numpy()
        skip = flags != 0
        by = db.algorithmic_bytes(skip=skip, tags=tags) + append_bytes
        med, p10, p90 = _median_times(ms)
        med = reduce_max(med, world, dev)
        results[name] = {"ms_per_step": round(med, 5), "p10_ms": round(p10, 5),
                         "p90_ms": round(p90, 5), "bytes_per_step": int(by),
                         "gbs": round(by * world / (med / 1e3) / 1e9, 2),
                         "requests_aborted": int(skip.sum())}
    name0, p0, tags0 = variants[0]
    split_ms = timed(p0, split_only=True)
    clocks = sampler.stop() if sampler else None
    split_med = _median_times(split_ms)[0]
    flags = db.flags[:spec.B].cpu().numpy()
    skip = flags != 0
    lens = db._lens(skip)
    split_bytes = (db.kv_bytes(skip) + int(((lens + 15) // 16).sum())
                   * (4 + (8 if spec.kv_dtype == "fp8" else 0)) + 2 * spec.B * spec.Hq * spec.D * 2)
    split_gbs = split_bytes / (split_med / 1e3) / 1e9
    peak, peak_kind = peaks()
    r0 = results[name0]
    med_s = r0["ms_per_step"] / 1e3
    cfg = {"workload": f"{spec.name}" + ("-full" if args.workload != "tiny" else ""),
           "batch": spec.B, "num_q_heads": spec.Hq, "num_kv_heads": spec.Hkv,
           "head_dim": spec.D, "page_size": 16, "num_pages": spec.num_pages,
           "kv_dtype": spec.kv_dtype, "tags": tags0, "split_tokens": spec.split_tokens,
           "per_head_tables": spec.per_head, "append": spec.append,
           "live_kv_mb": round(db.kv_bytes() / 1e6, 1),
           "l2": "L2 flushed between timed steps (512 MB write + 512 MB read, outside the "
                 "timed interval)",
           "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}
    if args.workload == "sweep":
        adm = sweep_admissible(spec)
        cfg["seq_len"] = int(spec.lens[0])
        cfg["admissible_batch_80gb_32_layers"] = adm
        cfg["admissible"] = spec.B <= adm
    line = {
        "metric": "paged decode attention KV GB/s (" + spec.name + ")",
        "value": round(r0["gbs"], 2), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": r0["ms_per_step"], "p10_ms": r0["p10_ms"],
        "p90_ms": r0["p90_ms"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None,
        "dtype": path_dtype(spec),
        "data": "synthetic", "config": cfg,
        "tokens_per_s": round(world * spec.B / (N_LAYERS * med_s), 1),
        "tokens_per_s_per_layer": round(world * spec.B / med_s, 1),
        "pct_of_hbm_peak": round(100 * r0["gbs"] / world / peak, 2),
        "roofline": {"kernel": "decode_split", "bound": "hbm", "achieved": round(split_gbs, 1),
                     "peak": peak, "unit": "GB/s", "frac": round(split_gbs / peak, 4),
                     "traffic": workload_traffic(args.workload, split_bytes),
                     "peak_kind": peak_kind,
                     "avg_launch_us": round(split_med * 1e3, 3), "stat": "median",
                     "bytes_per_launch": int(split_bytes), "timed_launches": len(split_ms)},
        "variants": results if len(results) > 1 else None,
        "gpu_launches": K * (len(variants) * (3 if spec.append else 2) + 3) + sum(
            K for _, p, t in variants if t and not p.opt) + sum(
            K for _, p, _ in variants if isinstance(p, PreparedMassStep)),
        "clocks": clocks,
    }
    if "tags_all_match" in results and "no_tags" in results:
        b = results["no_tags"]["ms_per_step"]
        a = results["tags_all_match"]["ms_per_step"]
        line["tag_overhead_pct"] = round(100 * (a - b) / b, 2)
        a = results["fused_tags_all_match"]["ms_per_step"]
        line["fused_tag_overhead_pct"] = round(100 * (a - b) / b, 2)
        a = results["tags_all_match_attn_mass"]["ms_per_step"]
        c = results["tags_all_match"]["ms_per_step"]
        line["attn_mass_overhead_pct"] = round(100 * (a - c) / c, 2)
    line["e2e"] = run_e2e_flushed(args, p0, B, stream, r0["bytes_per_step"], world, dev, flush)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_spec(spec)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def run_e2e_flushed(args, p, B, stream, step_bytes, world, dev, flush):
    """End to end through the public API with host buffers, L2 flushed before
    each step outside the host-timed interval."""
    import torch
    K = max(1, min(args.e2e_steps, args.steps))
    g = E2EStepGraph(p.db, B, bool(p.opt))
    h2d, d2h = e2e_bytes(p.db)
    total = 0.0
    for i in range(K + 2):
        flush()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        g.replay()
        stream.synchronize()
        if i >= 2:
            total += time.perf_counter() - t0
    total = reduce_max(total, world, dev)
    return {"value": round(aggregate(step_bytes, K, total, world), 2), "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "steps": K, "ms_per_step": round(total / K * 1e3, 4), "api": E2E_API}


def run_graph(args):
    """One JSON line: decode steps of a stack of --graph-layers layers (the
    Llama-shaped FP8 layer, each with its own pool and query, shared tables)
    replayed from one CUDA graph per step."""
    import torch
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import dataclasses
    import __graft_entry__
    __graft_entry__.build()
    from paged_fp8_kv_decode_gb300 import binding as B
    from paged_fp8_kv_decode_gb300 import workloads as W
    from paged_fp8_kv_decode_gb300.device_batch import DeviceBatch
    n = args.graph_layers
    spec = W.spec_llama8b("full", seed=rank_seed(W.BASE_SEED + 2, rank, 0))
    spec.split_tokens = args.split
    if args.no_tags:
        spec.tags = False
    batch = W.make_batch(spec)
    T = int(batch.fill_lens.max())
    dbs = []
    for l in range(n):
        sl = dataclasses.replace(spec, seed=spec.seed + 7 * (l + 1))
        rows = (W.draw_kv_rows(sl, T, "k", device=dev), W.draw_kv_rows(sl, T, "v", device=dev))
        db = DeviceBatch(batch, device=dev, rows=rows, q=W.draw_q(sl, device=dev))
        del rows
        dbs.append(db)
    torch.cuda.synchronize()
    d0 = dbs[0]
    layers = [B.Layer(cache=d.cache, q=d.q, out=d.out, k_new=d.k_new, v_new=d.v_new, flags=d.flags)
              for d in dbs]
    graph = B.pfkv_step_graph_create(layers, d0.pages, d0.positions, None, 1, d0.append_flags,
                                     spec.Hq, spec.sm_scale, spec.split_tokens, d0.max_seq_len,
                                     d0.workspace, B.PFKV_STAGE_FUSED_TAGS if args.fused_tags else 0)
    stream = torch.cuda.current_stream(dev)
    for _ in range(max(3, args.warmup)):
        graph.launch(stream)
    torch.cuda.synchronize()
    K = args.steps
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(K)]
    sampler = None
    if rank == 0 and not args.no_clocks:
        sampler = ClockSampler(local, clocks_path(args))
        sampler.start()
        time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(K):
        evs[i][0].record(stream)
        graph.launch(stream)
        evs[i][1].record(stream)
    t1.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop() if sampler else None
    total = reduce_max(t0.elapsed_time(t1) / 1e3, world, dev)
    ms = sorted(a.elapsed_time(b) for a, b in evs)
    med, p10, p90 = _median_times(ms)
    if any(int(d.flags[:spec.B].sum()) for d in dbs) or int(d0.append_flags[:spec.B].sum()):
        raise RuntimeError("benchmark workload flagged a request")
    attn = sum(d.algorithmic_bytes() for d in dbs)
    append = n * (spec.B * spec.Hkv * spec.D * (2 * 2 + 2) + spec.B * spec.Hkv * 8)
    step_bytes = attn + append
    graph.close()
    if rank == 0:
        line = {
            "metric": f"decode tokens/s ({n} Llama-3.1-8B-shaped FP8 attention layers per step, "
                      f"one CUDA graph per step)",
            "value": round(world * spec.B * K / total, 1), "unit": "tokens/s", "n_gpus": world,
            "steps": K, "warmup": max(3, args.warmup),
            "ms_per_step": round(total / K * 1e3, 4), "median_ms": round(med, 4),
            "p10_ms": round(p10, 4), "p90_ms": round(p90, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": FP8_DTYPE, "data": "synthetic",
            "config": {"workload": "llama8b-fp8-decode-stack", "layers": n, "batch": spec.B,
                       "num_q_heads": spec.Hq, "num_kv_heads": spec.Hkv, "head_dim": spec.D,
                       "page_size": 16, "num_pages_per_layer": spec.num_pages,
                       "tags": spec.tags, "tag_check": ("none" if not spec.tags else
                                                        "fused into attention" if args.fused_tags
                                                        else "separate pass"),
                       "l2": "inputs larger than L2: %d layers, %.0f MB live KV each"
                             % (n, dbs[0].kv_bytes() / 1e6),
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
            "kv_gbs": round(world * step_bytes * K / total / 1e9, 2),
            "per_layer_us": round(total / K / n * 1e6, 3),
            "gpu_launches": K * n * (3 if (args.no_tags or args.fused_tags) else 4),
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def run_multi(args):
    """One JSON line: the verification step of speculative decoding on the
    Llama-shaped FP8 layer: kv_append of kq candidate tokens per request, then
    attention of all kq query tokens, causal among them, over rotating layer
    replicas (inputs larger than L2)."""
    import torch
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import dataclasses
    import __graft_entry__
    __graft_entry__.build()
    from paged_fp8_kv_decode_gb300 import binding as B
    from paged_fp8_kv_decode_gb300 import workloads as W
    from paged_fp8_kv_decode_gb300.device_batch import DeviceBatch
    kq = args.multi
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    L = B.lib()
    reps = []
    opt = B.PFKV_STAGE_FUSED_TAGS if args.fused_tags else 0
    for r in range(args.replicas):
        base = W.spec_llama8b("full", seed=rank_seed(W.BASE_SEED + 2, rank, r))
        # the cache holds the context and the kq candidates (the step rewrites them)
        spec = dataclasses.replace(base, append=False, lens=base.lens + kq, split_tokens=args.split,
                                   tags=not args.no_tags)
        db = DeviceBatch(W.make_batch(spec), device=dev)
        g = torch.Generator(device=dev).manual_seed(77 + r)
        q = torch.randn((spec.B, kq, spec.Hq, spec.D), generator=g, device=dev).to(torch.bfloat16)
        kn = torch.randn((spec.B, spec.Hkv, kq, spec.D), generator=g, device=dev).to(torch.bfloat16)
        vn = torch.randn((spec.B, spec.Hkv, kq, spec.D), generator=g, device=dev).to(torch.bfloat16)
        pos = (db.seq_lens - kq).contiguous()
        out = torch.empty_like(q)
        Lmax = db.max_seq_len
        ws = torch.empty(B.pfkv_decode_multi_workspace_size(db.cache, db.pages, spec.Hq, kq,
                                                            spec.split_tokens, Lmax),
                         dtype=torch.uint8, device=dev)
        c, p = db.cache.c_struct(), db.pages.c_struct()
        keep = (db, q, kn, vn, pos, out, ws, c, p)
        app = (ctypes.byref(c), ctypes.byref(p), pos.data_ptr(), None, kq, kn.data_ptr(),
               vn.data_ptr(), db.append_flags.data_ptr(), sh)
        att = (ctypes.byref(c), ctypes.byref(p), q.data_ptr(), spec.Hq, kq,
               ctypes.c_float(spec.sm_scale), spec.split_tokens, Lmax, ws.data_ptr(), ws.numel(),
               out.data_ptr(), db.flags.data_ptr(), opt, sh)
        reps.append((keep, app, att))
    spec0 = reps[0][0][0].spec

    def step(r):
        _, app, att = r
        if L.pfkv_kv_append(*app) or L.pfkv_paged_decode_attn_multi(*att):
            raise RuntimeError("multi-query step failed")

    for i in range(args.warmup):
        step(reps[i % len(reps)])
    torch.cuda.synchronize()
    K = args.steps
    sampler = None
    if rank == 0 and not args.no_clocks:
        sampler = ClockSampler(local, clocks_path(args))
        sampler.start()
        time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t0.record(stream)
    for i in range(K):
        step(reps[i % len(reps)])
    t1.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop() if sampler else None
    el = reduce_max(t0.elapsed_time(t1) / 1e3, world, dev)
    for (db, *_), _, _ in reps:
        if int(db.flags[:spec0.B].sum()) or int(db.append_flags[:spec0.B].sum()):
            raise RuntimeError("benchmark workload flagged a request")
    # algorithmic bytes: each request's KV once (all kq queries read the same
    # pages), tables and scales, kq rows of q and out, the appended candidates
    attn = statistics.mean(r[0][0].algorithmic_bytes() for r in reps)
    attn += 2 * spec0.B * (kq - 1) * spec0.Hq * spec0.D * 2
    append = spec0.B * spec0.Hkv * kq * spec0.D * (2 * 2 + 2) + spec0.B * spec0.Hkv * 8
    step_bytes = attn + append
    if rank == 0:
        line = {
            "metric": f"multi-query verify KV GB/s (Llama-3.1-8B-shaped FP8 layer, "
                      f"{kq} candidate tokens per request)",
            "value": round(aggregate(step_bytes, K, el, world), 2), "unit": "GB/s",
            "n_gpus": world, "steps": K, "warmup": args.warmup,
            "ms_per_step": round(el / K * 1e3, 5), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": FP8_DTYPE,
            "data": "synthetic",
            "config": {"workload": "llama8b-fp8-verify", "batch": spec0.B,
                       "query_tokens_per_request": kq, "num_q_heads": spec0.Hq,
                       "num_kv_heads": spec0.Hkv, "head_dim": spec0.D, "page_size": 16,
                       "seq_lens": f"U[512,8192]+{kq}", "replicas": args.replicas,
                       "tag_check": ("none" if args.no_tags else "fused into attention"
                                     if args.fused_tags else "separate pass"),
                       "l2": "inputs larger than L2: %d rotating replicas" % args.replicas,
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
            "verified_tokens_per_s": round(world * spec0.B * kq / (N_LAYERS * el / K), 1),
            "gpu_launches": K * (3 if (args.no_tags or args.fused_tags) else 4),
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        run_reference(args)
    elif args.multi > 0:
        run_multi(args)
    elif args.graph_layers > 0:
        run_graph(args)
    elif args.workload != "llama8b":
        run_workload(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
