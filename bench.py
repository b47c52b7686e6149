"""Benchmark: paged FP8-KV decode attention, effective HBM GB/s on GB300.

One step = one pass of the hot path over one batch of the workload: the
append of the step's new tokens into the paged cache (when the workload has
any), the split-KV decode / grouped-verify kernel and the LSE merge, all
through the C ABI (paged_fp8_kv_cache_gb300.binding -> libpfkv.so).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload ID] [--impl reference]

Prints ONE JSON line (rank 0). The headline workload is the q8 speculative
verify over 2 x 256K keys (1.07 GB of FP8 KV per step: the largest workload
of fixed size, and one of the two long-context workloads that carry the
75 %-of-peak target). ``value`` = algorithmic bytes of all ranks / max-over-ranks device
time of the K timed steps (inputs resident in HBM, L2 flushed between steps:
a 256 MiB write, then a 256 MiB read, so that the step starts on a cold L2
holding no dirty lines, whose write-back would otherwise compete with the
step's own HBM traffic). ``e2e`` repeats the measurement through the same
public calls with the step's inputs copied from pinned host memory (one
copy of one packed buffer) and the outputs copied back (one copy) inside the
timed region. ``roofline`` is the decode call (decode/verify kernel + merge)
timed alone with CUDA events on its stream. ``cpu_baseline`` times the CPU
oracle on a bounded sample of the same workload. ``per_config`` and
``extensions`` give the same objects for every other workload.
``--impl reference`` times the CPU oracle (the only reference arm this
project has) on a bounded sample of the headline workload.

Algorithmic bytes of a step: K+V cache bytes read (every key of every
(sequence, KV head) once) + Q + out + LSE + the block-table entries used +
seq_lens, plus for an append: the new fp16 K/V read, their cache bytes
written and the slot mapping. Split partials are not counted (they are
overhead of the implementation).
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import shutil
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from paged_fp8_kv_cache_gb300 import workloads  # noqa: E402

METRIC = "paged FP8-KV decode attention: effective HBM GB/s and % of GB300 peak"
# the q8 speculative verify, 2 x 262144 keys: the largest workload of fixed size
DEFAULT_WORKLOAD = 4
L2_FLUSH_BYTES = 256 << 20  # > 2x the 129 MB L2
FALLBACK_HBM_GBS = 6800.0
# sources of each kernel (the hash ties a committed ncu summary to the code it measured)
KERNEL_SOURCES = {
    "decode_kernel": ["decode_kernel.cuh", "device_utils.cuh", "frag_layout.h", "mask_span.h"],
    "decode_persist_kernel": ["decode_kernel.cuh", "device_utils.cuh", "frag_layout.h", "mask_span.h"],
    "verify_kernel": ["verify_kernel.cuh", "device_utils.cuh", "frag_layout.h", "verify_layout.h", "mask_span.h"],
}


# ----------------------------------------------------------------------------- helpers


class L2Flush:
    """Cold, clean L2 before a timed step: write a buffer larger than L2, then read another
    (the write-back of the written lines happens during the read, outside the timed region)."""

    def __init__(self, torch):
        n = L2_FLUSH_BYTES // 4
        self.torch = torch
        self.w = torch.zeros(n, dtype=torch.float32, device="cuda")
        self.r = torch.ones(n, dtype=torch.float32, device="cuda")
        self.sink = torch.zeros((), dtype=torch.float32, device="cuda")

    def __call__(self):
        self.w.add_(1)
        self.torch.sum(self.r, dim=0, out=self.sink)


def visible_span(spec, n: int):
    """Keys [lo, hi] some query row of a sequence of n keys sees under the workload's mask (its
    query tokens sit at positions n - T .. n - 1; a window of W keys ends each row's view W
    positions back from it)."""
    T = spec.num_q_tokens
    lo = max(0, n - T - spec.window + 1) if spec.window > 0 else 0
    return lo, n - 1


def useful_flops(case) -> int:
    """QK^T and PV multiply-adds of every query row over its visible keys: 4 * D per (row, key)."""
    s = case.spec
    T, W = s.num_q_tokens, s.window
    total = 0
    for n in case.seq_lens.astype(np.int64):
        p = n - T + np.arange(T)
        hi = np.minimum(p, n - 1) if s.causal else np.full(T, n - 1)
        lo = np.maximum(0, p - W + 1) if W > 0 else np.zeros(T, np.int64)
        total += int(np.maximum(0, hi - lo + 1).sum())
    return 4 * s.head_dim * s.num_q_heads * total


def algorithmic_bytes(case, with_append: bool) -> int:
    s = case.spec
    elt = 2 if s.kv_dtype == "fp16" else 1
    keys = pages = 0
    for n in case.seq_lens.astype(np.int64):
        lo, hi = visible_span(s, int(n))
        if hi >= lo:
            keys += hi - lo + 1
            pages += hi // s.page_size - lo // s.page_size + 1
    kv = keys * s.num_kv_heads * s.head_dim * elt * 2
    rows = case.B * s.num_q_tokens * s.num_q_heads
    q_out = rows * s.head_dim * 2 * 2
    lse = rows * 4
    meta = case.B * 4
    total = kv + q_out + lse + pages * 4 + meta
    if with_append and case.slot_new.size:
        n = case.slot_new.size
        total += n * s.num_kv_heads * s.head_dim * (2 * 2 + elt * 2) + n * 8
    return total


def kernel_of(spec) -> str:
    """The kernel a workload's decode call runs: the tcgen05 grouped verifier for FP8 caches with
    more than 16 query rows per CTA (a slab holds up to 64 rows), the mma.sync decode kernel
    otherwise."""
    g = spec.num_q_heads // spec.num_kv_heads
    tokens = spec.num_q_tokens if spec.num_q_tokens * g <= 64 else 64 // g
    return "verify_kernel" if spec.kv_dtype != "fp16" and tokens * g > 16 else "decode_kernel"


def kernel_source_hash(kernel: str = "decode_kernel") -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "paged_fp8_kv_cache_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


FALLBACK_BF16_TFLOPS = 1900.0


def measured_tensor_peak():
    """Dense bf16 tensor-core TFLOP/s (burst) measured on this machine, else the fallback."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        if "bf16_tflops" in d:
            return float(d["bf16_tflops"]), "measured"
    return FALLBACK_BF16_TFLOPS, "fallback"


def profiled_traffic(workload_id: int, kernel: str):
    """DRAM bytes per launch of the workload's kernel from the committed ncu summary, if it was
    taken on the current kernel sources; else None."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_workload{workload_id}.txt")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m_hash = re.search(r"kernel_source_hash:\s*([0-9a-f]+)", text)
    m_t = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not (m_hash and m_t) or m_hash.group(1) != kernel_source_hash(kernel):
        return None
    return float(m_t.group(1))


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"pfkv_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sm, smax, reasons, n = [], None, set(), 0
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            n += 1
            for nm, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": n}


def max_over_ranks(values, dist=None, device="cpu"):
    """Element-wise max of per-rank timings (every rank gets the result)."""
    import torch
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    if dist is not None and dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.cpu()]


def rank_seed(spec, rank: int) -> int:
    """Each rank decodes its own batch of the workload (weak scaling); rank 0 the canonical one."""
    return spec.seed + 1000 * rank


def aggregate_gbs(bytes_per_rank_step: int, world: int, steps: int, max_ms: float) -> float:
    """Whole-job effective GB/s: bytes every rank processed / the slowest rank's time."""
    return bytes_per_rank_step * world * steps / (max_ms * 1e-3) / 1e9


def packed_layout(sizes, align: int = 256):
    """Byte offsets of buffers packed one after another (each start aligned) and the total size."""
    offs, off = [], 0
    for n in sizes:
        offs.append(off)
        off += -(-int(n) // align) * align
    return offs, max(off, align)


# ----------------------------------------------------------------------------- GPU arm

class DeviceWorkload:
    """A workload resident on the GPU: caches populated through the append kernel.

    The step's inputs (Q, block table, sequence lengths, new K/V and their slots) are views of
    one device buffer with a pinned host twin, and the outputs (out, LSE) views of another, so
    the end-to-end step moves its inputs and results with one copy each way."""

    def __init__(self, case, torch, pf):
        self.torch, self.pf, self.case = torch, pf, case
        s = case.spec
        dev = "cuda"
        elt = torch.float16 if s.kv_dtype == "fp16" else torch.uint8
        shape = (case.num_blocks, s.num_kv_heads, s.page_size, s.head_dim)
        self.k_cache = torch.zeros(shape, dtype=elt, device=dev)
        self.v_cache = torch.zeros(shape, dtype=elt, device=dev)
        # one float per pool, or one per KV head (the binding then sets PFKV_KV_SCALES_PER_HEAD)
        self.k_scale = torch.tensor(np.asarray(case.k_scale, np.float32).reshape(-1), device=dev)
        self.v_scale = torch.tensor(np.asarray(case.v_scale, np.float32).reshape(-1), device=dev)
        n = case.k_fill.shape[0]
        step = max(1, (1 << 24) // (s.num_kv_heads * s.head_dim))
        for a in range(0, n, step):
            b = min(n, a + step)
            pf.pfkv_kv_cache_append(torch.from_numpy(case.k_fill[a:b]).to(dev),
                                    torch.from_numpy(case.v_fill[a:b]).to(dev), self.k_cache, self.v_cache,
                                    torch.from_numpy(case.slot_fill[a:b]).to(dev), s.page_size, s.kv_dtype,
                                    self.k_scale, self.v_scale)
        # per-step inputs: one pinned host buffer and its device twin
        ins = [("q", case.q), ("bt", case.block_table), ("sl", case.seq_lens), ("kn", case.k_new),
               ("vn", case.v_new), ("slot", case.slot_new)]
        offs, total = packed_layout([a.nbytes for _, a in ins])
        self.h_in = torch.empty(total, dtype=torch.uint8).pin_memory()
        self.d_in = torch.empty(total, dtype=torch.uint8, device=dev)
        self.d = {}
        for (name, a), off in zip(ins, offs):
            a = np.ascontiguousarray(a)
            self.h_in[off:off + a.nbytes].numpy()[:] = a.reshape(-1).view(np.uint8)
            tdt = {np.float16: torch.float16, np.int32: torch.int32, np.int64: torch.int64}[a.dtype.type]
            self.d[name] = self.d_in[off:off + a.nbytes].view(tdt).view(a.shape)
        self.d_in.copy_(self.h_in)
        self.max_seq_len = int(case.seq_lens.max()) if case.B else 0
        B, T, Hq = case.B, s.num_q_tokens, s.num_q_heads
        rows = B * T * Hq
        (o_out, o_lse), total = packed_layout([rows * s.head_dim * 2, rows * 4])
        self.d_out = torch.empty(total, dtype=torch.uint8, device=dev)
        self.h_out = torch.empty(total, dtype=torch.uint8).pin_memory()
        self.out = self.d_out[o_out:o_out + rows * s.head_dim * 2].view(torch.float16).view(B * T, Hq, s.head_dim)
        self.lse = self.d_out[o_lse:o_lse + rows * 4].view(torch.float32).view(B * T, Hq)
        ws = pf.pfkv_attention_workspace_bytes(B, T, Hq, s.num_kv_heads, s.head_dim, s.page_size, s.kv_dtype,
                                               self.max_seq_len, s.causal, s.window, 0)
        self.ws = torch.empty(max(ws, 256), dtype=torch.uint8, device=dev)
        self.ws_bytes = ws
        if ws:
            self.ws[ws - 16:ws].fill_(0xFF)  # the range counter reads -1 until a persistent grid runs
        self.splits, self.split_tokens = pf.pfkv_attention_plan(B, T, Hq, s.num_kv_heads, s.head_dim, s.page_size,
                                                                s.kv_dtype, self.max_seq_len, s.causal, s.window, 0)
        self.has_append = case.slot_new.size > 0
        merge = self.splits > 1 and ws > 0
        self.launches_per_step = (1 if self.has_append else 0) + 1 + (1 if merge else 0)

    def kernel(self):
        """The attention kernel the calls ran. The persistent decode grid (large ragged batches)
        is the one that writes the workspace's range counter (its last 16 bytes, -1 until then)."""
        base = kernel_of(self.case.spec)
        if base != "decode_kernel" or not self.ws_bytes:
            return base
        ctr = int(self.ws[self.ws_bytes - 16:self.ws_bytes - 12].view(self.torch.int32).item())
        return "decode_persist_kernel" if ctr >= 0 else base

    def append_step(self):
        s = self.case.spec
        if self.has_append:
            self.pf.pfkv_kv_cache_append(self.d["kn"], self.d["vn"], self.k_cache, self.v_cache, self.d["slot"],
                                         s.page_size, s.kv_dtype, self.k_scale, self.v_scale)

    def decode_step(self):
        s = self.case.spec
        self.pf.pfkv_paged_attention(self.out, self.lse, self.d["q"], self.k_cache, self.v_cache, self.d["bt"],
                                     self.d["sl"], s.num_q_tokens, s.num_kv_heads, s.page_size, s.kv_dtype,
                                     self.k_scale, self.v_scale, float(self.case.softmax_scale), self.max_seq_len,
                                     s.causal, s.window, 0, self.ws)

    def h2d(self):
        self.d_in.copy_(self.h_in, non_blocking=True)

    def d2h(self):
        self.h_out.copy_(self.d_out, non_blocking=True)

    def io_bytes(self):
        return self.h_in.numel(), self.h_out.numel()


def time_steps(dw, torch, K, W, flush, e2e=False):
    """Device time (ms) of K steps, L2 flushed before each; and decode-call times. A step with an
    append records a middle event before the decode call; without one the step is the decode call
    and no extra event sits inside it."""
    mid = dw.has_append and not e2e

    def step(ev=None):
        if e2e:
            dw.h2d()
        dw.append_step()
        if ev is not None:
            ev.record()
        dw.decode_step()
        if e2e:
            dw.d2h()

    for _ in range(W):
        flush()
        step()
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    mids = [torch.cuda.Event(enable_timing=True) for _ in range(K)] if mid else starts
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    for i in range(K):
        flush()
        starts[i].record()
        step(mids[i] if mid else None)
        ends[i].record()
    torch.cuda.synchronize()
    total = sum(s.elapsed_time(e) for s, e in zip(starts, ends))
    dec = [m.elapsed_time(e) for m, e in zip(mids, ends)] if not e2e else []
    return total, dec


def dtype_label(spec) -> str:
    kv = {"fp16": "fp16", "e4m3": "fp8-e4m3", "e5m2": "fp8-e5m2"}[spec.kv_dtype]
    if kernel_of(spec) == "verify_kernel":
        return f"tcgen05: {kv} K x e4m3 Q terms (S), f16 V x f16 P (O), f32 accumulate"
    return f"f16 mma / f32 accumulate over {kv} KV"


def is_prefill(spec) -> bool:
    return spec.num_q_tokens > 16


def roofline_obj(case, wid, dec_ms, peak, peak_kind, kernel):
    """The decode call (decode/verify kernel + merge) against the HBM copy peak; a prefill chunk
    (dense: thousands of query rows per key) against the measured bf16 tensor peak."""
    dec_avg = sum(dec_ms) / len(dec_ms)
    if is_prefill(case.spec):
        tpeak, tkind = measured_tensor_peak()
        fl = useful_flops(case)
        ach = fl / (dec_avg * 1e-3) / 1e12
        return {"bound": "tensor", "kernel": f"{kernel} + lse_merge_kernel (one attention call)",
                "achieved": round(ach, 2), "peak": tpeak, "unit": "TFLOP/s", "frac": round(ach / tpeak, 4),
                "peak_source": f"{tkind} (MEASURED_PEAKS.json bf16_tflops, burst): the PV product runs on f16; "
                               "QK^T runs on FP8 with Q as three E4M3 terms (1.5x the bf16-equivalent MMA work)",
                "traffic": profiled_traffic(wid, kernel), "useful_flops_per_launch": fl,
                "avg_launch_ms": round(dec_avg, 5),
                "median_launch_frac": round(fl / (statistics.median(dec_ms) * 1e-3) / 1e12 / tpeak, 4)}
    dec_bytes = algorithmic_bytes(case, with_append=False)
    achieved = dec_bytes / (dec_avg * 1e-3) / 1e9
    return {"bound": "hbm", "kernel": f"{kernel} + lse_merge_kernel (one decode call)",
            "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
            "peak_source": "measured (MEASURED_PEAKS.json hbm_gbs, burst copy)" if peak_kind == "measured"
            else "fallback 6.8 TB/s",
            "traffic": profiled_traffic(wid, kernel), "algorithmic_bytes_per_launch": dec_bytes,
            "avg_launch_ms": round(dec_avg, 5),
            "median_launch_frac": round(dec_bytes / (statistics.median(dec_ms) * 1e-3) / 1e9 / peak, 4)}


def measure_workload(torch, pf, flush, case, wid, peak, peak_kind, steps, warmup, clocks=None):
    """Device-resident steps, then end-to-end steps, of one workload: the objects of its line."""
    dw = DeviceWorkload(case, torch, pf)
    nbytes = algorithmic_bytes(case, dw.has_append)
    pf.pfkv_device_errors(clear=True)
    torch.cuda.synchronize()
    if clocks is not None:
        clocks.start()
    total_ms, dec_ms = time_steps(dw, torch, steps, warmup, flush)
    clk = clocks.stop() if clocks is not None else None
    torch.cuda.synchronize()
    e2e_ms, _ = time_steps(dw, torch, steps, warmup, flush, e2e=True)
    if pf.pfkv_device_errors(clear=True):
        raise RuntimeError(f"device error word set while timing workload {wid}")
    bi, bo = dw.io_bytes()
    res = {"total_ms": total_ms, "e2e_ms": e2e_ms, "nbytes": nbytes, "dec_ms": dec_ms,
           "splits": dw.splits, "split_tokens": dw.split_tokens,
           # the persistent decode grid adds the kernel that zeroes its range counter
           "launches": dw.launches_per_step + (1 if dw.kernel() == "decode_persist_kernel" else 0),
           "io": (bi, bo), "clocks": clk,
           "roofline": roofline_obj(case, wid, dec_ms, peak, peak_kind, dw.kernel())}
    del dw
    torch.cuda.empty_cache()
    return res


def run_gpu(args):
    import torch
    import torch.distributed as dist

    from paged_fp8_kv_cache_gb300 import binding as pf
    from paged_fp8_kv_cache_gb300 import build

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    build.build()
    pf.load()

    wid = args.workload
    spec = workloads.ALL[wid]
    case = workloads.make_case(spec, seed=rank_seed(spec, rank))
    # the oracle on a sample of the same workload (spawned worker processes)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = oracle_baseline(case, args.cpu_budget)
    flush = L2Flush(torch)
    peak, peak_kind = measured_peaks()

    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    r = measure_workload(torch, pf, flush, case, wid, peak, peak_kind, args.steps, args.warmup,
                         clocks=ClockSampler(local))
    total_ms, e2e_ms = max_over_ranks([r["total_ms"], r["e2e_ms"]], dist, "cuda")
    if world > 1:
        dist.barrier()
    value = aggregate_gbs(r["nbytes"], world, args.steps, total_ms)
    e2e_val = aggregate_gbs(r["nbytes"], world, args.steps, e2e_ms)
    del case

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    bi, bo = r["io"]
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(total_ms / args.steps, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": dtype_label(spec),
        "data": "synthetic (seeded generator, " + spec.name + ")",
        "config": {"workload": spec.name, "workload_id": wid,
                   "l2": "flushed before every step (256 MiB write, then 256 MiB read: cold and clean)",
                   "algorithmic_bytes_per_step": r["nbytes"], "num_splits": r["splits"],
                   "split_tokens": r["split_tokens"],
                   "parallelism": f"replicas x{world} (independent batches, no collective on the data path)"},
        "calls_per_s": round(args.steps / (total_ms * 1e-3), 1),
        "frac_of_peak": round(value / peak, 4),
        "roofline": r["roofline"],
        "e2e": {"value": round(e2e_val, 2), "unit": "GB/s", "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
                "ms_per_step": round(e2e_ms / args.steps, 5), "copies_per_step": {"h2d": 1, "d2h": 1}},
        "gpu_launches": r["launches"] * args.steps,
        "clocks": r["clocks"],
        "cpu_baseline": cpu,
    }
    if world == 1 and not args.no_per_config:
        k = max(5, min(args.steps, 50))
        line["per_config"] = per_config(torch, pf, flush, wid, peak, peak_kind, args, workloads.CONFIGS, k)
        line["extensions"] = per_config(torch, pf, flush, wid, peak, peak_kind, args, workloads.EXTENSIONS, k)
        line["extensions"]["zero_blocks"] = zero_blocks_measure(torch, pf, flush, peak, args)
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def per_config(torch, pf, flush, skip, peak, peak_kind, args, configs, k):
    """Every other workload with the headline's objects: step rate, roofline of the decode call,
    e2e and the oracle on a sample."""
    res = {}
    for cid, spec in configs.items():
        if cid == skip or cid in args.skip_configs:
            continue
        case = workloads.make_case(spec)
        r = measure_workload(torch, pf, flush, case, cid, peak, peak_kind, k, 3)
        cpu = None if args.no_cpu_baseline else oracle_baseline(case, args.cpu_budget_per_config)
        bi, bo = r["io"]
        gbs = r["nbytes"] * k / (r["total_ms"] * 1e-3) / 1e9
        res[str(cid)] = {
            "workload": spec.name, "value": round(gbs, 2), "unit": "GB/s",
            "ms_per_step": round(r["total_ms"] / k, 5), "steps": k, "warmup": 3,
            "calls_per_s": round(k / (r["total_ms"] * 1e-3), 1),
            "frac_of_peak": round(gbs / peak, 4), "dtype": dtype_label(spec),
            "algorithmic_bytes_per_step": r["nbytes"], "num_splits": r["splits"], "split_tokens": r["split_tokens"],
            "roofline": r["roofline"],
            "e2e": {"value": round(r["nbytes"] * k / (r["e2e_ms"] * 1e-3) / 1e9, 2), "unit": "GB/s",
                    "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo, "ms_per_step": round(r["e2e_ms"] / k, 5)},
            "gpu_launches": r["launches"] * k,
            "cpu_baseline": cpu,
        }
        if is_prefill(spec):
            fl = useful_flops(case)
            res[str(cid)]["tflops"] = {"value": round(fl * k / (r["total_ms"] * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
                                       "useful_flops_per_step": fl,
                                       "note": "useful causal QK^T + PV flops of the step (append included in the time)"}
        del case
    return res


def zero_blocks_measure(torch, pf, flush, peak, args):
    """Zeroing of reused blocks: 64 of the 128 blocks of a pool shaped like the 128K decode's
    (Hkv 4, 2048-token pages, D 256, E4M3), both pools: 256 MiB written per call, timed like a
    step (L2 flushed before each call). The oracle zeroes 8 blocks of the same shape on the host
    beside it."""
    from oracle import append as oappend
    nb_pool, n, hkv, page, d = 128, 64, 4, 2048, 256
    k = torch.empty((nb_pool, hkv, page, d), dtype=torch.uint8, device="cuda")
    v = torch.empty_like(k)
    ids = torch.from_numpy(np.random.default_rng(7).permutation(nb_pool)[:n].astype(np.int32)).cuda()
    nbytes = 2 * n * hkv * page * d
    for _ in range(3):
        flush()
        pf.pfkv_kv_cache_zero_blocks(k, v, ids, "e4m3")
    steps = max(5, min(args.steps, 50))
    evs = []
    for _ in range(steps):
        flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        pf.pfkv_kv_cache_zero_blocks(k, v, ids, "e4m3")
        b.record()
        evs.append((a, b))
    torch.cuda.synchronize()
    ms = sum(a.elapsed_time(b) for a, b in evs) / steps
    assert pf.pfkv_device_errors(clear=True) == 0
    # the oracle beside it, on a host pool of the same block shape
    hk = np.ones((16, hkv, page, d), np.uint8)
    hv = np.ones_like(hk)
    t0 = time.perf_counter()
    oappend.zero_blocks(hk, hv, np.arange(0, 16, 2, dtype=np.int32))
    cpu_s = time.perf_counter() - t0
    cpu_bytes = 2 * 8 * hkv * page * d
    gbs = nbytes / (ms * 1e-3) / 1e9
    del k, v
    torch.cuda.empty_cache()
    return {"workload": "zero 64 reused blocks (Hkv4, page 2048, D256, E4M3), K and V pools: 256 MiB written",
            "value": round(gbs, 1), "unit": "GB/s", "ms_per_call": round(ms, 5), "frac_of_peak": round(gbs / peak, 4),
            "roofline": {"bound": "hbm (writes)", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(gbs / peak, 4), "traffic": None, "avg_launch_ms": round(ms, 5)},
            "steps": steps,
            "cpu_baseline": {"value": round(cpu_bytes / cpu_s / 1e9, 2), "unit": "GB/s", "cores": 1,
                             "kind": "oracle", "sample": "8 blocks of the same shape zeroed on the host"}}


# ----------------------------------------------------------------------------- oracle arm
#
# The oracle is timed on pieces of the workload: a piece is one (sequence, KV head) unit
# restricted to a range of at most PIECE_KEYS keys that ends at the sequence's last key (so a
# verify's causal rows are in it). Every worker process quantises the keys of its own piece
# into a host cache of just those pages (set-up, not timed), then evaluates
# oracle.attention.paged_attention on it, restricted to the piece's key range, as often as the
# budget allows. The pieces are written by the parent (the fp16 inputs of the range), so no
# worker builds the whole (up to 1 GB) workload.

PIECE_KEYS = 8192
PIECE_TOKENS = 16  # query tokens of a prefill chunk a piece evaluates
_OW = None


def _piece_arrays(case, b, kvh):
    """One unit's piece: fp16 K/V rows of its last <= PIECE_KEYS visible keys (page-aligned start),
    its Q rows, scales and mask; for a prefill chunk a spread of PIECE_TOKENS of its query tokens."""
    s = case.spec
    P, T, D = s.page_size, s.num_q_tokens, s.head_dim
    g = s.num_q_heads // s.num_kv_heads
    n = int(case.seq_lens[b])
    lo_vis, _ = visible_span(s, n)
    lo = max(0, n - PIECE_KEYS, lo_vis) // P * P
    pos = np.arange(lo, n)
    cached = int(case.cached[b])
    start = int(np.concatenate([[0], np.cumsum(case.cached.astype(np.int64))])[b])
    fill = pos < cached
    k16 = np.empty((n - lo, D), np.float16)
    v16 = np.empty((n - lo, D), np.float16)
    k16[fill] = case.k_fill[start + pos[fill], kvh]
    v16[fill] = case.v_fill[start + pos[fill], kvh]
    if (~fill).any():
        idx = b * s.append_new + (pos[~fill] - cached)
        k16[~fill] = case.k_new[idx, kvh]
        v16[~fill] = case.v_new[idx, kvh]
    ks = np.asarray(case.k_scale, np.float32).reshape(-1)
    vs = np.asarray(case.v_scale, np.float32).reshape(-1)
    tokens = np.unique(np.linspace(0, T - 1, PIECE_TOKENS).astype(np.int64)) if is_prefill(s) else np.arange(T)
    # useful flops of the piece: 4 * D per (row, visible key in [lo, n))
    p_t = n - T + tokens
    hi_t = np.minimum(p_t, n - 1) if s.causal else np.full(tokens.size, n - 1)
    lo_t = np.maximum(lo, np.maximum(0, p_t - s.window + 1) if s.window > 0 else 0)
    flops = 4 * D * g * int(np.maximum(0, hi_t - lo_t + 1).sum())
    return {"q": case.q[b * T:(b + 1) * T, kvh * g:(kvh + 1) * g, :], "k16": k16, "v16": v16,
            "ks": ks[kvh % ks.size], "vs": vs[kvh % vs.size], "sm": np.float32(case.softmax_scale),
            "lo": lo, "n": n, "T": T, "P": P, "kv": np.array(s.kv_dtype), "causal": s.causal, "window": s.window,
            "tokens": tokens, "all_tokens": not is_prefill(s), "keys": n - max(lo, lo_vis), "flops": flops}


def _oracle_init(tmpdir, npieces, counter, ready):
    global _OW
    from oracle import append as oappend
    with counter.get_lock():
        i = counter.value
        counter.value += 1
    d = dict(np.load(os.path.join(tmpdir, f"piece{i % npieces}.npz")))
    kv = str(d["kv"])
    lo, n, P, D = int(d["lo"]), int(d["n"]), int(d["P"]), d["k16"].shape[1]
    npages = -(-(n - lo) // P)
    dt = np.float16 if kv == "fp16" else np.uint8
    kc = np.zeros((npages, 1, P, D), dt)
    vc = np.zeros((npages, 1, P, D), dt)
    if kv == "fp16":
        kc.reshape(-1, D)[:n - lo] = d["k16"]
        vc.reshape(-1, D)[:n - lo] = d["v16"]
    else:
        kc.reshape(-1, D)[:n - lo] = oappend.quantise(d["k16"], d["ks"], kv)
        vc.reshape(-1, D)[:n - lo] = oappend.quantise(d["v16"], d["vs"], kv)
    bt = np.full((1, (n - 1) // P + 1 if n > 0 else 1), -1, np.int32)
    bt[0, lo // P:lo // P + npages] = np.arange(npages, dtype=np.int32)
    _OW = {"q": d["q"], "kc": kc, "vc": vc, "bt": bt, "sl": np.array([n], np.int32), "T": int(d["T"]), "P": P,
           "kv": kv, "ks": float(d["ks"]), "vs": float(d["vs"]), "sm": float(d["sm"]), "lo": lo, "n": n,
           "causal": bool(d["causal"]), "window": int(d["window"]),
           "tokens": None if bool(d["all_tokens"]) else [int(t) for t in d["tokens"]],
           "keys": int(d["keys"]), "flops": int(d["flops"])}
    with ready.get_lock():
        ready.value += 1


def _oracle_task(_):
    from oracle import attention as oatt
    w = _OW
    oatt.paged_attention(w["q"], w["kc"], w["vc"], w["bt"], w["sl"], w["T"], 1, w["P"], w["kv"], w["ks"], w["vs"],
                         w["sm"], units=[(0, 0)], token_range=(w["lo"], w["n"]), causal=w["causal"],
                         window=w["window"], tokens=w["tokens"])
    return w["keys"], w["flops"]


class OracleSampler:
    """The CPU oracle on a spawned process pool (one single-threaded worker per core, at most 16),
    timed on pieces of a workload (see above)."""

    def __init__(self, case):
        import multiprocessing as mp
        for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
            os.environ[var] = "1"
        s = case.spec
        self.case = case
        self.cores = max(1, min(16, len(os.sched_getaffinity(0))))
        units = [(b, h) for b in range(case.B) for h in range(s.num_kv_heads) if case.seq_lens[b] > 0]
        rng = np.random.default_rng(0)
        pick = [units[i] for i in rng.permutation(len(units))[:self.cores]]
        self.tmpdir = tempfile.mkdtemp(prefix="pfkv_oracle_")
        self.piece_keys = []
        for i, (b, h) in enumerate(pick):
            arr = _piece_arrays(case, b, h)
            self.piece_keys.append(int(arr["keys"]))
            np.savez(os.path.join(self.tmpdir, f"piece{i}.npz"), **arr)
        self.npieces = len(pick)
        ctx = mp.get_context("spawn")
        counter, ready = ctx.Value("i", 0), ctx.Value("i", 0)
        self.pool = ctx.Pool(self.cores, initializer=_oracle_init,
                             initargs=(self.tmpdir, self.npieces, counter, ready))
        t0 = time.time()
        while ready.value < self.cores:
            if time.time() - t0 > 180:
                self.close()
                raise RuntimeError("oracle worker processes did not start")
            time.sleep(0.05)
        elt = 2 if s.kv_dtype == "fp16" else 1
        self.key_bytes = s.head_dim * elt * 2  # K + V bytes of one key of one unit
        step_bytes = algorithmic_bytes(case, case.slot_new.size > 0)
        kv_visible = algorithmic_bytes(case, False) - case.B * s.num_q_tokens * s.num_q_heads * (s.head_dim * 4 + 4)
        self.overhead = step_bytes / max(1, kv_visible)  # algorithmic bytes per visible KV byte of a step

    def run(self, budget_s):
        """Evaluate pieces for about budget_s; effective GB/s (and TFLOP/s) of the oracle."""
        keys, flops, t_total, evals = 0, 0, 0.0, 0
        while t_total < budget_s:
            t0 = time.perf_counter()
            res = self.pool.map(_oracle_task, range(self.cores), chunksize=1)
            t_total += time.perf_counter() - t0
            keys += sum(r[0] for r in res)
            flops += sum(r[1] for r in res)
            evals += self.cores
        nbytes = keys * self.key_bytes * self.overhead
        s = self.case.spec
        rows = f"{PIECE_TOKENS} of its {s.num_q_tokens} query tokens, " if is_prefill(s) else ""
        out = {"value": round(nbytes / t_total / 1e9, 4), "unit": "GB/s", "cores": self.cores, "kind": "oracle",
               "sample": f"{evals} evaluations of {self.npieces} pieces of '{s.name}': one (sequence, KV head) "
                         f"unit each, {rows}restricted to its last <= {PIECE_KEYS} visible keys "
                         f"({min(self.piece_keys)}-{max(self.piece_keys)} keys), on {self.cores} single-threaded "
                         f"processes, {t_total:.2f} s wall; bytes scaled by the step's algorithmic/KV byte ratio "
                         f"({self.overhead:.4f})",
               "seconds": round(t_total, 3)}
        if is_prefill(s):
            out["tflops"] = round(flops / t_total / 1e12, 6)
        return out

    def close(self):
        self.pool.close()
        self.pool.join()
        shutil.rmtree(self.tmpdir, ignore_errors=True)


def oracle_baseline(case, budget_s=15.0):
    op = OracleSampler(case)
    try:
        return op.run(budget_s)
    finally:
        op.close()


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    spec = workloads.ALL[args.workload]
    case = workloads.make_case(spec)
    vals = []
    info = None
    per = max(1.0, min(20.0, 120.0 / max(1, args.steps + args.warmup)))
    op = OracleSampler(case)
    try:
        for i in range(args.warmup + args.steps):
            r = op.run(per)
            if i >= args.warmup:
                vals.append(r["value"])
                info = r
    finally:
        op.close()
    v = statistics.median(vals) if vals else 0.0
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "GB/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64 (numpy oracle)", "data": "synthetic (seeded generator, " + spec.name + ")",
            "config": {"workload": spec.name, "workload_id": args.workload,
                       "l2": "n/a (host memory)", "algorithmic_bytes_per_step": algorithmic_bytes(case, case.slot_new.size > 0),
                       "parallelism": "one single-threaded oracle process per host core"},
            "cpu_baseline": {"value": v, "unit": "GB/s", "cores": info["cores"] if info else None, "kind": "oracle",
                             "sample": info["sample"] if info else ""},
            "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", type=int, default=DEFAULT_WORKLOAD, choices=sorted(workloads.ALL))
    ap.add_argument("--impl", default="pfkv", choices=["pfkv", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true")
    ap.add_argument("--skip-configs", type=int, nargs="*", default=[])
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--cpu-budget-per-config", type=float, default=5.0)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
