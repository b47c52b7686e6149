"""Benchmark: paged FP8-KV decode attention, effective HBM GB/s on GB300.

One step = one pass of the hot path over one batch of the workload: the
append of the step's new tokens into the paged cache (when the workload has
any), the split-KV decode kernel and the LSE merge, all through the C ABI
(paged_fp8_kv_cache_gb300.binding -> libpfkv.so).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload ID] [--impl reference]

Prints ONE JSON line (rank 0). ``value`` = algorithmic bytes of all ranks /
max-over-ranks device time of the K timed steps (inputs resident in HBM, L2
flushed between steps: a 256 MiB write, then a 256 MiB read, so that the
step starts on a cold L2 holding no dirty lines, whose write-back would
otherwise compete with the step's own HBM traffic). ``e2e`` repeats the measurement through the same
public calls with the step's inputs copied from pinned host memory and the
outputs copied back inside the timed region. ``--impl reference`` times the
CPU oracle (the only reference arm this project has) on a bounded sample.

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
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from paged_fp8_kv_cache_gb300 import workloads  # noqa: E402

METRIC = "paged FP8-KV decode attention: effective HBM GB/s and % of GB300 peak"
DEFAULT_WORKLOAD = 2  # the batched-decode workload (the second of the five)
L2_FLUSH_BYTES = 256 << 20  # > 2x the 129 MB L2
FALLBACK_HBM_GBS = 6800.0
KERNEL_SOURCES = ["decode_kernel.cuh", "device_utils.cuh", "frag_layout.h"]  # the decode kernel


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

def algorithmic_bytes(case, with_append: bool) -> int:
    s = case.spec
    elt = 2 if s.kv_dtype == "fp16" else 1
    sl = case.seq_lens.astype(np.int64)
    kv = int(sl.sum()) * s.num_kv_heads * s.head_dim * elt * 2
    rows = case.B * s.num_q_tokens * s.num_q_heads
    q_out = rows * s.head_dim * 2 * 2
    lse = rows * 4
    pages = int((-(-sl // s.page_size)).sum()) * 4
    meta = case.B * 4
    total = kv + q_out + lse + pages + meta
    if with_append and case.slot_new.size:
        n = case.slot_new.size
        total += n * s.num_kv_heads * s.head_dim * (2 * 2 + elt * 2) + n * 8
    return total


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
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


def profiled_traffic(workload_id: int):
    """DRAM bytes per launch of the decode kernel from the committed ncu summary,
    if it was taken on the current kernel sources; else None."""
    path = os.path.join(ROOT, "profiles", f"decode_kernel_workload{workload_id}.txt")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m_hash = re.search(r"kernel_source_hash:\s*([0-9a-f]+)", text)
    m_t = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not (m_hash and m_t) or m_hash.group(1) != kernel_source_hash():
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


# ----------------------------------------------------------------------------- GPU arm

class DeviceWorkload:
    """A workload resident on the GPU: caches populated through the append kernel."""

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
        # per-step inputs: host (pinned) and device copies
        self.h = {
            "q": torch.from_numpy(case.q).pin_memory(),
            "bt": torch.from_numpy(case.block_table).pin_memory(),
            "sl": torch.from_numpy(case.seq_lens).pin_memory(),
            "kn": torch.from_numpy(case.k_new).pin_memory(),
            "vn": torch.from_numpy(case.v_new).pin_memory(),
            "slot": torch.from_numpy(case.slot_new).pin_memory(),
        }
        self.d = {k: v.to(dev) for k, v in self.h.items()}
        self.max_seq_len = int(case.seq_lens.max()) if case.B else 0
        B, T, Hq = case.B, s.num_q_tokens, s.num_q_heads
        self.out = torch.empty((B * T, Hq, s.head_dim), dtype=torch.float16, device=dev)
        self.lse = torch.empty((B * T, Hq), dtype=torch.float32, device=dev)
        self.h_out = torch.empty(self.out.shape, dtype=torch.float16).pin_memory()
        self.h_lse = torch.empty(self.lse.shape, dtype=torch.float32).pin_memory()
        ws = pf.pfkv_decode_workspace_bytes(B, T, Hq, s.num_kv_heads, s.head_dim, s.page_size, s.kv_dtype,
                                            self.max_seq_len, 0)
        self.ws = torch.empty(max(ws, 256), dtype=torch.uint8, device=dev)
        self.splits, self.split_tokens = pf.pfkv_decode_plan(B, T, Hq, s.num_kv_heads, s.head_dim, s.page_size,
                                                             s.kv_dtype, self.max_seq_len, 0)
        self.has_append = case.slot_new.size > 0
        # a split plan launches the merge kernel unless its ranges combine inside thread-block
        # clusters, in which case the library asks for no workspace
        merge = self.splits > 1 and ws > 0
        self.launches_per_step = (1 if self.has_append else 0) + 1 + (1 if merge else 0)

    def append_step(self):
        s = self.case.spec
        if self.has_append:
            self.pf.pfkv_kv_cache_append(self.d["kn"], self.d["vn"], self.k_cache, self.v_cache, self.d["slot"],
                                         s.page_size, s.kv_dtype, self.k_scale, self.v_scale)

    def decode_step(self):
        s = self.case.spec
        self.pf.pfkv_paged_attention_decode(self.out, self.lse, self.d["q"], self.k_cache, self.v_cache,
                                            self.d["bt"], self.d["sl"], s.num_q_tokens, s.num_kv_heads, s.page_size,
                                            s.kv_dtype, self.k_scale, self.v_scale,
                                            float(self.case.softmax_scale), self.max_seq_len, 0, self.ws)

    def h2d(self):
        for k in self.d:
            self.d[k].copy_(self.h[k], non_blocking=True)

    def d2h(self):
        self.h_out.copy_(self.out, non_blocking=True)
        self.h_lse.copy_(self.lse, non_blocking=True)

    def io_bytes(self):
        bi = sum(t.numel() * t.element_size() for t in self.h.values())
        bo = self.h_out.numel() * 2 + self.h_lse.numel() * 4
        return bi, bo


def time_steps(dw, torch, K, W, flush, e2e=False):
    """Device time (ms) of K steps, L2 flushed before each; and decode-call times."""
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
    mids = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    for i in range(K):
        flush()
        starts[i].record()
        step(mids[i])
        ends[i].record()
    torch.cuda.synchronize()
    total = sum(s.elapsed_time(e) for s, e in zip(starts, ends))
    dec = [m.elapsed_time(e) for m, e in zip(mids, ends)] if not e2e else []
    return total, dec


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

    # cpu_baseline before the first GPU work (its process pool is spawned)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = oracle_sample(args.workload, budget_s=args.cpu_budget)

    wid = args.workload
    spec = workloads.ALL[wid]
    case = workloads.make_case(spec, seed=rank_seed(spec, rank))
    dw = DeviceWorkload(case, torch, pf)
    flush = L2Flush(torch)
    nbytes = algorithmic_bytes(case, dw.has_append)
    pf.pfkv_device_errors(clear=True)

    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    sampler = ClockSampler(local)
    sampler.start()
    total_ms, dec_ms = time_steps(dw, torch, args.steps, args.warmup, flush)
    clocks = sampler.stop()
    torch.cuda.synchronize()
    e2e_ms, _ = time_steps(dw, torch, args.steps, args.warmup, flush, e2e=True)
    if pf.pfkv_device_errors(clear=True):
        raise RuntimeError("device error word set during the benchmark")

    total_ms, e2e_ms = max_over_ranks([total_ms, e2e_ms], dist, "cuda")
    if world > 1:
        dist.barrier()
    value = aggregate_gbs(nbytes, world, args.steps, total_ms)
    e2e_val = aggregate_gbs(nbytes, world, args.steps, e2e_ms)

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    peak, peak_kind = measured_peaks()
    dec_avg_ms = sum(dec_ms) / len(dec_ms)
    dec_bytes = algorithmic_bytes(case, with_append=False)
    achieved = dec_bytes / (dec_avg_ms * 1e-3) / 1e9
    bi, bo = dw.io_bytes()
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
        "dtype": "f16 mma / f32 accumulate over " + {"fp16": "fp16", "e4m3": "fp8-e4m3", "e5m2": "fp8-e5m2"}[spec.kv_dtype] + " KV",
        "data": "synthetic (seeded generator, " + spec.name + ")",
        "config": {"workload": spec.name, "workload_id": wid, "l2": "flushed before every step (256 MiB write, then 256 MiB read: cold and clean)",
                   "algorithmic_bytes_per_step": nbytes, "num_splits": dw.splits, "split_tokens": dw.split_tokens,
                   "parallelism": f"replicas x{world} (independent batches, no collective on the data path)"},
        "calls_per_s": round(args.steps / (total_ms * 1e-3), 1),
        "roofline": {"bound": "hbm", "kernel": "decode_kernel + lse_merge_kernel (one decode call)",
                     "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)"
                     if peak_kind == "measured" else "fallback 6.8 TB/s",
                     "traffic": profiled_traffic(wid), "algorithmic_bytes_per_launch": dec_bytes,
                     "avg_launch_ms": round(dec_avg_ms, 5)},
        "e2e": {"value": round(e2e_val, 2), "unit": "GB/s", "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
                "ms_per_step": round(e2e_ms / args.steps, 5)},
        "gpu_launches": dw.launches_per_step * args.steps,
        "clocks": clocks,
        "cpu_baseline": cpu,
    }
    del dw
    torch.cuda.empty_cache()
    if world == 1 and not args.no_per_config:
        line["per_config"] = per_config(torch, pf, flush, wid, peak, args, workloads.CONFIGS)
        line["extensions"] = per_config(torch, pf, flush, wid, peak, args, workloads.EXTENSIONS)
        line["extensions"]["zero_blocks"] = zero_blocks_measure(torch, pf, flush, peak, args)
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def per_config(torch, pf, flush, skip, peak, args, configs):
    res = {}
    for cid, spec in configs.items():
        if cid == skip or cid in args.skip_configs:
            continue
        case = workloads.make_case(spec)
        dw = DeviceWorkload(case, torch, pf)
        k = max(5, min(args.steps, 50))
        total_ms, dec = time_steps(dw, torch, k, 3, flush)
        nb = algorithmic_bytes(case, dw.has_append)
        db = algorithmic_bytes(case, False)
        dec_avg = sum(dec) / len(dec)
        res[str(cid)] = {"workload": spec.name, "GB/s": round(nb * k / (total_ms * 1e-3) / 1e9, 1),
                         "ms_per_step": round(total_ms / k, 5), "decode_call_GB/s": round(db / (dec_avg * 1e-3) / 1e9, 1),
                         "frac_of_peak": round(db / (dec_avg * 1e-3) / 1e9 / peak, 4),
                         # the same from the median call (robust to a slow outlier call)
                         "decode_call_GB/s_median": round(db / (statistics.median(dec) * 1e-3) / 1e9, 1),
                         "num_splits": dw.splits, "steps": k}
        del dw, case
        torch.cuda.empty_cache()
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
            "GB/s": round(gbs, 1), "ms_per_call": round(ms, 5), "frac_of_peak": round(gbs / peak, 4),
            "bound": "hbm (writes)", "steps": steps,
            "cpu_baseline": {"value": round(cpu_bytes / cpu_s / 1e9, 2), "unit": "GB/s", "cores": 1,
                             "kind": "oracle", "sample": "8 blocks of the same shape zeroed on the host"}}


# ----------------------------------------------------------------------------- oracle arm

def _oracle_worker_init(wid, seed):
    global _OW
    import numpy as _np  # noqa: F401
    from oracle import append as oappend
    case = workloads.make_case(workloads.ALL[wid], seed=seed)
    s = case.spec
    dt = np.float16 if s.kv_dtype == "fp16" else np.uint8
    shape = (case.num_blocks, s.num_kv_heads, s.page_size, s.head_dim)
    kc, vc = np.zeros(shape, dt), np.zeros(shape, dt)
    oappend.append_bulk(kc, case.k_fill, case.slot_fill, s.page_size, case.k_scale, s.kv_dtype)
    oappend.append_bulk(vc, case.v_fill, case.slot_fill, s.page_size, case.v_scale, s.kv_dtype)
    _OW = (case, kc, vc)


def _oracle_unit(u):
    from oracle import append as oappend
    from oracle import attention as oatt
    case, kc, vc = _OW
    s = case.spec
    b, kvh = u
    if case.slot_new.size:  # the step's append of this sequence's new token (this KV head's share)
        idx = [i for i in range(case.slot_new.size) if i // s.append_new == b]
        for i in idx:
            slot = int(case.slot_new[i])
            blk, off = divmod(slot, s.page_size)
            if s.kv_dtype == "fp16":
                kc[blk, kvh, off] = case.k_new[i, kvh]
                vc[blk, kvh, off] = case.v_new[i, kvh]
            else:
                ks = np.asarray(case.k_scale, np.float32).reshape(-1)
                vs = np.asarray(case.v_scale, np.float32).reshape(-1)
                kc[blk, kvh, off] = oappend.quantise(case.k_new[i, kvh], ks[kvh % ks.size], s.kv_dtype)
                vc[blk, kvh, off] = oappend.quantise(case.v_new[i, kvh], vs[kvh % vs.size], s.kv_dtype)
    oatt.paged_attention(case.q, kc, vc, case.block_table, case.seq_lens, s.num_q_tokens, s.num_kv_heads,
                         s.page_size, s.kv_dtype, case.k_scale, case.v_scale, case.softmax_scale, units=[u])
    elt = 2 if s.kv_dtype == "fp16" else 1
    return int(case.seq_lens[b]) * s.head_dim * elt * 2


class OraclePool:
    """The CPU oracle on a spawned process pool (one single-threaded worker per core)."""

    def __init__(self, wid, seed=None):
        import multiprocessing as mp
        for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
            os.environ[var] = "1"
        self.cores = len(os.sched_getaffinity(0))
        self.spec = workloads.ALL[wid]
        # every worker builds the whole seeded workload: on the 1 GB workloads a few workers keep
        # that set-up (and its host memory) bounded
        if workloads.kv_bytes_of(self.spec) > (256 << 20):
            self.cores = min(self.cores, 4)
        seed = self.spec.seed if seed is None else seed
        self.pool = mp.get_context("spawn").Pool(self.cores, initializer=_oracle_worker_init, initargs=(wid, seed))
        self.pool.map(abs, range(self.cores))  # wait until every worker holds its inputs
        self.case = workloads.make_case(self.spec, seed=seed)
        units = [(b, h) for b in range(self.case.B) for h in range(self.spec.num_kv_heads)]
        rng = np.random.default_rng(0)
        self.order = [units[i] for i in rng.permutation(len(units))]
        self.next = 0
        self.step_bytes = algorithmic_bytes(self.case, self.case.slot_new.size > 0)

    def run(self, budget_s):
        """Evaluate (sequence, KV head) units, cycling through the workload, for about budget_s."""
        kv_bytes, t_total, evals = 0, 0.0, 0
        n = self.cores
        while t_total < budget_s:
            batch = [self.order[(self.next + i) % len(self.order)] for i in range(n)]
            self.next = (self.next + n) % len(self.order)
            t0 = time.perf_counter()
            kv_bytes += sum(self.pool.map(_oracle_unit, batch, chunksize=1))
            t_total += time.perf_counter() - t0
            evals += n
            if t_total < budget_s / 8:
                n = min(n * 2, 64 * self.cores)
        frac = kv_bytes / max(1, self.case.kv_bytes())  # in units of whole steps
        return {"value": round(self.step_bytes * frac / t_total / 1e9, 4), "unit": "GB/s", "cores": self.cores,
                "kind": "oracle",
                "sample": f"{evals} (sequence, KV head) unit evaluations cycling over the {len(self.order)} units of "
                          f"'{self.spec.name}' (= {frac:.3g} steps of KV bytes) in {t_total:.2f} s wall on "
                          f"{self.cores} single-threaded processes",
                "seconds": round(t_total, 3)}

    def close(self):
        self.pool.close()
        self.pool.join()


def oracle_sample(wid, budget_s=15.0):
    op = OraclePool(wid)
    try:
        return op.run(budget_s)
    finally:
        op.close()


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    spec = workloads.ALL[args.workload]
    vals = []
    info = None
    per = max(1.0, min(20.0, 120.0 / max(1, args.steps + args.warmup)))
    op = OraclePool(args.workload)
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
            "vs_baseline": None, "dtype": "f64 (numpy oracle)", "data": "synthetic",
            "config": {"workload": spec.name, "workload_id": args.workload},
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
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
