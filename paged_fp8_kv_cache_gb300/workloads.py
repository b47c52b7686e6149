"""Seeded synthetic inputs for paged FP8-KV decode attention.

This module is the one piece the CUDA path's tests/bench and the CPU oracle
both consume. It draws random numbers and lays out the paged structure (which
token lives in which page); it holds none of the method's arithmetic: no FP8
encoding, no quantisation, no softmax. The per-tensor KV scale recipe
``amax(|x16|) / fmt_max`` is part of the input description of each workload
(static scales are inputs of the method: "1Cat-vLLM", section "Optional
experimental feature: FP8 KV cache"), so it is computed here.

Recipe (numpy ``Generator(PCG64(seed))``, fixed draw order: contexts, page
permutation, Q, K, V, outlier rows, new tokens). Values are drawn in float32
and rounded to fp16 (round-to-nearest-even).

* Each sequence b holds ``cached_b`` tokens in the cache and appends
  ``append_new`` more during the step, so it decodes over
  ``seq_len_b = cached_b + append_new`` keys. Its T query tokens are the last
  T positions of that range.
* Pages: ``pages_b = ceil(seq_len_b / P)``; the pool has
  ``ceil(pool_factor * sum_b pages_b)`` pages and the pages of all sequences
  are a seeded draw without replacement from it (a permutation when
  ``pool_factor == 1``). Unused block-table entries are -1.
* Outliers (``k_outlier_frac > 0``): exactly ``floor(frac * tokens * Hkv)``
  K rows (one (token, KV head) vector each) chosen without replacement are
  multiplied by ``k_outlier_mul`` in float32 before the fp16 rounding.
* Scales: ``k_scale = float32(amax|K16| / fmt_max)`` over every K value of
  the workload (cached and appended), fmt_max 448 (E4M3) or 57344 (E5M2);
  likewise ``v_scale``; 1.0 for an fp16 cache. ``softmax_scale =
  float32(1/sqrt(D))``. With ``scale_per_head`` the amax runs over each KV
  head's values alone and the scales are float32 arrays ``[Hkv]``.
* Head gains (``head_gain``, a tuple cycled over the KV heads): K and V of KV
  head h are multiplied by ``head_gain[h % len]`` in float32 before the fp16
  rounding (after the outliers), so that heads differ in magnitude.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import numpy as np

FMT_MAX = {"e4m3": 448.0, "e5m2": 57344.0}


@dataclass(frozen=True)
class CaseSpec:
    name: str
    contexts: tuple  # cached tokens per sequence, or ("loguniform", lo, hi, B)
    num_q_tokens: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    kv_dtype: str  # "fp16" | "e4m3" | "e5m2"
    k_dist: str = "normal"  # "normal"
    v_dist: str = "normal"  # "normal" | "uniform"
    k_outlier_frac: float = 0.0
    k_outlier_mul: float = 8.0
    pool_factor: float = 1.0
    append_new: int = 0
    seed: int = 0
    scale_per_head: bool = False
    head_gain: tuple = ()
    causal: bool = True  # the attention mask of the step's call (an input of the call, like T)
    window: int = 0      # sliding window of keys (0 = none)


# The five workloads of the benchmark (seed = 1000 + workload id).
CONFIGS = {
    1: CaseSpec("tiny decode: 1 seq x 1000, q1, Hq8/Hkv2, D128, fp16 KV, page 16",
                contexts=(1000,), num_q_tokens=1, num_q_heads=8, num_kv_heads=2,
                head_dim=128, page_size=16, kv_dtype="fp16", seed=1001),
    2: CaseSpec("batched decode: 4 seqs x 4096, q1, Hq32/Hkv8, D128, E4M3 KV, page 16",
                contexts=(4096,) * 4, num_q_tokens=1, num_q_heads=32, num_kv_heads=8,
                head_dim=128, page_size=16, kv_dtype="e4m3", seed=1002),
    3: CaseSpec("long-context decode: 1 seq x 131072, q1, Hq24/Hkv4, D256, E4M3 KV, page 2048",
                contexts=(131072,), num_q_tokens=1, num_q_heads=24, num_kv_heads=4,
                head_dim=256, page_size=2048, kv_dtype="e4m3", v_dist="uniform",
                k_outlier_frac=0.01, seed=1003),
    4: CaseSpec("speculative verify: 2 seqs x 262144, q8 causal, Hq24/Hkv4, D256, E5M2 KV, page 2048",
                contexts=(262144,) * 2, num_q_tokens=8, num_q_heads=24, num_kv_heads=4,
                head_dim=256, page_size=2048, kv_dtype="e5m2", seed=1004),
    5: CaseSpec("mixed serving batch: 64 seqs, log-uniform 1K-32K, q1, Hq32/Hkv8, D128, E4M3 KV, "
                "page 16 scattered pool, + append of 1 token per seq",
                contexts=("loguniform", 1024, 32768, 64), num_q_tokens=1, num_q_heads=32,
                num_kv_heads=8, head_dim=128, page_size=16, kv_dtype="e4m3",
                pool_factor=1.25, append_new=1, seed=1005),
}

# Workloads of rows built beyond the five, measured with the same harness and reported apart:
# a q16 verify (15 drafts + 1) at 256K keys, the q8 verifier's shape class with 16 query tokens
# per sequence and 4 query heads per KV head (64 rows per KV head); and the 128K decode with
# one static scale per KV head over heads of different magnitude.
EXTENSIONS = {
    6: CaseSpec("q16 speculative verify: 2 seqs x 262144, q16 causal, Hq16/Hkv4, D256, E5M2 KV, page 2048",
                contexts=(262144,) * 2, num_q_tokens=16, num_q_heads=16, num_kv_heads=4,
                head_dim=256, page_size=2048, kv_dtype="e5m2", seed=1006),
    7: CaseSpec("long-context decode with one scale per KV head: 1 seq x 131072, q1, Hq24/Hkv4, D256, E4M3 KV, "
                "page 2048, KV heads of magnitude x0.25/x1/x4/x0.5",
                contexts=(131072,), num_q_tokens=1, num_q_heads=24, num_kv_heads=4,
                head_dim=256, page_size=2048, kv_dtype="e4m3", v_dist="uniform",
                k_outlier_frac=0.01, seed=1007, scale_per_head=True, head_gain=(0.25, 1.0, 4.0, 0.5)),
}

# The draft's non-causal sliding-window attention: a block of 8 query tokens (7 drafts + the
# anchor) that see each other and the 4096 keys before them, at two context lengths (the cost
# must not depend on the context); and a chunked prefill: a 2048-token prompt chunk appended to a
# 129024-token context and attended causally (every token sees the context and the chunk's
# earlier tokens).
EXTENSIONS.update({
    8: CaseSpec("draft sliding-window attention: 2 seqs x 32768, q8 non-causal block, window 4096, Hq24/Hkv4, "
                "D256, E5M2 KV, page 2048",
                contexts=(32768,) * 2, num_q_tokens=8, num_q_heads=24, num_kv_heads=4, head_dim=256,
                page_size=2048, kv_dtype="e5m2", seed=1008, causal=False, window=4096),
    9: CaseSpec("draft sliding-window attention: 2 seqs x 262144, q8 non-causal block, window 4096, Hq24/Hkv4, "
                "D256, E5M2 KV, page 2048",
                contexts=(262144,) * 2, num_q_tokens=8, num_q_heads=24, num_kv_heads=4, head_dim=256,
                page_size=2048, kv_dtype="e5m2", seed=1009, causal=False, window=4096),
    10: CaseSpec("chunked prefill: 1 seq, 2048-token chunk appended to 129024 cached tokens (keys up to 131072), "
                 "causal, Hq24/Hkv4, D256, E4M3 KV, page 2048",
                 contexts=(129024,), num_q_tokens=2048, num_q_heads=24, num_kv_heads=4, head_dim=256,
                 page_size=2048, kv_dtype="e4m3", append_new=2048, seed=1010),
})

ALL = {**CONFIGS, **EXTENSIONS}


@dataclass
class Case:
    spec: CaseSpec
    seq_lens: np.ndarray        # int32 [B]: keys each sequence decodes over
    cached: np.ndarray          # int32 [B]: tokens already in the cache before the step
    block_table: np.ndarray     # int32 [B, max_blocks], -1 padded
    num_blocks: int
    q: np.ndarray               # fp16 [B*T, Hq, D]
    k_fill: np.ndarray          # fp16 [sum cached, Hkv, D]: tokens that populate the cache
    v_fill: np.ndarray
    slot_fill: np.ndarray       # int64 [sum cached]
    k_new: np.ndarray           # fp16 [B*append_new, Hkv, D]: tokens appended in the step
    v_new: np.ndarray
    slot_new: np.ndarray        # int64 [B*append_new]
    k_scale: np.float32
    v_scale: np.float32
    softmax_scale: np.float32
    extra: dict = field(default_factory=dict)

    @property
    def B(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def T(self) -> int:
        return self.spec.num_q_tokens

    def kv_bytes(self) -> int:
        """K+V cache bytes one decode pass reads (every key of every unit once)."""
        elt = 2 if self.spec.kv_dtype == "fp16" else 1
        return int(self.seq_lens.astype(np.int64).sum()) * self.spec.num_kv_heads * self.spec.head_dim * elt * 2


def kv_bytes_of(spec: CaseSpec) -> int:
    """Approximate K+V cache bytes of a workload (a log-uniform batch counted at its upper bound)."""
    c = spec.contexts
    total = c[2] * c[3] if len(c) and c[0] == "loguniform" else int(sum(c))
    elt = 2 if spec.kv_dtype == "fp16" else 1
    return int(total) * spec.num_kv_heads * spec.head_dim * elt * 2


def _contexts(spec: CaseSpec, rng) -> np.ndarray:
    c = spec.contexts
    if len(c) and c[0] == "loguniform":
        _, lo, hi, B = c
        u = rng.uniform(math.log(lo), math.log(hi), size=B)
        return np.floor(np.exp(u)).astype(np.int64)
    return np.asarray(c, dtype=np.int64)


def make_case(spec: CaseSpec, seed: int | None = None) -> Case:
    rng = np.random.Generator(np.random.PCG64(spec.seed if seed is None else seed))
    P, Hkv, Hq, D, T = spec.page_size, spec.num_kv_heads, spec.num_q_heads, spec.head_dim, spec.num_q_tokens
    # 1. contexts
    cached = _contexts(spec, rng)
    B = int(cached.shape[0])
    seq_lens = cached + spec.append_new
    # 2. page permutation
    pages = -(-seq_lens // P)
    total_pages = int(pages.sum())
    num_blocks = max(1, int(math.ceil(spec.pool_factor * total_pages)))
    perm = rng.permutation(num_blocks)[:total_pages].astype(np.int64)
    max_blocks = max(1, int(pages.max()) if B else 1)
    block_table = np.full((B, max_blocks), -1, dtype=np.int32)
    off = 0
    for b in range(B):
        block_table[b, :pages[b]] = perm[off:off + pages[b]]
        off += int(pages[b])
    # 3. Q
    q = rng.standard_normal((B * T, Hq, D), dtype=np.float32).astype(np.float16)
    # 4./5. K, V of the cached tokens (sequence-major, then position)
    n_fill = int(cached.sum())
    k = rng.standard_normal((n_fill, Hkv, D), dtype=np.float32)
    if spec.v_dist == "uniform":
        v = rng.uniform(-1.0, 1.0, size=(n_fill, Hkv, D)).astype(np.float32)
    else:
        v = rng.standard_normal((n_fill, Hkv, D), dtype=np.float32)
    # 6. outlier K rows
    if spec.k_outlier_frac > 0:
        n_rows = int(math.floor(spec.k_outlier_frac * n_fill * Hkv))
        rows = rng.choice(n_fill * Hkv, size=n_rows, replace=False)
        kr = k.reshape(n_fill * Hkv, D)
        kr[rows] *= np.float32(spec.k_outlier_mul)
    gain = None
    if spec.head_gain:
        gain = np.array([spec.head_gain[h % len(spec.head_gain)] for h in range(Hkv)], np.float32)[:, None]
        k *= gain
        v *= gain
    k16 = k.astype(np.float16)
    v16 = v.astype(np.float16)
    del k, v
    # 7. new tokens
    n_new = B * spec.append_new
    k_new = rng.standard_normal((n_new, Hkv, D), dtype=np.float32)
    v_new = rng.standard_normal((n_new, Hkv, D), dtype=np.float32)
    if gain is not None:
        k_new *= gain
        v_new *= gain
    k_new = k_new.astype(np.float16)
    v_new = v_new.astype(np.float16)

    def slots_for(b: int, positions: np.ndarray) -> np.ndarray:
        return block_table[b, positions // P].astype(np.int64) * P + positions % P

    slot_fill = np.concatenate([slots_for(b, np.arange(cached[b])) for b in range(B)]) if B else np.zeros(0, np.int64)
    slot_new = (np.concatenate([slots_for(b, np.arange(cached[b], seq_lens[b])) for b in range(B)])
                if n_new else np.zeros(0, np.int64))

    if spec.kv_dtype == "fp16":
        k_scale = v_scale = np.float32(1.0)
    elif spec.scale_per_head:
        fmax = FMT_MAX[spec.kv_dtype]

        def head_amax(a, b):
            out = np.zeros(Hkv)
            for arr in (a, b):
                if arr.shape[0]:
                    out = np.maximum(out, np.abs(arr).max(axis=(0, 2)).astype(np.float64))
            return out

        ka, va = head_amax(k16, k_new), head_amax(v16, v_new)
        k_scale = np.where(ka > 0, ka / fmax, 1.0).astype(np.float32)
        v_scale = np.where(va > 0, va / fmax, 1.0).astype(np.float32)
    else:
        fmax = FMT_MAX[spec.kv_dtype]
        kam = max(float(np.abs(k16).max()) if n_fill else 0.0, float(np.abs(k_new).max()) if n_new else 0.0)
        vam = max(float(np.abs(v16).max()) if n_fill else 0.0, float(np.abs(v_new).max()) if n_new else 0.0)
        k_scale = np.float32(kam / fmax) if kam > 0 else np.float32(1.0)
        v_scale = np.float32(vam / fmax) if vam > 0 else np.float32(1.0)
    return Case(spec=spec, seq_lens=seq_lens.astype(np.int32), cached=cached.astype(np.int32),
                block_table=block_table, num_blocks=num_blocks, q=q,
                k_fill=k16, v_fill=v16, slot_fill=slot_fill.astype(np.int64),
                k_new=k_new, v_new=v_new, slot_new=slot_new.astype(np.int64),
                k_scale=k_scale, v_scale=v_scale,
                softmax_scale=np.float32(1.0 / math.sqrt(D)))


def small_spec(cfg_id: int, **over) -> CaseSpec:
    """A reduced copy of a benchmark workload (same dtype/heads/page layout)."""
    return replace(ALL[cfg_id], **over)


def split_fill(case: Case, units: list[tuple[int, int]] | None = None):
    """Token index ranges of ``k_fill`` per sequence: list of (start, stop)."""
    starts = np.concatenate([[0], np.cumsum(case.cached.astype(np.int64))])
    return [(int(starts[b]), int(starts[b + 1])) for b in range(case.B)]
