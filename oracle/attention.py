"""Paged decode / grouped causal-verify attention over an FP8 cache (float64).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

What the pages fix: decode attention reads K/V from a paged cache stored as
FP8 and dequantised for compute ("1Cat-vLLM 1.5.0", section "Flash-V100
long-context improvements"; "1Cat-vLLM", "Optional experimental feature: FP8
KV cache"); speculative verification attends 8 query tokens per sequence (7
drafts + 1) "exactly" over the same cache ("1Cat-vLLM 1.5.0", "Production
DFlash2 on V100": exact grouped q8 verification over FP8 E5M2 KV); several
query heads share one KV head (grouped-query attention, same sections). The
attention itself is not an approximation, so this oracle is the plain
definition, computed in float64:

for sequence b, query token t < T and query head h:

* ``kvh = h // g`` with ``g = Hq // Hkv`` (contiguous head groups);
* query t sits at position ``p = N_b - T + t`` (``seq_lens[b] = N_b``
  already counts the T query tokens, whose K/V are in the cache) and sees
  the keys ``lo <= j <= hi`` with
  ``hi = p`` when causal (over its own drafts, the default) or ``hi = N_b - 1``
  when not (a draft block attending to all of its own tokens: the non-causal
  draft attention of "1Cat-vLLM 1.5.0", "Production DFlash2 on V100"), and
  ``lo = max(0, p - W + 1)`` for a sliding window of W keys (the draft's
  sliding-window attention, same page, "Flash-V100 long-context
  improvements") or ``lo = 0`` without one (W = 0). A window is read as a
  bound on how far back a query looks, relative to its own position; the
  causal flag alone bounds how far forward. Long T is the chunked prefill
  (the same attention for every token of a prompt chunk);
* key j lives at ``page = block_table[b][j // P]``, ``offset = j % P``;
* ``k_j = decode(K[page, kvh, offset]) * k_scale`` and likewise ``v_j``
  (``k_scale`` is the pool's static scale, or KV head kvh's when one scale
  per KV head is given: the per-head generalisation of the per-tensor
  scales, a reading of ours -- the pages use per-tensor scales only);
* ``s_j = softmax_scale * sum_d q_d k_jd``, ``m = max_j s_j``,
  ``w_j = exp(s_j - m)``, ``L = sum_j w_j``;
* ``out = sum_j w_j v_j / L`` and ``lse = m + ln L`` (natural log, the logits
  include both ``softmax_scale`` and ``k_scale``).

A row that sees no key (e.g. ``N_b - T + t < 0`` when causal, or an empty
sequence) has ``out = 0`` and ``lse = -inf`` (the empty-sum convention used
on both sides).

Evaluation order: per (sequence, KV head) all logits of all rows over the
whole key range are formed first, then the weights, then ``sum_j w_j v_j``.
This is the two-pass definition above; nothing is blocked, fused or rescaled
online.
"""

from __future__ import annotations

import numpy as np

from . import fp8


def _decode_pages(cache: np.ndarray, pages: np.ndarray, kvh: int, kv_dtype: str) -> np.ndarray:
    """float64 ``[len(pages) * P, D]`` of one KV head, unscaled."""
    chunk = cache[pages, kvh]  # [npages, P, D]
    flat = chunk.reshape(-1, chunk.shape[-1])
    if kv_dtype == "fp16":
        return flat.astype(np.float64)
    return fp8.decode(flat, kv_dtype)


def paged_attention(q: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray,
                    block_table: np.ndarray, seq_lens: np.ndarray,
                    num_q_tokens: int, num_kv_heads: int, page_size: int,
                    kv_dtype: str, k_scale: float, v_scale: float,
                    softmax_scale: float, units=None, token_range=None, causal=True, window=0,
                    tokens=None):
    """Attention for every (or the listed) (sequence, KV head) unit.

    q: fp16 ``[B*T, Hq, D]``. Caches ``[num_blocks, Hkv, P, D]`` (uint8 codes or
    fp16). Returns float64 ``out [B*T, Hq, D]`` and ``lse [B*T, Hq]``; rows of
    units not listed in ``units`` are left NaN.

    ``token_range=(lo, hi)`` restricts every row to keys ``lo <= j < hi`` (on
    top of its mask). It is how the split-KV partial results are defined: the
    attention of a row over one contiguous range of its keys.

    ``causal`` and ``window`` (W >= 0; 0 = no window) set each row's visible
    keys as stated at the top of this module. ``tokens`` (a list of query
    token indices) computes only those tokens' rows (the others stay NaN).
    """
    T = num_q_tokens
    q = np.asarray(q)
    BT, Hq, D = q.shape
    B = BT // T
    g = Hq // num_kv_heads
    out = np.full((BT, Hq, D), np.nan)
    lse = np.full((BT, Hq), np.nan)
    # one float32 scale per pool, or one per KV head (an array of num_kv_heads)
    ks_all = np.asarray(k_scale, dtype=np.float32).astype(np.float64).reshape(-1)
    vs_all = np.asarray(v_scale, dtype=np.float32).astype(np.float64).reshape(-1)
    for a in (ks_all, vs_all):
        if a.size not in (1, num_kv_heads):
            raise ValueError(f"{a.size} scales for {num_kv_heads} KV heads")
    sm = np.float64(np.float32(softmax_scale))
    if units is None:
        units = [(b, kvh) for b in range(B) for kvh in range(num_kv_heads)]
    for b, kvh in units:
        ks = ks_all[kvh if ks_all.size > 1 else 0]
        vs = vs_all[kvh if vs_all.size > 1 else 0]
        n = int(seq_lens[b])
        heads = list(range(kvh * g, (kvh + 1) * g))
        toks = list(range(T)) if tokens is None else [int(t) for t in tokens]
        nt = len(toks)
        # rows of this unit: (t, head) -> q vector
        qrows = q[b * T:(b + 1) * T, heads, :].astype(np.float64)[toks]  # [nt, g, D]
        qrows = qrows.reshape(nt * g, D)
        # per row: the first and last visible key
        pos = np.array([n - T + t for t in toks for _ in heads])
        last = pos if causal else np.full(nt * g, n - 1)
        first = np.maximum(0, pos - window + 1) if window > 0 else np.zeros(nt * g, dtype=np.int64)
        lo, hi = (0, n) if token_range is None else (max(0, token_range[0]), min(n, token_range[1]))
        if hi <= lo:
            o = np.zeros((nt * g, D))
            l_ = np.full(nt * g, -np.inf)
        else:
            first_page, last_page = lo // page_size, (hi - 1) // page_size
            pages = np.asarray(block_table[b, first_page:last_page + 1], dtype=np.int64)
            base = first_page * page_size
            # pass 1: all logits s[row, j] for j in [lo, hi)
            K = _decode_pages(k_cache, pages, kvh, kv_dtype)[lo - base:hi - base] * ks
            s = sm * (qrows @ K.T)  # [rows, hi-lo]
            j = np.arange(lo, hi)
            visible = (j[None, :] <= last[:, None]) & (j[None, :] >= first[:, None])
            s = np.where(visible, s, -np.inf)
            m = s.max(axis=1)
            has = np.isfinite(m)
            w = np.exp(s - np.where(has, m, 0.0)[:, None])
            w = np.where(visible, w, 0.0)
            L = w.sum(axis=1)
            # pass 2: weighted sum of V
            V = _decode_pages(v_cache, pages, kvh, kv_dtype)[lo - base:hi - base] * vs
            acc = w @ V
            o = np.where(has[:, None], acc / np.where(has, L, 1.0)[:, None], 0.0)
            l_ = np.where(has, m + np.log(np.where(has, L, 1.0)), -np.inf)
        o = o.reshape(nt, g, D)
        l_ = l_.reshape(nt, g)
        for i, t in enumerate(toks):
            out[b * T + t, heads, :] = o[i]
            lse[b * T + t, heads] = l_[i]
    return out, lse
