"""Shared helpers for tests: populate oracle caches from a workload case."""

import numpy as np

from oracle import append, attention


def cache_shape(case):
    s = case.spec
    return (case.num_blocks, s.num_kv_heads, s.page_size, s.head_dim)


def oracle_caches(case, include_new=True):
    """K/V caches (uint8 codes or fp16) holding every token the step decodes over."""
    s = case.spec
    dt = np.float16 if s.kv_dtype == "fp16" else np.uint8
    kc = np.zeros(cache_shape(case), dt)
    vc = np.zeros(cache_shape(case), dt)
    append.append_bulk(kc, case.k_fill, case.slot_fill, s.page_size, case.k_scale, s.kv_dtype)
    append.append_bulk(vc, case.v_fill, case.slot_fill, s.page_size, case.v_scale, s.kv_dtype)
    if include_new and case.slot_new.size:
        append.append_bulk(kc, case.k_new, case.slot_new, s.page_size, case.k_scale, s.kv_dtype)
        append.append_bulk(vc, case.v_new, case.slot_new, s.page_size, case.v_scale, s.kv_dtype)
    return kc, vc


def oracle_attention(case, kc, vc, units=None, token_range=None, seq_lens=None, q=None):
    s = case.spec
    return attention.paged_attention(
        case.q if q is None else q, kc, vc, case.block_table,
        case.seq_lens if seq_lens is None else seq_lens,
        s.num_q_tokens, s.num_kv_heads, s.page_size, s.kv_dtype,
        case.k_scale, case.v_scale, case.softmax_scale, units=units, token_range=token_range)
