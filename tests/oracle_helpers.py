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


# --------------------------------------------------------------------------- full-size helpers
#
# The oracle's quantisation is elementwise in the fp16 input (for a fixed scale), so evaluating
# it once on every finite fp16 value gives a table whose lookup is the oracle's function on any
# array of finite inputs. The full-size tests use it to check every cache byte of GB-sized
# workloads in seconds; tests/test_oracle_append.py pins the lookup against the direct call.

def quantise_table(scale, kv_dtype):
    """uint8[65536]: oracle.append.quantise of the fp16 value with bit pattern i (0 for the
    non-finite patterns, which the workloads never hold)."""
    codes = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16).view(np.float16)
    fin = np.isfinite(codes)
    tab = np.zeros(1 << 16, np.uint8)
    tab[fin] = append.quantise(codes[fin], np.float32(scale), kv_dtype)
    return tab


def head_tables(case):
    """Per KV head (k_table, v_table), or None for an fp16 cache."""
    s = case.spec
    if s.kv_dtype == "fp16":
        return None
    ks = np.asarray(case.k_scale, np.float32).reshape(-1)
    vs = np.asarray(case.v_scale, np.float32).reshape(-1)
    out = []
    for h in range(s.num_kv_heads):
        out.append((quantise_table(ks[h % ks.size], s.kv_dtype), quantise_table(vs[h % vs.size], s.kv_dtype)))
    return out


def expected_rows(x16, tables, which):
    """Expected cache rows of fp16 tokens ``[n, Hkv, D]``: codes by table lookup per KV head
    (``which`` 0 = K, 1 = V), or the fp16 values themselves for an fp16 cache."""
    if tables is None:
        return x16
    assert np.isfinite(x16).all()
    bits = x16.view(np.uint16)
    out = np.empty(x16.shape, np.uint8)
    for h, tab in enumerate(tables):
        out[:, h] = tab[which][bits[:, h]]
    return out


def unit_tokens(case, b):
    """fp16 K and V rows ``[seq_len_b, Hkv, D]`` of sequence b in position order (cached tokens,
    then the step's appended ones)."""
    starts = np.concatenate([[0], np.cumsum(case.cached.astype(np.int64))])
    k = case.k_fill[starts[b]:starts[b + 1]]
    v = case.v_fill[starts[b]:starts[b + 1]]
    a = case.spec.append_new
    if a:
        k = np.concatenate([k, case.k_new[b * a:(b + 1) * a]])
        v = np.concatenate([v, case.v_new[b * a:(b + 1) * a]])
    return k, v


def unit_caches(case, units, tables):
    """Host K/V pools holding, for each listed (sequence, KV head) unit, that head's rows of the
    sequence's pages as the oracle quantises them from the fp16 inputs; everything else zero."""
    s = case.spec
    P = s.page_size
    dt = np.float16 if s.kv_dtype == "fp16" else np.uint8
    kc = np.zeros(cache_shape(case), dt)
    vc = np.zeros(cache_shape(case), dt)
    for b, kvh in units:
        n = int(case.seq_lens[b])
        if n == 0:
            continue
        k16, v16 = unit_tokens(case, b)
        npg = -(-n // P)
        pad = npg * P - n
        for src, dst, which in ((k16, kc, 0), (v16, vc, 1)):
            rows = src[:, kvh:kvh + 1]
            codes = expected_rows(rows, None if tables is None else [tables[kvh]], which)[:, 0]
            if pad:
                codes = np.concatenate([codes, np.zeros((pad, s.head_dim), dt)])
            dst[case.block_table[b, :npg], kvh] = codes.reshape(npg, P, s.head_dim)
    return kc, vc
