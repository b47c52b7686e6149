"""Helpers for the GPU parity tests: run the CUDA path through the C ABI."""

import numpy as np
import torch

from paged_fp8_kv_cache_gb300 import binding as pf

DEV = "cuda"


def to_dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.to(dtype)
    return t.to(DEV)


class GpuCase:
    """Device-resident copy of a workload: caches populated by the append kernel."""

    def __init__(self, case, include_new=True, populate_chunk=1 << 22):
        s = case.spec
        self.case = case
        elt = torch.float16 if s.kv_dtype == "fp16" else torch.uint8
        shape = (case.num_blocks, s.num_kv_heads, s.page_size, s.head_dim)
        self.k_cache = torch.zeros(shape, dtype=elt, device=DEV)
        self.v_cache = torch.zeros(shape, dtype=elt, device=DEV)
        # one float per pool, or one per KV head (the binding then sets PFKV_KV_SCALES_PER_HEAD)
        self.k_scale = torch.tensor(np.asarray(case.k_scale, np.float32).reshape(-1), device=DEV)
        self.v_scale = torch.tensor(np.asarray(case.v_scale, np.float32).reshape(-1), device=DEV)
        self.q = to_dev(case.q)
        self.block_table = to_dev(case.block_table)
        self.seq_lens = to_dev(case.seq_lens)
        # populate through the append kernel, in chunks of tokens
        n = case.k_fill.shape[0]
        step = max(1, populate_chunk // (s.num_kv_heads * s.head_dim))
        for a in range(0, n, step):
            b = min(n, a + step)
            self.append(case.k_fill[a:b], case.v_fill[a:b], case.slot_fill[a:b])
        if include_new and case.slot_new.size:
            self.append(case.k_new, case.v_new, case.slot_new)

    def append(self, k, v, slots):
        s = self.case.spec
        pf.pfkv_kv_cache_append(to_dev(k), to_dev(v), self.k_cache, self.v_cache, to_dev(slots), s.page_size,
                                s.kv_dtype, self.k_scale, self.v_scale)

    def decode(self, num_splits=0, q=None, seq_lens=None, block_table=None, k_cache=None, v_cache=None,
               max_seq_len=None):
        s = self.case.spec
        q = self.q if q is None else q
        seq_lens = self.seq_lens if seq_lens is None else seq_lens
        bt = self.block_table if block_table is None else block_table
        kc = self.k_cache if k_cache is None else k_cache
        vc = self.v_cache if v_cache is None else v_cache
        msl = int(self.case.seq_lens.max()) if max_seq_len is None else max_seq_len
        B = seq_lens.shape[0]
        T = q.shape[0] // B
        out = torch.full(q.shape, float("nan"), dtype=torch.float16, device=DEV)
        lse = torch.full(q.shape[:2], float("nan"), dtype=torch.float32, device=DEV)
        ws_bytes = pf.pfkv_decode_workspace_bytes(B, T, q.shape[1], s.num_kv_heads, s.head_dim, s.page_size,
                                                  s.kv_dtype, msl, num_splits)
        ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=DEV)
        pf.pfkv_paged_attention_decode(out, lse, q, kc, vc, bt, seq_lens, T, s.num_kv_heads, s.page_size,
                                       s.kv_dtype, self.k_scale, self.v_scale, float(self.case.softmax_scale), msl,
                                       num_splits, ws)
        self.last_workspace = ws
        return out, lse

    def attention(self, causal=True, window=0, num_splits=0, max_seq_len=None):
        """pfkv_paged_attention over the whole case (any number of query tokens, a mask choice)."""
        s = self.case.spec
        msl = int(self.case.seq_lens.max()) if max_seq_len is None else max_seq_len
        B = self.seq_lens.shape[0]
        T = s.num_q_tokens
        out = torch.full(self.q.shape, float("nan"), dtype=torch.float16, device=DEV)
        lse = torch.full(self.q.shape[:2], float("nan"), dtype=torch.float32, device=DEV)
        ws_bytes = pf.pfkv_attention_workspace_bytes(B, T, s.num_q_heads, s.num_kv_heads, s.head_dim, s.page_size,
                                                     s.kv_dtype, msl, causal, window, num_splits)
        ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=DEV)
        pf.pfkv_paged_attention(out, lse, self.q, self.k_cache, self.v_cache, self.block_table, self.seq_lens, T,
                                s.num_kv_heads, s.page_size, s.kv_dtype, self.k_scale, self.v_scale,
                                float(self.case.softmax_scale), msl, causal, window, num_splits, ws)
        self.last_workspace = ws
        return out, lse


def assert_close(out, lse, o_ref, l_ref, rows=None, out_tol=2e-3, lse_tol=1e-4):
    o = out.float().cpu().numpy().astype(np.float64)
    l = lse.cpu().numpy().astype(np.float64)
    if rows is not None:
        o, l, o_ref, l_ref = o[rows], l[rows], o_ref[rows], l_ref[rows]
    ok = np.isfinite(l_ref)
    assert np.array_equal(np.isneginf(l), np.isneginf(l_ref)), "rows with no visible key differ"
    assert np.all(o[~ok] == 0), "rows with no visible key must be 0"
    do = np.abs(o - o_ref).max() if o.size else 0.0
    dl = np.abs(l[ok] - l_ref[ok]).max() if ok.any() else 0.0
    assert np.isfinite(do) and do <= out_tol, f"max |out - oracle| = {do:.3e} > {out_tol}"
    assert dl <= lse_tol, f"max |lse - oracle| = {dl:.3e} > {lse_tol}"
    return do, dl
