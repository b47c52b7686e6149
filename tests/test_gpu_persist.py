"""Ragged decode batches on the persistent grid: one wave of CTAs that claim the key ranges that
exist from a counter in the workspace (instead of a grid sized for the longest sequence the call
allows). Checked against the oracle with a workspace full of garbage, with one workspace serving
batches of different shapes, with empty and one-key sequences, and from a captured CUDA graph.

Which grid ran is read from the counter (documented in include/pfkv.h): after the persistent grid
it holds the number of key ranges; the one-CTA-per-range grid leaves it as it was."""

import numpy as np
import pytest
import torch

from paged_fp8_kv_cache_gb300 import binding as pf
from paged_fp8_kv_cache_gb300 import workloads
from oracle import attention
from tests.gpu_helpers import GpuCase, assert_close
from tests.oracle_helpers import oracle_caches

pytestmark = pytest.mark.gpu

GARBAGE = -0x2A2A2A2B  # int32 of the bytes 0xD5 0xD5 0xD5 0xD5


@pytest.fixture(autouse=True)
def _lib(pflib):
    pf.pfkv_device_errors(clear=True)
    yield
    assert pf.pfkv_device_errors(clear=True) == 0


def _spec(contexts, kv="e4m3", T=1, g=4, Hkv=8, D=128, P=16, seed=41, **kw):
    return workloads.CaseSpec("persistent grid", contexts=tuple(int(c) for c in contexts), num_q_tokens=T,
                              num_q_heads=g * Hkv, num_kv_heads=Hkv, head_dim=D, page_size=P, kv_dtype=kv,
                              seed=seed, **kw)


def _ragged(B, lo, hi, seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    return np.exp(rng.uniform(np.log(lo), np.log(hi), size=B)).astype(np.int64)


def _ranges(seq_lens, T, Hkv, split_tokens, causal=True, window=0, tile=64):
    """Key ranges of a one-slab call: per sequence and KV head, the split ranges of its span."""
    total = 0
    for N in (int(n) for n in seq_lens):
        p0, p1 = N - T, N - 1
        hi = p1 if (causal and p1 < N - 1) else N - 1
        lo = max(0, p0 - window + 1) if window > 0 else 0
        base = lo & ~(tile - 1)
        total += ((hi - base + split_tokens) // split_tokens if hi >= lo else 1) * Hkv
    return total


def _counter(ws, case, splits):
    s = case.spec
    rows = case.B * s.num_q_tokens * s.num_q_heads
    off = (rows * splits * s.head_dim * 4 + rows * splits * 4 + 15) & ~15
    return int(ws[off:off + 4].cpu().numpy().view(np.int32)[0])


class Ragged:
    def __init__(self, sp, causal=True, window=0, num_splits=0, max_seq_len=None):
        self.case = workloads.make_case(sp)
        kc, vc = oracle_caches(self.case)
        s = sp
        self.o_ref, self.l_ref = attention.paged_attention(
            self.case.q, kc, vc, self.case.block_table, self.case.seq_lens, s.num_q_tokens, s.num_kv_heads,
            s.page_size, s.kv_dtype, self.case.k_scale, self.case.v_scale, self.case.softmax_scale,
            causal=causal, window=window)
        self.g = GpuCase(self.case)
        self.causal, self.window, self.num_splits = causal, window, num_splits
        self.msl = int(self.case.seq_lens.max()) if max_seq_len is None else max_seq_len
        self.splits, self.split_tokens = pf.pfkv_attention_plan(self.case.B, s.num_q_tokens, s.num_q_heads,
                                                                s.num_kv_heads, s.head_dim, s.page_size, s.kv_dtype,
                                                                self.msl, causal, window, num_splits)
        self.ws_bytes = pf.pfkv_attention_workspace_bytes(self.case.B, s.num_q_tokens, s.num_q_heads,
                                                          s.num_kv_heads, s.head_dim, s.page_size, s.kv_dtype,
                                                          self.msl, causal, window, num_splits)
        self.ranges = _ranges(self.case.seq_lens, s.num_q_tokens, s.num_kv_heads, self.split_tokens, causal, window)
        self.out = torch.empty(self.g.q.shape, dtype=torch.float16, device="cuda")
        self.lse = torch.empty(self.g.q.shape[:2], dtype=torch.float32, device="cuda")

    def call(self, ws, stream=None):
        s = self.case.spec
        pf.pfkv_paged_attention(self.out, self.lse, self.g.q, self.g.k_cache, self.g.v_cache, self.g.block_table,
                                self.g.seq_lens, s.num_q_tokens, s.num_kv_heads, s.page_size, s.kv_dtype,
                                self.g.k_scale, self.g.v_scale, float(self.case.softmax_scale), self.msl,
                                self.causal, self.window, self.num_splits, ws, stream)

    def clear(self):
        self.out.fill_(float("nan"))
        self.lse.fill_(float("nan"))

    def check(self):
        assert_close(self.out, self.lse, self.o_ref, self.l_ref)


def _garbage(nbytes):
    return torch.full((nbytes,), 0xD5, dtype=torch.uint8, device="cuda")


@pytest.mark.parametrize("kv,D,P", [("e4m3", 128, 16), ("e5m2", 256, 16), ("fp16", 128, 32), ("fp16", 256, 64)])
def test_ragged_batch_runs_persistent_and_matches_oracle(kv, D, P):
    # 48 sequences x 8 KV heads, lengths log-uniform in [16, 5000]: the automatic plan cuts the
    # longest into several ranges, so the full grid would be mostly empty
    r = Ragged(_spec(_ragged(48, 16, 5000, seed=3), kv=kv, D=D, P=P))
    ws = _garbage(r.ws_bytes)
    r.clear()
    r.call(ws)
    torch.cuda.synchronize()
    r.check()
    assert _counter(ws, r.case, r.splits) == r.ranges


def test_small_batch_keeps_one_cta_per_range():
    r = Ragged(_spec((3000, 1, 700, 4100), Hkv=2), num_splits=4)
    ws = _garbage(r.ws_bytes)
    r.clear()
    r.call(ws)
    torch.cuda.synchronize()
    r.check()
    assert _counter(ws, r.case, r.splits) == GARBAGE


def test_empty_and_tiny_sequences_more_ctas_than_ranges():
    # mostly empty or one-key sequences and a long one: fewer ranges than resident CTAs, so
    # some CTAs find nothing to claim
    ctx = [0, 1, 0, 2, 63, 64, 65, 0] * 3 + [20000]
    r = Ragged(_spec(ctx, seed=42), num_splits=16)
    ws = _garbage(r.ws_bytes)
    r.clear()
    r.call(ws)
    torch.cuda.synchronize()
    r.check()
    assert _counter(ws, r.case, r.splits) == r.ranges


def test_sequences_shorter_than_the_query_block():
    # q4 rows of sequences with 0..3 keys (no key or only some of the block's own) among longer
    # ones, on the persistent grid
    ctx = [0, 0, 1, 2, 3, 1, 0, 2] * 6 + [3000, 1500]
    r = Ragged(_spec(ctx, T=4, g=2, seed=49), num_splits=8)
    ws = _garbage(r.ws_bytes)
    r.clear()
    r.call(ws)
    torch.cuda.synchronize()
    r.check()
    assert _counter(ws, r.case, r.splits) == r.ranges


@pytest.mark.parametrize("T,g,window", [(2, 4, 0), (1, 8, 1000), (4, 2, 300)])
def test_multi_token_and_window(T, g, window):
    r = Ragged(_spec(_ragged(40, 4, 6000, seed=7 + T), T=T, g=g, seed=43), causal=True, window=window,
               num_splits=8)
    ws = _garbage(r.ws_bytes)
    r.clear()
    r.call(ws)
    torch.cuda.synchronize()
    r.check()
    assert _counter(ws, r.case, r.splits) == r.ranges


def test_many_sequences():
    # more sequences than the grid orders by their last range's length (256): the last ranges
    # then follow in sequence order
    r = Ragged(_spec(_ragged(300, 1, 2000, seed=14), Hkv=2, seed=47), num_splits=4)
    ws = _garbage(r.ws_bytes)
    r.clear()
    r.call(ws)
    torch.cuda.synchronize()
    r.check()
    assert _counter(ws, r.case, r.splits) == r.ranges


@pytest.mark.parametrize("B", [1024, 1025])
def test_largest_batches(B):
    # 1024 sequences is the most the persistent grid takes (lengths and item prefix in shared
    # memory); one more runs the one-CTA-per-range grid
    r = Ragged(_spec(_ragged(B, 1, 300, seed=15), Hkv=2, seed=48), num_splits=2, max_seq_len=512)
    ws = _garbage(r.ws_bytes)
    r.clear()
    r.call(ws)
    torch.cuda.synchronize()
    r.check()
    assert _counter(ws, r.case, r.splits) == (r.ranges if B <= 1024 else GARBAGE)


def test_one_workspace_across_batches():
    # two batches of different shapes take turns on one workspace, with no synchronisation
    a = Ragged(_spec(_ragged(48, 16, 5000, seed=11), seed=44))
    b = Ragged(_spec(_ragged(96, 32, 2500, seed=12), Hkv=4, g=8, seed=45), num_splits=6)
    ws = _garbage(max(a.ws_bytes, b.ws_bytes))
    for r in (a, b):
        r.clear()
    a.call(ws)
    b.call(ws)
    a.out.fill_(float("nan"))
    a.call(ws)
    torch.cuda.synchronize()
    a.check()
    b.check()


def test_graph_replay():
    r = Ragged(_spec(_ragged(48, 16, 5000, seed=13), seed=46))
    ws = _garbage(r.ws_bytes)
    graph = torch.cuda.CUDAGraph()
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        r.call(ws, stream)  # outside the capture: library state set up
        torch.cuda.synchronize()
        with torch.cuda.graph(graph, stream=stream):
            r.call(ws, stream)
    torch.cuda.current_stream().wait_stream(stream)
    torch.cuda.synchronize()
    for _ in range(3):
        r.clear()
        ws[-16:].fill_(0xD5)
        graph.replay()
        torch.cuda.synchronize()
        r.check()
    assert _counter(ws, r.case, r.splits) == r.ranges
