"""Run-time claiming of each unit's last tiles (decode kernel): when every CTA of a call is
resident at once and the ranges are long, the CTAs of a (sequence, KV head) unit stream a static
share of its first 7/8 tiles and then take its last 1/8 one tile at a time from a counter in the
workspace, which the call zeroes. Each CTA still writes one partial result, so the merge is the
same. These tests check the results against the oracle, that the claiming really ran (every
counter ends at pool tiles + participating CTAs), and that it does not depend on what the
workspace held: garbage, a call with another batch in between, and CUDA-graph replays.
"""

import numpy as np
import pytest
import torch

from paged_fp8_kv_cache_gb300 import binding as pf
from paged_fp8_kv_cache_gb300 import workloads
from tests.gpu_helpers import GpuCase, assert_close
from tests.oracle_helpers import oracle_attention, oracle_caches

pytestmark = pytest.mark.gpu

TILE = 64


def spec(kv, T, g, Hkv, D, P, contexts, **kw):
    return workloads.CaseSpec("claims", contexts=tuple(contexts), num_q_tokens=T, num_q_heads=g * Hkv,
                              num_kv_heads=Hkv, head_dim=D, page_size=P, kv_dtype=kv, seed=kw.pop("seed", 21), **kw)


CASES = {
    "e4m3-d128-q1": (spec("e4m3", 1, 4, 2, 128, 16, (40000, 25013)), 6),
    "e5m2-d256-q4": (spec("e5m2", 4, 2, 2, 256, 2048, (30001, 8000)), 5),
    "fp16-d128-q2": (spec("fp16", 2, 4, 2, 128, 64, (20000,)), 4),
}


@pytest.fixture(autouse=True)
def _lib(pflib):
    pf.pfkv_device_errors(clear=True)
    yield
    assert pf.pfkv_device_errors(clear=True) == 0


def expected_counts(case, splits):
    """Final value of each unit's counter: its pool tiles plus the CTAs that took part."""
    s = case.spec
    msl = int(case.seq_lens.max())
    S, C = pf.pfkv_decode_plan(case.B, s.num_q_tokens, s.num_q_heads, s.num_kv_heads, s.head_dim, s.page_size,
                               s.kv_dtype, msl, splits)
    out = []
    for n in case.seq_lens:
        n = int(n)
        total = -(-n // TILE)
        parts = max(1, -(-n // C))
        out.extend([total // 8 + parts] * s.num_kv_heads)
    return np.array(out), S


def counters(ws, case, S):
    s = case.spec
    rows = case.B * s.num_q_tokens * s.num_q_heads
    off = (rows * S * s.head_dim * 4 + rows * S * 4 + 15) // 16 * 16
    n = case.B * s.num_kv_heads
    return ws[off:off + 4 * n].view(torch.int32).cpu().numpy()


@pytest.mark.parametrize("name", list(CASES))
def test_claimed_tiles_match_oracle(name):
    sp, splits = CASES[name]
    case = workloads.make_case(sp)
    kc, vc = oracle_caches(case)
    o_ref, l_ref = oracle_attention(case, kc, vc)
    g = GpuCase(case)
    out, lse = g.decode(num_splits=splits)
    torch.cuda.synchronize()
    assert_close(out, lse, o_ref, l_ref)
    want, S = expected_counts(case, splits)
    assert np.array_equal(counters(g.last_workspace, case, S), want), "tile claiming did not run as planned"


def test_claims_do_not_depend_on_the_workspace_contents():
    """Garbage in the workspace, a call with another batch in between, the first call again."""
    sp_a, splits_a = CASES["e4m3-d128-q1"]
    case_a = workloads.make_case(sp_a)
    kc, vc = oracle_caches(case_a)
    o_a, l_a = oracle_attention(case_a, kc, vc)
    sp_b = spec("e4m3", 1, 4, 2, 128, 16, (3000, 50000, 12), seed=22)
    case_b = workloads.make_case(sp_b)
    kcb, vcb = oracle_caches(case_b)
    o_b, l_b = oracle_attention(case_b, kcb, vcb)
    ga, gb = GpuCase(case_a), GpuCase(case_b)
    s = sp_a
    need_a = pf.pfkv_decode_workspace_bytes(case_a.B, 1, s.num_q_heads, s.num_kv_heads, s.head_dim, s.page_size,
                                            s.kv_dtype, int(case_a.seq_lens.max()), splits_a)
    need_b = pf.pfkv_decode_workspace_bytes(case_b.B, 1, s.num_q_heads, s.num_kv_heads, s.head_dim, s.page_size,
                                            s.kv_dtype, int(case_b.seq_lens.max()), 8)
    ws = torch.full((max(need_a, need_b),), 0xFF, dtype=torch.uint8, device="cuda")  # every counter -1

    def call(g, case, splits):
        out = torch.empty(g.q.shape, dtype=torch.float16, device="cuda")
        lse = torch.empty(g.q.shape[:2], dtype=torch.float32, device="cuda")
        pf.pfkv_paged_attention_decode(out, lse, g.q, g.k_cache, g.v_cache, g.block_table, g.seq_lens, 1,
                                       s.num_kv_heads, s.page_size, s.kv_dtype, g.k_scale, g.v_scale,
                                       float(case.softmax_scale), int(case.seq_lens.max()), splits, ws)
        return out, lse

    for g, case, splits, o, l in ((ga, case_a, splits_a, o_a, l_a), (gb, case_b, 8, o_b, l_b),
                                  (ga, case_a, splits_a, o_a, l_a)):
        out, lse = call(g, case, splits)
        torch.cuda.synchronize()
        assert_close(out, lse, o, l)


def test_claims_in_a_cuda_graph_replay():
    """The counters are zeroed by a node of the captured graph, so every replay claims afresh."""
    sp, splits = CASES["e5m2-d256-q4"]
    case = workloads.make_case(sp)
    kc, vc = oracle_caches(case)
    g = GpuCase(case)
    s = sp
    msl = int(case.seq_lens.max())
    need = pf.pfkv_decode_workspace_bytes(case.B, s.num_q_tokens, s.num_q_heads, s.num_kv_heads, s.head_dim,
                                          s.page_size, s.kv_dtype, msl, splits)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    out = torch.empty(g.q.shape, dtype=torch.float16, device="cuda")
    lse = torch.empty(g.q.shape[:2], dtype=torch.float32, device="cuda")
    q = g.q.clone()

    def step():
        pf.pfkv_paged_attention_decode(out, lse, q, g.k_cache, g.v_cache, g.block_table, g.seq_lens,
                                       s.num_q_tokens, s.num_kv_heads, s.page_size, s.kv_dtype, g.k_scale,
                                       g.v_scale, float(case.softmax_scale), msl, splits, ws)

    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        step()  # warm-up outside the capture (tensor maps, occupancy)
    torch.cuda.current_stream().wait_stream(stream)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    rng = np.random.default_rng(5)
    want, S = expected_counts(case, splits)
    for _ in range(3):
        qn = rng.standard_normal(case.q.shape, dtype=np.float32).astype(np.float16)
        q.copy_(torch.from_numpy(qn))
        graph.replay()
        torch.cuda.synchronize()
        o_ref, l_ref = oracle_attention(case, kc, vc, q=qn)
        assert_close(out, lse, o_ref, l_ref)
        assert np.array_equal(counters(ws, case, S), want)
