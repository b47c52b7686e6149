"""Split-KV decode with a caller workspace: the partial results of the key
ranges and their LSE merge, checked against the oracle when the workspace
starts out holding garbage, when one workspace serves calls with different
split counts, and when the call is replayed from a captured CUDA graph."""

import pytest
import torch

from paged_fp8_kv_cache_gb300 import binding as pf
from paged_fp8_kv_cache_gb300 import workloads
from tests.gpu_helpers import GpuCase, assert_close
from tests.oracle_helpers import oracle_attention, oracle_caches

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _lib(pflib):
    pf.pfkv_device_errors(clear=True)
    yield
    assert pf.pfkv_device_errors(clear=True) == 0


def _case(kv="e4m3", T=1, g=4, D=128, P=16, contexts=(3000, 1, 700, 4100)):
    sp = workloads.CaseSpec("split-merge", contexts=contexts, num_q_tokens=T, num_q_heads=g * 2, num_kv_heads=2,
                            head_dim=D, page_size=P, kv_dtype=kv, seed=23)
    case = workloads.make_case(sp)
    kc, vc = oracle_caches(case)
    o, l = oracle_attention(case, kc, vc)
    return case, GpuCase(case), o, l


def _call(g, out, lse, ws, splits):
    s = g.case.spec
    pf.pfkv_paged_attention_decode(out, lse, g.q, g.k_cache, g.v_cache, g.block_table, g.seq_lens,
                                   s.num_q_tokens, s.num_kv_heads, s.page_size, s.kv_dtype, g.k_scale, g.v_scale,
                                   float(g.case.softmax_scale), int(g.case.seq_lens.max()), splits, ws)


@pytest.mark.parametrize("kv,T,g,D", [("e4m3", 1, 4, 128), ("fp16", 8, 6, 256), ("e5m2", 2, 3, 256)])
def test_garbage_workspace_and_changing_split_counts(kv, T, g, D):
    case, gc, o_ref, l_ref = _case(kv, T, g, D)
    s = case.spec
    msl = int(case.seq_lens.max())
    need = max(pf.pfkv_decode_workspace_bytes(case.B, T, s.num_q_heads, 2, D, s.page_size, kv, msl, n)
               for n in (2, 3, 7, 16, 0))
    ws = torch.randint(0, 256, (need,), dtype=torch.uint8, device="cuda")  # garbage, counters included
    out = torch.empty(gc.q.shape, dtype=torch.float16, device="cuda")
    lse = torch.empty(gc.q.shape[:2], dtype=torch.float32, device="cuda")
    for n in (7, 2, 16, 0, 3, 7):
        out.fill_(float("nan"))
        lse.fill_(float("nan"))
        _call(gc, out, lse, ws, n)
        torch.cuda.synchronize()
        assert_close(out, lse, o_ref, l_ref)


def test_graph_replay():
    case, gc, o_ref, l_ref = _case()
    s = case.spec
    msl = int(case.seq_lens.max())
    splits = 9
    need = pf.pfkv_decode_workspace_bytes(case.B, 1, s.num_q_heads, 2, 128, s.page_size, "e4m3", msl, splits)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    out = torch.empty(gc.q.shape, dtype=torch.float16, device="cuda")
    lse = torch.empty(gc.q.shape[:2], dtype=torch.float32, device="cuda")
    graph = torch.cuda.CUDAGraph()
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        _call(gc, out, lse, ws, splits)  # outside the capture: library state set up
        torch.cuda.synchronize()
        with torch.cuda.graph(graph, stream=stream):
            _call(gc, out, lse, ws, splits)
    torch.cuda.current_stream().wait_stream(stream)
    torch.cuda.synchronize()
    for _ in range(3):
        out.fill_(float("nan"))
        lse.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert_close(out, lse, o_ref, l_ref)
