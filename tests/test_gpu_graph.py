"""A serving step -- append the step's new tokens, then decode -- captured once
as a CUDA graph and replayed: the library allocates nothing and never
synchronises, so both calls are capturable. Each replay is checked against the
oracle (cache bytes bit-exact, outputs within tolerance), including a replay
after the step's new K/V values were changed in place."""

from dataclasses import replace

import numpy as np
import pytest
import torch

from paged_fp8_kv_cache_gb300 import binding as pf
from paged_fp8_kv_cache_gb300 import workloads
from tests.gpu_helpers import GpuCase, assert_close, to_dev
from tests.oracle_helpers import oracle_attention, oracle_caches

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _lib(pflib):
    pf.pfkv_device_errors(clear=True)
    yield
    assert pf.pfkv_device_errors(clear=True) == 0


# the mixed batch (one new token per sequence; 12 sequences on the one-CTA-per-range grid, 64 on
# the persistent grid, whose step chains append, counter reset and attention by programmatic
# launch) and the q8 verifier (the 8 drafts' K/V appended)
@pytest.mark.parametrize("cfg,contexts,new", [(5, ("loguniform", 30, 900, 12), 1), (5, ("loguniform", 30, 3000, 64), 1),
                                              (4, (700, 300), 8)])
def test_append_and_decode_replayed_from_a_graph(cfg, contexts, new):
    case = workloads.make_case(workloads.small_spec(cfg, contexts=contexts, append_new=new))
    s = case.spec
    assert case.slot_new.size > 0
    gc = GpuCase(case, include_new=False)  # the cache before the step
    kn, vn, slots = to_dev(case.k_new), to_dev(case.v_new), to_dev(case.slot_new)
    msl = int(case.seq_lens.max())
    ws_b = pf.pfkv_decode_workspace_bytes(case.B, s.num_q_tokens, s.num_q_heads, s.num_kv_heads, s.head_dim,
                                          s.page_size, s.kv_dtype, msl, 0)
    ws = torch.empty(max(ws_b, 256), dtype=torch.uint8, device="cuda")
    out = torch.empty(gc.q.shape, dtype=torch.float16, device="cuda")
    lse = torch.empty(gc.q.shape[:2], dtype=torch.float32, device="cuda")

    def step():
        pf.pfkv_kv_cache_append(kn, vn, gc.k_cache, gc.v_cache, slots, s.page_size, s.kv_dtype, gc.k_scale,
                                gc.v_scale)
        pf.pfkv_paged_attention_decode(out, lse, gc.q, gc.k_cache, gc.v_cache, gc.block_table, gc.seq_lens,
                                       s.num_q_tokens, s.num_kv_heads, s.page_size, s.kv_dtype, gc.k_scale,
                                       gc.v_scale, float(case.softmax_scale), msl, 0, ws)

    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        step()  # outside the capture: per-shape library state set up
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            step()
    torch.cuda.current_stream().wait_stream(stream)
    torch.cuda.synchronize()

    for variant in range(2):
        c = case
        if variant == 1:  # new K/V values for the same slots, written into the captured buffers
            c = replace(case, k_new=(-case.k_new).astype(np.float16), v_new=(case.v_new * 0.5).astype(np.float16))
            kn.copy_(to_dev(c.k_new))
            vn.copy_(to_dev(c.v_new))
        kc, vc = oracle_caches(c)
        o_ref, l_ref = oracle_attention(c, kc, vc)
        for _ in range(2):
            out.fill_(float("nan"))
            lse.fill_(float("nan"))
            graph.replay()
            torch.cuda.synchronize()
            assert np.array_equal(gc.k_cache.cpu().numpy(), kc)
            assert np.array_equal(gc.v_cache.cpu().numpy(), vc)
            assert_close(out, lse, o_ref, l_ref)
