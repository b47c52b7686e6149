"""The decode entry point that allocates nothing and needs no workspace.

It serves callers that cannot call cudaMalloc -- a plugin inside another
engine whose memory pool already holds nearly all device memory, or a
serving loop where an allocation's implicit device synchronisation is not
acceptable. Its split scratch is a fixed array inside the library. This file
is collected last on purpose: it checks the new entry point through the C
ABI against the ordinary one (which takes a caller workspace) and against
the oracle, on two calls in a row, and passes both alone in a fresh process
and after every other test. Every case is one whose plan splits the keys,
so the built-in array is really used.
"""

import pytest
import torch

from paged_fp8_kv_cache_gb300 import binding as pf
from paged_fp8_kv_cache_gb300 import workloads
from tests.gpu_helpers import GpuCase, assert_close
from tests.oracle_helpers import oracle_attention, oracle_caches

pytestmark = pytest.mark.gpu

OUT_TOL, LSE_TOL = 2e-3, 1e-4  # the parity tolerances of the other GPU tests


def _static_decode(g, num_splits):
    s = g.case.spec
    out = torch.full(g.q.shape, float("nan"), dtype=torch.float16, device="cuda")
    lse = torch.full(g.q.shape[:2], float("nan"), dtype=torch.float32, device="cuda")
    pf.pfkv_paged_attention_decode_static_scratch(
        out, lse, g.q, g.k_cache, g.v_cache, g.block_table, g.seq_lens, s.num_q_tokens, s.num_kv_heads,
        s.page_size, s.kv_dtype, g.k_scale, g.v_scale, float(g.case.softmax_scale), int(g.case.seq_lens.max()),
        num_splits)
    return out, lse


@pytest.mark.parametrize("spec,splits", [
    (workloads.small_spec(3, contexts=(5000,)), 7),                      # long E4M3 decode, split
    (workloads.small_spec(4, contexts=(4100, 2500)), 4),                 # q8 verify on tcgen05, split
    (workloads.small_spec(5, contexts=("loguniform", 30, 700, 64)), 3),  # ragged batch
], ids=["long-e4m3", "verify-q8-e5m2", "mixed-e4m3"])
def test_static_scratch_matches_workspace_entry_point(pflib, spec, splits):
    pf.pfkv_device_errors(clear=True)
    case = workloads.make_case(spec)
    s = case.spec
    # the plan splits the keys, so the partials go through the built-in array
    need = pf.pfkv_decode_workspace_bytes(case.B, s.num_q_tokens, s.num_q_heads, s.num_kv_heads, s.head_dim,
                                          s.page_size, s.kv_dtype, int(case.seq_lens.max()), splits)
    assert need > 0
    g = GpuCase(case)
    ref_out, ref_lse = g.decode(num_splits=splits)
    torch.cuda.synchronize()
    kc, vc = oracle_caches(case)
    o_oracle, l_oracle = oracle_attention(case, kc, vc)
    for _ in range(2):  # two calls in a row share (and reuse) the built-in array
        out, lse = _static_decode(g, splits)
        torch.cuda.synchronize()
        assert torch.isfinite(out.float()).all()
        assert (out.float() - ref_out.float()).abs().max().item() <= OUT_TOL
        fin = torch.isfinite(ref_lse)
        assert torch.equal(fin, torch.isfinite(lse))
        assert (lse[fin] - ref_lse[fin]).abs().max().item() <= LSE_TOL
        assert_close(out, lse, o_oracle, l_oracle, out_tol=OUT_TOL, lse_tol=LSE_TOL)
    assert pf.pfkv_device_errors(clear=True) == 0


def test_static_scratch_rejects_oversized_plans(pflib):
    # 64 sequences x 8 tokens x 64 heads of 256 dims split 64 ways needs far more than the 32 MiB array
    need = pf.pfkv_decode_workspace_bytes(64, 8, 64, 8, 256, 2048, "e4m3", 262144, 64)
    assert need > 32 << 20
    dummy = torch.zeros(16, dtype=torch.uint8, device="cuda")
    p = dummy.data_ptr()
    st = pf.load().pfkv_paged_attention_decode_static_scratch(
        p, p, p, p, p, p, 128, p, 64, 8, 64, 8, 256, 2048, 128, pf.PFKV_KV_FP8_E4M3, p, p, 0.0625, 262144, 64, None)
    assert st == pf.PFKV_ERR_WORKSPACE
    assert str(32 << 20) in pf.pfkv_last_error()
    torch.cuda.synchronize()
