"""Few long sequences: the automatic plan gives each SM one CTA with a long key range (one wave of
ranges twice as long as at full occupancy). Checked against the oracle for FP8 and fp16 caches at
both head dims."""

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


# 16 KV heads of one query head each: few (sequence, head) units, so the plan runs one CTA per
# SM once a sequence is some tens of thousands of keys long
@pytest.mark.parametrize("kv,D,P,n", [("e4m3", 128, 16, 48000), ("e5m2", 256, 2048, 36000),
                                      ("fp16", 128, 64, 40000), ("e4m3", 256, 256, 36001)])
def test_one_cta_per_sm_long_ranges(kv, D, P, n):
    sp = workloads.CaseSpec("long ranges", contexts=(n,), num_q_tokens=1, num_q_heads=16, num_kv_heads=16,
                            head_dim=D, page_size=P, kv_dtype=kv, seed=61)
    case = workloads.make_case(sp)
    kc, vc = oracle_caches(case)
    o_ref, l_ref = oracle_attention(case, kc, vc)
    g = GpuCase(case)
    splits, _ = pf.pfkv_decode_plan(1, 1, 16, 16, D, P, kv, n, 0)
    assert splits < 40  # one range per SM-sized share, not two waves
    out, lse = g.decode()
    torch.cuda.synchronize()
    assert_close(out, lse, o_ref, l_ref)
