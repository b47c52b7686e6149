"""Verification with up to 16 query tokens per sequence (a q16 verify: 15 drafts + 1) on both
kernels: the tcgen05 grouped verifier (FP8, more than 16 rows per KV head) and the mma.sync
decode kernel (16 rows or fewer, or an fp16 cache), against the oracle, with causal edge lengths
(fewer keys than query tokens, exactly T, tile boundaries) and with the automatic split plan and
explicit ranges."""

import numpy as np
import pytest
import torch

from paged_fp8_kv_cache_gb300 import binding as pf
from paged_fp8_kv_cache_gb300 import workloads
from tests.gpu_helpers import GpuCase, assert_close
from tests.oracle_helpers import oracle_attention, oracle_caches

pytestmark = pytest.mark.gpu

# (kv dtype, head_dim, query tokens, group size, page size): rows per KV head = T * g
SHAPES = [
    ("e5m2", 256, 16, 4, 2048),  # 64 rows, tcgen05
    ("e4m3", 128, 16, 4, 16),    # 64 rows, tcgen05, small pages
    ("e4m3", 256, 12, 4, 2048),  # 48 rows, tcgen05
    ("e5m2", 128, 9, 2, 16),     # 18 rows, tcgen05 (32 padded)
    ("e4m3", 256, 16, 1, 2048),  # 16 rows, mma.sync decode kernel
    ("fp16", 128, 16, 2, 16),    # 32 rows, fp16 cache: mma.sync decode kernel
    ("fp16", 256, 16, 4, 2048),  # 64 rows, fp16 cache
]


@pytest.fixture(autouse=True)
def _lib(pflib):
    pf.pfkv_device_errors(clear=True)
    yield
    assert pf.pfkv_device_errors(clear=True) == 0


@pytest.mark.parametrize("kv,D,T,g,P", SHAPES)
def test_q16_shapes(kv, D, T, g, P):
    contexts = (max(1, T - 5), T, T + 1, 127, 128, 129, 900)
    sp = workloads.CaseSpec("q16", contexts=contexts, num_q_tokens=T, num_q_heads=g * 2, num_kv_heads=2,
                            head_dim=D, page_size=P, kv_dtype=kv, seed=77 + T * 10 + g)
    case = workloads.make_case(sp)
    kc, vc = oracle_caches(case)
    o_ref, l_ref = oracle_attention(case, kc, vc)
    gc = GpuCase(case)
    torch.cuda.synchronize()
    assert np.array_equal(gc.k_cache.cpu().numpy(), kc)
    assert np.array_equal(gc.v_cache.cpu().numpy(), vc)
    for splits in (0, 3):
        out, lse = gc.decode(num_splits=splits)
        torch.cuda.synchronize()
        assert_close(out, lse, o_ref, l_ref)
