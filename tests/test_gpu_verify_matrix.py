"""The tcgen05 grouped-verify kernel (FP8 caches, more than 16 query rows per
KV head) across its shape variants: 32/48/64 padded rows, head_dim 128 and
256, E4M3 and E5M2, small and large pages, and causal edge lengths (a
sequence shorter than the query-token count, so that some rows see no key;
exactly T keys; tile boundaries at 127/128/129 keys), each against the
oracle with the automatic split plan and with explicit ranges."""

import numpy as np
import pytest
import torch

from paged_fp8_kv_cache_gb300 import binding as pf
from paged_fp8_kv_cache_gb300 import workloads
from tests.gpu_helpers import GpuCase, assert_close
from tests.oracle_helpers import oracle_attention, oracle_caches

pytestmark = pytest.mark.gpu

# (query tokens, group size): rows = T * g = 24 / 32 -> 32 padded, 48, 64
SHAPES = [(4, 6), (8, 4), (8, 6), (6, 8), (8, 8)]


@pytest.fixture(autouse=True)
def _lib(pflib):
    pf.pfkv_device_errors(clear=True)
    yield
    assert pf.pfkv_device_errors(clear=True) == 0


@pytest.mark.parametrize("P", [16, 2048])
@pytest.mark.parametrize("T,g", SHAPES)
@pytest.mark.parametrize("kv,D", [("e4m3", 128), ("e5m2", 256), ("e4m3", 256), ("e5m2", 128)])
def test_verify_shapes(kv, D, T, g, P):
    contexts = (max(1, T - 3), T, 127, 128, 129, 700)
    sp = workloads.CaseSpec("verify-matrix", contexts=contexts, num_q_tokens=T, num_q_heads=g * 2, num_kv_heads=2,
                            head_dim=D, page_size=P, kv_dtype=kv, seed=31 + T * 10 + g)
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
