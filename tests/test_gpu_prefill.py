"""Chunked prefill over the paged FP8 cache (pfkv_paged_attention with many query tokens per
sequence, causal): every token of a prompt chunk attends to the cached context and to the
chunk's earlier tokens ("1Cat-vLLM 1.5.0", "Flash-V100 long-context improvements": the
long-prefill GQA path that packs the heads of a group into wider tensor-core work). The chunk
is cut into slabs of up to 64 rows (tokens x the group's heads) per CTA.

Reduced sizes compare every row with the oracle; chunks of 128 / 512 / 2048 tokens over 32K /
64K / 128K contexts compare a seeded sample of query tokens (slab boundaries included) of every
KV head.
"""

import numpy as np
import pytest
import torch

from oracle import attention as oatt
from paged_fp8_kv_cache_gb300 import binding as pf
from paged_fp8_kv_cache_gb300 import workloads
from tests.gpu_helpers import GpuCase, assert_close
from tests.oracle_helpers import head_tables, oracle_caches, unit_caches

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _lib(pflib):
    pf.pfkv_device_errors(clear=True)
    yield
    assert pf.pfkv_device_errors(clear=True) == 0


def spec(kv, T, g, Hkv, D, P, contexts, seed=31):
    return workloads.CaseSpec("prefill", contexts=tuple(contexts), num_q_tokens=T, num_q_heads=g * Hkv,
                              num_kv_heads=Hkv, head_dim=D, page_size=P, kv_dtype=kv, seed=seed)


SMALL = {
    # GQA-6 on FP8: 10-token slabs of 60 rows on the tcgen05 kernel (64-row tile, 4 padding rows)
    "e4m3-g6-T128": (spec("e4m3", 128, 6, 4, 256, 64, (1500, 300)), True, 0),
    # MHA: 64-token slabs
    "e5m2-g1-T200": (spec("e5m2", 200, 1, 8, 128, 16, (700, 210)), True, 0),
    # GQA-8: 8-token slabs
    "e4m3-g8-T64-window": (spec("e4m3", 64, 8, 4, 256, 128, (2000,)), False, 100),
    # fp16 cache: the decode kernel with four 16-row groups per CTA
    "fp16-g4-T100": (spec("fp16", 100, 4, 4, 128, 32, (400, 150)), True, 0),
    # the first chunk of a prompt: the chunk is the whole sequence (a causal triangle)
    "e5m2-g6-first-chunk": (spec("e5m2", 256, 6, 2, 256, 2048, (256,)), True, 0),
}


@pytest.mark.parametrize("name", list(SMALL))
def test_prefill_matches_oracle(name):
    sp, causal, window = SMALL[name]
    case = workloads.make_case(sp)
    kc, vc = oracle_caches(case)
    o_ref, l_ref = oatt.paged_attention(case.q, kc, vc, case.block_table, case.seq_lens, sp.num_q_tokens,
                                        sp.num_kv_heads, sp.page_size, sp.kv_dtype, case.k_scale, case.v_scale,
                                        case.softmax_scale, causal=causal, window=window)
    g = GpuCase(case)
    for splits in (0, 1, 2):
        out, lse = g.attention(causal=causal, window=window, num_splits=splits)
        torch.cuda.synchronize()
        assert_close(out, lse, o_ref, l_ref)


@pytest.mark.parametrize("T,N", [(128, 32768), (512, 65536), (2048, 131072)])
def test_prefill_chunk_at_long_context(T, N):
    """A chunk of T prompt tokens whose last token is at position N - 1 (E4M3, Hq24/Hkv4, D256,
    2048-token pages), in the automatic launch configuration; sampled tokens of every KV head."""
    sp = spec("e4m3", T, 6, 4, 256, 2048, (N,), seed=T)
    case = workloads.make_case(sp)
    g = GpuCase(case)
    out, lse = g.attention(causal=True)
    torch.cuda.synchronize()
    rng = np.random.default_rng(T)
    ts = 10  # tokens per slab at a group of 6
    pick = sorted(set([0, 1, ts - 1, ts, T - ts, T - 1] + list(rng.choice(T, 10, replace=False))))
    units = [(0, h) for h in range(sp.num_kv_heads)]
    kc, vc = unit_caches(case, units, head_tables(case))
    o_ref, l_ref = oatt.paged_attention(case.q, kc, vc, case.block_table, case.seq_lens, T, sp.num_kv_heads,
                                        sp.page_size, sp.kv_dtype, case.k_scale, case.v_scale, case.softmax_scale,
                                        causal=True, tokens=pick)
    assert_close(out, lse, o_ref, l_ref, rows=pick)
