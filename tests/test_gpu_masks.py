"""Parity of the masked attention (pfkv_paged_attention: causal or not, sliding window) with the
oracle, on both kernels: the mma.sync decode kernel (up to 16 rows per KV head, or an fp16
cache) and the tcgen05 verifier (FP8, more rows). Windows span a single key, tile boundaries
(64 and 128 keys), one long window and one longer than every sequence; sequences are ragged and
include one shorter than the query block. The non-causal sliding window is the draft attention
of a block-diffusion drafter ("1Cat-vLLM 1.5.0", "Production DFlash2 on V100"); its cost must not
grow with the context, which tests/test_gpu_masks.py::test_window_reads_only_the_window checks
through the plan.
"""

import pytest
import torch

from paged_fp8_kv_cache_gb300 import binding as pf
from paged_fp8_kv_cache_gb300 import workloads
from oracle import attention as oatt
from tests.gpu_helpers import GpuCase, assert_close
from tests.oracle_helpers import oracle_caches

pytestmark = pytest.mark.gpu

KERNELS = {
    # 16 rows per KV head: the decode kernel with two 8-row tiles per warp
    "decode-e4m3-16rows": dict(kv="e4m3", T=8, g=2, Hkv=2, D=128, P=16, contexts=(5000, 130, 8, 1)),
    # 8 rows: the decode kernel with one 8-row tile, D 256
    "decode-e5m2-8rows": dict(kv="e5m2", T=4, g=2, Hkv=2, D=256, P=2048, contexts=(4500, 70)),
    # 48 rows on FP8: the tcgen05 verifier (a q8 draft block of a GQA-6 model)
    "verify-e5m2-48rows": dict(kv="e5m2", T=8, g=6, Hkv=2, D=256, P=64, contexts=(5000, 130, 9)),
    # fp16 cache, 24 rows: the decode kernel with row groups
    "decode-fp16-24rows": dict(kv="fp16", T=8, g=3, Hkv=2, D=128, P=32, contexts=(3000, 200)),
}
WINDOWS = [1, 64, 127, 128, 4096, 10 ** 6]

_cache = {}


def prepared(name):
    if name not in _cache:
        k = dict(KERNELS[name])
        sp = workloads.CaseSpec(name, contexts=k.pop("contexts"), num_q_tokens=k.pop("T"),
                                num_q_heads=k["g"] * k["Hkv"], num_kv_heads=k["Hkv"], head_dim=k["D"],
                                page_size=k["P"], kv_dtype=k["kv"], seed=77)
        case = workloads.make_case(sp)
        kc, vc = oracle_caches(case)
        _cache[name] = (case, kc, vc, GpuCase(case))
    return _cache[name]


@pytest.fixture(autouse=True)
def _lib(pflib):
    pf.pfkv_device_errors(clear=True)
    yield
    assert pf.pfkv_device_errors(clear=True) == 0


@pytest.mark.parametrize("causal", [True, False], ids=["causal", "noncausal"])
@pytest.mark.parametrize("window", WINDOWS)
@pytest.mark.parametrize("name", list(KERNELS))
def test_mask_matches_oracle(name, window, causal):
    case, kc, vc, g = prepared(name)
    s = case.spec
    o_ref, l_ref = oatt.paged_attention(case.q, kc, vc, case.block_table, case.seq_lens, s.num_q_tokens,
                                        s.num_kv_heads, s.page_size, s.kv_dtype, case.k_scale, case.v_scale,
                                        case.softmax_scale, causal=causal, window=window)
    for splits in (0, 1, 3):
        out, lse = g.attention(causal=causal, window=window, num_splits=splits)
        torch.cuda.synchronize()
        assert_close(out, lse, o_ref, l_ref)


def test_decode_entry_point_equals_the_causal_unwindowed_mask():
    case, kc, vc, g = prepared("verify-e5m2-48rows")
    o1, l1 = g.decode(num_splits=3)
    o2, l2 = g.attention(causal=True, window=0, num_splits=3)
    torch.cuda.synchronize()
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(l1.view(torch.int32), l2.view(torch.int32))


@pytest.mark.parametrize("kv,T,g", [("e5m2", 8, 6), ("e4m3", 1, 4)])
def test_window_reads_only_the_window(kv, T, g):
    """The key ranges of a windowed call cover the window (plus the query block and one tile),
    whatever the context: the same plan at 32K and at 256K keys."""
    plans = [pf.pfkv_attention_plan(1, T, 4 * g, 4, 256, 2048, kv, n, False, 4096, 0) for n in (32768, 262144)]
    assert plans[0] == plans[1]
    S, C = plans[0]
    assert S * C <= 4096 + T + 2 * 128 + C
