"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Sizes here are ones the oracle finishes in seconds but that still span
several 64-key tiles, several split ranges, and a ragged last tile / page.
Bar: cache bytes bit-exact; |out - oracle| <= 2e-3 (fp16 output of
unit-scale inputs); |lse - oracle| <= 1e-4.
"""

import numpy as np
import pytest
import torch

from oracle import merge
from paged_fp8_kv_cache_gb300 import binding as pf
from paged_fp8_kv_cache_gb300 import workloads
from tests.gpu_helpers import GpuCase, assert_close, to_dev
from tests.oracle_helpers import oracle_attention, oracle_caches

pytestmark = pytest.mark.gpu

SMALL = {
    "c1-tiny-fp16": workloads.CONFIGS[1],
    "c2-batched-e4m3": workloads.CONFIGS[2],
    "c3-long-e4m3-small": workloads.small_spec(3, contexts=(5000,)),
    "c4-verify-q8-e5m2-small": workloads.small_spec(4, contexts=(4100, 2500)),
    "c5-mixed-e4m3-small": workloads.small_spec(5, contexts=("loguniform", 30, 700, 64)),
    "x6-verify-q16-e5m2-small": workloads.small_spec(6, contexts=(4100, 2500)),
}

_cache = {}


def prepared(name):
    if name not in _cache:
        case = workloads.make_case(SMALL[name])
        kc, vc = oracle_caches(case)
        o, l = oracle_attention(case, kc, vc)
        _cache[name] = (case, kc, vc, o, l)
    return _cache[name]


@pytest.fixture(autouse=True)
def _lib(pflib):
    pf.pfkv_device_errors(clear=True)
    yield
    assert pf.pfkv_device_errors(clear=True) == 0


@pytest.mark.parametrize("name", list(SMALL))
def test_append_bit_exact(name):
    case, kc, vc, _, _ = prepared(name)
    g = GpuCase(case)
    torch.cuda.synchronize()
    gk = g.k_cache.cpu().numpy()
    gv = g.v_cache.cpu().numpy()
    assert np.array_equal(gk.view(np.uint8), kc.view(np.uint8))
    assert np.array_equal(gv.view(np.uint8), vc.view(np.uint8))


@pytest.mark.parametrize("splits", [0, 1, 2, 7])
@pytest.mark.parametrize("name", list(SMALL))
def test_decode_matches_oracle(name, splits):
    case, kc, vc, o_ref, l_ref = prepared(name)
    g = GpuCase(case)
    out, lse = g.decode(num_splits=splits)
    torch.cuda.synchronize()
    assert_close(out, lse, o_ref, l_ref)


def test_page_shuffle_is_bitwise_invariant():
    """Moving physical pages (and the block table with them) changes no output bit."""
    case, _, _, _, _ = prepared("c5-mixed-e4m3-small")
    g = GpuCase(case)
    out1, lse1 = g.decode(num_splits=3)
    perm = torch.from_numpy(np.random.default_rng(0).permutation(case.num_blocks)).to("cuda")
    kc2 = torch.empty_like(g.k_cache)
    vc2 = torch.empty_like(g.v_cache)
    kc2[perm] = g.k_cache
    vc2[perm] = g.v_cache
    bt = g.block_table.long()
    bt2 = torch.where(bt >= 0, perm[bt.clamp(min=0)], bt).int()
    out2, lse2 = g.decode(num_splits=3, block_table=bt2, k_cache=kc2, v_cache=vc2)
    torch.cuda.synchronize()
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))
    assert torch.equal(lse1.view(torch.int32), lse2.view(torch.int32))


def test_split_partials_match_oracle_ranges():
    """The workspace holds, per split range, the attention restricted to that range."""
    name = "c3-long-e4m3-small"
    case, kc, vc, _, _ = prepared(name)
    s = case.spec
    g = GpuCase(case)
    S, C = pf.pfkv_decode_plan(case.B, s.num_q_tokens, s.num_q_heads, s.num_kv_heads, s.head_dim, s.page_size,
                               s.kv_dtype, int(case.seq_lens.max()), 3)
    assert S == 3
    g.decode(num_splits=3)
    torch.cuda.synchronize()
    rows = case.B * s.num_q_tokens * s.num_q_heads
    ws = g.last_workspace.view(torch.float32).cpu().numpy()
    o_part = ws[:rows * S * s.head_dim].reshape(rows, S, s.head_dim)
    l_part = ws[rows * S * s.head_dim:rows * S * s.head_dim + rows * S].reshape(rows, S)
    for si in range(S):
        o_r, l_r = oracle_attention(case, kc, vc, token_range=(si * C, (si + 1) * C))
        assert np.abs(o_part[:, si] - o_r.reshape(rows, -1)).max() <= 2e-3
        fin = np.isfinite(l_r.reshape(rows))
        assert np.abs(l_part[:, si][fin] - l_r.reshape(rows)[fin]).max() <= 1e-4
    # and the oracle's own merge of those partials reproduces the full result
    mo, ml = merge.lse_merge(o_part.astype(np.float64), l_part.astype(np.float64))
    o_full, l_full = oracle_attention(case, kc, vc)
    assert np.abs(mo - o_full.reshape(rows, -1)).max() <= 2e-3


@pytest.mark.parametrize("rows,S,D", [(7, 1, 128), (33, 5, 256), (64, 64, 128), (3, 200, 256)])
def test_lse_merge_kernel(rows, S, D):
    rng = np.random.default_rng(rows * S)
    o = rng.standard_normal((rows, S, D)).astype(np.float32)
    l = (rng.standard_normal((rows, S)) * 5).astype(np.float32)
    l[rng.random((rows, S)) < 0.2] = -np.inf  # empty ranges
    l[0, :] = -np.inf  # a row with no key at all
    out = torch.empty((rows, D), dtype=torch.float16, device="cuda")
    lse = torch.empty(rows, dtype=torch.float32, device="cuda")
    pf.pfkv_lse_merge(out, lse, to_dev(o), to_dev(l))
    torch.cuda.synchronize()
    mo, ml = merge.lse_merge(o.astype(np.float64), l.astype(np.float64))
    assert_close(out, lse, mo, ml)
