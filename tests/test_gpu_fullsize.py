"""The five benchmark workloads and the extension workloads (q16 verify, one scale per KV
head) at full size, in the launch configuration the benchmark times (automatic split plan),
checked against the oracle.

The oracle computes whole (sequence, KV head) units; for the large
workloads a seeded sample of units is checked (every row and head-dim
element of each sampled unit), and cache bytes are compared on a seeded
sample of tokens. With one scale per KV head (heads of different magnitude) the tolerances are
taken in each head's units: outputs divided by the head's gain, LSEs against 1e-4 * max(1, gain).
"""

import numpy as np
import pytest
import torch

from oracle import append as oappend
from paged_fp8_kv_cache_gb300 import binding as pf
from paged_fp8_kv_cache_gb300 import workloads
from tests.gpu_helpers import GpuCase
from tests.oracle_helpers import oracle_attention

pytestmark = pytest.mark.gpu

UNITS_CHECKED = {1: None, 2: None, 3: None, 4: 2, 5: 6, 6: 2, 7: None}


@pytest.fixture(autouse=True)
def _lib(pflib):
    pf.pfkv_device_errors(clear=True)
    yield
    assert pf.pfkv_device_errors(clear=True) == 0


def _gather_cache(gpu_cache, case, units):
    """Host copy of the pages the sampled units touch (others stay zero)."""
    s = case.spec
    dt = np.float16 if s.kv_dtype == "fp16" else np.uint8
    host = np.zeros((case.num_blocks, s.num_kv_heads, s.page_size, s.head_dim), dt)
    for b, kvh in units:
        npg = -(-int(case.seq_lens[b]) // s.page_size)
        pages = torch.from_numpy(case.block_table[b, :npg].astype(np.int64)).cuda()
        host[case.block_table[b, :npg], kvh] = gpu_cache[pages, kvh].cpu().numpy()
    return host


@pytest.mark.parametrize("cfg", [1, 2, 3, 4, 5, 6, 7])
def test_full_size_workload(cfg):
    case = workloads.make_case(workloads.ALL[cfg])
    s = case.spec
    g = GpuCase(case)
    out, lse = g.decode()
    torch.cuda.synchronize()

    # cache bytes: sampled tokens against the oracle's quantisation
    rng = np.random.default_rng(cfg)
    all_k = np.concatenate([case.k_fill, case.k_new])
    all_v = np.concatenate([case.v_fill, case.v_new])
    all_slots = np.concatenate([case.slot_fill, case.slot_new])
    pick = rng.choice(all_slots.size, size=min(2048, all_slots.size), replace=False)
    slots = all_slots[pick]
    blk = torch.from_numpy(slots // s.page_size).cuda()
    off = torch.from_numpy(slots % s.page_size).cuda()
    got_k = g.k_cache[blk, :, off, :].cpu().numpy()
    got_v = g.v_cache[blk, :, off, :].cpu().numpy()
    if s.kv_dtype == "fp16":
        assert np.array_equal(got_k.view(np.uint16), all_k[pick].view(np.uint16))
        assert np.array_equal(got_v.view(np.uint16), all_v[pick].view(np.uint16))
    else:
        ks = oappend.head_scales(case.k_scale, s.num_kv_heads)
        vs = oappend.head_scales(case.v_scale, s.num_kv_heads)
        assert np.array_equal(got_k, oappend.quantise(all_k[pick], ks, s.kv_dtype))
        assert np.array_equal(got_v, oappend.quantise(all_v[pick], vs, s.kv_dtype))

    # attention: every unit (small workloads) or a seeded sample of units
    all_units = [(b, h) for b in range(case.B) for h in range(s.num_kv_heads)]
    n = UNITS_CHECKED[cfg]
    units = all_units if n is None else [all_units[i] for i in rng.choice(len(all_units), n, replace=False)]
    kc = _gather_cache(g.k_cache, case, units)
    vc = _gather_cache(g.v_cache, case, units)
    o_ref, l_ref = oracle_attention(case, kc, vc, units=units)
    T, g_ = s.num_q_tokens, s.num_q_heads // s.num_kv_heads
    rows = np.zeros(o_ref.shape[:2], bool)
    for b, kvh in units:
        rows[b * T:(b + 1) * T, kvh * g_:(kvh + 1) * g_] = True
    o = out.float().cpu().numpy().astype(np.float64)
    l = lse.cpu().numpy().astype(np.float64)
    # each query head's KV-head gain (1 without head gains)
    hg = s.head_gain or (1.0,)
    gain = np.array([hg[(h // g_) % len(hg)] for h in range(s.num_q_heads)])[None, :].repeat(o.shape[0], 0)
    do = (np.abs(o - o_ref) / gain[:, :, None])[rows].max()
    dl = (np.abs(l - l_ref) / np.maximum(1.0, gain))[rows].max()
    assert do <= 2e-3, f"max |out - oracle| = {do:.3e}"
    assert dl <= 1e-4, f"max |lse - oracle| = {dl:.3e}"
    # every row is finite (all sequences are non-empty)
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()
