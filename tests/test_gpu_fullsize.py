"""The five benchmark workloads and the extension workloads (q16 verify, one scale per KV
head, the draft's non-causal sliding window at 32K and 256K keys, a 2048-token prefill chunk at
128K keys) at full size, in the launch configuration the benchmark times (automatic split
plan), checked against the oracle.

* Cache bytes: every byte the append kernel wrote, over every token of the workload, compared
  chunk by chunk with the oracle's quantisation of the same fp16 inputs (read off a table of
  the oracle's quantise over all fp16 values; see tests/oracle_helpers.py).
* Attention: the oracle computes whole (sequence, KV head) units on its own caches (built from
  the fp16 inputs, not from GPU bytes); every unit of the small workloads is checked, a seeded
  sample of units of the large ones (every row and head-dim element of each sampled unit).
With one scale per KV head (heads of different magnitude) the tolerances are taken in each
head's units: outputs divided by the head's gain, LSEs against 1e-4 * max(1, gain).
"""

import numpy as np
import pytest
import torch

from paged_fp8_kv_cache_gb300 import binding as pf
from paged_fp8_kv_cache_gb300 import workloads
from tests.gpu_helpers import GpuCase
from oracle import attention
from tests.oracle_helpers import expected_rows, head_tables, unit_caches

pytestmark = pytest.mark.gpu

UNITS_CHECKED = {1: None, 2: None, 3: None, 4: 3, 5: 64, 6: 3, 7: None, 8: 4, 9: 3, 10: None}
TOKENS_CHECKED = 24  # query tokens sampled per unit of a prefill chunk (the oracle's cost grows with rows x keys)
CHUNK_TOKENS = 1 << 15


@pytest.fixture(autouse=True)
def _lib(pflib):
    pf.pfkv_device_errors(clear=True)
    yield
    assert pf.pfkv_device_errors(clear=True) == 0


def check_every_cache_byte(g, case, tables):
    """Every token's K and V rows in the GPU pools equal the oracle's quantisation."""
    s = case.spec
    for src_k, src_v, slots in ((case.k_fill, case.v_fill, case.slot_fill),
                                (case.k_new, case.v_new, case.slot_new)):
        for a in range(0, slots.size, CHUNK_TOKENS):
            sl = slots[a:a + CHUNK_TOKENS]
            blk = torch.from_numpy(sl // s.page_size).cuda()
            off = torch.from_numpy(sl % s.page_size).cuda()
            got_k = g.k_cache[blk, :, off, :].cpu().numpy()
            got_v = g.v_cache[blk, :, off, :].cpu().numpy()
            want_k = expected_rows(src_k[a:a + CHUNK_TOKENS], tables, 0)
            want_v = expected_rows(src_v[a:a + CHUNK_TOKENS], tables, 1)
            if s.kv_dtype == "fp16":
                got_k, got_v, want_k, want_v = (x.view(np.uint16) for x in (got_k, got_v, want_k, want_v))
            assert np.array_equal(got_k, want_k), f"K cache bytes differ in tokens {a}..{a + sl.size}"
            assert np.array_equal(got_v, want_v), f"V cache bytes differ in tokens {a}..{a + sl.size}"


@pytest.mark.parametrize("cfg", sorted(workloads.ALL))
def test_full_size_workload(cfg):
    case = workloads.make_case(workloads.ALL[cfg])
    s = case.spec
    g = GpuCase(case)
    out, lse = g.attention(causal=s.causal, window=s.window)
    torch.cuda.synchronize()

    tables = head_tables(case)
    check_every_cache_byte(g, case, tables)

    # attention: every unit (small workloads) or a seeded sample of units, on the oracle's caches
    rng = np.random.default_rng(cfg)
    all_units = [(b, h) for b in range(case.B) for h in range(s.num_kv_heads)]
    n = UNITS_CHECKED[cfg]
    units = all_units if n is None else [all_units[i] for i in rng.choice(len(all_units), n, replace=False)]
    kc, vc = unit_caches(case, units, tables)
    T, g_ = s.num_q_tokens, s.num_q_heads // s.num_kv_heads
    tokens = None
    if T > 16:  # a prefill chunk: slab boundaries, the ends and a seeded sample of its tokens
        ts = 64 // g_
        tokens = sorted(set([0, 1, ts - 1, ts, T - ts - 1, T - 1] +
                            [int(t) for t in rng.choice(T, TOKENS_CHECKED, replace=False)]))
    o_ref, l_ref = attention.paged_attention(case.q, kc, vc, case.block_table, case.seq_lens, T, s.num_kv_heads,
                                             s.page_size, s.kv_dtype, case.k_scale, case.v_scale, case.softmax_scale,
                                             units=units, causal=s.causal, window=s.window, tokens=tokens)
    rows = np.zeros(o_ref.shape[:2], bool)
    for b, kvh in units:
        for t in (range(T) if tokens is None else tokens):
            rows[b * T + t, kvh * g_:(kvh + 1) * g_] = True
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
