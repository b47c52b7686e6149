"""Structure of the seeded synthetic inputs (CPU only)."""

import numpy as np
import pytest

from paged_fp8_kv_cache_gb300 import workloads


SMALL5 = workloads.small_spec(5, contexts=("loguniform", 64, 2048, 64))


@pytest.mark.parametrize("spec", [workloads.CONFIGS[1], workloads.CONFIGS[2], SMALL5], ids=["1", "2", "5-small"])
def test_deterministic_and_well_formed(spec):
    a = workloads.make_case(spec)
    b = workloads.make_case(spec)
    assert np.array_equal(a.q.view(np.uint16), b.q.view(np.uint16))
    assert np.array_equal(a.block_table, b.block_table)
    s = a.spec
    P = s.page_size
    used = a.block_table[a.block_table >= 0]
    assert len(np.unique(used)) == used.size, "a page is shared"
    assert used.max() < a.num_blocks
    for bb in range(a.B):
        npg = -(-int(a.seq_lens[bb]) // P)
        assert np.all(a.block_table[bb, :npg] >= 0) and np.all(a.block_table[bb, npg:] == -1)
    all_slots = np.concatenate([a.slot_fill, a.slot_new])
    assert len(np.unique(all_slots)) == all_slots.size
    assert a.k_fill.shape == (int(a.cached.sum()), s.num_kv_heads, s.head_dim)
    if s.kv_dtype != "fp16":
        fmax = workloads.FMT_MAX[s.kv_dtype]
        kam = max(np.abs(a.k_fill).max(), np.abs(a.k_new).max() if a.k_new.size else 0)
        assert a.k_scale == np.float32(float(kam) / fmax)


def test_config5_shape():
    c = workloads.make_case(SMALL5)
    assert c.B == 64 and np.all(c.cached >= 64) and np.all(c.cached < 2048)
    assert np.all(c.seq_lens == c.cached + 1)
    pages = -(-c.seq_lens.astype(np.int64) // 16)
    assert c.num_blocks == int(np.ceil(1.25 * pages.sum()))


def test_outlier_rows_exact_count():
    spec = workloads.small_spec(3, contexts=(4096,))
    c = workloads.make_case(spec)
    # K ~ N(0,1) -> |k| > 6 is (almost) only reachable through the x8 rows;
    # the rows hit are exactly floor(1% of rows) many distinct rows
    n_rows = int(np.floor(0.01 * 4096 * 4))
    rows = c.k_fill.reshape(-1, 256).astype(np.float32)
    big = np.abs(rows).max(axis=1) > 8.0
    assert big.sum() <= n_rows and big.sum() >= 0.9 * n_rows
