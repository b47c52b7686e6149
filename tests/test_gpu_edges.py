"""Edge cases and shape coverage of the CUDA path against the oracle."""

import numpy as np
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


def spec(kv, T, g, Hkv, D, P, contexts, **kw):
    return workloads.CaseSpec("edge", contexts=tuple(contexts), num_q_tokens=T, num_q_heads=g * Hkv,
                              num_kv_heads=Hkv, head_dim=D, page_size=P, kv_dtype=kv, seed=kw.pop("seed", 5), **kw)


def run_and_compare(sp, splits=(0, 3)):
    case = workloads.make_case(sp)
    kc, vc = oracle_caches(case)
    o, l = oracle_attention(case, kc, vc)
    g = GpuCase(case)
    torch.cuda.synchronize()
    assert np.array_equal(g.k_cache.cpu().numpy().view(np.uint8), kc.view(np.uint8))
    for s in splits:
        out, lse = g.decode(num_splits=s)
        torch.cuda.synchronize()
        assert_close(out, lse, o, l)
    assert pf.pfkv_device_errors(clear=True) == 0


@pytest.mark.parametrize("P", [16, 32, 64, 128, 256, 2048])
@pytest.mark.parametrize("kv,D", [("e4m3", 128), ("e5m2", 256), ("fp16", 256), ("fp16", 128)])
def test_page_sizes(kv, D, P):
    run_and_compare(spec(kv, 1, 4, 2, D, P, (300, 97, 1025)))


@pytest.mark.parametrize("T,g", [(1, 1), (1, 8), (2, 3), (3, 5), (5, 2), (8, 1), (8, 6), (8, 8), (4, 16)])
def test_group_and_query_token_counts(T, g):
    run_and_compare(spec("e4m3", T, g, 2, 128, 16, (200, 77, 130)))


@pytest.mark.parametrize("kv", ["e4m3", "e5m2", "fp16"])
def test_q8_verify_head_dim_256_ragged(kv):
    run_and_compare(spec(kv, 8, 6, 2, 256, 64, (8, 9, 63, 64, 65, 700)), splits=(0, 1, 5))


def test_short_and_empty_sequences():
    # seq_len 0 (empty), below T, exactly T, one more, tile boundaries
    run_and_compare(spec("e4m3", 4, 2, 2, 128, 16, (0, 2, 4, 5, 64, 65, 128, 129)), splits=(0, 1, 2))


def test_single_key():
    run_and_compare(spec("e5m2", 1, 4, 2, 128, 16, (1, 1, 1)), splits=(0, 1))


def test_outliers_and_uniform_v():
    run_and_compare(spec("e4m3", 1, 6, 4, 256, 2048, (3000,), v_dist="uniform", k_outlier_frac=0.01))


def test_zero_sequences_is_a_no_op():
    case = workloads.make_case(spec("e4m3", 1, 4, 2, 128, 16, (40,)))
    g = GpuCase(case)
    q = torch.empty((0, 8, 128), dtype=torch.float16, device="cuda")
    out = torch.empty_like(q)
    lse = torch.empty((0, 8), dtype=torch.float32, device="cuda")
    pf.pfkv_paged_attention_decode(out, lse, q, g.k_cache, g.v_cache, g.block_table[:0],
                                   g.seq_lens[:0], 1, 2, 16, "e4m3", g.k_scale, g.v_scale, 0.1, 40)
    torch.cuda.synchronize()


def test_bad_block_id_is_flagged_not_faulted():
    case = workloads.make_case(spec("e4m3", 1, 4, 2, 128, 16, (100, 50)))
    g = GpuCase(case)
    bt = g.block_table.clone()
    bt[1, 0] = case.num_blocks + 7  # outside the pool
    g.decode(num_splits=1, block_table=bt)
    flags = pf.pfkv_device_errors(clear=True)
    assert flags & pf.PFKV_DEVERR_BLOCK_ID
    assert pf.pfkv_device_errors(clear=True) == 0


def test_seq_len_beyond_capacity_is_flagged_and_clamped():
    case = workloads.make_case(spec("e5m2", 1, 4, 2, 128, 16, (100, 50)))
    g = GpuCase(case)
    sl = g.seq_lens.clone()
    sl[0] = 10 ** 6
    g.decode(num_splits=1, seq_lens=sl)
    assert pf.pfkv_device_errors(clear=True) & pf.PFKV_DEVERR_SEQ_LEN


def test_bad_slot_is_flagged_and_skipped():
    case = workloads.make_case(spec("e4m3", 1, 4, 2, 128, 16, (20,)))
    g = GpuCase(case)
    before = g.k_cache.clone()
    bad = np.array([case.num_blocks * 16 + 3, -1], dtype=np.int64)
    g.append(case.k_fill[:2], case.v_fill[:2], bad)
    assert pf.pfkv_device_errors(clear=True) & pf.PFKV_DEVERR_SLOT
    assert torch.equal(before, g.k_cache)


def test_host_rejections_with_real_buffers():
    case = workloads.make_case(spec("e4m3", 1, 4, 2, 128, 16, (3000,)))
    g = GpuCase(case)
    s = case.spec
    need = pf.pfkv_decode_workspace_bytes(1, 1, 8, 2, 128, 16, "e4m3", 3000, 4)
    assert need > 0
    small = torch.empty(need - 16, dtype=torch.uint8, device="cuda")
    out = torch.empty_like(g.q)
    lse = torch.empty(g.q.shape[:2], dtype=torch.float32, device="cuda")
    with pytest.raises(pf.PfkvError) as ei:
        pf.pfkv_paged_attention_decode(out, lse, g.q, g.k_cache, g.v_cache, g.block_table, g.seq_lens, 1, 2, 16,
                                       "e4m3", g.k_scale, g.v_scale, 0.1, 3000, 4, small)
    assert ei.value.status == pf.PFKV_ERR_WORKSPACE
    with pytest.raises(pf.PfkvError) as ei:
        pf.pfkv_paged_attention_decode(out, lse, g.q, g.k_cache, g.v_cache, g.block_table, g.seq_lens, 1, 2, 16,
                                       "e4m3", None, None, 0.1, 3000, 1, None)
    assert ei.value.status == pf.PFKV_ERR_INVALID_ARG


@pytest.mark.parametrize("kv,T,g,D", [("e5m2", 8, 6, 256), ("e4m3", 8, 6, 128), ("e4m3", 1, 4, 256), ("fp16", 2, 4, 256)])
def test_out_8_byte_aligned_and_q_alignment_checked(kv, T, g, D):
    # the ABI asks 8-byte alignment of out and 16-byte alignment of q: out at 8 bytes past a
    # 16-byte boundary is served; such a q is refused on the host, before anything is enqueued
    case = workloads.make_case(spec(kv, T, g, 2, D, 64, (700, 129, 5)))
    kc, vc = oracle_caches(case)
    o_ref, l_ref = oracle_attention(case, kc, vc)
    gc = GpuCase(case)
    n = gc.q.numel()
    out_buf = torch.full((n + 4,), float("nan"), dtype=torch.float16, device="cuda")
    out8 = out_buf[4:].view(gc.q.shape)
    assert out8.data_ptr() % 16 == 8
    lse = torch.full(gc.q.shape[:2], float("nan"), dtype=torch.float32, device="cuda")
    s = case.spec
    msl = int(case.seq_lens.max())
    ws = torch.empty(max(pf.pfkv_decode_workspace_bytes(case.B, T, s.num_q_heads, 2, D, 64, kv, msl, 0), 16),
                     dtype=torch.uint8, device="cuda")

    def call(q, out):
        pf.pfkv_paged_attention_decode(out, lse, q, gc.k_cache, gc.v_cache, gc.block_table, gc.seq_lens, T, 2, 64,
                                       kv, gc.k_scale, gc.v_scale, float(case.softmax_scale), msl, 0, ws)

    call(gc.q, out8)
    torch.cuda.synchronize()
    assert_close(out8, lse, o_ref, l_ref)
    q_buf = torch.empty(n + 4, dtype=torch.float16, device="cuda")
    q8 = q_buf[4:].view(gc.q.shape)
    assert q8.data_ptr() % 16 == 8
    with pytest.raises(pf.PfkvError):
        call(q8, out8)
    assert pf.pfkv_device_errors(clear=True) == 0
