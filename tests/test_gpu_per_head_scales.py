"""One static scale per KV head (PFKV_KV_SCALES_PER_HEAD) on KV heads of different magnitude:
the appended FP8 bytes bit-exact against the oracle, and attention within tolerance on both
kernels (mma.sync decode kernel, tcgen05 grouped verifier), with the automatic split plan and
explicit ranges; and the per-tensor call on the same cache bytes as a cross-check of the flag.

The tolerances are the unit-scale ones (2e-3 on the fp16 output, 1e-4 on the LSE) taken in each
head's own units: KV head h's K and V are its unit-scale values times gain_h, so its outputs are
gain_h times larger (and so is their fp16 rounding) and its logits gain_h times larger (and so is
the rounding of their fp32 sums); outputs are compared after dividing by gain_h, LSEs against
1e-4 * max(1, gain_h)."""

import numpy as np
import pytest
import torch

from paged_fp8_kv_cache_gb300 import binding as pf
from paged_fp8_kv_cache_gb300 import workloads
from tests.gpu_helpers import GpuCase
from tests.oracle_helpers import oracle_attention, oracle_caches

pytestmark = pytest.mark.gpu

GAINS = (0.25, 4.0, 1.0, 2.0)
# (kv dtype, head_dim, query tokens, group size, KV heads, page size)
SHAPES = [
    ("e4m3", 128, 1, 4, 4, 16),     # 4 rows: decode kernel
    ("e5m2", 256, 2, 4, 2, 2048),   # 8 rows: decode kernel
    ("e5m2", 256, 8, 6, 2, 2048),   # 48 rows: tcgen05 verify
    ("e4m3", 128, 4, 8, 4, 16),     # 32 rows: tcgen05 verify
]


@pytest.fixture(autouse=True)
def _lib(pflib):
    pf.pfkv_device_errors(clear=True)
    yield
    assert pf.pfkv_device_errors(clear=True) == 0


@pytest.mark.parametrize("kv,D,T,g,hkv,P", SHAPES)
def test_per_head_scales(kv, D, T, g, hkv, P):
    sp = workloads.CaseSpec("per-head", contexts=(max(1, T - 1), 130, 1500), num_q_tokens=T, num_q_heads=g * hkv,
                            num_kv_heads=hkv, head_dim=D, page_size=P, kv_dtype=kv, seed=5 + D + T * g,
                            append_new=T, scale_per_head=True, head_gain=GAINS)
    case = workloads.make_case(sp)
    assert np.asarray(case.k_scale).shape == (hkv,)
    kc, vc = oracle_caches(case)
    o_ref, l_ref = oracle_attention(case, kc, vc)
    gc = GpuCase(case)
    torch.cuda.synchronize()
    assert np.array_equal(gc.k_cache.cpu().numpy(), kc)
    assert np.array_equal(gc.v_cache.cpu().numpy(), vc)
    gain = np.array([GAINS[(h // g) % len(GAINS)] for h in range(g * hkv)])  # of query head h's KV head
    for splits in (0, 3):
        out, lse = gc.decode(num_splits=splits)
        torch.cuda.synchronize()
        o = out.float().cpu().numpy().astype(np.float64)
        l = lse.cpu().numpy().astype(np.float64)
        ok = np.isfinite(l_ref)
        assert np.array_equal(np.isneginf(l), np.isneginf(l_ref))
        assert np.all(o[~ok] == 0)
        do = np.abs((o - o_ref) / gain[None, :, None]).max()
        dl = (np.abs(l - l_ref) / np.maximum(1.0, gain)[None, :])[ok].max()
        assert do <= 2e-3, f"max |out - oracle| / gain = {do:.3e}"
        assert dl <= 1e-4, f"max |lse - oracle| / max(1, gain) = {dl:.3e}"


def test_per_head_flag_with_equal_scales_matches_per_tensor():
    # the same cache and one scale per KV head, all equal to the pool's: the same outputs, bitwise
    sp = workloads.small_spec(2, contexts=(700, 3000))
    case = workloads.make_case(sp)
    gc = GpuCase(case)
    out1, lse1 = gc.decode(num_splits=0)
    hkv = sp.num_kv_heads
    gc.k_scale = gc.k_scale.repeat(hkv).contiguous()
    gc.v_scale = gc.v_scale.repeat(hkv).contiguous()
    out2, lse2 = gc.decode(num_splits=0)
    torch.cuda.synchronize()
    assert torch.equal(out1, out2) and torch.equal(lse1, lse2)
