"""Zeroing of reused KV blocks through the C ABI against the oracle: listed blocks become all
zero bytes in both pools, every other byte is unchanged, negative ids are skipped, and an id past
the pool is skipped and reported in the device error word."""

import numpy as np
import pytest
import torch

from oracle import append as oappend
from paged_fp8_kv_cache_gb300 import binding as pf

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _lib(pflib):
    pf.pfkv_device_errors(clear=True)
    yield


def _pools(kv, nb, hkv, page, d, seed):
    rng = np.random.default_rng(seed)
    if kv == "fp16":
        k = rng.integers(0, 1 << 16, size=(nb, hkv, page, d), dtype=np.uint16).view(np.float16)
        v = rng.integers(0, 1 << 16, size=(nb, hkv, page, d), dtype=np.uint16).view(np.float16)
    else:
        k = rng.integers(0, 256, size=(nb, hkv, page, d), dtype=np.uint8)
        v = rng.integers(0, 256, size=(nb, hkv, page, d), dtype=np.uint8)
    return k, v


@pytest.mark.parametrize("kv", ["fp16", "e4m3", "e5m2"])
@pytest.mark.parametrize("nb,hkv,page,d", [(40, 2, 16, 128), (6, 4, 2048, 256)])
def test_zero_blocks_matches_oracle(kv, nb, hkv, page, d):
    k, v = _pools(kv, nb, hkv, page, d, seed=nb + d)
    ids = np.array([3, -1, nb - 1, 3, 0, -7], dtype=np.int32)
    gk, gv = torch.from_numpy(k.copy()).cuda(), torch.from_numpy(v.copy()).cuda()
    pf.pfkv_kv_cache_zero_blocks(gk, gv, torch.from_numpy(ids).cuda(), kv)
    torch.cuda.synchronize()
    oappend.zero_blocks(k, v, ids)
    assert np.array_equal(gk.cpu().numpy().view(np.uint8), k.view(np.uint8))
    assert np.array_equal(gv.cpu().numpy().view(np.uint8), v.view(np.uint8))
    assert pf.pfkv_device_errors(clear=True) == 0


def test_zero_blocks_reports_an_id_past_the_pool():
    k, v = _pools("e4m3", 8, 2, 16, 128, seed=3)
    ids = np.array([2, 8, 1000], dtype=np.int32)  # 8 and 1000 are past the pool
    gk, gv = torch.from_numpy(k.copy()).cuda(), torch.from_numpy(v.copy()).cuda()
    pf.pfkv_kv_cache_zero_blocks(gk, gv, torch.from_numpy(ids).cuda(), "e4m3")
    torch.cuda.synchronize()
    oappend.zero_blocks(k, v, ids)
    assert np.array_equal(gk.cpu().numpy(), k) and np.array_equal(gv.cpu().numpy(), v)
    assert pf.pfkv_device_errors(clear=True) == pf.PFKV_DEVERR_BLOCK_ID


def test_zero_blocks_empty_list_is_a_no_op():
    k, v = _pools("e5m2", 4, 2, 16, 128, seed=4)
    gk, gv = torch.from_numpy(k.copy()).cuda(), torch.from_numpy(v.copy()).cuda()
    pf.pfkv_kv_cache_zero_blocks(gk, gv, torch.zeros(0, dtype=torch.int32, device="cuda"), "e5m2")
    torch.cuda.synchronize()
    assert np.array_equal(gk.cpu().numpy(), k) and np.array_equal(gv.cpu().numpy(), v)
