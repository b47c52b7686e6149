"""One append call large enough that the append kernel's grid-stride loop iterates (its grid is
capped at 64 CTAs of 256 threads per SM, one thread per 8 elements), checked byte for byte
against the oracle's append over the whole pool; a prefill-sized append takes this path."""

import numpy as np
import pytest
import torch

from oracle import append as oappend
from paged_fp8_kv_cache_gb300 import binding as pf

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("kv,n_tok,hkv,d,page,per_head", [
    ("e4m3", 32768, 4, 256, 2048, False),   # 33.5M elements per pool in one call
    ("e5m2", 40000, 8, 128, 16, True),      # 41M elements, one scale per KV head
    ("fp16", 65536, 4, 128, 64, False),    # 33.5M elements
    ("e4m3", 80000, 3, 96, 48, False),     # 23M elements: page size and head dim not powers of two
])
def test_single_large_append_is_bit_exact(pflib, kv, n_tok, hkv, d, page, per_head):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    threads_needed = n_tok * hkv * d // 8
    assert threads_needed > sms * 64 * 256, "the call must make the grid-stride loop iterate"
    rng = np.random.default_rng(n_tok)
    num_blocks = -(-n_tok // page) + 3
    slots = rng.permutation(num_blocks * page)[:n_tok].astype(np.int64)
    slots[rng.random(n_tok) < 0.01] = -1  # skipped tokens
    k16 = rng.standard_normal((n_tok, hkv, d), dtype=np.float32).astype(np.float16)
    v16 = (rng.standard_normal((n_tok, hkv, d), dtype=np.float32) * 3).astype(np.float16)
    if kv == "fp16":
        ks = vs = np.float32(1.0)
    elif per_head:
        fmax = 448.0 if kv == "e4m3" else 57344.0
        ks = (np.abs(k16).max(axis=(0, 2)).astype(np.float32) / np.float32(fmax)).astype(np.float32)
        vs = (np.abs(v16).max(axis=(0, 2)).astype(np.float32) / np.float32(fmax)).astype(np.float32)
    else:
        fmax = 448.0 if kv == "e4m3" else 57344.0
        ks = np.float32(float(np.abs(k16).max()) / fmax)
        vs = np.float32(float(np.abs(v16).max()) / fmax)
    dt_t = torch.float16 if kv == "fp16" else torch.uint8
    dt_n = np.float16 if kv == "fp16" else np.uint8
    shape = (num_blocks, hkv, page, d)
    kc = torch.zeros(shape, dtype=dt_t, device="cuda")
    vc = torch.zeros(shape, dtype=dt_t, device="cuda")
    kst = torch.tensor(np.asarray(ks, np.float32).reshape(-1), device="cuda")
    vst = torch.tensor(np.asarray(vs, np.float32).reshape(-1), device="cuda")
    pf.pfkv_device_errors(clear=True)
    pf.pfkv_kv_cache_append(torch.from_numpy(k16).cuda(), torch.from_numpy(v16).cuda(), kc, vc,
                            torch.from_numpy(slots).cuda(), page, kv, kst, vst)
    torch.cuda.synchronize()
    assert pf.pfkv_device_errors(clear=True) == 0
    okc = np.zeros(shape, dt_n)
    ovc = np.zeros(shape, dt_n)
    oappend.append_bulk(okc, k16, slots, page, ks, kv)
    oappend.append_bulk(ovc, v16, slots, page, vs, kv)
    assert np.array_equal(kc.cpu().numpy().view(np.uint8), okc.view(np.uint8))
    assert np.array_equal(vc.cpu().numpy().view(np.uint8), ovc.view(np.uint8))
