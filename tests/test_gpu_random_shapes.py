"""Seeded random shapes through pfkv_paged_attention, each against the oracle: cache dtype, head
dim, page size, GQA group, query tokens (decode, verify and prefill slabs), ragged and empty
sequences, causal or not, sliding windows and forced split counts drawn together, so that
combinations no hand-written case names (a windowed prefill on the fp16 cache, a 3-head group at
13 tokens on 32-token pages, ...) meet the same 2e-3 / 1e-4 bar as the rest. A second set draws
large ragged decode batches with random masks and split counts, which run on the persistent grid
when their one-CTA-per-range grid would exceed two waves."""

import numpy as np
import pytest
import torch

from oracle import attention as oatt
from paged_fp8_kv_cache_gb300 import binding as pf
from paged_fp8_kv_cache_gb300 import workloads
from tests.gpu_helpers import GpuCase, assert_close
from tests.oracle_helpers import oracle_caches

pytestmark = pytest.mark.gpu

N_CASES = 120
ORACLE_BUDGET = 1.5e9  # multiply-adds the float64 oracle is given per case


def _draw(i):
    rng = np.random.Generator(np.random.PCG64(9000 + i))
    while True:
        kv = ["e4m3", "e5m2", "fp16"][rng.integers(3)]
        D = [128, 256][rng.integers(2)]
        P = [16, 32, 64, 128, 256, 2048][rng.integers(6)]
        Hkv = [1, 2, 4][rng.integers(3)]
        g = [1, 2, 3, 4, 6, 8][rng.integers(6)]
        if rng.random() < 0.75:  # decode / verify: all rows of a KV head in one CTA
            T = min(int(rng.integers(1, 64 // g + 1)), 16)
        else:  # prefill chunk: several query slabs
            T = int(rng.integers(17, 97))
        B = int(rng.integers(1, 6))
        contexts = []
        for _ in range(B):
            u = rng.random()
            contexts.append(0 if u < 0.08 else int(rng.integers(1, 64)) if u < 0.25 else int(rng.integers(64, 3000)))
        causal = bool(rng.random() < 0.7)
        window = 0 if rng.random() < 0.5 else int(rng.integers(1, 2000))
        splits = 0 if rng.random() < 0.6 else int(rng.integers(1, 9))
        N = max(contexts) + T
        if B * T * g * Hkv * N * D * 2 <= ORACLE_BUDGET:
            return dict(kv=kv, D=D, P=P, Hkv=Hkv, g=g, T=T, contexts=tuple(contexts), causal=causal,
                        window=window, splits=splits, seed=9000 + i)


CASES = [_draw(i) for i in range(N_CASES)]


def _id(c):
    return (f"{c['kv']}-D{c['D']}-P{c['P']}-Hkv{c['Hkv']}-g{c['g']}-T{c['T']}-B{len(c['contexts'])}"
            f"-{'c' if c['causal'] else 'nc'}-w{c['window']}-s{c['splits']}")


@pytest.fixture(autouse=True)
def _lib(pflib):
    pf.pfkv_device_errors(clear=True)
    yield
    assert pf.pfkv_device_errors(clear=True) == 0


@pytest.mark.parametrize("c", CASES, ids=[_id(c) for c in CASES])
def test_random_shape_matches_oracle(c):
    # the cached tokens of each sequence, then its T query tokens appended (their K/V are in the
    # cache when the attention runs)
    sp = workloads.CaseSpec("random shape", contexts=c["contexts"], num_q_tokens=c["T"],
                            num_q_heads=c["g"] * c["Hkv"], num_kv_heads=c["Hkv"], head_dim=c["D"],
                            page_size=c["P"], kv_dtype=c["kv"], append_new=c["T"], seed=c["seed"])
    case = workloads.make_case(sp)
    kc, vc = oracle_caches(case)
    o_ref, l_ref = oatt.paged_attention(case.q, kc, vc, case.block_table, case.seq_lens, c["T"], c["Hkv"], c["P"],
                                        c["kv"], case.k_scale, case.v_scale, case.softmax_scale,
                                        causal=c["causal"], window=c["window"])
    g = GpuCase(case)
    out, lse = g.attention(causal=c["causal"], window=c["window"], num_splits=c["splits"])
    torch.cuda.synchronize()
    assert np.array_equal(g.k_cache.cpu().numpy().view(np.uint8), kc.view(np.uint8))
    assert_close(out, lse, o_ref, l_ref)


def _draw_batch(i):
    # large ragged decode batches (one row tile per KV head, so that the call may run the
    # persistent grid) with random masks and split counts
    rng = np.random.Generator(np.random.PCG64(9500 + i))
    kv = ["e4m3", "e5m2", "fp16"][rng.integers(3)]
    D = [128, 256][rng.integers(2)]
    P = [16, 64, 2048][rng.integers(3)]
    Hkv = [2, 4, 8][rng.integers(3)]
    g = [1, 2, 4, 8][rng.integers(4)]
    T = int(rng.integers(1, 8 // g + 1))
    B = int(rng.integers(40, 97))
    contexts = tuple(int(c) for c in np.exp(rng.uniform(0, np.log(3000), size=B)).astype(np.int64) - 1)
    causal = bool(rng.random() < 0.7)
    window = 0 if rng.random() < 0.6 else int(rng.integers(1, 1500))
    splits = int(rng.integers(2, 9))
    return dict(kv=kv, D=D, P=P, Hkv=Hkv, g=g, T=T, contexts=contexts, causal=causal, window=window,
                splits=splits, seed=9500 + i)


BATCHES = [_draw_batch(i) for i in range(16)]


@pytest.mark.parametrize("c", BATCHES, ids=[_id(c) for c in BATCHES])
def test_random_ragged_batch_matches_oracle(c):
    test_random_shape_matches_oracle(c)
