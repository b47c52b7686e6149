"""Pins of the oracle's quantise-and-append step (CPU only)."""

from fractions import Fraction

import numpy as np
import pytest

from oracle import append, fp8
from paged_fp8_kv_cache_gb300 import workloads


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_quantise_division_is_correctly_rounded_fp32(fmt):
    """float64-then-float32 quotient == numpy's IEEE float32 division == exact rounding."""
    rng = np.random.default_rng(3)
    x16 = (rng.standard_normal(50000) * 3).astype(np.float16)
    scale = np.float32(0.0123456)
    q_np32 = (x16.astype(np.float32) / scale).astype(np.float32)  # IEEE fp32 division
    assert np.array_equal(append.quantise(x16, scale, fmt), fp8.encode(q_np32, fmt))
    # exact rational check of the rounding on a sample
    for x in x16[:300]:
        exact = Fraction(float(np.float32(x))) / Fraction(float(scale))
        r = np.float32(float(exact))  # nearest double, then float32
        lo = np.nextafter(r, np.float32(-np.inf), dtype=np.float32)
        hi = np.nextafter(r, np.float32(np.inf), dtype=np.float32)
        d = abs(Fraction(float(r)) - exact)
        assert d <= abs(Fraction(float(lo)) - exact) and d <= abs(Fraction(float(hi)) - exact)


def test_quantise_in_range_never_saturates_with_amax_scale():
    rng = np.random.default_rng(4)
    x16 = rng.standard_normal(10000).astype(np.float16)
    scale = np.float32(float(np.abs(x16).max()) / 448.0)
    codes = append.quantise(x16, scale, "e4m3")
    vals = fp8.decode(codes, "e4m3") * float(scale)
    # relative error of a 3-bit mantissa round-to-nearest: <= 2^-4 for normals
    big = np.abs(x16.astype(np.float64)) > 2.0 ** -6 * float(scale)
    rel = np.abs(vals[big] - x16[big]) / np.abs(x16[big].astype(np.float64))
    assert rel.max() <= 2.0 ** -4 + 1e-12


@pytest.mark.parametrize("kv", ["fp16", "e4m3", "e5m2"])
def test_append_layout_and_skip(kv):
    P, Hkv, D, nb = 4, 3, 8, 5
    rng = np.random.default_rng(5)
    n = 9
    new = rng.standard_normal((n, Hkv, D)).astype(np.float16)
    slots = rng.permutation(nb * P)[:n].astype(np.int64)
    slots[2] = -1
    dt = np.float16 if kv == "fp16" else np.uint8
    cache = np.zeros((nb, Hkv, P, D), dt)
    append.append(cache, new, slots, P, np.float32(0.01), kv)
    for i in range(n):
        s = slots[i]
        if s < 0:
            continue
        got = cache[s // P, :, s % P, :]
        if kv == "fp16":
            assert np.array_equal(got.view(np.uint16), new[i].view(np.uint16))
        else:
            assert np.array_equal(got, append.quantise(new[i], np.float32(0.01), kv))
    # untouched slots stay zero
    touched = {int(s) for s in slots if s >= 0}
    for s in range(nb * P):
        if s not in touched:
            assert not cache[s // P, :, s % P, :].any()


@pytest.mark.parametrize("cfg", [1, 2, 5])
def test_append_bulk_equals_token_loop(cfg):
    spec = workloads.small_spec(cfg, contexts=(37, 5, 64) if cfg != 5 else ("loguniform", 8, 60, 3))
    case = workloads.make_case(spec)
    dt = np.float16 if spec.kv_dtype == "fp16" else np.uint8
    shape = (case.num_blocks, spec.num_kv_heads, spec.page_size, spec.head_dim)
    a = np.zeros(shape, dt)
    b = np.zeros(shape, dt)
    append.append(a, case.k_fill, case.slot_fill, spec.page_size, case.k_scale, spec.kv_dtype)
    append.append_bulk(b, case.k_fill, case.slot_fill, spec.page_size, case.k_scale, spec.kv_dtype)
    assert np.array_equal(a.view(np.uint8), b.view(np.uint8))


@pytest.mark.parametrize("kv", ["fp16", "e4m3", "e5m2"])
def test_zero_blocks_clears_listed_blocks_only(kv):
    # the reused-block zeroing: listed blocks become all-zero bytes, which decode to +0 in every
    # cache format; every other block keeps its bytes; negative and out-of-pool ids are skipped
    from oracle import append as oappend, fp8
    rng = np.random.default_rng(5)
    shape = (9, 2, 4, 8)
    if kv == "fp16":
        kc0 = rng.integers(0, 1 << 16, size=shape, dtype=np.uint16).view(np.float16)
        vc0 = rng.integers(0, 1 << 16, size=shape, dtype=np.uint16).view(np.float16)
    else:
        kc0 = rng.integers(0, 256, size=shape, dtype=np.uint8)
        vc0 = rng.integers(0, 256, size=shape, dtype=np.uint8)
    kc, vc = kc0.copy(), vc0.copy()
    ids = [3, -1, 7, 3, 9, 120, 0]
    oappend.zero_blocks(kc, vc, ids)
    listed = {0, 3, 7}
    for b in range(shape[0]):
        if b in listed:
            assert not kc[b].view(np.uint8).any() and not vc[b].view(np.uint8).any()
        else:
            assert np.array_equal(kc[b].view(np.uint8), kc0[b].view(np.uint8))
            assert np.array_equal(vc[b].view(np.uint8), vc0[b].view(np.uint8))
    if kv == "fp16":
        z = np.zeros(1, np.uint16).view(np.float16)[0]
        assert z == 0 and not np.signbit(z)
    else:
        fmt = fp8.E4M3 if kv == "e4m3" else fp8.E5M2
        z = fp8.decode(np.zeros(1, np.uint8), fmt)[0]
        assert z == 0 and not np.signbit(z)


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_quantise_table_lookup_is_the_oracle_call(fmt):
    """The full-size GPU tests read the oracle's quantisation off a table of all 65536 fp16
    inputs; a lookup must equal the direct call on any finite input."""
    from tests.oracle_helpers import quantise_table
    rng = np.random.default_rng(11)
    scale = np.float32(0.0371)
    tab = quantise_table(scale, fmt)
    x = np.concatenate([(rng.standard_normal(20000) * 40).astype(np.float16),
                        np.array([0.0, -0.0, 65504.0, -65504.0, 6e-8, -6e-8], np.float16)])
    assert np.array_equal(tab[x.view(np.uint16)], append.quantise(x, scale, fmt))
    every = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16).view(np.float16)
    fin = np.isfinite(every)
    assert np.array_equal(tab[fin], append.quantise(every[fin], scale, fmt))


@pytest.mark.parametrize("cfg,heads", [(5, False), (3, True)])
def test_unit_caches_equal_the_oracle_append(cfg, heads):
    """Per-unit host caches built by table lookup hold the bytes oracle.append writes."""
    from tests.oracle_helpers import head_tables, oracle_caches, unit_caches
    over = {"contexts": ("loguniform", 30, 300, 6)} if cfg == 5 else {"contexts": (2100,)}
    if heads:
        over.update(scale_per_head=True, head_gain=(0.5, 2.0, 1.0, 4.0))
    case = workloads.make_case(workloads.small_spec(cfg, **over))
    kc, vc = oracle_caches(case)
    units = [(b, h) for b in range(case.B) for h in range(case.spec.num_kv_heads)][::3]
    uk, uv = unit_caches(case, units, head_tables(case))
    P = case.spec.page_size
    for b, h in units:
        n = int(case.seq_lens[b])
        pages = case.block_table[b, :-(-n // P)]
        a = kc[pages, h].reshape(-1, case.spec.head_dim)[:n]
        assert np.array_equal(uk[pages, h].reshape(-1, case.spec.head_dim)[:n], a)
        assert np.array_equal(uv[pages, h].reshape(-1, case.spec.head_dim)[:n],
                              vc[pages, h].reshape(-1, case.spec.head_dim)[:n])
