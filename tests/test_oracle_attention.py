"""Pins of the oracle's paged attention and LSE merge (CPU only).

What pins the oracle, none of which is the oracle itself:

* a brute-force restatement (pure-Python loops, ``math.fsum``/``math.exp``,
  gather through the block table key by key) on tiny inputs, all three cache
  dtypes, GQA groups 1-3, 1 or 3 causal query tokens;
* closed forms: constant V gives V; all-zero K gives the mean of the visible
  V and ``lse = ln(#visible)``; one key gives that key's V and logit;
* invariances: permuting physical pages (with the block table), splitting
  the keys and merging, GQA group vs a single head, causal row t vs a
  one-token decode of the shorter sequence;
* planted mistakes: each plausible bug, inserted into a copy of the oracle's
  source, must fail at least one of the pins above.
"""

import inspect
import math
import types

import numpy as np
import pytest

import oracle.attention as oatt
from oracle import append as oappend
from oracle import fp8, merge
from paged_fp8_kv_cache_gb300 import workloads
from tests.oracle_helpers import oracle_caches


def tiny_spec(kv, T=1, g=2, Hkv=2, D=8, P=4, contexts=(13, 27), **kw):
    return workloads.CaseSpec("tiny", contexts=contexts, num_q_tokens=T, num_q_heads=g * Hkv,
                              num_kv_heads=Hkv, head_dim=D, page_size=P, kv_dtype=kv, seed=kw.pop("seed", 99), **kw)


def run(att, case, kc, vc, **kw):
    s = case.spec
    args = dict(q=case.q, k_cache=kc, v_cache=vc, block_table=case.block_table, seq_lens=case.seq_lens,
                num_q_tokens=s.num_q_tokens, num_kv_heads=s.num_kv_heads, page_size=s.page_size,
                kv_dtype=s.kv_dtype, k_scale=case.k_scale, v_scale=case.v_scale,
                softmax_scale=case.softmax_scale)
    args.update(kw)
    return att(**args)


def brute(case, kc, vc, causal=True, window=0):
    """Plain loops over (b, t, h, key, d); shares nothing with the vectorised oracle. A key j
    is visible to query t (position p = n - T + t) when it is not after p (if causal) and not
    W or more positions before it (with a window of W keys)."""
    s = case.spec
    T, Hq, Hkv, D, P = s.num_q_tokens, s.num_q_heads, s.num_kv_heads, s.head_dim, s.page_size
    g = Hq // Hkv
    sm = float(case.softmax_scale)
    ksa = np.asarray(case.k_scale, dtype=np.float32).reshape(-1)
    vsa = np.asarray(case.v_scale, dtype=np.float32).reshape(-1)

    def val(cache, page, kvh, off, d):
        x = cache[page, kvh, off, d]
        return float(x) if s.kv_dtype == "fp16" else fp8.decode_code(int(x), s.kv_dtype)

    out = np.zeros((case.B * T, Hq, D))
    lse = np.zeros((case.B * T, Hq))
    for b in range(case.B):
        n = int(case.seq_lens[b])
        for t in range(T):
            for h in range(Hq):
                kvh = h // g
                ks = float(ksa[kvh % ksa.size])  # one scale per pool, or KV head kvh's
                vs = float(vsa[kvh % vsa.size])
                qv = [float(case.q[b * T + t, h, d]) for d in range(D)]
                p = n - T + t
                keys = [j for j in range(n) if (not causal or j <= p) and (window == 0 or p - j < window)]
                if not keys:
                    out[b * T + t, h] = 0.0
                    lse[b * T + t, h] = -math.inf
                    continue
                logits = []
                for j in keys:
                    page = int(case.block_table[b, j // P])
                    logits.append(sm * math.fsum(qv[d] * val(kc, page, kvh, j % P, d) * ks for d in range(D)))
                m = max(logits)
                w = [math.exp(x - m) for x in logits]
                L = math.fsum(w)
                for d in range(D):
                    acc = math.fsum(w[i] * val(vc, int(case.block_table[b, j // P]), kvh, j % P, d) * vs
                                    for i, j in enumerate(keys))
                    out[b * T + t, h, d] = acc / L
                lse[b * T + t, h] = m + math.log(L)
    return out, lse


BRUTE_CASES = [
    dict(kv="fp16", T=1, g=2, D=4, P=4, contexts=(13, 27)),
    dict(kv="e4m3", T=1, g=3, D=8, P=4, contexts=(1, 40)),
    dict(kv="e5m2", T=3, g=2, D=8, P=16, contexts=(19, 3)),
    dict(kv="e4m3", T=3, g=1, D=4, P=16, contexts=(33,), Hkv=3),
    dict(kv="e5m2", T=1, g=2, D=8, P=4, contexts=(40, 17), v_dist="uniform", k_outlier_frac=0.1),
    dict(kv="e4m3", T=16, g=2, D=4, P=4, contexts=(21, 16)),  # q16 verify: 15 drafts + 1
    # one scale per KV head, heads of different magnitude
    dict(kv="e5m2", T=2, g=2, Hkv=3, D=8, P=4, contexts=(25, 9), scale_per_head=True, head_gain=(0.25, 4.0, 1.0)),
]


# (case, causal, window): the draft masks (sliding window, non-causal) and a prefill-length T
BRUTE_MASK_CASES = [
    (dict(kv="e4m3", T=3, g=2, D=8, P=4, contexts=(19, 7)), False, 0),
    (dict(kv="e5m2", T=8, g=2, D=4, P=4, contexts=(30, 11)), False, 5),
    (dict(kv="fp16", T=4, g=1, D=4, P=16, contexts=(26, 4)), True, 3),
    (dict(kv="e4m3", T=8, g=3, D=4, P=4, contexts=(17,)), True, 1),
    (dict(kv="e5m2", T=16, g=2, D=4, P=4, contexts=(40, 18)), False, 9),
    (dict(kv="e4m3", T=40, g=2, D=4, P=16, contexts=(61, 40)), True, 0),   # a chunk of 40 prompt tokens
    (dict(kv="e5m2", T=40, g=1, D=4, P=4, contexts=(50,)), True, 13),
]


def pin_brute(att):
    for c in BRUTE_CASES:
        case = workloads.make_case(tiny_spec(**dict(c)))
        kc, vc = oracle_caches(case)
        o, l = run(att, case, kc, vc)
        bo, bl = brute(case, kc, vc)
        if not (np.allclose(o, bo, rtol=0, atol=1e-12) and np.allclose(l, bl, rtol=0, atol=1e-12)):
            return False
    for c, causal, window in BRUTE_MASK_CASES:
        case = workloads.make_case(tiny_spec(**dict(c)))
        kc, vc = oracle_caches(case)
        o, l = run(att, case, kc, vc, causal=causal, window=window)
        bo, bl = brute(case, kc, vc, causal=causal, window=window)
        if not (np.allclose(o, bo, rtol=0, atol=1e-12) and np.allclose(l, bl, rtol=0, atol=1e-12)):
            return False
    return True


# Visible key sets of a 10-key sequence with 3 query tokens (positions 7, 8, 9), written out by
# hand for each mask: (causal, window) -> one set per query token.
VISIBLE_SETS_N10_T3 = {
    (True, 0): [set(range(0, 8)), set(range(0, 9)), set(range(0, 10))],
    (True, 4): [{4, 5, 6, 7}, {5, 6, 7, 8}, {6, 7, 8, 9}],
    (True, 1): [{7}, {8}, {9}],
    (False, 0): [set(range(10))] * 3,
    (False, 4): [{4, 5, 6, 7, 8, 9}, {5, 6, 7, 8, 9}, {6, 7, 8, 9}],
    (False, 1): [{7, 8, 9}, {8, 9}, {9}],
    (False, 12): [set(range(10))] * 3,
}


def pin_visible_sets(att):
    """Zero K (equal weights) and one-hot V (key j's V is the unit vector e_j): each output row is
    the indicator of its visible keys divided by their number, and lse = ln(number)."""
    case = workloads.make_case(tiny_spec("fp16", T=3, g=1, Hkv=1, D=16, P=4, contexts=(10,)))
    kc, vc = oracle_caches(case)
    kc[:] = 0
    vc[:] = 0
    for j in range(10):
        vc[case.block_table[0, j // 4], 0, j % 4, j] = 1.0
    for (causal, window), sets in VISIBLE_SETS_N10_T3.items():
        o, l = run(att, case, kc, vc, causal=causal, window=window)
        for t, vis in enumerate(sets):
            want = np.zeros(16)
            want[sorted(vis)] = 1.0 / len(vis)
            if not (np.allclose(o[t, 0], want, rtol=0, atol=1e-15) and math.isclose(l[t, 0], math.log(len(vis)))):
                return False
    return True


def pin_mask_reductions(att):
    """A causal window at least as long as the sequence is no window; non-causal rows all see the
    whole sequence, i.e. each is a one-token decode at the last position; a causal windowed row
    is that query's one-token decode restricted to its last W keys."""
    case = workloads.make_case(tiny_spec("e5m2", T=4, g=2, P=4, contexts=(23, 9)))
    kc, vc = oracle_caches(case)
    o, l = run(att, case, kc, vc)
    ow, lw = run(att, case, kc, vc, window=23)
    if not (np.array_equal(o, ow) and np.array_equal(l, lw)):
        return False
    onc, lnc = run(att, case, kc, vc, causal=False)
    T = 4
    for t in range(T):
        q1 = case.q.reshape(case.B, T, *case.q.shape[1:])[:, t]
        o1, l1 = run(att, case, kc, vc, q=q1, num_q_tokens=1)
        if not (np.allclose(o1, onc.reshape(case.B, T, *o.shape[1:])[:, t], rtol=0, atol=1e-14)
                and np.allclose(l1, lnc.reshape(case.B, T, -1)[:, t], rtol=0, atol=1e-14)):
            return False
    W = 3
    ocw, lcw = run(att, case, kc, vc, window=W)
    for b in range(case.B):
        n = int(case.seq_lens[b])
        for t in range(T):
            p = n - T + t
            if p < 0:
                continue
            q1 = case.q[b * T + t:b * T + t + 1]
            o1, l1 = run(att, case, kc, vc, q=q1, num_q_tokens=1, seq_lens=np.array([p + 1], np.int32),
                         block_table=case.block_table[b:b + 1], token_range=(p - W + 1, p + 1))
            if not (np.allclose(o1[0], ocw[b * T + t], rtol=0, atol=1e-14)
                    and np.allclose(l1[0], lcw[b * T + t], rtol=0, atol=1e-14)):
                return False
    return True


def pin_page_permutation(att):
    case = workloads.make_case(tiny_spec("e4m3", T=3, g=2, P=4, contexts=(23, 30)))
    kc, vc = oracle_caches(case)
    o1, l1 = run(att, case, kc, vc)
    rng = np.random.default_rng(0)
    perm = rng.permutation(case.num_blocks)  # physical page p moves to perm[p]
    kc2 = np.empty_like(kc)
    vc2 = np.empty_like(vc)
    kc2[perm] = kc
    vc2[perm] = vc
    bt2 = np.where(case.block_table >= 0, perm[np.maximum(case.block_table, 0)], -1).astype(np.int32)
    o2, l2 = run(att, case, kc2, vc2, block_table=bt2)
    return np.array_equal(o1, o2) and np.array_equal(l1, l2)


def pin_constant_v(att):
    case = workloads.make_case(tiny_spec("e5m2", T=3, g=2, P=4, contexts=(21, 9)))
    kc, vc = oracle_caches(case)
    code = 0x3D  # 1.25 in E5M2
    vc[:] = code
    o, _ = run(att, case, kc, vc)
    return np.allclose(o, 1.25 * float(case.v_scale), rtol=1e-14, atol=0)


def pin_zero_k(att):
    case = workloads.make_case(tiny_spec("e4m3", T=3, g=2, P=4, contexts=(21, 9)))
    kc, vc = oracle_caches(case)
    kc[:] = 0
    o, l = run(att, case, kc, vc)
    T, g, Hkv = 3, 2, 2
    for b in range(case.B):
        n = int(case.seq_lens[b])
        for t in range(T):
            vis = n - T + t + 1
            for h in range(g * Hkv):
                kvh = h // g
                js = np.arange(vis)
                pages = case.block_table[b, js // 4]
                v = fp8.decode(vc[pages, kvh, js % 4, :], "e4m3") * float(case.v_scale)
                if not np.allclose(o[b * T + t, h], v.mean(axis=0), rtol=0, atol=1e-13):
                    return False
                if not math.isclose(l[b * T + t, h], math.log(vis), abs_tol=1e-13):
                    return False
    return True


def pin_single_key(att):
    case = workloads.make_case(tiny_spec("fp16", T=1, g=2, P=4, contexts=(1, 1)))
    kc, vc = oracle_caches(case)
    o, l = run(att, case, kc, vc)
    for b in range(2):
        page = case.block_table[b, 0]
        for h in range(4):
            kvh = h // 2
            v = vc[page, kvh, 0].astype(np.float64)
            s0 = float(case.softmax_scale) * float(np.dot(case.q[b, h].astype(np.float64), kc[page, kvh, 0].astype(np.float64)))
            if not (np.array_equal(o[b, h], v) and math.isclose(l[b, h], s0, rel_tol=1e-15, abs_tol=1e-15)):
                return False
    return True


def pin_causal_rows_are_shorter_decodes(att):
    for T, contexts in ((3, (22, 11)), (16, (30, 17))):
        case = workloads.make_case(tiny_spec("e5m2", T=T, g=2, P=4, contexts=contexts))
        kc, vc = oracle_caches(case)
        o, l = run(att, case, kc, vc)
        for t in range(T):
            q1 = case.q.reshape(case.B, T, *case.q.shape[1:])[:, t]
            sl = case.seq_lens - (T - 1 - t)
            o1, l1 = run(att, case, kc, vc, q=q1, num_q_tokens=1, seq_lens=sl)
            if not (np.allclose(o1, o.reshape(case.B, T, *o.shape[1:])[:, t], rtol=0, atol=1e-14)
                    and np.allclose(l1, l.reshape(case.B, T, -1)[:, t], rtol=0, atol=1e-14)):
                return False
    return True


def pin_gqa_head_alone(att):
    case = workloads.make_case(tiny_spec("e4m3", T=1, g=3, Hkv=2, P=4, contexts=(17, 25)))
    kc, vc = oracle_caches(case)
    o, l = run(att, case, kc, vc)
    g, Hkv = 3, 2
    for h in range(g * Hkv):
        kvh = h // g
        # MHA view: one query head against one KV head (a pool holding just that head)
        o1, l1 = run(att, case, kc[:, kvh:kvh + 1], vc[:, kvh:kvh + 1], q=case.q[:, h:h + 1], num_kv_heads=1)
        if not (np.allclose(o1[:, 0], o[:, h], rtol=0, atol=1e-14) and np.allclose(l1[:, 0], l[:, h], rtol=0, atol=1e-14)):
            return False
    return True


def pin_split_merge(att):
    case = workloads.make_case(tiny_spec("e4m3", T=3, g=2, P=4, contexts=(37, 30)))
    kc, vc = oracle_caches(case)
    o, l = run(att, case, kc, vc)
    for cuts in ([0, 5, 36, 40], [0, 12, 24, 35, 36, 37, 40], [0, 40]):
        parts = [run(att, case, kc, vc, token_range=(a, b)) for a, b in zip(cuts[:-1], cuts[1:])]
        rows = o.shape[0] * o.shape[1]
        op = np.stack([p[0].reshape(rows, -1) for p in parts], axis=1)
        lp = np.stack([p[1].reshape(rows) for p in parts], axis=1)
        mo, ml = merge.lse_merge(op, lp)
        if not (np.allclose(mo, o.reshape(rows, -1), rtol=0, atol=1e-13) and np.allclose(ml, l.reshape(rows), rtol=0, atol=1e-13)):
            return False
    return True


def pin_long_chunk_rows_are_shorter_decodes(att):
    """A prefill chunk of 200 query tokens: causal row t is the one-token decode of the sequence
    cut after position n - T + t (sampled rows)."""
    T = 200
    case = workloads.make_case(tiny_spec("e4m3", T=T, g=2, D=8, P=16, contexts=(260,)))
    kc, vc = oracle_caches(case)
    pick = [0, 1, 57, 123, 198, 199]
    o, l = run(att, case, kc, vc, tokens=pick)
    for t in pick:
        q1 = case.q[t:t + 1]
        o1, l1 = run(att, case, kc, vc, q=q1, num_q_tokens=1, seq_lens=case.seq_lens - (T - 1 - t))
        if not (np.allclose(o1[0], o[t], rtol=0, atol=1e-14) and np.allclose(l1[0], l[t], rtol=0, atol=1e-14)):
            return False
    return bool(np.isnan(o[2]).all())  # rows not asked for stay NaN


PINS = [pin_brute, pin_page_permutation, pin_constant_v, pin_zero_k, pin_single_key,
        pin_causal_rows_are_shorter_decodes, pin_gqa_head_alone, pin_split_merge, pin_visible_sets,
        pin_mask_reductions, pin_long_chunk_rows_are_shorter_decodes]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_oracle_passes_pin(pin):
    assert pin(oatt.paged_attention)


def test_weights_sum_to_one_and_lse_definition():
    case = workloads.make_case(tiny_spec("e5m2", T=3, g=2, P=4, contexts=(31, 8)))
    kc, vc = oracle_caches(case)
    vc[:] = 0x3C  # V = 1 everywhere -> out = sum_j w_j / L * v_scale
    o, l = oatt.paged_attention(case.q, kc, vc, case.block_table, case.seq_lens, 3, 2, 4, "e5m2",
                                case.k_scale, np.float32(1.0), case.softmax_scale)
    assert np.allclose(o, 1.0, rtol=0, atol=1e-14)


def test_empty_and_short_sequences():
    case = workloads.make_case(tiny_spec("e4m3", T=3, g=2, P=4, contexts=(0, 2)))
    kc, vc = oracle_caches(case)
    o, l = oatt.paged_attention(case.q, kc, vc, case.block_table, case.seq_lens, 3, 2, 4, "e4m3",
                                case.k_scale, case.v_scale, case.softmax_scale)
    # sequence 0 is empty: every row sees nothing
    assert np.all(o[0:3] == 0) and np.all(np.isneginf(l[0:3]))
    # sequence 1 has 2 keys and 3 query tokens: row t=0 sees nothing, t=1 one key, t=2 two
    assert np.all(o[3] == 0) and np.all(np.isneginf(l[3]))
    assert np.all(np.isfinite(l[4:6]))


MUTANTS = {
    "drop k_scale": ("[lo - base:hi - base] * ks", "[lo - base:hi - base]"),
    "drop v_scale": ("[lo - base:hi - base] * vs", "[lo - base:hi - base]"),
    "drop softmax scale": ("s = sm * (qrows @ K.T)", "s = (qrows @ K.T)"),
    "causal off by one": ("j[None, :] <= last[:, None]", "j[None, :] < last[:, None]"),
    "reversed draft order": ("pos = np.array([n - T + t", "pos = np.array([n - 1 - t"),
    "rows head-major vs limits token-major": ("for t in toks for _ in heads", "for _ in heads for t in toks"),
    "window off by one": ("np.maximum(0, pos - window + 1)", "np.maximum(0, pos - window)"),
    "window ignored": ("first = np.maximum(0, pos - window + 1) if window > 0",
                       "first = np.zeros(nt * g, dtype=np.int64) if window > 0"),
    "window anchored at the block end": ("np.maximum(0, pos - window + 1)", "np.maximum(0, n - window + 0 * pos)"),
    "non-causal mask still causal": ("last = pos if causal else np.full(nt * g, n - 1)", "last = pos"),
    "non-causal bound one short": ("np.full(nt * g, n - 1)", "np.full(nt * g, n - 2)"),
    "token subset takes the first rows": ("[toks]  # [nt, g, D]", "[:len(toks)]  # [nt, g, D]"),
    "interleaved GQA map": ("heads = list(range(kvh * g, (kvh + 1) * g))", "heads = list(range(kvh, Hq, num_kv_heads))"),
    "pages taken in sorted order": ("pages = np.asarray(block_table[b, first_page:last_page + 1], dtype=np.int64)",
                                    "pages = np.sort(np.asarray(block_table[b, first_page:last_page + 1], dtype=np.int64))"),
    "log base 2 in lse": ("m + np.log(np.where(has, L, 1.0))", "m + np.log2(np.where(has, L, 1.0))"),
    "missing max subtraction in weights": ("w = np.exp(s - np.where(has, m, 0.0)[:, None])", "w = np.exp(s)"),
    "no normalisation": ("acc / np.where(has, L, 1.0)[:, None]", "acc"),
    "per-head scales: head 0's for every head": ("ks = ks_all[kvh if ks_all.size > 1 else 0]", "ks = ks_all[0]"),
    "per-head scales: K's scale for V": ("vs = vs_all[kvh if vs_all.size > 1 else 0]",
                                         "vs = ks_all[kvh if ks_all.size > 1 else 0]"),
}


def _mutant(old, new):
    src = inspect.getsource(oatt)
    assert src.count(old) == 1, old
    mod = types.ModuleType("oracle_attention_mutant")
    mod.__dict__["__name__"] = "oracle.attention_mutant"
    code = compile(src.replace(old, new).replace("from . import fp8", "from oracle import fp8"), "mutant", "exec")
    exec(code, mod.__dict__)
    return mod.paged_attention


@pytest.mark.parametrize("name", list(MUTANTS))
def test_planted_mistake_fails_a_pin(name):
    att = _mutant(*MUTANTS[name])
    failed = [p.__name__ for p in PINS if not p(att)]
    assert failed, f"planted mistake '{name}' passed every pin"


def test_merge_closed_forms():
    rng = np.random.default_rng(1)
    o = rng.standard_normal((5, 4, 3))
    lse = rng.standard_normal((5, 4))
    # equal lse: plain mean, lse + ln S
    mo, ml = merge.lse_merge(o, np.zeros((5, 4)))
    assert np.allclose(mo, o.mean(axis=1)) and np.allclose(ml, math.log(4))
    # one dominant part (others -inf): that part unchanged
    l2 = np.full((5, 4), -np.inf)
    l2[:, 2] = lse[:, 2]
    mo, ml = merge.lse_merge(o, l2)
    assert np.array_equal(mo, o[:, 2]) and np.array_equal(ml, lse[:, 2])
    # all empty
    mo, ml = merge.lse_merge(o, np.full((5, 4), -np.inf))
    assert np.all(mo == 0) and np.all(np.isneginf(ml))
    # a shift of every lse by c shifts the merged lse by c and keeps out
    mo1, ml1 = merge.lse_merge(o, lse)
    mo2, ml2 = merge.lse_merge(o, lse + 3.0)
    assert np.allclose(mo1, mo2) and np.allclose(ml2, ml1 + 3.0)


@pytest.mark.parametrize("kv", ["e4m3", "e5m2"])
def test_per_head_scales_all_equal_reduce_to_the_per_tensor_scale(kv):
    # one scale per KV head, all equal to the pool's scale: the same cache bytes and the same
    # attention as the per-tensor scale, exactly
    case = workloads.make_case(tiny_spec(kv, T=3, g=2, Hkv=3, P=4, contexts=(23, 30)))
    Hkv = case.spec.num_kv_heads
    kc, vc = oracle_caches(case)
    ks = np.full(Hkv, case.k_scale, np.float32)
    vs = np.full(Hkv, case.v_scale, np.float32)
    kc2, vc2 = np.zeros_like(kc), np.zeros_like(vc)
    oappend.append_bulk(kc2, case.k_fill, case.slot_fill, case.spec.page_size, ks, kv)
    oappend.append_bulk(vc2, case.v_fill, case.slot_fill, case.spec.page_size, vs, kv)
    assert np.array_equal(kc, kc2) and np.array_equal(vc, vc2)
    o1, l1 = run(oatt.paged_attention, case, kc, vc)
    o2, l2 = run(oatt.paged_attention, case, kc2, vc2, k_scale=ks, v_scale=vs)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


@pytest.mark.parametrize("kv", ["e4m3", "e5m2"])
def test_per_head_scale_commutes_with_power_of_two_head_gains(kv):
    # multiplying KV head h's fp16 values and its scale by the same power of two leaves its FP8
    # bytes unchanged (the float32 quotient is the same number), so each head is quantised
    # against its own scale only
    rng = np.random.default_rng(11)
    x = rng.standard_normal((50, 3, 16)).astype(np.float16)
    s = np.array([0.01, 0.02, 0.005], np.float32)
    gains = np.array([1.0, 2.0, 8.0], np.float32)
    a = oappend.quantise(x, oappend.head_scales(s, 3), kv)
    b = oappend.quantise((x.astype(np.float32) * gains[:, None]).astype(np.float16),
                         oappend.head_scales(s * gains, 3), kv)
    assert np.array_equal(a, b)
    # and a head quantised alone with its scale gives the same bytes
    for h in range(3):
        assert np.array_equal(a[:, h], oappend.quantise(x[:, h], s[h], kv))
