"""CPU oracle for paged FP8-KV decode attention.

TEST INFRASTRUCTURE ONLY. Nothing in the product path may import, call or
execute anything in this package: only the tests, ``__graft_entry__.smoke()``
and the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.
It shares no code, headers, tables or constant generators with the CUDA path
in ``paged_fp8_kv_cache_gb300/csrc``; the only thing both sides consume is the
seeded input generator in ``paged_fp8_kv_cache_gb300/workloads.py``, which holds
none of the method's arithmetic.

What it computes (plain definitions, numpy float64):

* ``fp8``       -- bitwise E4M3 ("fn") and E5M2 codecs written from the two
                   formats' bit-field definitions (sign, biased exponent,
                   mantissa; subnormals; E4M3 has no infinity).
* ``append``    -- quantise-and-append of new fp16 K/V into a paged cache
                   laid out ``[num_blocks, Hkv, P, D]`` through an int64 slot
                   mapping (the reshape-and-cache step). Also the zeroing of
                   reused blocks.
* ``attention`` -- paged decode / grouped causal verify attention over that
                   cache: gather by block table, FP8 decode, per-tensor
                   scales, scaled softmax with natural-log LSE.
* ``merge``     -- the log-sum-exp merge of split-KV partial results.

Parity status: every function here is pinned by the ``-m "not gpu"`` tests in
``tests/test_oracle_*.py`` (exhaustive codec anchors and nearest-value search,
library-cast special cases, brute force on tiny inputs, closed forms and
invariants, planted-mistake checks). No function is "parity unpinned".
"""

from . import fp8, append, attention, merge  # noqa: F401
