"""Log-sum-exp merge of split-KV partial attention results (float64 oracle).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

The long-context E4M3 decode route of "1Cat-vLLM 1.5.0" (section "Flash-V100
long-context improvements") splits a 128K-256K key range across workers; the
pages do not spell out how partial results are combined. The plain reading is
the identity that makes a split exact: if a row's keys are cut into disjoint
ranges s with partial results ``o_s = sum_{j in s} w_j v_j / L_s`` and
``lse_s = m + ln L_s`` (the attention restricted to range s), then with
``M = max_s lse_s`` and ``w_s = exp(lse_s - M)``:

* ``out = sum_s w_s o_s / sum_s w_s``
* ``lse = M + ln sum_s w_s``

Ranges with no visible key carry ``lse_s = -inf`` and weight 0; a row with no
visible key at all gets ``out = 0``, ``lse = -inf``.
"""

from __future__ import annotations

import numpy as np


def lse_merge(o_parts: np.ndarray, lse_parts: np.ndarray):
    """Merge partials ``o_parts [rows, S, D]``, ``lse_parts [rows, S]`` (float64)."""
    o_parts = np.asarray(o_parts, dtype=np.float64)
    lse_parts = np.asarray(lse_parts, dtype=np.float64)
    M = lse_parts.max(axis=1)
    has = np.isfinite(M)
    w = np.exp(lse_parts - np.where(has, M, 0.0)[:, None])
    w = np.where(np.isfinite(lse_parts), w, 0.0)
    W = w.sum(axis=1)
    num = np.einsum("rs,rsd->rd", w, np.where(np.isfinite(lse_parts)[:, :, None], o_parts, 0.0))
    out = np.where(has[:, None], num / np.where(has, W, 1.0)[:, None], 0.0)
    lse = np.where(has, M + np.log(np.where(has, W, 1.0)), -np.inf)
    return out, lse
