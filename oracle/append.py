"""Quantise-and-append of new K/V tokens into a paged cache (float64 oracle).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

The pages name the KV write path only as a module imported next to the
attention extension ("1Cat-vLLM", section on the source build / runtime
notes: ``paged_kv_utils``) and fix two of its parameters: the cache stores FP8
with static per-tensor scales that are never computed online ("1Cat-vLLM",
"Optional experimental feature: FP8 KV cache": do not add
``--calculate-kv-scales``), in pages of 2048 tokens ("SM70 release profile
and acceleration status": 2048-token KV blocks) or 16 (its override table:
``--block-size 16``). Everything else is a reading, stated here:

* cache layout ``[num_blocks, Hkv, P, D]`` (one contiguous ``P x D`` chunk per
  page and KV head), separate K and V pools;
* token i goes to ``slot = slot_mapping[i]``, ``block = slot // P``,
  ``offset = slot % P``; a negative slot means "skip this token";
* the stored byte is ``encode(float32(float32(x16) / scale))``: the fp16 input
  widened to float32, divided (not multiplied by a reciprocal) by the float32
  scale with one IEEE round-to-nearest, then FP8 round-to-nearest-even with
  saturation to the largest finite value;
* an fp16 cache (no quantisation) stores the fp16 bits unchanged.

The float32 quotient is formed as the float64 quotient rounded once to
float32. That is the correctly rounded float32 quotient: for p-bit operands a
2p+2-bit intermediate makes the second rounding innocuous, and float64 has
53 >= 2*24+2 bits.
"""

from __future__ import annotations

import numpy as np

from . import fp8


def quantise(x16: np.ndarray, scale, fmt) -> np.ndarray:
    """uint8 codes of fp16 values divided by a float32 scale (a scalar, or an array that
    broadcasts against ``x16``, e.g. ``[Hkv, 1]`` for one scale per KV head)."""
    x32 = np.asarray(x16, dtype=np.float16).astype(np.float32)
    s32 = np.asarray(scale, dtype=np.float32)
    q = (x32.astype(np.float64) / s32.astype(np.float64)).astype(np.float32)
    return fp8.encode(q, fmt)


def head_scales(scale, num_kv_heads: int):
    """A per-tensor scale as a float32 scalar, or one scale per KV head (an array of
    ``num_kv_heads``, the per-head generalisation of the pages' per-tensor static scales) as a
    float32 ``[Hkv, 1]`` column that broadcasts over ``[..., Hkv, D]``."""
    s = np.asarray(scale, dtype=np.float32)
    if s.size == 1:
        return np.float32(s.reshape(()))
    if s.size != num_kv_heads:
        raise ValueError(f"{s.size} scales for {num_kv_heads} KV heads")
    return s.reshape(num_kv_heads, 1)


def append(cache: np.ndarray, new: np.ndarray, slot_mapping: np.ndarray,
           page_size: int, scale, kv_dtype: str) -> None:
    """Write ``new[i]`` (fp16 ``[Hkv, D]``) into ``cache`` at ``slot_mapping[i]``.

    ``scale`` is one float32 for the pool or one per KV head (``[Hkv]``).

    ``cache`` is ``uint8 [num_blocks, Hkv, P, D]`` for ``kv_dtype`` in
    ``{"e4m3", "e5m2"}`` or ``float16 [num_blocks, Hkv, P, D]`` for ``"fp16"``.
    Updated in place. Tokens are visited in order, so a slot named twice ends
    with the later token (the GPU path makes no promise there; tests never
    repeat a slot).
    """
    new = np.asarray(new, dtype=np.float16)
    n_tok = new.shape[0]
    num_blocks = cache.shape[0]
    scale = head_scales(scale, cache.shape[1])
    for i in range(n_tok):
        slot = int(slot_mapping[i])
        if slot < 0:
            continue
        block, off = divmod(slot, page_size)
        if block >= num_blocks:
            raise IndexError(f"slot {slot} outside a pool of {num_blocks} pages")
        if kv_dtype == "fp16":
            cache[block, :, off, :] = new[i]
        else:
            cache[block, :, off, :] = quantise(new[i], scale, kv_dtype)


def append_bulk(cache: np.ndarray, new: np.ndarray, slot_mapping: np.ndarray,
                page_size: int, scale, kv_dtype: str) -> None:
    """Same result as :func:`append` for distinct slots, vectorised over tokens.

    Used to populate large caches; ``tests/test_oracle_append.py`` checks it
    equals the token-by-token loop.
    """
    new = np.asarray(new, dtype=np.float16)
    slots = np.asarray(slot_mapping, dtype=np.int64)
    keep = slots >= 0
    slots = slots[keep]
    if slots.size == 0:
        return
    if np.any(slots // page_size >= cache.shape[0]):
        raise IndexError("slot outside the pool")
    block = slots // page_size
    off = slots % page_size
    vals = new[keep]
    if kv_dtype != "fp16":
        vals = quantise(vals, head_scales(scale, cache.shape[1]), kv_dtype)
    # cache[block, :, off, :] with fancy indices on axes 0 and 2
    cache[block, :, off, :] = vals


def zero_blocks(k_cache: np.ndarray, v_cache: np.ndarray, block_ids) -> None:
    """Clear the listed blocks of both pools in place ("1Cat-vLLM 1.5.0", section "Reliability
    and correctness fixes": newly reused KV blocks are zeroed before attention).

    Pools are ``[num_blocks, Hkv, P, D]``; every element of a listed block becomes the zero
    byte pattern (+0 in fp16, E4M3 and E5M2 alike). A negative id means "no block" and is
    skipped, as is an id past the pool (the device path reports that one).
    """
    nb = k_cache.shape[0]
    for bid in np.asarray(block_ids, dtype=np.int64).ravel():
        if 0 <= bid < nb:
            k_cache[bid] = 0
            v_cache[bid] = 0
