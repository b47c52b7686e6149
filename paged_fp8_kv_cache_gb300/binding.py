"""ctypes binding of libpfkv.so: the C ABI of include/pfkv.h, same names.

Argument marshalling only. Functions take torch tensors (device memory
allocated by PyTorch) or plain ints and pass raw pointers, sizes and the
current CUDA stream to the library; every step of the computation runs in
the library's kernels. A non-OK status raises :class:`PfkvError`. The
library is loaded on first use; if it has not been built, loading raises
(there is no CPU fallback).
"""

from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_lib", "libpfkv.so")

PFKV_OK = 0
PFKV_ERR_INVALID_ARG = 1
PFKV_ERR_UNSUPPORTED = 2
PFKV_ERR_WORKSPACE = 3
PFKV_ERR_CUDA = 4
PFKV_ERR_DEVICE_CHECK = 5

PFKV_KV_FP16 = 0
PFKV_KV_FP8_E4M3 = 1
PFKV_KV_FP8_E5M2 = 2
KV_DTYPES = {"fp16": PFKV_KV_FP16, "e4m3": PFKV_KV_FP8_E4M3, "e5m2": PFKV_KV_FP8_E5M2}

PFKV_DEVERR_SLOT = 0x1
PFKV_DEVERR_BLOCK_ID = 0x2
PFKV_DEVERR_SEQ_LEN = 0x4
PFKV_DEVERR_TIMEOUT = 0x8
PFKV_KV_SCALES_PER_HEAD = 0x100  # OR into an FP8 dtype: one scale per KV head
PFKV_MASK_CAUSAL = 0x1

# every entry point declared in include/pfkv.h
EXPORTS = [
    "pfkv_kv_cache_append",
    "pfkv_kv_cache_zero_blocks",
    "pfkv_decode_plan",
    "pfkv_decode_workspace_bytes",
    "pfkv_paged_attention_decode",
    "pfkv_paged_attention",
    "pfkv_attention_plan",
    "pfkv_attention_workspace_bytes",
    "pfkv_paged_attention_decode_static_scratch",
    "pfkv_lse_merge",
    "pfkv_device_errors",
    "pfkv_capabilities",
    "pfkv_status_string",
    "pfkv_last_error",
]


class PfkvError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{_status_name(status)}: {message}")
        self.status = status


_lib = None


def _status_name(st: int) -> str:
    return {0: "PFKV_OK", 1: "PFKV_ERR_INVALID_ARG", 2: "PFKV_ERR_UNSUPPORTED", 3: "PFKV_ERR_WORKSPACE",
            4: "PFKV_ERR_CUDA", 5: "PFKV_ERR_DEVICE_CHECK"}.get(st, f"status {st}")


def load(path: str | None = None):
    """Load the library (once) and declare its signatures."""
    global _lib
    if _lib is not None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"libpfkv.so not built ({p} missing): run paged_fp8_kv_cache_gb300.build.build()")
    lib = ctypes.CDLL(p)
    vp, i32, i64p, f32p, u32p = ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.POINTER(ctypes.c_uint32)
    lib.pfkv_kv_cache_append.argtypes = [vp, vp, vp, vp, i64p, i32, i32, i32, i32, i32, i32, f32p, f32p, vp]
    lib.pfkv_kv_cache_append.restype = i32
    lib.pfkv_kv_cache_zero_blocks.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, i32, vp]
    lib.pfkv_kv_cache_zero_blocks.restype = i32
    lib.pfkv_decode_plan.argtypes = [i32, i32, i32, i32, i32, i32, i32, i32, i32,
                                     ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int)]
    lib.pfkv_decode_plan.restype = i32
    lib.pfkv_decode_workspace_bytes.argtypes = [i32, i32, i32, i32, i32, i32, i32, i32, i32]
    lib.pfkv_decode_workspace_bytes.restype = ctypes.c_size_t
    lib.pfkv_paged_attention_decode.argtypes = [vp, vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i32, i32, i32,
                                                i32, vp, vp, ctypes.c_float, i32, i32, vp, ctypes.c_size_t, vp]
    lib.pfkv_paged_attention_decode.restype = i32
    lib.pfkv_paged_attention.argtypes = [vp, vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i32, i32, i32,
                                         i32, vp, vp, ctypes.c_float, i32, i32, i32, i32, vp, ctypes.c_size_t, vp]
    lib.pfkv_paged_attention.restype = i32
    lib.pfkv_attention_plan.argtypes = [i32] * 11 + [ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int)]
    lib.pfkv_attention_plan.restype = i32
    lib.pfkv_attention_workspace_bytes.argtypes = [i32] * 11
    lib.pfkv_attention_workspace_bytes.restype = ctypes.c_size_t
    lib.pfkv_paged_attention_decode_static_scratch.argtypes = [vp, vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, i32,
                                                               i32, i32, i32, i32, vp, vp, ctypes.c_float, i32,
                                                               i32, vp]
    lib.pfkv_paged_attention_decode_static_scratch.restype = i32
    lib.pfkv_lse_merge.argtypes = [vp, vp, vp, vp, i32, i32, i32, vp]
    lib.pfkv_lse_merge.restype = i32
    lib.pfkv_device_errors.argtypes = [u32p, i32]
    lib.pfkv_device_errors.restype = i32
    lib.pfkv_capabilities.argtypes = []
    lib.pfkv_capabilities.restype = ctypes.c_uint32
    lib.pfkv_status_string.argtypes = [i32]
    lib.pfkv_status_string.restype = ctypes.c_char_p
    lib.pfkv_last_error.argtypes = []
    lib.pfkv_last_error.restype = ctypes.c_char_p
    _lib = lib
    return lib


def _check(st: int):
    if st != PFKV_OK:
        raise PfkvError(st, _lib.pfkv_last_error().decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _kv(dtype) -> int:
    return KV_DTYPES[dtype] if isinstance(dtype, str) else int(dtype)


def _kv_scaled(dtype, k_scale, v_scale, num_kv_heads) -> int:
    """The dtype argument, with PFKV_KV_SCALES_PER_HEAD when the scale tensors hold one float per KV head."""
    kv = _kv(dtype)
    n = [t.numel() for t in (k_scale, v_scale) if t is not None]
    if n and max(n) > 1:
        if any(x != num_kv_heads for x in n):
            raise PfkvError(PFKV_ERR_INVALID_ARG, f"scales of {n} floats: one per pool or one per KV head "
                                                  f"({num_kv_heads}) expected")
        kv |= PFKV_KV_SCALES_PER_HEAD
    return kv


def pfkv_kv_cache_zero_blocks(k_cache, v_cache, block_ids, kv_dtype, stream=None):
    """Zero the listed blocks of both pools [num_blocks, Hkv, P, D]; block_ids int32 [n] (negative = skip)."""
    lib = load()
    nb, hkv, page, d = k_cache.shape
    _check(lib.pfkv_kv_cache_zero_blocks(_ptr(k_cache), _ptr(v_cache), _ptr(block_ids), block_ids.numel(), hkv, d,
                                         page, nb, _kv(kv_dtype), _stream(stream)))


def pfkv_kv_cache_append(k_new, v_new, k_cache, v_cache, slot_mapping, page_size, kv_dtype,
                         k_scale=None, v_scale=None, stream=None):
    """k_new/v_new fp16 [n_tok, Hkv, D]; caches [num_blocks, Hkv, P, D]; slot_mapping int64 [n_tok]."""
    lib = load()
    n_tok, hkv, d = k_new.shape
    _check(lib.pfkv_kv_cache_append(_ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), _ptr(slot_mapping),
                                    n_tok, hkv, d, page_size, k_cache.shape[0],
                                    _kv_scaled(kv_dtype, k_scale, v_scale, hkv), _ptr(k_scale), _ptr(v_scale),
                                    _stream(stream)))


def pfkv_decode_plan(num_seqs, num_q_tokens, num_q_heads, num_kv_heads, head_dim, page_size, kv_dtype,
                     max_seq_len, num_splits_request=0):
    lib = load()
    ns, st = ctypes.c_int(0), ctypes.c_int(0)
    _check(lib.pfkv_decode_plan(num_seqs, num_q_tokens, num_q_heads, num_kv_heads, head_dim, page_size,
                                _kv(kv_dtype), max_seq_len, num_splits_request, ctypes.byref(ns), ctypes.byref(st)))
    return ns.value, st.value


def pfkv_decode_workspace_bytes(num_seqs, num_q_tokens, num_q_heads, num_kv_heads, head_dim, page_size, kv_dtype,
                                max_seq_len, num_splits_request=0) -> int:
    lib = load()
    return int(lib.pfkv_decode_workspace_bytes(num_seqs, num_q_tokens, num_q_heads, num_kv_heads, head_dim,
                                               page_size, _kv(kv_dtype), max_seq_len, num_splits_request))


def pfkv_paged_attention_decode(out, lse, q, k_cache, v_cache, block_table, seq_lens, num_q_tokens, num_kv_heads,
                                page_size, kv_dtype, k_scale, v_scale, softmax_scale, max_seq_len, num_splits=0,
                                workspace=None, stream=None):
    """q/out fp16 [B*T, Hq, D]; lse float32 [B*T, Hq]; block_table int32 [B, max_blocks]; seq_lens int32 [B]."""
    lib = load()
    num_seqs = seq_lens.shape[0]
    hq, d = q.shape[1], q.shape[2]
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib.pfkv_paged_attention_decode(
        _ptr(out), _ptr(lse), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), block_table.shape[1],
        _ptr(seq_lens), num_seqs, num_q_tokens, hq, num_kv_heads, d, page_size, k_cache.shape[0],
        _kv_scaled(kv_dtype, k_scale, v_scale, num_kv_heads), _ptr(k_scale), _ptr(v_scale), float(softmax_scale),
        max_seq_len, num_splits, _ptr(workspace), ws_bytes,
        _stream(stream)))


def _mask(causal) -> int:
    return PFKV_MASK_CAUSAL if causal else 0


def pfkv_attention_plan(num_seqs, num_q_tokens, num_q_heads, num_kv_heads, head_dim, page_size, kv_dtype,
                        max_seq_len, causal=True, window=0, num_splits_request=0):
    lib = load()
    ns, st = ctypes.c_int(0), ctypes.c_int(0)
    _check(lib.pfkv_attention_plan(num_seqs, num_q_tokens, num_q_heads, num_kv_heads, head_dim, page_size,
                                   _kv(kv_dtype), _mask(causal), window, max_seq_len, num_splits_request,
                                   ctypes.byref(ns), ctypes.byref(st)))
    return ns.value, st.value


def pfkv_attention_workspace_bytes(num_seqs, num_q_tokens, num_q_heads, num_kv_heads, head_dim, page_size, kv_dtype,
                                   max_seq_len, causal=True, window=0, num_splits_request=0) -> int:
    lib = load()
    return int(lib.pfkv_attention_workspace_bytes(num_seqs, num_q_tokens, num_q_heads, num_kv_heads, head_dim,
                                                  page_size, _kv(kv_dtype), _mask(causal), window, max_seq_len,
                                                  num_splits_request))


def pfkv_paged_attention(out, lse, q, k_cache, v_cache, block_table, seq_lens, num_q_tokens, num_kv_heads, page_size,
                         kv_dtype, k_scale, v_scale, softmax_scale, max_seq_len, causal=True, window=0, num_splits=0,
                         workspace=None, stream=None):
    """Paged attention with a mask choice (causal or not, sliding window of ``window`` keys, 0 = none) and up to
    8192 query tokens per sequence (chunked prefill); tensors as pfkv_paged_attention_decode."""
    lib = load()
    num_seqs = seq_lens.shape[0]
    hq, d = q.shape[1], q.shape[2]
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib.pfkv_paged_attention(
        _ptr(out), _ptr(lse), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), block_table.shape[1],
        _ptr(seq_lens), num_seqs, num_q_tokens, hq, num_kv_heads, d, page_size, k_cache.shape[0],
        _kv_scaled(kv_dtype, k_scale, v_scale, num_kv_heads), _ptr(k_scale), _ptr(v_scale), float(softmax_scale),
        _mask(causal), window, max_seq_len, num_splits, _ptr(workspace), ws_bytes, _stream(stream)))


def pfkv_paged_attention_decode_static_scratch(out, lse, q, k_cache, v_cache, block_table, seq_lens, num_q_tokens,
                                               num_kv_heads, page_size, kv_dtype, k_scale, v_scale, softmax_scale,
                                               max_seq_len, num_splits=0, stream=None):
    """Decode with the library's built-in split scratch (for callers that cannot allocate device memory)."""
    lib = load()
    num_seqs = seq_lens.shape[0]
    hq, d = q.shape[1], q.shape[2]
    _check(lib.pfkv_paged_attention_decode_static_scratch(
        _ptr(out), _ptr(lse), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), block_table.shape[1],
        _ptr(seq_lens), num_seqs, num_q_tokens, hq, num_kv_heads, d, page_size, k_cache.shape[0],
        _kv_scaled(kv_dtype, k_scale, v_scale, num_kv_heads), _ptr(k_scale), _ptr(v_scale), float(softmax_scale),
        max_seq_len, num_splits, _stream(stream)))


def pfkv_lse_merge(out, lse, o_parts, lse_parts, stream=None):
    """o_parts float32 [rows, S, D], lse_parts float32 [rows, S] -> out fp16 [rows, D], lse float32 [rows]."""
    lib = load()
    rows, s, d = o_parts.shape
    _check(lib.pfkv_lse_merge(_ptr(out), _ptr(lse), _ptr(o_parts), _ptr(lse_parts), rows, s, d, _stream(stream)))


def pfkv_device_errors(clear: bool = True) -> int:
    """Error bits of the current device (synchronises); never raises for set bits."""
    lib = load()
    flags = ctypes.c_uint32(0)
    st = lib.pfkv_device_errors(ctypes.byref(flags), 1 if clear else 0)
    if st not in (PFKV_OK, PFKV_ERR_DEVICE_CHECK):
        _check(st)
    return flags.value


def pfkv_capabilities() -> int:
    return int(load().pfkv_capabilities())


def pfkv_status_string(status: int) -> str:
    return load().pfkv_status_string(status).decode()


def pfkv_last_error() -> str:
    return load().pfkv_last_error().decode()
