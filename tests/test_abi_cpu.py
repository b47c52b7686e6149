"""The C-ABI library builds, loads and exports what include/pfkv.h declares;
host-side validation and split planning work without a GPU (CPU only)."""

import ctypes
import os
import re
import shutil
import subprocess

import pytest

from paged_fp8_kv_cache_gb300 import binding as pf

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pfkv.h")
CSRC = os.path.join(ROOT, "paged_fp8_kv_cache_gb300", "csrc")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pfkv_[a-z0-9_]+)\s*\(", text)))


def test_binding_lists_every_declared_function():
    assert sorted(pf.EXPORTS) == declared_functions()


def test_library_exports_every_declared_symbol(pflib):
    lib = ctypes.CDLL(pf.LIB_PATH)
    missing = [f for f in declared_functions() if not hasattr(lib, f)]
    assert not missing, missing


def test_exports_nothing_else(pflib):
    nm = shutil.which("nm")
    if nm is None:
        pytest.skip("nm not available")
    out = subprocess.run([nm, "-D", "--defined-only", pf.LIB_PATH], capture_output=True, text=True).stdout
    pfkv = sorted({ln.split()[-1] for ln in out.splitlines() if " T pfkv_" in ln})
    assert pfkv == declared_functions()


def test_status_strings_and_capabilities(pflib):
    for st, name in [(0, "PFKV_OK"), (1, "PFKV_ERR_INVALID_ARG"), (2, "PFKV_ERR_UNSUPPORTED"),
                     (3, "PFKV_ERR_WORKSPACE"), (4, "PFKV_ERR_CUDA"), (5, "PFKV_ERR_DEVICE_CHECK")]:
        assert pf.pfkv_status_string(st) == name
    caps = pf.pfkv_capabilities()
    for bit in (0x1, 0x2, 0x4, 0x10, 0x20, 0x100, 0x200, 0x1000, 0x2000, 0x4000, 0x10000, 0x20000, 0x40000):
        assert caps & bit


@pytest.mark.parametrize("args,status", [
    (dict(T=17), pf.PFKV_ERR_UNSUPPORTED),
    (dict(T=0), pf.PFKV_ERR_UNSUPPORTED),
    (dict(D=64), pf.PFKV_ERR_UNSUPPORTED),
    (dict(P=24), pf.PFKV_ERR_UNSUPPORTED),
    (dict(P=4096), pf.PFKV_ERR_UNSUPPORTED),
    (dict(Hq=30), pf.PFKV_ERR_INVALID_ARG),
    (dict(T=8, Hq=72, Hkv=8), pf.PFKV_ERR_UNSUPPORTED),  # 8 tokens x group 9 = 72 rows > 64
    (dict(T=16, Hq=40, Hkv=8), pf.PFKV_ERR_UNSUPPORTED),  # 16 tokens x group 5 = 80 rows > 64
    (dict(B=-1), pf.PFKV_ERR_INVALID_ARG),
    (dict(kv=7), pf.PFKV_ERR_INVALID_ARG),
])
def test_plan_rejects_bad_shapes(pflib, args, status):
    a = dict(B=2, T=1, Hq=32, Hkv=8, D=128, P=16, kv=1, msl=4096, S=4)
    a.update(args)
    with pytest.raises(pf.PfkvError) as ei:
        pf.pfkv_decode_plan(a["B"], a["T"], a["Hq"], a["Hkv"], a["D"], a["P"], a["kv"], a["msl"], a["S"])
    assert ei.value.status == status


@pytest.mark.parametrize("T,Hq,Hkv", [(9, 16, 4), (16, 16, 4), (16, 8, 8), (12, 40, 8)])
def test_plan_accepts_q16_verify_shapes(pflib, T, Hq, Hkv):
    # up to 16 query tokens per sequence while the rows per KV head (T * g) stay within 64
    S, C = pf.pfkv_decode_plan(2, T, Hq, Hkv, 256, 2048, "e5m2", 262144, 19)
    assert S == 19 and S * C >= 262144


@pytest.mark.parametrize("msl,req,exp", [
    (4096, 1, (1, 4096)), (4096, 2, (2, 2048)), (5000, 7, (7, 768)), (100, 7, (2, 64)),
    (0, 3, (1, 64)), (262144, 38, (38, 6912)), (1, 1, (1, 64)),
])
def test_split_plan_with_explicit_count(pflib, msl, req, exp):
    # explicit counts need no device query: ranges are whole 64-key tiles
    assert pf.pfkv_decode_plan(4, 1, 32, 8, 128, 16, "e4m3", msl, req) == exp
    S, C = exp
    assert S * C >= msl and (S - 1) * C < max(msl, 1)


@pytest.mark.parametrize("args,status", [
    (dict(T=8193), pf.PFKV_ERR_UNSUPPORTED),     # more query tokens than one call takes
    (dict(Hq=65, Hkv=1), pf.PFKV_ERR_UNSUPPORTED),  # one token's heads must fit a 64-row slab
    (dict(mask=2), pf.PFKV_ERR_INVALID_ARG),
    (dict(window=-1), pf.PFKV_ERR_INVALID_ARG),
])
def test_attention_plan_rejects_bad_arguments(pflib, args, status):
    a = dict(B=1, T=8, Hq=24, Hkv=4, D=256, P=2048, kv=2, mask=1, window=0, msl=262144, S=4)
    a.update(args)
    lib = pf.load()
    ns, st = ctypes.c_int(0), ctypes.c_int(0)
    got = lib.pfkv_attention_plan(a["B"], a["T"], a["Hq"], a["Hkv"], a["D"], a["P"], a["kv"], a["mask"], a["window"],
                                  a["msl"], a["S"], ctypes.byref(ns), ctypes.byref(st))
    assert got == status


@pytest.mark.parametrize("T,causal,window,req,exp", [
    (8, True, 0, 19, (19, 13824)),      # the q8 verify: ranges over the whole sequence
    (8, False, 4096, 5, (5, 896)),      # a window: ranges over window + block + one tile only
    (8, True, 4096, 2, (2, 2176)),
    (2048, True, 0, 1, (1, 262144)),    # a prefill chunk of 2048 tokens, 10-token slabs
    (2048, True, 0, 3, (3, 87424)),
])
def test_attention_plan_spans(pflib, T, causal, window, req, exp):
    # explicit split counts need no device query (E5M2, group of 6: the tcgen05 kernel, 128-key tiles)
    assert pf.pfkv_attention_plan(1, T, 24, 4, 256, 2048, "e5m2", 262144, causal, window, req) == exp


def test_decode_entry_points_keep_their_token_limit(pflib):
    with pytest.raises(pf.PfkvError) as ei:
        pf.pfkv_decode_plan(1, 17, 8, 8, 128, 16, "e4m3", 4096, 2)
    assert ei.value.status == pf.PFKV_ERR_UNSUPPORTED
    assert pf.pfkv_decode_workspace_bytes(1, 17, 8, 8, 128, 16, "e4m3", 4096, 2) == 0
    assert pf.pfkv_attention_plan(1, 17, 8, 8, 128, 16, "e4m3", 4096, True, 0, 2) == (2, 2048)


def test_decode_validation_before_any_launch(pflib):
    lib = pf.load()
    # null pointers with a valid shape and an explicit split count: rejected on the host
    st = lib.pfkv_paged_attention_decode(None, None, None, None, None, None, 4, None, 2, 1, 32, 8, 128, 16, 64,
                                         1, None, None, ctypes.c_float(0.1), 64, 1, None, 0, None)
    assert st == pf.PFKV_ERR_INVALID_ARG
    # zero sequences is a no-op
    st = lib.pfkv_paged_attention_decode(None, None, None, None, None, None, 4, None, 0, 1, 32, 8, 128, 16, 64,
                                         1, None, None, ctypes.c_float(0.1), 64, 1, None, 0, None)
    assert st == pf.PFKV_OK
    # append: zero tokens is a no-op; bad head_dim is unsupported; null pointers invalid
    assert lib.pfkv_kv_cache_append(None, None, None, None, None, 0, 8, 128, 16, 10, 1, None, None, None) == 0
    assert lib.pfkv_kv_cache_append(None, None, None, None, None, 4, 8, 100, 16, 10, 1, None, None, None) == \
        pf.PFKV_ERR_UNSUPPORTED
    assert lib.pfkv_kv_cache_append(None, None, None, None, None, 4, 8, 128, 16, 10, 1, None, None, None) == \
        pf.PFKV_ERR_INVALID_ARG
    assert "null" in pf.pfkv_last_error()
    # merge: bad sizes
    assert lib.pfkv_lse_merge(None, None, None, None, 4, 0, 128, None) == pf.PFKV_ERR_INVALID_ARG
    assert lib.pfkv_lse_merge(None, None, None, None, 0, 3, 128, None) == pf.PFKV_OK


def test_fragment_layout_checker(tmp_path):
    gxx = shutil.which("g++") or shutil.which("c++")
    if gxx is None:
        pytest.skip("no host C++ compiler")
    exe = tmp_path / "layout_check"
    subprocess.run([gxx, "-std=c++17", "-O1", os.path.join(CSRC, "layout_check.cpp"), "-o", str(exe)], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    assert "layout ok" in r.stdout


def test_zero_blocks_validation_before_any_launch(pflib):
    lib = pf.load()
    # no ids: a no-op; bad head_dim: unsupported; null pointers / misaligned pools: invalid
    assert lib.pfkv_kv_cache_zero_blocks(None, None, None, 0, 8, 128, 16, 10, 1, None) == pf.PFKV_OK
    assert lib.pfkv_kv_cache_zero_blocks(None, None, None, 4, 8, 100, 16, 10, 1, None) == pf.PFKV_ERR_UNSUPPORTED
    assert lib.pfkv_kv_cache_zero_blocks(None, None, None, 4, 8, 128, 16, 10, 1, None) == pf.PFKV_ERR_INVALID_ARG
    assert lib.pfkv_kv_cache_zero_blocks(None, None, None, -1, 8, 128, 16, 10, 1, None) == pf.PFKV_ERR_INVALID_ARG
    assert lib.pfkv_kv_cache_zero_blocks(ctypes.c_void_p(16), ctypes.c_void_p(24), ctypes.c_void_p(32), 4, 8, 128,
                                         16, 10, 1, None) == pf.PFKV_ERR_INVALID_ARG
    assert "aligned" in pf.pfkv_last_error()
    assert lib.pfkv_kv_cache_zero_blocks(None, None, None, 4, 8, 128, 16, 10, 9, None) == pf.PFKV_ERR_INVALID_ARG


def test_zero_blocks_rejects_rows_of_partial_16_byte_stores(pflib):
    lib = pf.load()
    # FP8 rows of 8 bytes (head_dim 8) would need an 8-byte tail store: unsupported; fp16 rows of 16 bytes are fine
    assert lib.pfkv_kv_cache_zero_blocks(None, None, None, 4, 1, 8, 1, 10, 1, None) == pf.PFKV_ERR_UNSUPPORTED
    assert lib.pfkv_kv_cache_zero_blocks(None, None, None, 4, 1, 8, 1, 10, 0, None) == pf.PFKV_ERR_INVALID_ARG


def test_per_head_scale_flag_on_the_host(pflib):
    lib = pf.load()
    per_head = pf.PFKV_KV_SCALES_PER_HEAD
    assert pf.pfkv_capabilities() & 0x8000
    # plan and workspace accept and ignore the flag
    assert pf.pfkv_decode_plan(2, 1, 24, 4, 256, 2048, 1 | per_head, 131072, 38) == \
        pf.pfkv_decode_plan(2, 1, 24, 4, 256, 2048, 1, 131072, 38)
    assert pf.pfkv_decode_workspace_bytes(2, 1, 24, 4, 256, 2048, 2 | per_head, 131072, 38) == \
        pf.pfkv_decode_workspace_bytes(2, 1, 24, 4, 256, 2048, 2, 131072, 38) > 0
    # with an fp16 cache the flag is an invalid argument (there is no scale)
    assert lib.pfkv_kv_cache_append(None, None, None, None, None, 4, 8, 128, 16, 10, 0 | per_head, None, None,
                                    None) == pf.PFKV_ERR_INVALID_ARG
    assert "dtype" in pf.pfkv_last_error()
    with pytest.raises(pf.PfkvError) as ei:
        pf.pfkv_decode_plan(2, 1, 24, 4, 256, 2048, 0 | per_head, 4096, 2)
    assert ei.value.status == pf.PFKV_ERR_INVALID_ARG
    # an unknown format with the flag is still unknown
    assert lib.pfkv_kv_cache_append(None, None, None, None, None, 4, 8, 128, 16, 10, 3 | per_head, None, None,
                                    None) == pf.PFKV_ERR_INVALID_ARG


def test_binding_sets_the_per_head_flag_from_the_scale_tensors():
    import torch
    one, four, three = torch.ones(1), torch.ones(4), torch.ones(3)
    assert pf._kv_scaled("e4m3", one, one, 4) == pf.PFKV_KV_FP8_E4M3
    assert pf._kv_scaled("e5m2", four, four, 4) == pf.PFKV_KV_FP8_E5M2 | pf.PFKV_KV_SCALES_PER_HEAD
    assert pf._kv_scaled("fp16", None, None, 4) == pf.PFKV_KV_FP16
    for k, v in ((three, three), (four, one), (one, four)):  # a count that is neither 1 nor num_kv_heads
        with pytest.raises(pf.PfkvError) as ei:
            pf._kv_scaled("e4m3", k, v, 4)
        assert ei.value.status == pf.PFKV_ERR_INVALID_ARG


def test_header_is_plain_c_and_links_against_the_library(tmp_path, pflib):
    # the boundary is a C ABI: the header compiles as strict C99 and a C program links and calls it
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not available")
    src = tmp_path / "abi.c"
    src.write_text(
        '#include "pfkv.h"\n'
        "#include <stdio.h>\n"
        "int main(void) {\n"
        "  pfkv_kv_dtype d = (pfkv_kv_dtype)(PFKV_KV_FP8_E4M3 | PFKV_KV_SCALES_PER_HEAD);\n"
        "  int ns = 0, st = 0;\n"
        "  pfkv_status s = pfkv_decode_plan(4, 1, 32, 8, 128, 16, d, 4096, 13, &ns, &st);\n"
        '  printf("%d %d %d %s\\n", (int)s, ns, st, pfkv_status_string(s));\n'
        "  return s != PFKV_OK || (pfkv_capabilities() & PFKV_CAP_SCALES_PER_HEAD) == 0;\n"
        "}\n")
    exe = tmp_path / "abi"
    libdir = os.path.dirname(pf.LIB_PATH)
    subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I", os.path.join(ROOT, "include"),
                    str(src), "-o", str(exe), "-L", libdir, "-lpfkv", f"-Wl,-rpath,{libdir}"], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()
    assert out[0] == "0" and out[1] == "13" and int(out[2]) * 13 >= 4096 and out[3] == "PFKV_OK"
