"""The bounded-wait failure path, exercised without a GPU fault.

Every pipeline wait of the library's kernels is an mbarrier wait with a time limit; when the
limit passes, the waiting thread stops waiting, the kernel sets PFKV_DEVERR_TIMEOUT and the
CTA abandons its work instead of spinning on. The product kernels' waits cannot be made to run
out safely (their waits guard copies in flight), so a test-only probe (tests/cuda/
wait_timeout_probe.cu, compiled here, not linked into the library) runs the same wait routine
with a 1 ms limit on an mbarrier that nothing arrives at, and checks that the wait returns
false after the limit, sets the timeout bit and leaves the context usable; a control with an
arrival checks that a completed phase passes at once.
"""

import ctypes
import os
import subprocess

import pytest
import torch

from paged_fp8_kv_cache_gb300 import binding as pf
from paged_fp8_kv_cache_gb300 import build

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def probe(tmp_path_factory):
    so = str(tmp_path_factory.mktemp("waitprobe") / "libwaitprobe.so")
    cmd = [build._nvcc(), *build.ARCH, "-O3", "-std=c++17", "-Xcompiler", "-fPIC", "-shared",
           os.path.join(HERE, "cuda", "wait_timeout_probe.cu"), "-o", so]
    subprocess.run(cmd, check=True, capture_output=True)
    lib = ctypes.CDLL(so)
    lib.pfkv_test_wait_probe.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_ulonglong, ctypes.c_int, ctypes.c_int,
                                                                 ctypes.c_void_p]
    lib.pfkv_test_wait_probe.restype = ctypes.c_int
    return lib


def run_probe(lib, limit_ns, arrive, ctas=4):
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    elapsed = torch.zeros(ctas, dtype=torch.int64, device="cuda")
    ok = torch.full((ctas,), -1, dtype=torch.int32, device="cuda")
    st = lib.pfkv_test_wait_probe(err.data_ptr(), elapsed.data_ptr(), ok.data_ptr(), limit_ns, arrive, ctas,
                                  torch.cuda.current_stream().cuda_stream)
    assert st == 0
    torch.cuda.synchronize()
    return int(err.item()), elapsed.cpu().tolist(), ok.cpu().tolist()


def test_wait_that_nothing_completes_gives_up_and_flags_timeout(probe):
    limit = 1_000_000  # 1 ms
    err, elapsed, ok = run_probe(probe, limit, arrive=0)
    assert ok == [0] * 4
    assert err & pf.PFKV_DEVERR_TIMEOUT
    assert all(limit <= e < 50 * limit for e in elapsed), elapsed
    # the context is still usable afterwards
    x = torch.arange(1000, device="cuda", dtype=torch.float32)
    assert float(x.sum().item()) == 499500.0


def test_completed_phase_passes_at_once(probe):
    err, elapsed, ok = run_probe(probe, 1_000_000, arrive=1)
    assert ok == [1] * 4 and err == 0
    assert all(e < 1_000_000 for e in elapsed), elapsed
