"""pfkv: paged FP8 KV-cache decode attention for GB300 (sm_103a).

The compute path lives in the CUDA library ``libpfkv.so`` (sources in
``csrc/``, C ABI in ``include/pfkv.h``). ``binding`` is a thin ctypes layer
over that ABI with the same entry-point names; it loads the library on first
use and raises if it is missing (there is no CPU fallback). ``workloads``
holds the seeded synthetic inputs.
"""

__all__ = ["binding", "workloads"]
