"""libverkv: VerKV's decode-time hot path (PoissonComp, shrinkage-estimator attention, Bernstein
certificate, fetch and refine) as hand-written CUDA for sm_103a behind a C ABI.

`binding` is the thin ctypes layer over libverkv.so (same names as include/verkv.h); `inputs`
holds the seeded synthetic workloads.  Importing the package loads nothing; the CUDA library is
loaded on first use of `binding.lib()` and raises if it is missing.
"""
__all__ = ["binding", "inputs"]
