"""DualKV shared-prompt exact attention (forward + backward) for GB300 (sm_103a).

The compute path is the C-ABI library ``libdualkv.so`` (hand-written CUDA
kernels); ``dualkv`` is its thin ctypes binding.  ``workloads`` draws seeded
synthetic inputs.  Importing this package does not load the library; the
binding loads it on first use and raises if it is missing.
"""
__all__ = ["dualkv", "workloads"]
