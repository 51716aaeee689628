"""BaKron solver (Kronecker-factored GPTQ) for GB300 (sm_103a).

The compute path is the C-ABI library ``libbakron.so`` built from
``csrc/``; :mod:`kronecker_factored_gptq_gb300.bakron` is a thin ctypes
binding over it.  Importing this package does not load the library; the first
call into the binding does, and raises if it has not been built.
"""

__all__ = ["bakron", "workloads"]
