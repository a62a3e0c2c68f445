"""paged_kv_gqa_table_gb300: paged-KV GQA decode attention and MLA paged causal
prefill for GB300 (sm_103a), as hand-written CUDA kernels behind a C-ABI
library (``libpkv.so``).

The Python layer marshals arguments only; every step of the computation runs
in the library's kernels.  Importing this package does not load the library:
the first call through :mod:`paged_kv_gqa_table_gb300.binding` does, and it
raises if the library is missing.
"""
__all__ = ["binding", "synth"]
