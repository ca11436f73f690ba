"""paged_fp8_kv_decode_gb300: decode attention over a paged FP8/BF16 KV cache on GB300.

The compute lives in ``libpfkv.so`` (hand-written CUDA for sm_103a behind a C
ABI, declared in ``include/pfkv.h``).  ``binding`` marshals arguments to it;
``workloads`` draws seeded synthetic batches.  Importing this package does not
load the library; the first call into ``binding`` does, and fails loudly if the
library has not been built.
"""
__all__ = ["binding", "workloads"]
