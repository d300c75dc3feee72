"""FP8 (E4M3FN) per-token/per-head KV cache for BF16 attention on one GB300 GPU.

The compute path is the C-ABI library ``libftkv.so`` (hand-written sm_103a CUDA kernels, declared in
``include/ftkv.h``); ``fp8_kv_cache_ftkv_gb300.ops`` marshals torch CUDA tensors into it.  Importing
this package does not load the library; the first call does, and fails loudly if it is missing.
"""
