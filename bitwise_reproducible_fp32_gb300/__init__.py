"""Bit-exact fixed-order FP32 hot path (GEMM, RMSNorm, softmax cross-entropy,
AdamW) for GB300 (sm_103a): ctypes binding over the C-ABI library
``libdetfp32.so``. The library is loaded on first use; a missing or unbuilt
library raises instead of falling back to anything else."""
