"""GB300-native TMA-fed bf16 GEMM and TMA tile copy (sm_103a).

The compute path is the C-ABI library `libtg.so` (hand-written CUDA for sm_103a);
`tma_pipelined_tensor_gb300.tg` is its thin ctypes binding.  Importing the package does
not load the library; the binding loads it on first use and raises if it is missing.
"""
__all__ = ["inputs", "tg"]
