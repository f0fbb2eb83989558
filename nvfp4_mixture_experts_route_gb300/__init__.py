"""Routed NVFP4 mixture-of-experts expert block for GB300 (sm_103a).

The compute runs in hand-written CUDA kernels behind the C-ABI library
``libmoe_nvfp4.so`` (declared in ``include/moe_nvfp4.h``); ``binding`` loads
it with ctypes and marshals pointers. PyTorch supplies device memory and
streams only.
"""
