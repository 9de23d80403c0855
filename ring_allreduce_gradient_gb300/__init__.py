"""GB300-native data-parallel collective data path (virtual ranks on one GPU).

The work runs in hand-written sm_103a CUDA kernels behind the C ABI declared
in ``include/dp.h`` (library ``libdp_gb300.so``); ``binding`` marshals
arguments to it through ctypes.  PyTorch supplies device memory and streams.
"""
