"""GB300 (sm_103a) HiSA sparse-attention step: CUDA kernels behind a C-ABI library.

The compiled library ``libhisa.so`` is loaded lazily by ``binding``; importing
this package does not touch the GPU.
"""
