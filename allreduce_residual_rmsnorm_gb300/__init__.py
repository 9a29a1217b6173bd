"""GB300-native allreduce-fusion epilogue: R-way rank sum + residual add +
RMSNorm (+ FP8 E4M3 / NVFP4 quantisation), single GPU.

The compute runs in the C-ABI library ``libarfusion.so`` (hand-written sm_103a
CUDA kernels); :mod:`.binding` marshals torch tensors into it.  The library is
loaded on first use and there is no fallback: if it is missing, calls raise.
"""
__all__ = ["binding", "workloads"]
