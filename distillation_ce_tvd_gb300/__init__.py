"""GB300-native fused cross-entropy + total-variation-distance distillation loss.

The compute path is the C-ABI library ``libfused_ce_tvd.so`` (CUDA kernels for
sm_103a, declared in ``include/fused_ce_tvd.h``).  ``binding`` marshals torch
tensors into it, ``autograd`` ties forward and backward together for
``torch.autograd``, and ``workloads`` draws the seeded synthetic inputs.

The library is loaded on first use; calling an op without it raises.
"""
__all__ = ["binding", "autograd", "workloads"]
