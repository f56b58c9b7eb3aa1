"""GB300 (sm_103a) Lightning Attention RNN mixer: CUDA kernels behind a C ABI
(``include/hla.h``, ``libhla.so``) and a thin PyTorch binding.

The mixer is the RNN layer of HypeNet (arXiv 2601.22156, Appendix A, Eq. 18-19):
QK-RMSNorm, RoPE, the fixed-decay linear recurrence S_t = gamma_h S_{t-1} +
k~_t^T v_t, o_t = q~_t S_t, then the output RMSNorm and sigmoid gate.
"""
from .api import (backward_workspace_size, decode_step, gamma_schedule, make_shape, prefill,
                  prefill_backward, prefill_workspace_size)

__all__ = [
    "prefill", "decode_step", "prefill_backward", "gamma_schedule", "make_shape",
    "prefill_workspace_size", "backward_workspace_size",
]
