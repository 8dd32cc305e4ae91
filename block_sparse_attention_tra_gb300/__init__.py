"""GB300-native fused causal attention forwards.

Two forwards that never materialise the T x T score matrix, each one CUDA
kernel for sm_103a behind a C ABI (``include/bsa.h``, ``libbsa.so``):

* ``tra_forward``        -- threshold rectified attention,
  ``out = ReLU(Q K^T - tau(i))^p V`` with ``tau(i) = beta sqrt(2 ln(i+1)/D)``,
  causal and unnormalised (page "triton_threshold_attention.py").
* ``nsa_select_forward`` -- NSA selection-branch attention over gathered key
  blocks, GQA, causal, scaled softmax (page "nsa_selection_kernel.py").
* ``nsa_select_forward_fsa`` -- the same result in the page's block-outer
  split-K form: each selected block's K/V read once, per-pair softmax
  partials, a log-sum-exp combine.
* ``tra_forward_host`` -- ``tra_forward`` on host tensors, streamed through
  the GPU in chunks of heads with overlapped copies.
* ``tra_backward`` and ``tra_attention`` -- the gradients of ``tra_forward``,
  and the forward as a ``torch.autograd.Function`` whose backward runs them
  (the page's ThresholdRelaFunction); ``tra_diff_forward``,
  ``tra_diff_backward`` and ``tra_diff_attention`` -- the page's differential
  form, its gradients and the two as an autograd function.

The binding in ``bsa`` only marshals arguments; every step runs in the CUDA
library, which is loaded on first use and must be built (``build.build()``).
"""

from .bsa import (  # noqa: F401
    BsaError,
    device_error,
    library_path,
    load_library,
    nsa_select_forward,
    nsa_select_forward_fsa,
    nsa_select_forward_fsa_raw,
    nsa_select_forward_raw,
    nsa_select_fsa_workspace_size,
    status_string,
    tra_attention,
    tra_backward,
    tra_backward_raw,
    tra_diff_attention,
    tra_diff_backward,
    tra_diff_backward_raw,
    tra_diff_forward,
    tra_diff_forward_raw,
    tra_forward,
    tra_forward_ex_raw,
    tra_forward_host,
    tra_forward_host_raw,
    tra_forward_host_workspace_size,
    tra_forward_raw,
)

__all__ = [
    "BsaError",
    "device_error",
    "library_path",
    "load_library",
    "tra_forward",
    "tra_forward_raw",
    "tra_forward_ex_raw",
    "tra_forward_host",
    "tra_forward_host_raw",
    "tra_forward_host_workspace_size",
    "tra_attention",
    "tra_backward",
    "tra_backward_raw",
    "tra_diff_attention",
    "tra_diff_backward",
    "tra_diff_backward_raw",
    "tra_diff_forward",
    "tra_diff_forward_raw",
    "nsa_select_forward",
    "nsa_select_forward_raw",
    "nsa_select_forward_fsa",
    "nsa_select_forward_fsa_raw",
    "nsa_select_fsa_workspace_size",
    "status_string",
]
