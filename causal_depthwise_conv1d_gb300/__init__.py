"""GB300-native causal depthwise conv1d: forward pass, decode-step update and
backward pass.

The compute lives in hand-written sm_103a CUDA kernels behind a C ABI
(``include/ccv.h``, built into ``libccv.so`` next to this file).  The binding in
``binding.py`` only marshals torch tensors into that ABI.  Importing the
package is cheap; the shared library is loaded on first use of a binding
name and a missing library raises immediately (there is no CPU fallback).
"""
_BINDING_NAMES = ("ccv_fwd", "ccv_fwd_ptr", "ccv_update", "ccv_bwd", "ccv_bwd_ptr", "ccv_bwd_workspace_size",
                  "ccv_last_error", "ccv_last_kernel", "ccv_version", "ccv_device_fault", "ccv_test_bounded_wait",
                  "load_library",
                  "CcvError", "causal_conv1d_fwd", "causal_conv1d_update", "causal_conv1d_bwd")


def __getattr__(name):
    if name in _BINDING_NAMES:
        from . import binding
        return getattr(binding, name)
    raise AttributeError(name)
