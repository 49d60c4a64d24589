"""Exact tiled attention with online softmax for one GB300 (sm_103a).

The compute lives in the CUDA library ``libfa_gb300.so`` (C ABI in
``include/fa_gb300.h``); this package builds it, loads it and marshals torch
tensors to it.  Importing the package does not load the library; the first call
does, and fails loudly if the library was not built.
"""
from ._lib import build, load  # noqa: F401
from .api import (FaError, attention_backward, attention_forward, attention_forward_fp8,  # noqa: F401
                  attention_forward_splitkv, fa_bwd, fa_bwd_main, fa_bwd_postprocess, fa_bwd_preprocess,
                  fa_bwd_workspace_size, fa_fwd, fa_fwd_fp8, fa_fwd_splitkv, fa_fwd_splitkv_pick_splits,
                  fa_fwd_splitkv_workspace_size, fa_get_device_status, new_workspace)
