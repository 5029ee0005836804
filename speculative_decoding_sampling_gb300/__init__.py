"""GB300 (sm_103a) speculative-sampling verification.

One call verifies a batch: softmax of the target logits at temperature T,
left-to-right accept test u < min(1, p(x)/q(x)), first rejection, and the
final token drawn by inverse CDF from max(0, p - q) (after a rejection) or
from p_{K+1} (all drafts accepted).  The work runs in the CUDA kernels of
libspecverify.so (C ABI: include/spec_verify.h); this package is the thin
PyTorch binding.  There is no CPU fallback: if the library is not built,
every call raises.
"""
from ._native import (SV_BAD_Q, SV_BAD_ROW, SV_BAD_TOKEN, SV_BAD_U, SV_BF16,
                      SV_DEGENERATE_RESIDUAL, SV_EINVAL, SV_ECUDA,
                      SV_EUNSUPPORTED, SV_FP32, SV_MAX_V, SV_OK,
                      NativeLibraryMissing)
from .binding import (SpecVerifyError, SpecVerifyResult, default_workspace,
                      spec_verify, sv_filter_logits, sv_kernel_launches, sv_sample_survivors,
                      sv_status_string, sv_verify_rows, sv_workspace_bytes,
                      spec_verify_lm_head, sv_lm_head_logits, sv_lm_head_workspace_bytes,
                      TreeResult, spec_verify_tree, sv_tree_workspace_bytes)
from . import adaptive

__all__ = [
    "spec_verify", "sv_verify_rows", "sv_sample_survivors",
    "spec_verify_lm_head", "sv_lm_head_logits", "sv_lm_head_workspace_bytes",
    "spec_verify_tree", "sv_tree_workspace_bytes", "TreeResult",
    "sv_workspace_bytes", "sv_filter_logits", "sv_kernel_launches", "sv_status_string", "default_workspace",
    "SpecVerifyResult", "SpecVerifyError", "NativeLibraryMissing",
    "SV_OK", "SV_EINVAL", "SV_ECUDA", "SV_EUNSUPPORTED", "SV_BF16", "SV_FP32",
    "SV_BAD_U", "SV_BAD_TOKEN", "SV_BAD_Q", "SV_BAD_ROW",
    "SV_DEGENERATE_RESIDUAL", "SV_MAX_V", "adaptive",
]
