"""Document-masked (varlen) causal grouped-query attention for GB300 (sm_103a).

The compute lives in the C-ABI library libvsw_attn.so (include/attn_varlen.h,
include/gdn_varlen.h and include/kda_varlen.h for the Gated DeltaNet and Kimi
Delta local layers);
``binding`` marshals torch CUDA tensors into it.  ``synth`` generates the
seeded packed-document workloads.  ``layer`` wraps one attention layer
(projections, the library's attention on strided views, a small loss, and the
backward) for CUDA-graph replay.
"""
from importlib import import_module

_BINDING_NAMES = {
    "attn_varlen_fwd", "attn_varlen_bwd", "attn_varlen_bwd_workspace_bytes", "attn_varlen_get_status",
    "attn_varlen_strerror", "attn_varlen_mask_ranges", "attn_varlen_bwd_preprocess", "attn_varlen_bwd_plan",
    "attn_varlen_bwd_dkdv", "attn_varlen_bwd_dq", "attn_varlen_bwd_noalloc", "attn_varlen_fwd_strided",
    "attn_varlen_bwd_strided", "attn_varlen_set_workspace", "attn_varlen_workspace_bytes", "load_library",
    "AttnError", "gdn_varlen_fwd", "gdn_varlen_workspace_bytes", "gdn_varlen_bwd", "gdn_varlen_bwd_workspace_bytes",
    "kda_varlen_fwd", "kda_varlen_workspace_bytes", "kda_varlen_bwd", "kda_varlen_bwd_workspace_bytes",
}


def __getattr__(name):
    if name in _BINDING_NAMES:
        return getattr(import_module(".binding", __name__), name)
    raise AttributeError(name)
