"""GB300-native grouped-query-attention AV decode reduction.

    out[b, q_h, d] = sum_{c < L_b} attn[b, c, q_h] * V[b, c, q_h // G, d]

computed by hand-written sm_103a kernels behind a C ABI (include/gqa_av.h),
the decode score step before it (include/gqa_qk.h):

    attn[b, c, q_h] = softmax over c < L_b of scale * q[b, q_h, :] . K[b, c, q_h // G, :]

and both fused in one pass over the KV cache (include/gqa_attn.h).

``workloads`` (seeded inputs) imports without the CUDA library; the binding
functions below need the built library and raise ImportError without it.
"""
from . import workloads  # noqa: F401

_BINDING = ("gqa_av_decode", "gqa_av_decode_per_head", "gqa_av_decode_tuned",
            "gqa_av_decode_noalloc", "gqa_av_plan",
            "gqa_av_workspace_bytes", "gqa_av_set_workspace", "gqa_av_device_status",
            "gqa_av_status_string", "gqa_av_last_error", "GqaAvError", "MODE_AUTO",
            "MODE_PER_HEAD", "MODE_GQA", "GQA_AV_BF16", "GQA_AV_FP16",
            "gqa_qk_softmax_decode", "gqa_qk_device_status", "gqa_av_decode_paged",
            "gqa_attn_decode", "gqa_attn_plan", "gqa_attn_device_status")


def __getattr__(name):
    if name in _BINDING or name == "native":
        from . import _native
        return _native if name == "native" else getattr(_native, name)
    raise AttributeError(name)
