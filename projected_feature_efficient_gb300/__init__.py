"""GB300 (sm_103a) projected-feature softmax attention.

    Qp = Q P_h,  Kp = K P_h,  O = softmax(Qp Kp^T / sqrt(m)) V

Thin Python binding of ``libspa.so`` (C ABI in include/spa.h).  The binding
only marshals torch tensors into pointers and sizes; every step of the
computation runs in the library's CUDA kernels.  There is no fallback: the
first use of any binding name loads ``libspa.so`` and raises ImportError if it
has not been built (``python -m projected_feature_efficient_gb300.build``).
"""
import importlib

__all__ = [
    "SPA_BF16", "SPA_F32", "SPA_OK", "SPA_ERR_TIMEOUT", "SpaError", "device_error", "lib",
    "lib_path", "selftest_wait_timeout", "selftest_bwd_wait_timeout", "selftest_proj_wait_timeout",
    "selftest_copy_wait_timeout",
    "spa_attention_fwd", "spa_attention_fwd_host",
    "spa_attention_fwd_ws", "spa_attention_workspace_size", "spa_attention_prepare",
    "spa_attention_apply", "spa_project", "status_str", "kcache_new", "spa_kcache_append",
    "spa_attention_decode", "spa_topk_features", "spa_sfa_attention_fwd", "spa_attention_bwd",
    "spa_attention_fwd_lse", "spa_attention_bwd_lse", "spa_attention_bwd_workspace_size",
    "spa_attention_bwd_prepare", "spa_attention_bwd_apply", "spa_attention_bwd_finish",
    "host_pool_trim",
]


def __getattr__(name):
    if name in __all__:
        return getattr(importlib.import_module("._binding", __name__), name)
    raise AttributeError(name)
