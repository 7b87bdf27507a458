"""Gated delta rule kernels for GB300 (sm_103a): chunked prefill, one-token decode, gated norm.

The compute lives in libgdn.so (hand-written CUDA, C ABI in include/gdn.h); this package only
builds it and binds it.  Import is cheap: the library is loaded on the first call.
"""
from ._binding import (  # noqa: F401
    GDN_BF16,
    GDN_F32,
    GDN_FORM_AUTO,
    GDN_FORM_OFF,
    GDN_FORM_ON,
    GdnError,
    gdn_chunk_fwd,
    gdn_chunk_fwd_noalloc,
    gdn_decay_from_logits,
    gdn_gate_rmsnorm_silu,
    gdn_get_device_error,
    gdn_recurrent_multi_step,
    gdn_recurrent_step,
    gdn_selftest_bounded_wait,
    gdn_set_kernel_forms,
    lib,
)

__all__ = ["gdn_chunk_fwd", "gdn_chunk_fwd_noalloc", "gdn_recurrent_step", "gdn_recurrent_multi_step",
           "gdn_gate_rmsnorm_silu", "gdn_decay_from_logits", "gdn_get_device_error",
           "gdn_selftest_bounded_wait", "gdn_set_kernel_forms", "GdnError", "lib", "GDN_F32", "GDN_BF16",
           "GDN_FORM_AUTO", "GDN_FORM_OFF", "GDN_FORM_ON"]
