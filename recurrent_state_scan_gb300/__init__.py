"""Gated delta-rule recurrent state scan (Gated DeltaNet) on NVIDIA GB300.

The compute lives in libgdn (CUDA for sm_103a, C ABI declared in include/gdn.h);
this package builds it in-tree and binds it with ctypes.
"""
from .gdn import (GdnError, GdnShape, gdn_causal_conv, gdn_causal_conv_slots,  # noqa: F401
                  gdn_decode_layer, gdn_decode_step, gdn_prefill_layer, gdn_decode_step_slots, gdn_gated_rmsnorm,
                  gdn_last_device_status,
                  gdn_prefill, gdn_prefill_noalloc, gdn_prefill_norm, gdn_prefill_variant,
                  gdn_prefill_variant_plan, gdn_prefill_variant_workspace_bytes,
                  gdn_prefill_workspace_bytes,
                  gdn_scan_variant, gdn_scan_window, gdn_status_string, load)
