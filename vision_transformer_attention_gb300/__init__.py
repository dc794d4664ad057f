"""GB300-native relative-position attention on a 2D patch grid.

The product is the C-ABI CUDA library ``libvta_gb300.so`` (include/rpe_attn.h):
iRPE contextual Product attention and Swin window attention with the relative
bias, hand-written for sm_103a. ``api`` is the thin Python binding; the
library is loaded on first call and its absence is an error, never a
fallback.
"""
from .api import (rpe_attn_bias_fwd, rpe_attn_fwd, rpe_build_bucket_ids, rpe_device_status,  # noqa: F401
                  rpe_release_stream, rpe_shutdown, rpe_wait_probe, swin_window_attn_fwd,
                  swin_window_attn_fwd_fmap)
from ._lib import RPE_TERM_K, RPE_TERM_Q, RPE_TERM_V, RpeError  # noqa: F401
