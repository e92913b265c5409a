"""B300 (sm_103a) gated delta rule and causal linear attention prefill.

The computation runs in hand-written CUDA kernels in libgdn_b300.so behind the
C ABI of include/gdn.h; this package is its thin PyTorch-tensor binding.
"""
from ._lib import (CHUNK, GdnError, chunk_fwd_workspace_size, gdn_chunk_fwd,  # noqa: F401
                   gdn_chunk_fwd_staged, gdn_chunk_prepare, gdn_recurrent_step, lib,
                   linear_attn_fwd, set_wait_limit, staged_workspace_size, status_string,
                   two_level_segments, linear_attn_variant,
                   version, workspace_status, workspace_timeout_site, LIB_PATH)
