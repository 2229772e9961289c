"""GB300-native chunkwise gated delta rule (Gated DeltaNet recurrence).

    S_t = alpha_t S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,   o_t = S_t q_t

The computation lives in ``libgdn.so`` (hand-written sm_103a CUDA kernels behind
the C ABI of ``include/gdn.h``); :mod:`.gdn` is its thin Python binding.
"""
from .gdn import (GdnError, gdn_bwd, gdn_bwd_raw, gdn_bwd_workspace_bytes, gdn_fwd,  # noqa: F401
                  gdn_fwd_raw, gdn_fwd_workspace_bytes, gdn_last_error, gdn_saved_bytes,
                  gdn_status_string, gdn_version, load_library, make_problem)
