"""GB300-native batched speculative-decoding verification (accept-or-resample).

The work runs in libspecverify.so (hand-written sm_103a CUDA behind the C ABI of
include/spec_verify.h); this package is its thin ctypes binding.
"""
from ._binding import (SV_DTYPE_BF16, SV_DTYPE_F32, SV_MAX_GAMMA, SV_OK, SpecVerifyError,  # noqa: F401
                       SV_ERR_SCRATCH_TOO_SMALL, SV_NOALLOC_SCRATCH_BYTES,
                       lib, spec_verify, spec_verify_ex, spec_verify_noalloc, spec_verify_onehot,
                       spec_verify_filtered, spec_verify_filter_thresholds,
                       spec_verify_tree_greedy, verify_tree, spec_verify_kv_rollback,
                       spec_verify_status_string,
                       spec_verify_version, spec_verify_workspace_size,
                       spec_verify_filtered_workspace_size,
                       spec_verify_workspace_status, verify, workspace_for,
                       spec_verify_staging_size, spec_verify_staged, spec_verify_staged_h2d_bytes,
                       verify_staged)
from .build import LIB_PATH, build_library  # noqa: F401
