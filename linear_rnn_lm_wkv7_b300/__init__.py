"""WKV7 state recurrence for B300 (sm_103a): forward with chunk checkpoints,
checkpointed backward and single-token decode, as hand-written CUDA kernels
behind a C ABI (include/wkv7.h).  This package is the thin Python binding.
"""
from ._binding import (BF16, D_HEAD, F32, LIBRARY_PATH, MAX_CHUNK, SIGNATURES, STATUS, WKV7Error,  # noqa: F401
                       backward, backward_from_forward, backward_workspace_size, debug_enabled, debug_status, decode, forward,
                       forward_workspace_size, lib, num_chunks, version)
