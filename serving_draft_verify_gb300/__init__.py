"""DSpark draft / schedule / verify / accept-rate path on one GB300 (sm_103a).

The compute lives in libdspark.so (CUDA kernels behind a C ABI, declared in
include/dspark.h); this package holds its build script, the ctypes binding
(same names as the C entry points) and the seeded synthetic workloads.
"""
from ._binding import (  # noqa: F401
    DSparkError,
    LIB_PATH,
    MAX_GAMMA,
    dspark_accept_rate_tv,
    dspark_training_loss,
    dspark_decode_rounds,
    dspark_draft_block_ex,
    dspark_verify_ex,
    HEAD_MARKOV,
    HEAD_GATED,
    HEAD_RNN,
    dspark_draft_block,
    dspark_schedule_prefix,
    dspark_set_l2_residency,
    dspark_verify,
    exported_symbols,
    load,
    status_string,
    workspace_status,
)
