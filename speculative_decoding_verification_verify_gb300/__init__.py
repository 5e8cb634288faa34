"""Batched speculative-decoding verifier for NVIDIA GB300 (sm_103a).

The compute lives in libspecverify.so (hand-written CUDA, C ABI in include/spec_verify.h);
`binding` marshals torch tensors into it and `workloads` builds seeded synthetic inputs.
"""
from .binding import (  # noqa: F401
    BF16,
    FP32,
    MODE_GREEDY,
    MODE_REJECTION,
    MODE_TREE,
    MODE_BLOCK,
    Options,
    Result,
    SpecVerifyError,
    load_debug_library,
    load_library,
    spec_verify_block,
    spec_verify_debug_fault,
    spec_verify_greedy,
    spec_verify_kv_compact,
    spec_verify_philox,
    spec_verify_plan_budget,
    spec_verify_rejection,
    spec_verify_rejection_ex,
    spec_verify_strerror,
    spec_verify_tree,
    spec_verify_tree_ex,
    spec_verify_wait_timeouts,
    spec_verify_workspace_bytes,
    using_library,
)
