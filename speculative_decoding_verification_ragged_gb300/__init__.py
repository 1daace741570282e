"""GB300-native batched draft-token verification for speculative decoding.

The compute path is libspecverify.so (hand-written sm_103a CUDA behind the C
ABI in include/spec_verify.h); this package holds its sources (csrc/), the
in-tree build (_build.py) and a thin ctypes binding (binding.py).
"""
from ._build import build  # noqa: F401
from .binding import (  # noqa: F401
    EXPORTS, SpecError, StepController, draft_confidence, load_library, new_workspace,
    prefix_stats, restore_rows, step_cost_additive, step_cost_sps,
    verify_greedy, verify_greedy_active, verify_greedy_margin, verify_greedy_noalloc, verify_relaxed_topk,
    verify_sample, workspace_bytes,
)

__all__ = ["build", "load_library", "new_workspace", "workspace_bytes", "verify_greedy",
           "verify_greedy_noalloc", "verify_greedy_margin", "verify_greedy_active",
           "verify_relaxed_topk", "verify_sample", "draft_confidence", "prefix_stats",
           "restore_rows", "StepController", "step_cost_sps", "step_cost_additive", "SpecError", "EXPORTS"]
