"""GB300-native batched speculative-decoding verification (sm_103a CUDA, C ABI).

The compute path is libspecverify.so (see include/spec_verify.h); this package
is its build step, a ctypes binding and a torch-tensor front end.
"""
from .api import (BoundSample, SamplingParams, VerifyOutput, alloc_outputs, greedy_workspace_size,  # noqa: F401
                  new_workspace, rules_tensor, set_early_logits_reads, transform_probs, tree_sample_workspace_size,
                  tree_workspace_size, verify_greedy, verify_greedy_early, verify_greedy_tree, verify_sample,
                  verify_sample_tree, workspace_size)
from . import _lib  # noqa: F401
