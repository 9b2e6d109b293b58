"""B300-native (sm_103a) Medusa decode-step library.

The compute lives in libmedusa_b300.so (CUDA, C ABI in include/medusa.h);
this package is its thin Python binding.  Importing it without the built
library raises ImportError: there is no CPU fallback.
"""
from ._binding import (  # noqa: F401
    DEV_BAD_TOKEN, DEV_KV_OVERFLOW, DEV_NAN, DEV_TIMEOUT, MEDUSA_BF16, MEDUSA_F32, MedusaError, Tree, lib,
    medusa_build_tree, medusa_heads_topk, medusa_heads_topk_tree, medusa_heads_topk_tree_workspace_size,
    medusa_heads_topk_workspace_size, kernel_launches, medusa_kv_commit,
    medusa_tree_attention, medusa_tree_attention_workspace_size, medusa_verify_accept,
    medusa_sample_next, medusa_verify_accept_workspace_size, workspace,
)
from .step import MedusaStep  # noqa: F401

LIB_PATH = lib._name
