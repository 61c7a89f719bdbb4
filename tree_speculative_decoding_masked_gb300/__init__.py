"""GB300-native verification of speculative-decoding draft trees.

The compute path is libtreeverify.so (hand-written sm_103a CUDA behind a C ABI, see
include/treeverify.h); this package is its Python binding.  The binding only marshals
arguments; if the library is missing, calls raise instead of falling back to anything.
"""
from ._binding import (  # noqa: F401
    TV_BF16,
    TV_DEV_BAD_TOKEN,
    TV_DEV_BAD_TREE,
    TV_DEV_TIMEOUT,
    TV_F32,
    TreeVerifyError,
    commit_accepted_kv,
    expand_children,
    expand_workspace_size,
    exported_symbols,
    frontier_topw,
    library_path,
    load_library,
    philox4x32_10,
    prune_tree,
    select_subtree,
    select_workspace_size,
    selftest_bounded_wait,
    set_attention_splits,
    set_attention_variant,
    set_sm_partition,
    status_string,
    tree_attention,
    tree_attention_plan,
    tree_attention_workspace_size,
    tree_prep,
    verify_greedy,
    verify_greedy_static,
    verify_sample,
    verify_workspace_size,
    vocab_stats,
)
