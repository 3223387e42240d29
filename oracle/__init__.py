"""CPU oracle for the tree-verify step (test infrastructure only).

Only the test suite, the package smoke check and the benchmark's CPU
baseline / reference leg use this package; the product path never does.
"""
from .tree_verify import (  # noqa: F401
    accept, ancestors, argmax_row, argmax_rows, attention_one_sequence, check_tree,
    commit, depths, gather_pages, prefix_kv, seq_capacity, tree_attention, verify_step,
)
