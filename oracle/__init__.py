"""CPU oracle for tree-masked attention (TEST INFRASTRUCTURE ONLY).

This package is the slow, plain, independent definition that the CUDA path is checked
against.  Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import it; the library (``tree_masked_attention_plan_gb300``) never does,
and this package imports nothing from the library.  Everything here is NumPy (fp64 for
floating point, int64 for counts), written from the Tree Training explainer
("Tree Training 技术详解", tingdeliu.github.io) and, for the online-softmax merge, the
Tree Attention page (t6page "Tree Attention", the associativity equation).

Modules
-------
``tree``       tree validation, root-to-leaf path enumeration, the plan (DFS order and
               intervals, depth positions, path counts g_t and weights g_t/K), the
               128x128 tile classes, CSR lists and the heaviest-first work orders.
``attention``  fp64 RoPE, path-expanded causal attention forward+backward (the
               definition), the per-node tree-mask formulation used for large trees,
               and the associative (max, numerator, denominator) softmax merge.
``hybrid``     section 9: the path-expanded causal convolution (forward and backward)
               and the parent-routed recurrent state with its transpose.
``ce``         sections 6.2, 6.3, 12: the path-averaged next-token cross-entropy with ignore
               labels (loss, logsumexp, gradients of the hidden states and the vocabulary
               matrix), whole and restricted to sampled rows.

Parity status: every function here is pinned by ``tests/test_oracle_*.py`` against the
pages' worked example, closed forms, brute force on tiny inputs, library routines in
special cases or finite differences; none is "parity unpinned".
"""
from .tree import (TreeError, validate_tree, root_to_leaf_paths, plan, tile_classes,
                   tree_stats, TILE)
from .attention import (rope, rope_transpose, attention_paths, attention_nodes,
                        merge_softmax_state, softmax_state)
from .hybrid import conv_paths, route_states, route_states_bwd
from .ce import ce_paths, ce_rows

__all__ = ["TreeError", "validate_tree", "root_to_leaf_paths", "plan", "tile_classes",
           "tree_stats", "TILE", "rope", "rope_transpose", "attention_paths",
           "attention_nodes", "merge_softmax_state", "softmax_state", "conv_paths",
           "route_states", "route_states_bwd", "ce_paths", "ce_rows"]
