"""Seeded synthetic inputs shared by the CPU oracle tests, the GPU tests and the bench.

This package holds only input generation: tree shapes (parent[], node_len[]) and
random tensors.  It contains none of the tree-attention arithmetic (no DFS order,
no positions, no masks, no path counts); both the oracle and the CUDA path take
what is generated here as plain inputs.
"""
from .trees import (CONFIGS, Workload, tiny_tree, caterpillar_tree, rollout_tree,
                    forest_tree, large_tree, random_tree, make_workload)
from .tensors import make_conv_tensors, make_tensors

__all__ = ["CONFIGS", "Workload", "tiny_tree", "caterpillar_tree", "rollout_tree",
           "forest_tree", "large_tree", "random_tree", "make_workload", "make_tensors", "make_conv_tensors"]
