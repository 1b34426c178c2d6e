"""Seeded synthetic inputs for the verify step.

This package only draws random inputs.  It holds none of the verify step's
arithmetic (no softmax, no accept test, no residual, no inverse CDF), so the
CUDA path and the CPU oracle can both be fed from it without sharing code.
"""
from .workloads import (CONFIGS, FUSED_CONFIGS, TREE_CONFIGS, FusedWorkload, TreeWorkload, Workload,  # noqa: F401
                        config, make_fused_workload, make_tree_workload, make_workload, tree_config)
