"""Seeded synthetic inputs for the verify step.

This package only draws random inputs.  It holds none of the verify step's
arithmetic (no softmax, no accept test, no residual, no inverse CDF), so the
CUDA path and the CPU oracle can both be fed from it without sharing code.
"""
from .workloads import (CONFIGS, TREE_CONFIGS, TreeWorkload, Workload, config, make_tree_workload,  # noqa: F401
                        make_workload, tree_config)
