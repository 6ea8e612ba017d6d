"""Seeded synthetic inputs for CSR SpMM (shared by the oracle tests and the CUDA path).

No product arithmetic lives here: only counter-based random numbers
(:mod:`synth.rng`) and the problem generators (:mod:`synth.workloads`).
"""
from .workloads import (Problem, WORKLOADS, distinct_sorted_columns, knn_kernel_graph,
                        laplacian_2d, power_law, uniform_rows, zipf_lengths)

__all__ = ["Problem", "WORKLOADS", "distinct_sorted_columns", "knn_kernel_graph",
           "laplacian_2d", "power_law", "uniform_rows", "zipf_lengths"]
