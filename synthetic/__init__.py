"""Seeded synthetic inputs shared by the oracle, the tests and the benchmark.

This package holds no decoder arithmetic: it only defines the workload shapes
and produces seeded FP16 (or FP8 E4M3 + per-row scale) weights and prompt token
ids.  Both the CPU oracle and
the CUDA path receive the tensors it returns as plain data.
"""
from .configs import ModelConfig, Workload, MODELS, WORKLOADS, workload  # noqa: F401
from .inputs import (make_weights, make_weights_fp8, make_prompt, normal_table, fp8_code_table,  # noqa: F401
                     WEIGHT_ORDER, FP8_MATRICES)
