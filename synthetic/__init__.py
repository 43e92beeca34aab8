"""Seeded synthetic inputs shared by the oracle, the tests and the benchmark.

This package holds no decoder arithmetic: it only defines the workload shapes
and produces seeded FP16 weights and prompt token ids.  Both the CPU oracle and
the CUDA path receive the tensors it returns as plain data.
"""
from .configs import ModelConfig, Workload, MODELS, WORKLOADS, workload  # noqa: F401
from .inputs import make_weights, make_prompt, normal_table, WEIGHT_ORDER  # noqa: F401
