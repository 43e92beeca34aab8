"""Seeded synthetic inputs shared by the oracle, the tests and the benchmark.

This package holds no decoder arithmetic: it only defines the workload shapes
and produces seeded FP16 (or FP8 E4M3 + per-row scale, or MXFP4 codes + block
scale) weights and prompt token ids.  Both the CPU oracle and
the CUDA path receive the tensors it returns as plain data.
"""
from .configs import ModelConfig, Workload, MODELS, WORKLOADS, workload  # noqa: F401
from .inputs import (make_weights, make_weights_fp8, make_weights_mxfp4, make_prompt, normal_table,  # noqa: F401
                     fp8_code_table, mxfp4_byte_table, WEIGHT_ORDER, FP8_MATRICES)
