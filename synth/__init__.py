"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle checks."""
from .inputs import (WORKLOADS, Workload, Inputs, generate, normal_bf16, f32_to_bf16_bits, to_bits,
                     bf16_bits_to_f32, random_importance, sweep_points)
