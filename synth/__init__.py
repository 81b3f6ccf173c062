"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle checks."""
from .workloads import (CANARY_BF16_BITS, SPECS, Spec, Workload, bf16_bits, decode_queries, generate,
                        host_subset, sweep_spec)

__all__ = ["CANARY_BF16_BITS", "SPECS", "Spec", "Workload", "bf16_bits", "decode_queries", "generate",
           "host_subset", "sweep_spec"]
