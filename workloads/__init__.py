"""Seeded synthetic workloads for the KDA forward (input generation only)."""
from .synthetic import (DECODE_WORKLOADS, WORKLOADS, Workload, custom, make_decode_inputs,
                        make_inputs, token_heads, varlen_lengths)

__all__ = ["WORKLOADS", "DECODE_WORKLOADS", "Workload", "custom", "make_inputs",
           "make_decode_inputs", "token_heads", "varlen_lengths"]
