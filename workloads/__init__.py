"""Seeded synthetic workloads for the KDA forward (input generation only)."""
from .synthetic import WORKLOADS, Workload, custom, make_inputs, token_heads, varlen_lengths

__all__ = ["WORKLOADS", "Workload", "custom", "make_inputs", "token_heads", "varlen_lengths"]
