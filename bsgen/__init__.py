"""Seeded synthetic inputs shared by the CUDA-path tests, the bench and the oracle.

Only structure descriptions (sector axes, rule parameters, layout names) and
value draws live here; nothing in this package evaluates a rule, builds a
layout or contracts blocks.
"""
from . import rng
from .configs import (CONFIGS, OP_A, OP_B, Axis, Rule, Workload, chain2, config1, config2, config3,
                      config4, config5, get, tiny_random)

__all__ = ["rng", "CONFIGS", "OP_A", "OP_B", "Axis", "Rule", "Workload", "config1", "config2",
           "config3", "config4", "config5", "get", "tiny_random", "chain2"]
