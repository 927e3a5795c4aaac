"""Seeded synthetic workloads shared by the tests, the bench and the oracle's checks."""
from .synth import (Adapter, MoeWorkload, ProjWorkload, CONFIGS, bf16_to_f32, f32_to_bf16,
                    make, random_small)

__all__ = ["Adapter", "MoeWorkload", "ProjWorkload", "CONFIGS", "bf16_to_f32",
           "f32_to_bf16", "make", "random_small"]
