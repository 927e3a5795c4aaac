"""Seeded synthetic workloads shared by the tests, the bench and the oracle's checks."""
from .synth import (Adapter, EmbedWorkload, MoeWorkload, ProjWorkload, CONFIGS, bf16_to_f32,
                    embed, f32_to_bf16, make, random_small)

__all__ = ["Adapter", "EmbedWorkload", "MoeWorkload", "ProjWorkload", "CONFIGS", "bf16_to_f32",
           "embed", "f32_to_bf16", "make", "random_small"]
