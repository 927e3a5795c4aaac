"""Seeded synthetic workloads shared by the tests, the bench and the oracle's checks."""
from .synth import (Adapter, EmbedWorkload, MoeGatherWorkload, MoeWorkload, ProjWorkload, StackWorkload,
                    CONFIGS, bf16_to_f32, embed, f32_to_bf16, make, moe_gather, random_small, stacked)

__all__ = ["Adapter", "EmbedWorkload", "MoeGatherWorkload", "MoeWorkload", "ProjWorkload", "CONFIGS",
           "bf16_to_f32", "embed", "f32_to_bf16", "make", "moe_gather", "random_small", "StackWorkload",
           "stacked"]
