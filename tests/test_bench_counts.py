"""The benchmark's algorithmic byte and flop counts (the roofline numerators),
checked on small workloads against counts written out by hand (CPU only)."""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import workloads  # noqa: E402


def test_projection_counts_touched_slots_at_true_rank():
    wl = workloads.random_small(seed=3, M=6, K=16, N=24, L=3, R=8, ranks=[2, 5, 0])
    wl.seq_slot[:] = [0, 0, 1, -1, 2, 7]  # slot 2 is empty, 7 is past max_loras
    byts, flops = bench.proj_algorithmic(wl)
    M, K, N = 6, 16, 24
    want_b = N * K * 2 + M * K * 2 + M * N * 2 + M * 4 + (2 * K + N * 2) * 2 + (5 * K + N * 5) * 2
    want_f = 2.0 * M * N * K + 2 * (2.0 * 2 * (K + N)) + 2.0 * 5 * (K + N)
    assert byts == want_b and flops == want_f


def test_stack_counts_members_without_zero_scale():
    wl = workloads.stacked(seed=4, M=5, K=16, N=8, L=2, R=16, ranks=(1, 3), max_members=3,
                           zero_member_slot=0)
    wl.seq_slot[:] = [0, 0, 1, -1, 1]
    byts, flops = bench.stack_algorithmic(wl)
    M, K, N = 5, 16, 8
    want_b = N * K * 2 + M * K * 2 + M * N * 2 + M * 4
    want_f = 2.0 * M * N * K
    for s in (0, 1):
        live = [m for m in wl.stacks[s] if m.adapter_scale != 0.0]
        want_b += sum((m.rank * K + N * m.rank) * 2 for m in live)
        rows = int(np.sum(wl.seq_slot == s))
        want_f += rows * sum(2.0 * m.rank * (K + N) for m in live)
    assert any(m.adapter_scale == 0.0 for m in wl.stacks[0])  # the zero-scale member is left out
    assert byts == want_b and flops == want_f


def test_moe_gather_counts_each_named_expert_once():
    wl = workloads.moe_gather(seed=5, tokens=3, E=4, top_k=2, K=16, N=8, n_adapters=2, rank=4)
    wl.indices[:] = [0, 2, 2, 0, 0, 2]  # experts 1 and 3 are never named
    wl.seq_slot[:] = [1, 1, -1, -1, 0, 0]
    byts, flops = bench.moe_gather_algorithmic(wl)
    T, K, N = 6, 16, 8
    want_b = T * K * 2 + 3 * N * 2 + T * 4 * 3 + 2 * N * K * 2
    # expert 0: slot-rows 0 (slot 1) and 4 (slot 0); expert 2: slot-rows 1 (slot 1) and 5 (slot 0)
    want_b += 4 * ((4 * K + N * 4) * 2)
    want_f = 2.0 * T * N * K + 4 * 2.0 * 4 * (K + N)
    assert byts == want_b and flops == want_f


def test_embedding_counts_rows_gathered_and_touched_slots():
    wl = workloads.embed(seed=8, M=6, vocab=40, n_embd=16, L=3, R=8, ranks=[2, 5, 3])
    wl.seq_slot[:] = [0, 0, 1, -1, 5, 0]  # slot 2 is never named, 5 is past max_loras
    byts, flops = bench.embed_algorithmic(wl)
    M, n = 6, 16
    # E rows in, y rows out, tokens and slots; one B row per adapted row; A of slots 0 and 1
    want_b = 2 * M * n * 2 + M * 4 * 2 + (3 * 2 + 1 * 5) * 2 + (2 * n + 5 * n) * 2
    want_f = 3 * 2.0 * 2 * n + 2.0 * 5 * n
    assert byts == want_b and flops == want_f


def test_moe_counts_only_experts_with_rows_and_live_adapters():
    wl = workloads.make("moe", seed=9, tokens=6, E=3, top_k=2, K=16, N=8, n_adapters=2, rank=4)
    wl.expert_offsets[:] = [0, 5, 5, 12]  # expert 1 has no rows
    wl.seq_slot[:] = [0, 0, 1, -1, 1, 1, 1, -1, 0, 7, 0, 1]
    wl.adapters[2][0].adapter_scale = 0.0  # expert 2's slot 0 is switched off
    byts, flops = bench.moe_algorithmic(wl)
    T, E, K, N = 12, 3, 16, 8
    pair = (4 * K + N * 4) * 2
    want_b = T * K * 2 + T * N * 2 + T * 4 + (E + 1) * 4 + 2 * N * K * 2 + 3 * pair
    # expert 0: four adapted rows over slots {0, 1}; expert 2: three rows of slot 1
    want_f = 2.0 * T * N * K + 7 * 2.0 * 4 * (K + N)
    assert byts == want_b and flops == want_f


def test_gate_up_writes_the_activation_not_the_halves():
    wl = workloads.random_small(seed=10, M=5, K=16, N=24, L=2, R=8, ranks=[3, 4])
    wl.seq_slot[:] = [0, 1, 1, -1, 0]
    byts, flops = bench.gate_up_algorithmic(wl)
    M, K, N, I = 5, 16, 24, 12
    want_b = N * K * 2 + M * K * 2 + M * I * 2 + M * 4 + (3 * K + N * 3) * 2 + (4 * K + N * 4) * 2
    want_f = 2.0 * M * N * K + 2 * 2.0 * 3 * (K + N) + 2 * 2.0 * 4 * (K + N)
    assert byts == want_b and flops == want_f
