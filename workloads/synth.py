"""Seeded synthetic inputs for the multi-adapter LoRA projection.

This module is shared by the CUDA path's tests/bench and by the oracle's
tests. It draws inputs only: it holds none of the method's arithmetic
(no scale rule, no product, no routing sort). Every floating-point input is
drawn in fp32 and rounded once, round-to-nearest-even, to bf16; both sides
consume the same bf16 bytes (held here as ``numpy.uint16``).

Workloads follow the five shapes the pages' engines run:

* ``tiny``    -- 8 rows, 256x256 base, 4 adapters of rank 8 (seed 0);
* ``decode``  -- 64 rows, 4096x4096 base, 16 adapters of ranks {8,16,32,64},
                 pool rank 64, 10% of rows without an adapter (seed 1);
* ``qkv``     -- 256 rows, fused q/k/v base 6144x4096 (4096+1024+1024 rows),
                 32 adapters of rank 16, Zipf(1.1) routing, 5% rows without
                 an adapter, adapter scales from {0, 0.5, 1} (seed 2);
* ``prefill`` -- 8192 rows as 8 sequences of 1024, 14336x4096 gate/up base,
                 8 adapters of rank 64 under rsLoRA, one per sequence (seed 3);
* ``moe``     -- 8 experts of 4096x14336 (down projection), 512 tokens routed
                 top-2 (1024 slot-rows grouped by expert), 4 adapters of rank 16
                 per expert (seed 4).

Draw order inside each generator is fixed and documented in the function, so
a given seed always yields the same bytes (numpy ``PCG64``).
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional

import numpy as np

# ----------------------------------------------------------------------------
# bf16 helpers (storage format only)
# ----------------------------------------------------------------------------


def f32_to_bf16(a: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest, ties to even); returns uint16 bits.

    Inputs here are finite, so no NaN special-casing is needed.
    """
    a = np.ascontiguousarray(a, dtype=np.float32)
    out = np.empty(a.shape, dtype=np.uint16)
    flat_in = a.reshape(-1)
    flat_out = out.reshape(-1)
    step = 1 << 24
    for s in range(0, flat_in.size, step):
        u = flat_in[s:s + step].view(np.uint32).astype(np.uint64)
        u += ((u >> 16) & 1) + 0x7FFF
        flat_out[s:s + step] = (u >> 16).astype(np.uint16)
    return out


def bf16_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bits (uint16) to fp32 exactly."""
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


# ----------------------------------------------------------------------------
# Containers
# ----------------------------------------------------------------------------


@dataclass
class Adapter:
    """One adapter's pair at its true rank, PEFT layout.

    ``A`` is ``[rank][n_in]`` and ``B`` is ``[n_out][rank]`` (bf16 bits).
    ``alpha`` is the file's alpha (0 = absent), ``use_rslora`` selects the
    square-root rule, ``adapter_scale`` is the runtime multiplier.
    """

    A: np.ndarray
    B: np.ndarray
    rank: int
    alpha: float
    use_rslora: bool = False
    adapter_scale: float = 1.0


@dataclass
class ProjWorkload:
    name: str
    seed: int
    M: int
    K: int
    N: int
    max_loras: int
    max_rank: int
    W: np.ndarray               # [N][K] bf16 bits
    x: np.ndarray               # [M][K] bf16 bits
    seq_slot: np.ndarray        # [M] int32, <0 = no adapter
    adapters: List[Optional[Adapter]]  # length max_loras
    splits: Optional[List[int]] = None  # row blocks of a fused base (q, k, v)
    note: str = ""


@dataclass
class MoeWorkload:
    name: str
    seed: int
    E: int
    T: int                      # slot-rows (tokens x top_k)
    K: int                      # n_in of one expert (intermediate size)
    N: int                      # n_out of one expert (hidden size)
    max_loras: int
    max_rank: int
    W: List[np.ndarray]         # E x [N][K] bf16 bits
    x: np.ndarray               # [T][K] bf16 bits, rows grouped by expert
    expert_offsets: np.ndarray  # [E+1] int32
    seq_slot: np.ndarray        # [T] int32 (a token's slot on both its rows)
    adapters: List[List[Optional[Adapter]]]  # [E][max_loras]
    token_of_row: np.ndarray = field(default=None)  # [T] source token id
    note: str = ""


@dataclass
class MoeGatherWorkload:
    """Decode-path MoE fold: slot-rows in token order, expert per slot-row."""
    name: str
    seed: int
    E: int
    T: int                      # slot-rows = tokens x top_k, token-major
    K: int
    N: int
    max_loras: int
    max_rank: int
    top_k: int
    W: List[np.ndarray]         # E x [N][K] bf16 bits
    x: np.ndarray               # [T][K] bf16 bits, slot-row j = token j // top_k
    indices: np.ndarray         # [T] int32 expert of each slot-row
    seq_slot: np.ndarray        # [T] int32 (a token's slot on all its rows)
    combine: np.ndarray         # [T] float32 combine weight of each slot-row
    adapters: List[List[Optional[Adapter]]]  # [E][max_loras]
    note: str = ""


@dataclass
class EmbedWorkload:
    """Token-embedding gather through an adapted matrix E + s B A (rows = vocab)."""
    name: str
    seed: int
    M: int
    vocab: int
    n_embd: int
    max_loras: int
    max_rank: int
    E: np.ndarray               # [vocab][n_embd] bf16 bits
    tokens: np.ndarray          # [M] int32 token ids
    seq_slot: np.ndarray        # [M] int32, <0 = no adapter
    adapters: List[Optional[Adapter]]  # A [rank][n_embd], B [vocab][rank]
    note: str = ""


# ----------------------------------------------------------------------------
# Drawing helpers
# ----------------------------------------------------------------------------


def _normal_bf16(rng: np.random.Generator, shape, var: float) -> np.ndarray:
    """N(0, var) drawn in fp32, then rounded to bf16."""
    out = np.empty(shape, dtype=np.uint16)
    flat = out.reshape(-1)
    std = np.float32(np.sqrt(var))
    step = 1 << 24
    for s in range(0, flat.size, step):
        n = min(step, flat.size - s)
        v = rng.standard_normal(n, dtype=np.float32)
        v *= std
        flat[s:s + n] = f32_to_bf16(v)
    return out


def _uniform_bf16(rng: np.random.Generator, shape, bound: float) -> np.ndarray:
    """U(-bound, +bound) drawn in fp32, then rounded to bf16."""
    v = rng.uniform(-bound, bound, size=shape).astype(np.float32)
    return f32_to_bf16(v)


def _adapter(rng, n_in, n_out, rank, a_bound, b_var, alpha, rslora=False, adapter_scale=1.0):
    A = _uniform_bf16(rng, (rank, n_in), a_bound)
    B = _normal_bf16(rng, (n_out, rank), b_var)
    return Adapter(A=A, B=B, rank=rank, alpha=float(alpha), use_rslora=rslora,
                   adapter_scale=float(adapter_scale))


def _mark_no_adapter(rng, slots: np.ndarray, frac: float) -> np.ndarray:
    """Set exactly round(frac*M) rows, chosen by a seeded permutation, to -1."""
    m = slots.shape[0]
    k = int(round(frac * m))
    idx = rng.permutation(m)[:k]
    slots = slots.copy()
    slots[idx] = -1
    return slots


# ----------------------------------------------------------------------------
# The five workloads
# ----------------------------------------------------------------------------


def tiny(seed: int = 0) -> ProjWorkload:
    """256x256 base, 8 rows, 4 adapters of rank 8, alpha 16.

    Draw order: W, x, then (A, B) per adapter, then seq_slot.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    M, K, N, L, R = 8, 256, 256, 4, 8
    W = _normal_bf16(rng, (N, K), 1.0 / K)
    x = _normal_bf16(rng, (M, K), 1.0)
    ads = [_adapter(rng, K, N, 8, 1.0 / 16, 0.02, alpha=16.0) for _ in range(L)]
    seq_slot = rng.integers(-1, L, size=M, dtype=np.int64).astype(np.int32)
    return ProjWorkload("tiny", seed, M, K, N, L, R, W, x, seq_slot, ads,
                        note="W~N(0,1/256) x~N(0,1) A~U(+-1/16) B~N(0,0.02) r=8 alpha=16")


def decode(seed: int = 1, M: int = 64) -> ProjWorkload:
    """4096x4096 base, 64 rows, 16 adapters with ranks from {8,16,32,64}.

    Pool rank 64; alpha = 2*rank. Draw order: W, x, ranks, (A, B) per
    adapter, slot per row, then the 10% no-adapter rows.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    K, N, L, R = 4096, 4096, 16, 64
    W = _normal_bf16(rng, (N, K), 1.0 / K)
    x = _normal_bf16(rng, (M, K), 1.0)
    ranks = rng.choice(np.array([8, 16, 32, 64]), size=L)
    ads = [_adapter(rng, K, N, int(r), 1.0 / 64, 0.02, alpha=2.0 * int(r)) for r in ranks]
    seq_slot = rng.integers(0, L, size=M, dtype=np.int64).astype(np.int32)
    seq_slot = _mark_no_adapter(rng, seq_slot, 0.10)
    return ProjWorkload("decode", seed, M, K, N, L, R, W, x, seq_slot, ads,
                        note="W~N(0,1/4096) x~N(0,1) r~U{8,16,32,64} R=64 "
                             "A~U(+-1/64) B~N(0,0.02) alpha=2r, 10% rows -1")


def zipf_slots(rng: np.random.Generator, m: int, n_adapters: int, s: float) -> np.ndarray:
    """Slot k-1 with probability proportional to k^-s, k = 1..n_adapters."""
    k = np.arange(1, n_adapters + 1, dtype=np.float64)
    p = k ** (-s)
    p /= p.sum()
    return rng.choice(n_adapters, size=m, p=p).astype(np.int32)


def qkv(seed: int = 2, M: int = 256) -> ProjWorkload:
    """Fused q/k/v base [6144][4096] = q 4096 + k 1024 + v 1024 rows.

    32 adapters of rank 16, one A per adapter and B over all 6144 rows;
    adapter scales from {0, 0.5, 1.0}, alpha 32. Draw order: W, x, per
    adapter (A, B, adapter scale), Zipf slots, the 5% no-adapter rows.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    K, N, L, R = 4096, 6144, 32, 16
    W = _normal_bf16(rng, (N, K), 1.0 / K)
    x = _normal_bf16(rng, (M, K), 1.0)
    ads = []
    for _ in range(L):
        ad = _adapter(rng, K, N, 16, 1.0 / 64, 0.02, alpha=32.0)
        ad.adapter_scale = float(rng.choice(np.array([0.0, 0.5, 1.0])))
        ads.append(ad)
    seq_slot = zipf_slots(rng, M, L, 1.1)
    seq_slot = _mark_no_adapter(rng, seq_slot, 0.05)
    return ProjWorkload("qkv", seed, M, K, N, L, R, W, x, seq_slot, ads,
                        splits=[4096, 1024, 1024],
                        note="W~N(0,1/4096) x~N(0,1) r=16 A~U(+-1/64) B~N(0,0.02) "
                             "alpha=32 adapter_scale~U{0,0.5,1} Zipf(1.1) 5% rows -1")


def gated_q(seed: int = 6, M: int = 64) -> ProjWorkload:
    """Gated attention query: one fused base [q 4096 | gate 4096][4096] whose
    output is twice the query width (q rows, then the gate rows), 16 adapters
    of rank 16 with one A each and B over all 8192 rows. Draw order: W, x,
    per adapter (A, B), Zipf slots, the 10% no-adapter rows.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    K, N, L, R = 4096, 8192, 16, 16
    W = _normal_bf16(rng, (N, K), 1.0 / K)
    x = _normal_bf16(rng, (M, K), 1.0)
    ads = [_adapter(rng, K, N, 16, 1.0 / 64, 0.02, alpha=32.0) for _ in range(L)]
    seq_slot = zipf_slots(rng, M, L, 1.1)
    seq_slot = _mark_no_adapter(rng, seq_slot, 0.10)
    return ProjWorkload("gated_q", seed, M, K, N, L, R, W, x, seq_slot, ads,
                        splits=[4096, 4096],
                        note="W~N(0,1/4096) x~N(0,1) r=16 A~U(+-1/64) B~N(0,0.02) alpha=32 "
                             "Zipf(1.1) 10% rows -1; output [q | gate]")


def prefill(seed: int = 3, seq_len: int = 1024, n_seq: int = 8) -> ProjWorkload:
    """Gate/up base [14336][4096], 8 contiguous sequences of 1024 rows.

    Sequence i uses adapter i; rank 64, rsLoRA, alpha 16. Draw order: W,
    x, then (A, B) per adapter.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    K, N, L, R = 4096, 14336, n_seq, 64
    M = seq_len * n_seq
    W = _normal_bf16(rng, (N, K), 1.0 / K)
    x = _normal_bf16(rng, (M, K), 1.0)
    ads = [_adapter(rng, K, N, 64, 1.0 / 64, 0.02, alpha=16.0, rslora=True) for _ in range(L)]
    seq_slot = np.repeat(np.arange(n_seq, dtype=np.int32), seq_len)
    return ProjWorkload("prefill", seed, M, K, N, L, R, W, x, seq_slot, ads,
                        note="W~N(0,1/4096) x~N(0,1) r=64 rsLoRA alpha=16 "
                             "A~U(+-1/64) B~N(0,0.02), 8 sequences x 1024 rows")


def moe(seed: int = 4, tokens: int = 512, E: int = 8, top_k: int = 2,
        K: int = 14336, N: int = 4096, n_adapters: int = 4, rank: int = 16) -> MoeWorkload:
    """Expert down projection: E experts of [N][K], tokens routed top-k.

    Routing: logits [tokens][E] ~ N(0,1); a token goes to the top_k largest
    logits (a softmax does not change the order; ties go to the lower
    expert id). Slot-rows are ordered by (expert, token), stably, and
    ``expert_offsets`` is the exclusive scan of the per-expert counts. Each
    slot-row has its own input row ~ N(0,1). A token's slot (uniform over
    {-1, 0..n_adapters-1}) is shared by its top_k slot-rows.

    Draw order: per expert W_e; logits; token slots; x; per expert and
    adapter (A, B).
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    W = [_normal_bf16(rng, (N, K), 1.0 / K) for _ in range(E)]
    logits = rng.standard_normal((tokens, E), dtype=np.float32)
    order = np.argsort(-logits, axis=1, kind="stable")[:, :top_k]
    tok_slot = rng.integers(-1, n_adapters, size=tokens, dtype=np.int64).astype(np.int32)
    pairs = [(int(order[t, j]), t) for t in range(tokens) for j in range(top_k)]
    pairs.sort()  # (expert, token): stable grouping by expert
    T = len(pairs)
    expert_of_row = np.array([p[0] for p in pairs], dtype=np.int32)
    token_of_row = np.array([p[1] for p in pairs], dtype=np.int32)
    counts = np.bincount(expert_of_row, minlength=E)
    offsets = np.zeros(E + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(counts)
    seq_slot = tok_slot[token_of_row].astype(np.int32)
    x = _normal_bf16(rng, (T, K), 1.0)
    ads = [[_adapter(rng, K, N, rank, 1.0 / 64, 0.02, alpha=32.0) for _ in range(n_adapters)]
           for _ in range(E)]
    return MoeWorkload("moe", seed, E, T, K, N, n_adapters, rank, W, x, offsets, seq_slot, ads,
                       token_of_row=token_of_row,
                       note="W_e~N(0,1/14336) x~N(0,1) per slot-row, top-2 of N(0,1) logits, "
                            "r=16 alpha=32 A~U(+-1/64) B~N(0,0.02), slot~U{-1,0..3} per token")


def moe_gather(seed: int = 6, tokens: int = 64, E: int = 8, top_k: int = 2, K: int = 14336,
               N: int = 4096, n_adapters: int = 4, rank: int = 16) -> MoeGatherWorkload:
    """Decode-path MoE down projection, slot-rows left in token order.

    Routing as in ``moe``: logits [tokens][E] ~ N(0,1), a token's top_k
    largest (ties to the lower id); slot-row t*top_k + i holds the token's
    i-th choice. Combine weights: the softmax of the token's top_k logits (the
    chosen experts' probabilities renormalised to sum 1), in fp32. Each
    slot-row has its own input row ~ N(0,1); a token's slot (uniform over
    {-1, 0..n_adapters-1}) is shared by its top_k slot-rows.

    Draw order: per expert W_e; logits; token slots; x; per expert and
    adapter (A, B).
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    W = [_normal_bf16(rng, (N, K), 1.0 / K) for _ in range(E)]
    logits = rng.standard_normal((tokens, E), dtype=np.float32)
    order = np.argsort(-logits, axis=1, kind="stable")[:, :top_k]
    tok_slot = rng.integers(-1, n_adapters, size=tokens, dtype=np.int64).astype(np.int32)
    T = tokens * top_k
    indices = order.reshape(T).astype(np.int32)
    top = np.take_along_axis(logits, order, axis=1).astype(np.float64)
    w = np.exp(top - top.max(axis=1, keepdims=True))
    combine = (w / w.sum(axis=1, keepdims=True)).reshape(T).astype(np.float32)
    seq_slot = np.repeat(tok_slot, top_k).astype(np.int32)
    x = _normal_bf16(rng, (T, K), 1.0)
    ads = [[_adapter(rng, K, N, rank, 1.0 / 64, 0.02, alpha=32.0) for _ in range(n_adapters)]
           for _ in range(E)]
    return MoeGatherWorkload("moe_gather", seed, E, T, K, N, n_adapters, rank, top_k, W, x, indices,
                             seq_slot, combine, ads,
                             note="W_e~N(0,1/14336) x~N(0,1) per slot-row, top-2 of N(0,1) logits in "
                                  "token order, combine = softmax of the top-2, r=16 alpha=32")


def random_small(seed: int, M: int, K: int, N: int, L: int, R: int,
                 ranks=None, alpha=None, rslora=False, p_none: float = 0.25,
                 adapter_scales=None) -> ProjWorkload:
    """Small random case for brute-force and edge checks (any shapes).

    Draw order: W, x, per slot (rank if not given, A, B), slot per row.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    W = _normal_bf16(rng, (N, K), 1.0 / max(K, 1))
    x = _normal_bf16(rng, (M, K), 1.0)
    ads: List[Optional[Adapter]] = []
    for s in range(L):
        r = int(ranks[s]) if ranks is not None else int(rng.integers(1, R + 1))
        if r == 0:
            ads.append(None)
            continue
        a = float(alpha[s]) if alpha is not None else 2.0 * r
        sc = float(adapter_scales[s]) if adapter_scales is not None else 1.0
        ads.append(_adapter(rng, K, N, r, 1.0 / np.sqrt(max(K, 1)), 0.02, alpha=a,
                            rslora=rslora, adapter_scale=sc))
    seq_slot = rng.integers(-1, max(L, 1), size=M, dtype=np.int64).astype(np.int32)
    if p_none == 0.0:
        seq_slot[seq_slot < 0] = 0
    return ProjWorkload(f"random{seed}", seed, M, K, N, L, R, W, x, seq_slot, ads)


@dataclass
class StackWorkload:
    """A projection whose slots each hold a stack of adapters (several
    adapters on one base matrix, all applied to the slot's rows)."""
    name: str
    seed: int
    M: int
    K: int
    N: int
    max_loras: int
    max_rank: int
    W: np.ndarray               # [N][K] bf16 bits
    x: np.ndarray               # [M][K] bf16 bits
    seq_slot: np.ndarray        # [M] int32, <0 = no adapter
    stacks: List[List[Adapter]]  # per slot, its members in order (empty: no adapter)
    note: str = ""


def stacked(seed: int = 7, M: int = 64, K: int = 4096, N: int = 4096, L: int = 8, R: int = 64,
            ranks=(8, 16, 32), max_members: int = 3, p_none: float = 0.1,
            a_bound: float = 1.0 / 64, zero_member_slot: int = 1) -> StackWorkload:
    """Base [N][K] ~ N(0, 1/K), M rows of x ~ N(0, 1), L slots each holding a
    stack of 1..max_members adapters with ranks from ``ranks`` (A ~ U(+-a_bound),
    B ~ N(0, 0.02), alpha = 2 rank, adapter scale from {0.5, 1}), the members'
    ranks summing to at most R; slot ``zero_member_slot`` (if any) gets one more
    member with adapter scale 0. Slots uniform over the L slots, round(p_none M)
    rows set to -1.

    Draw order: W, x, per slot (member count, then per member: rank, adapter
    scale, A, B), slot per row, the -1 rows.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    W = _normal_bf16(rng, (N, K), 1.0 / K)
    x = _normal_bf16(rng, (M, K), 1.0)
    stacks: List[List[Adapter]] = []
    for s in range(L):
        n_m = int(rng.integers(1, max_members + 1))
        members: List[Adapter] = []
        used = 0
        for _ in range(n_m):
            r = int(rng.choice(np.array(ranks)))
            sc = float(rng.choice(np.array([0.5, 1.0])))
            if used + r > R:
                break
            members.append(_adapter(rng, K, N, r, a_bound, 0.02, alpha=2.0 * r, adapter_scale=sc))
            used += r
        if s == zero_member_slot and used + min(ranks) <= R:
            members.append(_adapter(rng, K, N, int(min(ranks)), a_bound, 0.02, alpha=2.0 * min(ranks),
                                    adapter_scale=0.0))
        stacks.append(members)
    seq_slot = rng.integers(0, L, size=M, dtype=np.int64).astype(np.int32)
    seq_slot = _mark_no_adapter(rng, seq_slot, p_none)
    return StackWorkload("stacked", seed, M, K, N, L, R, W, x, seq_slot, stacks,
                         note="W~N(0,1/K) x~N(0,1); per slot 1-3 adapters r in {8,16,32} (sum <= R), "
                              "A~U(+-1/64) B~N(0,0.02) alpha=2r, adapter scale {0.5,1}; one member at scale 0")


def embed(seed: int = 5, M: int = 64, vocab: int = 32000, n_embd: int = 4096, L: int = 16,
          R: int = 64, ranks=None, p_none: float = 0.1) -> EmbedWorkload:
    """Token embedding [vocab][n_embd] ~ N(0, 0.02) gathered for M tokens drawn
    uniformly from the vocabulary, L adapters (ranks from {8,16,32,64} unless
    given; A ~ U(+-1/64), B ~ N(0, 0.02), alpha = 2 rank), slots uniform over
    the adapters with round(p_none M) rows set to -1.

    Draw order: E, then (rank, A, B) per adapter, tokens, slots, the -1 rows.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    E = _normal_bf16(rng, (vocab, n_embd), 0.02)
    ads: List[Optional[Adapter]] = []
    for s in range(L):
        r = int(ranks[s]) if ranks is not None else int(rng.choice([8, 16, 32, 64]))
        ads.append(_adapter(rng, n_embd, vocab, r, 1.0 / 64, 0.02, alpha=2.0 * r))
    tokens = rng.integers(0, vocab, size=M, dtype=np.int64).astype(np.int32)
    seq_slot = rng.integers(0, L, size=M, dtype=np.int64).astype(np.int32)
    seq_slot = _mark_no_adapter(rng, seq_slot, p_none)
    return EmbedWorkload("embed", seed, M, vocab, n_embd, L, R, E, tokens, seq_slot, ads,
                         note="E~N(0,0.02) A~U(+-1/64) B~N(0,0.02) alpha=2r, uniform tokens")


CONFIGS = {
    "tiny": tiny,
    "decode": decode,
    "qkv": qkv,
    "gated_q": gated_q,
    "prefill": prefill,
    "moe": moe,
}


def make(name: str, **kw):
    return CONFIGS[name](**kw)
