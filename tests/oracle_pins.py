"""Checks that pin the oracle to things other than itself.

Each ``check_*`` raises AssertionError on failure. ``test_oracle_pins.py``
runs them against the oracle as built; ``test_oracle_mutants.py`` runs them
against copies of the oracle with a plausible mistake planted, and requires
every mutant to fail at least one check.

Pins (what fixes the expected value):
  * fp64 brute force of the materialised (W + s B A) x -- a different
    association of the same product (ferrox-core weight_matrix/lora.rs test
    ``dense_delta``, tolerance 1e-4);
  * worked examples under tests/golden/ (page-printed scale factors; a hand
    derivation with exact arithmetic);
  * byte identities the pages state: scale 0 and slot -1 equal the base-only
    product (ferrox lora.rs module doc, 'Cost when absent'); a fused q/k/v base
    with one copy of A and split B rows equals the stacked split calls
    (frink lora_attach.rs module doc); zero-padded rank equals true rank
    (spark_model lora_delta.rs, LoraPair doc); a batch equals its rows
    (ferrox test ``batch_delta_is_the_matvec_delta_per_position``);
  * closed forms: alpha/sqrt(r) = (alpha/r) * sqrt(r) exactly at r = 4, 16, 64;
    doubling the adapter scale doubles the delta exactly;
  * numpy's stable argsort for the routing sort.
"""
from __future__ import annotations

import json
import os

import numpy as np

import oracle
import workloads
from workloads import Adapter, bf16_to_f32, f32_to_bf16

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _bf(a):
    return f32_to_bf16(np.asarray(a, dtype=np.float32))


def _f64(u16):
    return bf16_to_f32(u16).astype(np.float64)


def brute_force_fp64(wl, scales=None) -> np.ndarray:
    """y = (W + s_i B A) x_i with the delta matrix materialised, in fp64."""
    W = _f64(wl.W)
    x = _f64(wl.x)
    y = np.empty((wl.M, wl.N), dtype=np.float64)
    for i in range(wl.M):
        s = int(wl.seq_slot[i])
        Weff = W
        if 0 <= s < len(wl.adapters) and wl.adapters[s] is not None:
            ad = wl.adapters[s]
            sc = scales[s] if scales is not None else oracle.scale(ad.alpha, ad.rank, ad.use_rslora,
                                                                     ad.adapter_scale)
            if sc != 0.0:
                Weff = W + np.float64(sc) * (_f64(ad.B) @ _f64(ad.A))
        y[i] = Weff @ x[i]
    return y


def check_scale_examples():
    with open(os.path.join(GOLDEN, "scale_examples.json")) as f:
        g = json.load(f)
    for alpha, rank, rs, asc, want in g["rows"]:
        got = oracle.scale(alpha, rank, bool(rs), asc)
        assert abs(got - want) < 1e-7, (alpha, rank, rs, asc, got, want)


def check_hand_example():
    with open(os.path.join(GOLDEN, "hand_example.json")) as f:
        g = json.load(f)
    ads = [Adapter(A=_bf(a["A"]), B=_bf(a["B"]), rank=a["rank"], alpha=a["alpha"],
                   use_rslora=bool(a["use_rslora"]), adapter_scale=a["adapter_scale"])
           for a in g["adapters"]]
    y = oracle.proj(_bf(g["x"]), _bf(g["W"]), np.array(g["seq_slot"], np.int32), ads)
    want = np.array(g["expected_y"], dtype=np.float32)
    assert np.array_equal(y, want), (y, want)


def check_brute_force(wl, tol=1e-4):
    y = oracle.workload_proj(wl)
    ref = brute_force_fp64(wl)
    err = np.abs(y.astype(np.float64) - ref)
    assert err.max() <= tol * (1.0 + np.abs(ref)).max(), (wl.name, err.max())


def check_brute_force_suite():
    check_brute_force(workloads.make("tiny"))
    cases = [
        dict(seed=11, M=5, K=7, N=9, L=3, R=4),
        dict(seed=12, M=16, K=16, N=16, L=4, R=8, alpha=[0.0, 3.0, 0.0, 5.0]),
        dict(seed=13, M=9, K=13, N=6, L=2, R=3, rslora=True),
        dict(seed=14, M=3, K=16, N=11, L=5, R=2, adapter_scales=[0.5, -1.0, 2.0, 0.0, 0.25]),
        dict(seed=15, M=12, K=1, N=4, L=2, R=1),
    ]
    for c in cases:
        check_brute_force(workloads.random_small(**c))


def check_no_delta_rows_are_base_bytes():
    wl = workloads.make("tiny")
    y = oracle.workload_proj(wl)
    base = oracle.proj(wl.x, wl.W, np.full(wl.M, -1, np.int32), wl.adapters)
    none = wl.seq_slot < 0
    assert none.any() and (~none).any()
    assert np.array_equal(y[none].view(np.uint32), base[none].view(np.uint32))
    # adapted rows differ from base (the delta is really applied)
    assert not np.array_equal(y[~none], base[~none])
    # adapter scale 0 (every slot): byte-identical to base
    zero = [Adapter(a.A, a.B, a.rank, a.alpha, a.use_rslora, 0.0) for a in wl.adapters]
    y0 = oracle.proj(wl.x, wl.W, wl.seq_slot, zero)
    assert np.array_equal(y0.view(np.uint32), base.view(np.uint32))
    # a slot at or past max_loras is treated as no adapter
    far = wl.seq_slot.copy()
    far[:] = len(wl.adapters) + 3
    yf = oracle.proj(wl.x, wl.W, far, wl.adapters)
    assert np.array_equal(yf.view(np.uint32), base.view(np.uint32))
    # an empty slot (no pair) is no adapter
    empty = [None] * len(wl.adapters)
    ye = oracle.proj(wl.x, wl.W, wl.seq_slot, empty)
    assert np.array_equal(ye.view(np.uint32), base.view(np.uint32))


def check_fused_split_exact(wl=None, rows=None):
    if wl is None:
        wl = workloads.random_small(seed=21, M=10, K=24, N=20, L=3, R=4)
        splits = [12, 4, 4]
    else:
        splits = wl.splits
    fused = oracle.proj(wl.x, wl.W, wl.seq_slot, wl.adapters, rows=rows)
    parts = []
    row0 = 0
    for n in splits:
        ads = []
        for a in wl.adapters:
            if a is None:
                ads.append(None)
                continue
            ads.append(Adapter(a.A, np.ascontiguousarray(a.B[row0:row0 + n]), a.rank, a.alpha,
                               a.use_rslora, a.adapter_scale))
        parts.append(oracle.proj(wl.x, np.ascontiguousarray(wl.W[row0:row0 + n]), wl.seq_slot,
                                 ads, rows=rows))
        row0 += n
    stacked = np.concatenate(parts, axis=1)
    assert np.array_equal(fused.view(np.uint32), stacked.view(np.uint32))


def check_rslora_closed_form():
    for r in (4, 16, 64):
        wl = workloads.random_small(seed=30 + r, M=6, K=32, N=10, L=2, R=r, ranks=[r, r],
                                    alpha=[8.0, 3.0])
        zeroW = np.zeros_like(wl.W)
        plain = oracle.proj(wl.x, zeroW, wl.seq_slot, wl.adapters)
        rs = [Adapter(a.A, a.B, a.rank, a.alpha, True, a.adapter_scale) for a in wl.adapters]
        root = oracle.proj(wl.x, zeroW, wl.seq_slot, rs)
        k = np.float32(np.sqrt(r))
        assert np.array_equal(root.view(np.uint32), (plain * k).view(np.uint32)), r
        assert np.any(plain != 0)


def check_zero_padding_exact():
    wl = workloads.random_small(seed=41, M=8, K=40, N=12, L=3, R=8, ranks=[3, 5, 8])
    pads = []
    scales = []
    for a in wl.adapters:
        R = 8
        A = np.zeros((R, wl.K), np.uint16)
        A[:a.rank] = a.A
        B = np.zeros((wl.N, R), np.uint16)
        B[:, :a.rank] = a.B
        pads.append(Adapter(A, B, R, a.alpha, a.use_rslora, a.adapter_scale))
        scales.append(oracle.scale(a.alpha, a.rank, a.use_rslora, a.adapter_scale))
    y_true = oracle.workload_proj(wl)
    y_pad = oracle.proj(wl.x, wl.W, wl.seq_slot, pads, scales=scales)
    assert np.array_equal(y_true.view(np.uint32), y_pad.view(np.uint32))


def check_linear_in_scale():
    wl = workloads.random_small(seed=51, M=7, K=20, N=9, L=2, R=4, p_none=0.0)
    zeroW = np.zeros_like(wl.W)
    one = oracle.proj(wl.x, zeroW, wl.seq_slot, wl.adapters)
    dbl = [Adapter(a.A, a.B, a.rank, a.alpha, a.use_rslora, 2.0 * a.adapter_scale)
           for a in wl.adapters]
    two = oracle.proj(wl.x, zeroW, wl.seq_slot, dbl)
    assert np.array_equal(two.view(np.uint32), (one * np.float32(2)).view(np.uint32))
    assert np.any(one != 0)


def check_batch_is_rows():
    wl = workloads.make("tiny")
    y = oracle.workload_proj(wl)
    for i in range(wl.M):
        yi = oracle.workload_proj(wl, rows=[i])
        assert np.array_equal(y[i:i + 1].view(np.uint32), yi.view(np.uint32)), i
    cols = np.array([255, 0, 17, 128], np.int32)
    yc = oracle.workload_proj(wl, rows=[3, 1], cols=cols)
    assert np.array_equal(yc.view(np.uint32), y[[3, 1]][:, cols].view(np.uint32))


def check_slot_sort():
    rng = np.random.default_rng(7)
    for M, L in [(0, 3), (1, 1), (64, 16), (257, 5), (1000, 33)]:
        s = rng.integers(-3, L + 3, size=M).astype(np.int32)
        perm, seg = oracle.slot_sort(s, L)
        key = np.where((s >= 0) & (s < L), s + 1, 0)
        want = np.argsort(key, kind="stable").astype(np.int32)
        assert np.array_equal(perm, want)
        assert np.array_equal(np.sort(perm), np.arange(M))
        counts = np.bincount(key, minlength=L + 1)
        assert np.array_equal(np.diff(seg), counts) and seg[0] == 0 and seg[-1] == M


def small_moe():
    return workloads.synth.moe(seed=5, tokens=24, E=3, top_k=2, K=40, N=24, n_adapters=3, rank=4)


def check_moe_segments():
    wl = small_moe()
    y = oracle.workload_moe(wl)
    for e in range(wl.E):
        a, b = int(wl.expert_offsets[e]), int(wl.expert_offsets[e + 1])
        if a == b:
            continue
        seg = oracle.proj(wl.x[a:b], wl.W[e], wl.seq_slot[a:b], wl.adapters[e])
        assert np.array_equal(y[a:b].view(np.uint32), seg.view(np.uint32)), e
    perm, seg = oracle.moe_slot_sort(wl.expert_offsets, wl.seq_slot, wl.max_loras)
    ex = np.repeat(np.arange(wl.E), np.diff(wl.expert_offsets))
    key = np.where((wl.seq_slot >= 0) & (wl.seq_slot < wl.max_loras), wl.seq_slot + 1, 0)
    want = np.lexsort((key, ex)).astype(np.int32)  # primary expert, then key, stable
    assert np.array_equal(perm, want)


# --------------------------------------------------------------------------
# Embedding row gather (ferrox-core lora.rs, LoraDelta::add_row_to)
# --------------------------------------------------------------------------


def small_embed_cases():
    return [
        workloads.embed(seed=21, M=9, vocab=40, n_embd=24, L=3, ranks=[4, 8, 16]),
        workloads.embed(seed=22, M=16, vocab=7, n_embd=33, L=4, ranks=[1, 2, 3, 5], p_none=0.25),
    ]


def check_embed_brute_force(tol=1e-4):
    """y[i] = E[t_i] + s B[t_i] A in fp64 (the delta row of the materialised
    s B A, as ferrox's add_row_to defines it)."""
    for wl in small_embed_cases():
        y = oracle.workload_embed(wl)
        E = _f64(wl.E)
        for i in range(wl.M):
            t, s = int(wl.tokens[i]), int(wl.seq_slot[i])
            ref = E[t].copy()
            if 0 <= s < wl.max_loras:
                ad = wl.adapters[s]
                sc = oracle.scale(ad.alpha, ad.rank, ad.use_rslora, ad.adapter_scale)
                ref += np.float64(sc) * (_f64(ad.B)[t] @ _f64(ad.A))
            err = np.abs(y[i].astype(np.float64) - ref).max()
            assert err <= tol * (1.0 + np.abs(ref).max()), (wl.seed, i, err)


def check_embed_row_gather_identity():
    """With E = 0 the gathered row t equals the projection of the unit vector
    e_t through the flipped pair (A' = B^T, B' = A^T) with a zero base -- the
    same products in the same order, so byte for byte."""
    wl = small_embed_cases()[0]
    E0 = np.zeros_like(wl.E)
    y = oracle.embed(wl.tokens, E0, wl.seq_slot, wl.adapters)
    flipped = [Adapter(A=np.ascontiguousarray(ad.B.T), B=np.ascontiguousarray(ad.A.T), rank=ad.rank,
                       alpha=ad.alpha, use_rslora=ad.use_rslora, adapter_scale=ad.adapter_scale)
               for ad in wl.adapters]
    one = _bf([1.0])[0]
    for i in range(wl.M):
        x = np.zeros((1, wl.vocab), dtype=np.uint16)
        x[0, int(wl.tokens[i])] = one
        W0 = np.zeros((wl.n_embd, wl.vocab), dtype=np.uint16)
        yp = oracle.proj(x, W0, wl.seq_slot[i:i + 1], flipped)
        assert np.array_equal(y[i].view(np.uint32), yp[0].view(np.uint32)), i


def check_embed_no_delta_rows_are_the_embedding():
    """Slot -1, a slot >= L, scale 0: the row is E[t] exactly; a token outside
    the vocabulary gives a zero row."""
    wl = small_embed_cases()[1]
    slots = wl.seq_slot.copy()
    slots[0], slots[1] = -1, wl.max_loras + 2
    scales = [0.0] + [oracle.scale(a.alpha, a.rank, a.use_rslora, a.adapter_scale)
                      for a in wl.adapters[1:]]
    toks = wl.tokens.copy()
    toks[2] = wl.vocab
    y = oracle.embed(toks, wl.E, slots, wl.adapters, scales=scales)
    Ef = bf16_to_f32(wl.E)
    for i in range(wl.M):
        if i == 2:
            assert not y[i].any()
        elif slots[i] < 0 or slots[i] >= wl.max_loras or slots[i] == 0:
            assert np.array_equal(y[i].view(np.uint32), Ef[int(toks[i])].view(np.uint32)), i


# --------------------------------------------------------------------------
# Gated MLP input: fused [gate|up] projection, then silu(gate) * up
# (frink lora_attach.rs, parts_mut: the fused ffn_up is gate rows then up rows)
# --------------------------------------------------------------------------


def small_gate_up(seed=31, M=9, K=40, I=24, L=3, R=16):
    """A fused [gate|up] workload: W [2I][K], adapters with B [2I][r]."""
    return workloads.random_small(seed, M=M, K=K, N=2 * I, L=L, R=R)


def check_silu_mul_closed_forms():
    """silu(g) * u against g * (1 + tanh(g/2)) / 2 * u in fp64 (the logistic
    function written through tanh), and the exact points silu(0) = 0, u = 0."""
    rng = np.random.default_rng(7)
    I = 16
    y = rng.normal(0.0, 3.0, size=(5, 2 * I)).astype(np.float32)
    y[0, :I] = 0.0
    y[1, I:] = 0.0
    y[2, :4] = [30.0, -30.0, 1e-3, -1e-3]
    act = oracle.silu_mul(y, I)
    g = y[:, :I].astype(np.float64)
    u = y[:, I:].astype(np.float64)
    ref = g * (1.0 + np.tanh(g / 2.0)) / 2.0 * u
    assert np.all(act[0] == 0.0) and np.all(act[1] == 0.0)
    err = np.abs(act.astype(np.float64) - ref)
    assert np.all(err <= 1e-6 * (1.0 + np.abs(ref))), err.max()


def check_gate_up_is_the_split_projections():
    """The gate half of the fused projection is the projection through the gate
    rows of W and of every B (one shared A), the up half likewise, byte for
    byte; act is silu of the one times the other."""
    wl = small_gate_up()
    I = wl.N // 2
    act = oracle.gate_up(wl.x, wl.W, wl.seq_slot, wl.adapters)
    halves = []
    for lo in (0, I):
        ads = [None if a is None else Adapter(A=a.A, B=np.ascontiguousarray(a.B[lo:lo + I]), rank=a.rank,
                                              alpha=a.alpha, use_rslora=a.use_rslora,
                                              adapter_scale=a.adapter_scale) for a in wl.adapters]
        halves.append(oracle.proj(wl.x, np.ascontiguousarray(wl.W[lo:lo + I]), wl.seq_slot, ads))
    both = np.concatenate(halves, axis=1)
    assert np.array_equal(act.view(np.uint32), oracle.silu_mul(both, I).view(np.uint32))
    g, u = halves[0].astype(np.float64), halves[1].astype(np.float64)
    ref = g * (1.0 + np.tanh(g / 2.0)) / 2.0 * u
    with np.errstate(invalid="ignore", over="ignore"):
        assert np.all(np.abs(act - ref) <= 1e-5 * (1.0 + np.abs(ref)))


# --------------------------------------------------------------------------
# Decode-path MoE fold keyed by per-slot-row expert indices, with combine
# weights (spark_model lora_delta.rs, LoraKernels moe_gather)
# --------------------------------------------------------------------------


def small_moe_gather(seed=51, tokens=5, E=3, top_k=2, K=24, N=16):
    return workloads.moe_gather(seed=seed, tokens=tokens, E=E, top_k=top_k, K=K, N=N, n_adapters=3, rank=4)


def check_moe_gather_brute_force(tol=1e-4):
    """y[t] = sum_i w_ti (W_e + s B A) x_ti in fp64 with the delta matrix
    materialised; an index outside [0, E) contributes nothing."""
    wl = small_moe_gather()
    wl.indices[3] = wl.E  # out of range: that slot-row adds nothing
    y = oracle.workload_moe_gather(wl)
    x = _f64(wl.x)
    for t in range(wl.T // wl.top_k):
        ref = np.zeros(wl.N)
        for i in range(wl.top_k):
            j = t * wl.top_k + i
            e, s = int(wl.indices[j]), int(wl.seq_slot[j])
            if not 0 <= e < wl.E:
                continue
            Weff = _f64(wl.W[e])
            if 0 <= s < wl.max_loras:
                ad = wl.adapters[e][s]
                sc = oracle.scale(ad.alpha, ad.rank, ad.use_rslora, ad.adapter_scale)
                Weff = Weff + np.float64(sc) * (_f64(ad.B) @ _f64(ad.A))
            ref += np.float64(wl.combine[j]) * (Weff @ x[j])
        assert np.abs(y[t] - ref).max() <= tol * (1.0 + np.abs(ref).max()), t


def check_moe_gather_is_the_grouped_fold():
    """Without combine weights the slot-rows equal the grouped (expert_offsets)
    fold over the same rows sorted stably by expert, byte for byte; with
    one-hot weights a token's row is its chosen slot-row exactly."""
    wl = small_moe_gather(seed=52, tokens=7)
    rows = oracle.workload_moe_gather(wl, with_combine=False)
    order = np.argsort(wl.indices, kind="stable").astype(np.int32)
    offs = np.zeros(wl.E + 1, dtype=np.int32)
    offs[1:] = np.cumsum(np.bincount(wl.indices, minlength=wl.E))
    grouped = oracle.moe(wl.x[order], wl.W, offs, wl.seq_slot[order], wl.adapters)
    assert np.array_equal(rows[order].view(np.uint32), grouped.view(np.uint32))
    onehot = np.zeros_like(wl.combine)
    onehot[1::wl.top_k] = 1.0  # every token's second choice
    y = oracle.moe_gather(wl.x, wl.W, wl.indices, wl.seq_slot, wl.adapters, combine=onehot, top_k=wl.top_k)
    assert np.array_equal(y.view(np.uint32), (rows[1::wl.top_k] + 0.0).view(np.uint32))


# --------------------------------------------------------------------------
# several adapters on one matrix (ferrox-core weight_matrix/lora.rs, LoraStack)
# --------------------------------------------------------------------------


def small_stack(seed=61, M=11, K=24, N=16, L=4, R=16):
    wl = workloads.stacked(seed=seed, M=M, K=K, N=N, L=L, R=R, ranks=(1, 3, 4), max_members=3,
                           p_none=0.2, a_bound=0.3, zero_member_slot=1)
    # one member under the square-root rule and one without alpha
    st = wl.stacks[0]
    st[0] = Adapter(st[0].A, st[0].B, st[0].rank, 8.0, True, st[0].adapter_scale)
    if len(wl.stacks[2]) > 0:
        m = wl.stacks[2][0]
        wl.stacks[2][0] = Adapter(m.A, m.B, m.rank, 0.0, False, 0.75)
    return wl


def check_stack_brute_force(tol=1e-4):
    """y = (W + sum_m s_m B_m A_m) x_i with the delta matrix materialised, fp64."""
    for seed in (61, 62, 63):
        wl = small_stack(seed=seed)
        y = oracle.proj_stack(wl.x, wl.W, wl.seq_slot, wl.stacks)
        W, x = _f64(wl.W), _f64(wl.x)
        for i in range(wl.M):
            s = int(wl.seq_slot[i])
            Weff = W.copy()
            if 0 <= s < wl.max_loras:
                for m in wl.stacks[s]:
                    sc = oracle.scale(m.alpha, m.rank, m.use_rslora, m.adapter_scale)
                    Weff += np.float64(sc) * (_f64(m.B) @ _f64(m.A))
            ref = Weff @ x[i]
            assert np.abs(y[i] - ref).max() <= tol * (1.0 + np.abs(ref).max()), (seed, i)


def check_stack_reductions():
    """A stack of one adapter is that adapter, byte for byte; a member at scale
    0 adds nothing (the stack without it, byte for byte); rows whose slot is
    -1, past max_loras or empty, and stacks whose every scale is 0, are the
    base product byte for byte (ferrox lora.rs module doc, 'Cost when absent')."""
    wl = small_stack(seed=64)
    ss = wl.seq_slot
    one = [st[:1] for st in wl.stacks]
    y1 = oracle.proj_stack(wl.x, wl.W, ss, one)
    yp = oracle.proj(wl.x, wl.W, ss, [st[0] for st in wl.stacks])
    assert np.array_equal(y1.view(np.uint32), yp.view(np.uint32))
    y = oracle.proj_stack(wl.x, wl.W, ss, wl.stacks)
    nz = [[m for m in st if m.adapter_scale != 0.0] for st in wl.stacks]
    assert any(len(a) != len(b) for a, b in zip(nz, wl.stacks))
    ynz = oracle.proj_stack(wl.x, wl.W, ss, nz)
    assert np.array_equal(y.view(np.uint32), ynz.view(np.uint32))
    base = oracle.proj(wl.x, wl.W, np.full(wl.M, -1, np.int32), [None] * wl.max_loras)
    none = ss < 0
    assert none.any() and (~none).any()
    assert np.array_equal(y[none].view(np.uint32), base[none].view(np.uint32))
    assert not np.array_equal(y[~none], base[~none])
    zero = [[Adapter(m.A, m.B, m.rank, m.alpha, m.use_rslora, 0.0) for m in st] for st in wl.stacks]
    for stacks, slots in ((zero, ss), ([[] for _ in wl.stacks], ss),
                          (wl.stacks, np.full(wl.M, wl.max_loras + 2, np.int32))):
        yz = oracle.proj_stack(wl.x, wl.W, slots, stacks)
        assert np.array_equal(yz.view(np.uint32), base.view(np.uint32))


ALL_CHECKS = [
    check_scale_examples,
    check_hand_example,
    check_brute_force_suite,
    check_no_delta_rows_are_base_bytes,
    check_fused_split_exact,
    check_rslora_closed_form,
    check_zero_padding_exact,
    check_linear_in_scale,
    check_batch_is_rows,
    check_slot_sort,
    check_moe_segments,
    check_embed_brute_force,
    check_embed_row_gather_identity,
    check_embed_no_delta_rows_are_the_embedding,
    check_silu_mul_closed_forms,
    check_gate_up_is_the_split_projections,
    check_moe_gather_brute_force,
    check_moe_gather_is_the_grouped_fold,
    check_stack_brute_force,
    check_stack_reductions,
]
