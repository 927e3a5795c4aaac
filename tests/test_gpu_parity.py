"""CUDA path vs the oracle, through the C ABI (GPU only).

Tolerance for adapted rows: |gpu - oracle| <= 2e-2 + 1e-2 |oracle| per
element (bf16 inputs, fp32 accumulation on both sides, one bf16 rounding of
the GPU output). Rows with no delta must be byte-identical to the GPU's own
base-only run; the routing sort must equal the oracle's exactly.
"""
import numpy as np
import pytest
import torch

import oracle
import rank_delta_gb300 as rd
import workloads
from rank_delta_gb300 import build as rdbuild
from rank_delta_gb300 import torch_helpers as th
from tests.gpu_common import ProjRun, assert_close

pytestmark = pytest.mark.gpu

PATHS = [rd.LORA_PATH_SIMT, rd.LORA_PATH_TC, rd.LORA_PATH_TC_ONE]


@pytest.fixture(scope="module", autouse=True)
def lib():
    rdbuild.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return rd.lib()


@pytest.fixture(scope="module")
def tiny():
    return ProjRun(workloads.make("tiny"))


@pytest.fixture(scope="module")
def decode():
    return ProjRun(workloads.make("decode"))


@pytest.fixture(scope="module")
def decode_ref(decode):
    return oracle.workload_proj(decode.wl)


@pytest.mark.parametrize("path", PATHS)
def test_tiny_matches_oracle(tiny, path):
    y = tiny.apply(path=path)
    assert tiny.last_status == 0
    assert_close(y, oracle.workload_proj(tiny.wl), f"tiny path {path}")


@pytest.mark.parametrize("path", PATHS)
def test_decode_matches_oracle(decode, decode_ref, path):
    y = decode.apply(path=path)
    assert decode.last_status == 0
    assert_close(y, decode_ref, f"decode path {path}")


@pytest.mark.parametrize("path", PATHS)
def test_no_delta_rows_are_base_bytes(decode, path):
    y = decode.apply(path=path)
    base = decode.apply(slots=torch.full_like(decode.slots, -1), path=path)
    none = decode.wl.seq_slot < 0
    assert none.any()
    assert np.array_equal(y[none], base[none])
    assert not np.array_equal(y[~none], base[~none])


def test_routing_sort_equals_oracle(decode):
    decode.apply()
    perm, seg = rd.lora_proj_routing(decode.ws, decode.wl.M, decode.wl.max_loras)
    operm, oseg = oracle.slot_sort(decode.wl.seq_slot, decode.wl.max_loras)
    assert np.array_equal(perm, operm)
    assert np.array_equal(seg, oseg)


def test_routing_sort_large_and_ragged():
    rng = np.random.default_rng(3)
    M, L = 3000, 40
    wl = workloads.random_small(seed=5, M=M, K=64, N=64, L=L, R=8, ranks=[8] * L)
    wl.seq_slot = rng.integers(-2, L + 2, size=M).astype(np.int32)
    run = ProjRun(wl)
    run.apply(path=rd.LORA_PATH_SIMT)
    assert run.last_status & rd.LORA_FLAG_SLOT_RANGE
    perm, seg = rd.lora_proj_routing(run.ws, M, L)
    operm, oseg = oracle.slot_sort(wl.seq_slot, L)
    assert np.array_equal(perm, operm) and np.array_equal(seg, oseg)


@pytest.mark.parametrize("path", PATHS)
def test_batch_equals_single_rows(decode, path):
    y = decode.apply(path=path)
    for i in [0, 5, 17, 63]:
        yi = decode.apply(slots=decode.slots[i:i + 1], path=path, x=decode.x[i:i + 1])
        assert np.array_equal(yi[0], y[i]), i


def test_slot_past_max_loras_is_no_delta_and_flagged(decode):
    slots = decode.slots.clone()
    slots[3] = decode.wl.max_loras + 5
    y = decode.apply(slots=slots)
    assert decode.last_status & rd.LORA_FLAG_SLOT_RANGE
    base = decode.apply(slots=torch.full_like(decode.slots, -1))
    assert np.array_equal(y[3], base[3])


def test_set_scale_zero_gives_base_and_is_stream_ordered(decode, decode_ref):
    wl = decode.wl
    s = int(wl.seq_slot[0])
    assert s >= 0
    rd.lora_set_scale(decode.route.rt, s, 0.0)
    y0 = decode.apply()
    base = decode.apply(slots=torch.full_like(decode.slots, -1))
    rows = wl.seq_slot == s
    assert np.array_equal(y0[rows], base[rows])
    rd.lora_set_scale(decode.route.rt, s, wl.adapters[s].adapter_scale)
    y1 = decode.apply()
    assert_close(y1, decode_ref, "after restoring the scale")


def test_scale_table_equals_oracle_scale(decode):
    tab = decode.route.scale_table()
    for s, ad in enumerate(decode.wl.adapters):
        assert tab[s] == np.float32(oracle.scale(ad.alpha, ad.rank, ad.use_rslora, ad.adapter_scale))


def test_unpack_makes_slot_base_only(tiny):
    wl = tiny.wl
    s = int(wl.seq_slot[wl.seq_slot >= 0][0])
    rd.lora_pool_unpack(tiny.route.rt, s)
    y = tiny.apply()
    base = tiny.apply(slots=torch.full_like(tiny.slots, -1))
    rows = wl.seq_slot == s
    assert np.array_equal(y[rows], base[rows])
    tiny.route.pack(s, wl.adapters[s])
    assert_close(tiny.apply(), oracle.workload_proj(wl), "after repack")


def test_rows_closest_to_their_own_slot(decode, decode_ref):
    wl = decode.wl
    y = th.bf16_bits_to_f32(decode.apply())
    rows = np.where(wl.seq_slot >= 0)[0][:12]
    for i in rows:
        errs = []
        for s in range(wl.max_loras):
            alt = np.full(wl.M, -1, np.int32)
            alt[i] = s
            ref = oracle.proj(wl.x, wl.W, alt, wl.adapters, rows=[i])[0]
            errs.append(np.abs(y[i] - ref).max())
        assert int(np.argmin(errs)) == int(wl.seq_slot[i])


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("M,K,N,L,R", [(1, 64, 40, 2, 8), (17, 72, 200, 3, 16), (300, 136, 130, 5, 24),
                                       (64, 512, 384, 7, 64), (129, 256, 128, 1, 8)])
def test_ragged_shapes_match_oracle(path, M, K, N, L, R):
    wl = workloads.random_small(seed=M * 7 + K, M=M, K=K, N=N, L=L, R=R)
    run = ProjRun(wl)
    y = run.apply(path=path)
    assert_close(y, oracle.workload_proj(wl), f"M{M} K{K} N{N} path {path}")


def test_empty_batch_is_a_noop(tiny):
    wl = tiny.wl
    y = torch.full((4, wl.N), 7, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    rd.lora_proj_apply(tiny.x, tiny.x.stride(0), tiny.W, 0, wl.K, wl.N, tiny.slots, tiny.route.rt, y,
                       y.stride(0), tiny.ws, tiny.ws.numel())
    torch.cuda.synchronize()
    assert (y.view(torch.int16) == 7).all()


def test_alpha_zero_and_rslora_scales_on_gpu():
    wl = workloads.random_small(seed=77, M=24, K=128, N=96, L=3, R=16, ranks=[16, 4, 9],
                                alpha=[0.0, 8.0, 5.0], adapter_scales=[0.7, 1.0, 2.0])
    wl.adapters[1].use_rslora = True
    run = ProjRun(wl)
    for path in PATHS:
        assert_close(run.apply(path=path), oracle.workload_proj(wl), f"alpha/rslora path {path}")


@pytest.mark.parametrize("M,K,N,L,R", [(2100, 200, 136, 5, 24), (2048, 320, 128, 40, 16),
                                       (4096, 128, 64, 3, 64)])
def test_large_batch_tensor_core_shrink(M, K, N, L, R):
    """From 2048 rows h comes from the tensor-core shrink tiles inside the
    projection launch: ragged row
    tiles, K not a multiple of 64, a pool rank that is not a multiple of 16,
    and tiles holding more slots than one UMMA group (16 slots of rank 16)."""
    wl = workloads.random_small(seed=M + K + L, M=M, K=K, N=N, L=L, R=R)
    run = ProjRun(wl)
    y = run.apply(path=rd.LORA_PATH_TC)
    assert run.last_status == 0
    assert_close(y, oracle.workload_proj(wl), f"M{M} K{K} N{N} L{L} R{R}")
    base = run.apply(slots=torch.full_like(run.slots, -1), path=rd.LORA_PATH_TC)
    none = wl.seq_slot < 0
    assert np.array_equal(y.view(np.uint16)[none], base.view(np.uint16)[none])


def test_fully_adapted_wide_tiles_match_oracle():
    """Token tiles of 256 rows leave no TMEM for a separate delta accumulator:
    when every row of a tile is adapted the delta accumulates into the base
    accumulator. All rows adapted here (no -1 slots), ragged last tile."""
    wl = workloads.random_small(seed=600, M=600, K=192, N=160, L=4, R=32, p_none=0.0)
    run = ProjRun(wl)
    y = run.apply(path=rd.LORA_PATH_TC)
    assert run.last_status == 0
    assert_close(y, oracle.workload_proj(wl), "M600 all rows adapted")


@pytest.mark.parametrize("path", PATHS)
def test_pool_rank_256_needs_several_staging_passes(path):
    """max_rank 256 (the largest pool rank): a K part's slots span more k than
    both staging regions hold, so the expand runs in several passes; K 2048
    gives two K parts on the tensor-core path."""
    wl = workloads.random_small(seed=256, M=40, K=2048, N=256, L=6, R=256,
                                ranks=[256, 200, 129, 64, 250, 7])
    run = ProjRun(wl)
    y = run.apply(path=path)
    assert run.last_status == 0
    assert_close(y, oracle.workload_proj(wl), f"R256 path {path}")


def test_many_slots_in_one_tile_match_oracle():
    """200 slots, 256 rows in one token tile (more slots than the in-tile
    routing keeps, so the routing kernel's work list is used), three K parts."""
    wl = workloads.random_small(seed=200, M=256, K=3072, N=384, L=200, R=16)
    run = ProjRun(wl)
    y = run.apply(path=rd.LORA_PATH_TC)
    assert run.last_status == 0
    assert_close(y, oracle.workload_proj(wl), "L200 M256")
    base = run.apply(slots=torch.full_like(run.slots, -1), path=rd.LORA_PATH_TC)
    none = wl.seq_slot < 0
    assert np.array_equal(y.view(np.uint16)[none], base.view(np.uint16)[none])


def test_set_scales_lists_some_slots_and_zeroes_the_rest(decode, decode_ref):
    """Listed slots take their (last listed) scale, the others 0: their rows
    become the base product byte for byte; restoring every scale restores y."""
    wl = decode.wl
    rd.lora_set_scales(decode.route.rt, [(0, 0.25), (2, 1.0), (0, 2.0)])
    tab = decode.route.scale_table()
    for s, ad in enumerate(wl.adapters):
        want = {0: 2.0, 2: 1.0}.get(s, 0.0)
        assert tab[s] == np.float32(oracle.scale(ad.alpha, ad.rank, ad.use_rslora, want)), s
    y = decode.apply()
    base = decode.apply(slots=torch.full_like(decode.slots, -1))
    off = ~np.isin(wl.seq_slot, [0, 2])
    assert np.array_equal(y[off], base[off])
    rd.lora_set_scales(decode.route.rt, [(s, ad.adapter_scale) for s, ad in enumerate(wl.adapters)])
    assert_close(decode.apply(), decode_ref, "after restoring every scale")
