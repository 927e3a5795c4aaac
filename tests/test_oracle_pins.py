"""The oracle against its pins (CPU only). See tests/oracle_pins.py for what pins what."""
import numpy as np
import pytest

import oracle
import workloads
from tests import oracle_pins as P


def test_scale_worked_examples():
    P.check_scale_examples()


def test_hand_worked_example():
    P.check_hand_example()


def test_brute_force_fp64():
    P.check_brute_force_suite()


def test_no_delta_rows_are_base_bytes():
    P.check_no_delta_rows_are_base_bytes()


def test_fused_split_exact_small():
    P.check_fused_split_exact()


def test_fused_qkv_split_exact_on_qkv_workload():
    wl = workloads.make("qkv")
    rows = np.concatenate([np.where(wl.seq_slot < 0)[0][:3], np.arange(0, 256, 23)]).astype(np.int32)
    P.check_fused_split_exact(wl, rows=rows)


def test_rslora_closed_form():
    P.check_rslora_closed_form()


def test_zero_padding_exact():
    P.check_zero_padding_exact()


def test_linear_in_scale():
    P.check_linear_in_scale()


def test_batch_is_rows():
    P.check_batch_is_rows()


def test_slot_sort_is_stable_argsort():
    P.check_slot_sort()


def test_moe_segments_and_sort():
    P.check_moe_segments()


def test_workload_shapes_and_scales():
    """The generated workloads have the stated shapes and effective scales."""
    wl = workloads.make("tiny")
    assert (wl.M, wl.K, wl.N, wl.max_loras, wl.max_rank) == (8, 256, 256, 4, 8)
    assert {oracle.scale(a.alpha, a.rank, a.use_rslora, a.adapter_scale) for a in wl.adapters} == {2.0}
    d = workloads.make("decode")
    assert d.W.shape == (4096, 4096) and d.x.shape == (64, 4096)
    assert int((d.seq_slot < 0).sum()) == 6
    assert {oracle.scale(a.alpha, a.rank, a.use_rslora, a.adapter_scale) for a in d.adapters} == {2.0}
    assert set(a.rank for a in d.adapters) <= {8, 16, 32, 64}


@pytest.mark.parametrize("name", ["tiny"])
def test_oracle_deterministic(name):
    wl = workloads.make(name)
    a = oracle.workload_proj(wl)
    b = oracle.workload_proj(wl)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_embed_brute_force_fp64():
    P.check_embed_brute_force()


def test_embed_is_the_row_gather_of_the_flipped_projection():
    P.check_embed_row_gather_identity()


def test_embed_no_delta_rows_and_out_of_range_tokens():
    P.check_embed_no_delta_rows_are_the_embedding()


def test_silu_mul_closed_forms():
    P.check_silu_mul_closed_forms()


def test_gate_up_is_the_split_projections():
    P.check_gate_up_is_the_split_projections()


def test_moe_gather_brute_force_fp64():
    P.check_moe_gather_brute_force()


def test_moe_gather_is_the_grouped_fold():
    P.check_moe_gather_is_the_grouped_fold()


def test_stack_brute_force_fp64():
    P.check_stack_brute_force()


def test_stack_reductions_are_exact():
    P.check_stack_reductions()
