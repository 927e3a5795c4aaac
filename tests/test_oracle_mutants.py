"""Every plausible mistake planted in a copy of the oracle fails a pin.

Each mutant is a textual edit of oracle/lora_oracle.c compiled into a
temporary library; the oracle itself is never modified. The edits model the
mistakes a from-scratch implementation is likely to make: a dropped term, a
wrong sign, a transposed operand, a wrong index, the wrong scale rule, a
broken routing or grouping rule.
"""
import os
import subprocess

import pytest

import oracle
from tests import oracle_pins as P

SRC = os.path.join(os.path.dirname(oracle.__file__), "lora_oracle.c")

MUTANTS = {
    "drop_base_term": ("acc += widen(wrow[k]) * xr[k];", ";"),
    "delta_sign": ("acc += scale[s] * d;", "acc -= scale[s] * d;"),
    "drop_scale": ("acc += scale[s] * d;", "acc += d;"),
    "B_transposed": ("d += widen(brow[r]) * hr[r];",
                     "d += widen(B[s][(size_t)r * N + n]) * hr[r];"),
    "A_wrong_x_index": ("acc += widen(arow[k]) * xr[k];", "acc += widen(arow[k]) * xr[K - 1 - k];"),
    "scale_rank_over_alpha": ("factor = alpha / (float)rank;", "factor = (float)rank / alpha;"),
    "rslora_as_plain": ("factor = alpha / sqrtf((float)rank);", "factor = alpha / (float)rank;"),
    "alpha0_gives_zero": ("float factor = 1.0f;", "float factor = 0.0f;"),
    "ignore_adapter_scale": ("return adapter_scale * factor;", "return factor;"),
    "last_slot_dropped": ("if (slot < 0 || slot >= L)\n        return 0;",
                          "if (slot < 0 || slot >= L - 1)\n        return 0;"),
    "sort_unstable": ("for (int i = 0; i < M; i++) {\n            int s = seq_slot[i];",
                      "for (int i = M - 1; i >= 0; i--) {\n            int s = seq_slot[i];"),
    "sort_base_bucket_last": ("int key = (s >= 0 && s < L) ? s + 1 : 0;\n            if (key == b)\n                perm[p++] = i;\n        }\n    }\n    seg_off[L + 1] = p;",
                              "int key = (s >= 0 && s < L) ? s : L;\n            if (key == b)\n                perm[p++] = i;\n        }\n    }\n    seg_off[L + 1] = p;"),
    "moe_expert_off_by_one": ("if (expert_offsets[q] <= i && i < expert_offsets[q + 1])",
                              "if (expert_offsets[q] < i && i <= expert_offsets[q + 1])"),
    "widen_wrong_shift": ("uint32_t u = ((uint32_t)b) << 16;", "uint32_t u = ((uint32_t)b) << 15;"),
    "embed_B_row_of_the_row_index": ("const uint16_t *b_of_t = B[s] + (size_t)t * rank[s];",
                                     "const uint16_t *b_of_t = B[s] + (size_t)(i % vocab) * rank[s];"),
    "embed_drop_scale": ("v += scale[s] * dsum;", "v += dsum;"),
    "embed_A_transposed": ("widen(A[s][(size_t)r * n_embd + e]);",
                           "widen(A[s][(size_t)e * rank[s] + r]);"),
    "silu_sign": ("float sg = g / (1.0f + expf(-g));", "float sg = g / (1.0f + expf(g));"),
    "silu_halves_swapped": ("act[(size_t)i * I + n] = sg * ur[n];",
                            "act[(size_t)i * I + n] = gr[n] / (1.0f + expf(-ur[n])) * gr[n];"),
    "silu_without_up": ("act[(size_t)i * I + n] = sg * ur[n];", "act[(size_t)i * I + n] = sg;"),
    "gather_weight_of_the_token": ("float w = combine[j];", "float w = combine[j / top_k];"),
    "gather_expert_ignored": ("int e = indices[j];", "int e = indices[j] >= 0 ? 0 : -1;"),
    "gather_no_reset_per_token": ("if (j % top_k == 0)\n                for (int n = 0; n < N; n++)\n                    yt[n] = 0.0f;",
                                  "if (j == 0)\n                for (int n = 0; n < N; n++)\n                    yt[n] = 0.0f;"),
    "stack_first_member_dropped": ("for (int m = m0; m < m1; m++) {", "for (int m = m0 + 1; m < m1; m++) {"),
    "stack_first_scale_for_all": ("y[(size_t)j * n_cols + c] += scale[m] * dm;",
                                  "y[(size_t)j * n_cols + c] += scale[m0] * dm;"),
    "stack_h_from_the_first_member": ("const uint16_t *am = A[m] + (size_t)r * K;",
                                      "const uint16_t *am = A[m0] + (size_t)(r % rank[m0]) * K;"),
    "h_uses_pool_row_of_next_slot": ("const uint16_t *arow = A[s] + (size_t)r * K;",
                                     "const uint16_t *arow = A[(s + 1) % L] ? A[(s + 1) % L] + (size_t)r * K : A[s] + (size_t)r * K;"),
}


@pytest.fixture(scope="module")
def src_text():
    with open(SRC) as f:
        return f.read()


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, src_text, tmp_path):
    old, new = MUTANTS[name]
    assert src_text.count(old) == 1, f"mutation site for {name} not unique"
    c = tmp_path / f"{name}.c"
    c.write_text(src_text.replace(old, new))
    so = tmp_path / f"{name}.so"
    subprocess.run(["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared", "-o",
                    str(so), str(c), "-lm"], check=True)
    failed = []
    with oracle._use_library(str(so)):
        for check in P.ALL_CHECKS:
            try:
                check()
            except AssertionError:
                failed.append(check.__name__)
    assert failed, f"mutant {name} passed every pin"
