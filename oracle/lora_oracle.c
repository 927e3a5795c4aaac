/*
 * Oracle for the multi-adapter LoRA projection -- TEST INFRASTRUCTURE ONLY.
 *
 * Only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline leg may
 * load this library. It shares no code with the CUDA path: no headers, no
 * helpers, no tables. It is deliberately plain and slow.
 *
 * What it computes (the plain definition, no blocking or fusion):
 *
 *   y[i][n] = sum_k W[n][k] x[i][k]                       (base)
 *           + s * sum_r B_s[n][r] * (sum_k A_s[r][k] x[i][k])   (low-rank term)
 *
 * with s = seq_slot[i]'s scale, and the low-rank term skipped entirely (not
 * multiplied by zero) when row i has no adapter.
 *   - formula and layouts: ferrox-core `weight_matrix/lora.rs`, module doc
 *     ("Layouts": base [rows][cols], lora_a [rank][cols], lora_b [rows][rank])
 *     and `LoraDelta::project` / `LoraDelta::accumulate` / `LoraDelta::add_to`;
 *   - per-row routing through seq_slot, negative = no delta:
 *     spark_model `layers/ops/lora_delta.rs`, `apply_lora_bgmv`;
 *   - scale rule: ferrox-core `weight_matrix/lora.rs` module doc ("Scale") and
 *     `LoraDelta::new` / `effective_scale`; rsLoRA square-root rule:
 *     spark_model `lora_delta.rs`, `LoraPair` doc, and metrale
 *     `lora/slot_math.rs`, `scale_table_values`.
 *
 * Precision: inputs are bf16 (widened exactly to fp32); all sums are fp32,
 * accumulated in ascending index order, as the ferrox page's `dot` does.
 * Build with -ffp-contract=off so no multiply-add is fused and the result is
 * the same on every host.
 *
 * Parity pins live in tests/test_oracle_pins.py (brute force in fp64,
 * byte identities, closed forms and worked examples under tests/golden/).
 */
#include <math.h>
#include <omp.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

static float widen(uint16_t b)
{
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Threads of the OpenMP loops below (timing only; the result does not
 * depend on it: every output element is summed by one thread). */
void oracle_set_threads(int n)
{
    if (n > 0)
        omp_set_num_threads(n);
}

int oracle_max_threads(void) { return omp_get_max_threads(); }

/* adapter_scale * (alpha / rank), or * (alpha / sqrt(rank)) under rsLoRA,
 * or adapter_scale alone when alpha is 0 ("absent").
 * ferrox-core lora.rs `LoraDelta::new` computes alpha/rank in f32 once and
 * `effective_scale` multiplies the runtime scale by it; same order here. */
float oracle_scale(float alpha, int rank, int use_rslora, float adapter_scale)
{
    float factor = 1.0f;
    if (alpha != 0.0f) {
        if (use_rslora)
            factor = alpha / sqrtf((float)rank);
        else
            factor = alpha / (float)rank;
    }
    return adapter_scale * factor;
}

/* Does row `slot` get a low-rank term?  Negative or out-of-range slots, an
 * empty slot (no A) and a zero scale all mean "no delta"; the zero-scale case
 * is the ferrox `add_to` early return taken before any arithmetic. */
static int has_delta(int slot, int L, const uint16_t *const *A, const float *scale)
{
    if (slot < 0 || slot >= L)
        return 0;
    if (A[slot] == NULL)
        return 0;
    if (scale[slot] == 0.0f)
        return 0;
    return 1;
}

/* Stable grouping of rows by slot: bucket 0 holds the rows with no valid slot
 * (slot < 0 or slot >= L), bucket 1+s holds the rows of slot s; inside a
 * bucket rows keep their input order. seg_off has L+2 entries.
 * Written as one scan of the rows per bucket, so stability is evident. */
void oracle_slot_sort(const int32_t *seq_slot, int M, int L, int32_t *perm, int32_t *seg_off)
{
    int p = 0;
    for (int b = 0; b <= L; b++) {
        seg_off[b] = p;
        for (int i = 0; i < M; i++) {
            int s = seq_slot[i];
            int key = (s >= 0 && s < L) ? s + 1 : 0;
            if (key == b)
                perm[p++] = i;
        }
    }
    seg_off[L + 1] = p;
}

/*
 * y[row j][col c] for the selected rows and columns.
 *   x        [M][x_stride] bf16, row i starts at x + i*x_stride
 *   W        [N][K] bf16 row-major
 *   A[s]     [rank[s]][K] bf16 (true rank, no padding) or NULL
 *   B[s]     [N][rank[s]] bf16
 *   scale[s] effective scale of slot s (oracle_scale)
 *   rows     indices of the rows to compute (NULL = 0..M-1, n_rows = M)
 *   cols     indices of the columns to compute (NULL = 0..N-1, n_cols = N)
 *   y        [n_rows][n_cols] fp32
 */
void oracle_proj(const uint16_t *x, int64_t x_stride, const uint16_t *W, int M, int K, int N,
                 const int32_t *seq_slot, int L, const uint16_t *const *A,
                 const uint16_t *const *B, const int32_t *rank, const float *scale,
                 const int32_t *rows, int n_rows, const int32_t *cols, int n_cols, float *y)
{
    if (rows == NULL)
        n_rows = M;
    if (cols == NULL)
        n_cols = N;
    int rmax = 0;
    for (int s = 0; s < L; s++)
        if (A[s] != NULL && rank[s] > rmax)
            rmax = rank[s];
    if (n_rows <= 0 || n_cols <= 0)
        return;

    float *xf = (float *)malloc(sizeof(float) * (size_t)n_rows * (size_t)(K > 0 ? K : 1));
    float *h = (float *)malloc(sizeof(float) * (size_t)n_rows * (size_t)(rmax > 0 ? rmax : 1));

    /* Pass 1, per row: widen x, then h = A_s x (ferrox `project`). */
#pragma omp parallel for schedule(dynamic, 1)
    for (int j = 0; j < n_rows; j++) {
        int i = rows ? rows[j] : j;
        float *xr = xf + (size_t)j * K;
        for (int k = 0; k < K; k++)
            xr[k] = widen(x[(int64_t)i * x_stride + k]);
        int s = seq_slot[i];
        if (has_delta(s, L, A, scale)) {
            for (int r = 0; r < rank[s]; r++) {
                const uint16_t *arow = A[s] + (size_t)r * K;
                float acc = 0.0f;
                for (int k = 0; k < K; k++)
                    acc += widen(arow[k]) * xr[k];
                h[(size_t)j * rmax + r] = acc;
            }
        }
    }

    /* Pass 2, per output element: base dot product, then the low-rank term
     * s * (b_n . h) added once (ferrox `accumulate`). */
#pragma omp parallel for collapse(2) schedule(static)
    for (int j = 0; j < n_rows; j++) {
        for (int c = 0; c < n_cols; c++) {
            int i = rows ? rows[j] : j;
            int n = cols ? cols[c] : c;
            const float *xr = xf + (size_t)j * K;
            const uint16_t *wrow = W + (size_t)n * K;
            float acc = 0.0f;
            for (int k = 0; k < K; k++)
                acc += widen(wrow[k]) * xr[k];
            int s = seq_slot[i];
            if (has_delta(s, L, A, scale)) {
                const uint16_t *brow = B[s] + (size_t)n * rank[s];
                const float *hr = h + (size_t)j * rmax;
                float d = 0.0f;
                for (int r = 0; r < rank[s]; r++)
                    d += widen(brow[r]) * hr[r];
                acc += scale[s] * d;
            }
            y[(size_t)j * n_cols + c] = acc;
        }
    }
    free(xf);
    free(h);
}

/*
 * Several adapters on one base matrix (ferrox-core `weight_matrix/lora.rs`,
 * `LoraStack`: every adapter attached to a matrix is one term of the sum,
 * applied in order by `LoraStack::add_to`):
 *
 *   y[i][n] = sum_k W[n][k] x[i][k] + sum_m s_m * sum_r B_m[n][r] * (A_m x_i)[r]
 *
 * where m runs over the members of row i's slot, member_off[s] ..
 * member_off[s+1]-1, in order. A member whose scale is 0 is skipped before
 * any arithmetic (the `add_to` early return), so a stack whose every scale is
 * 0 -- or a slot with no members, or a row whose slot is negative or >= L --
 * leaves the base product untouched, byte for byte.
 *   A[m] [rank[m]][K], B[m] [N][rank[m]] bf16, scale[m] the member's
 *   effective scale (oracle_scale); rows / cols / y as in oracle_proj.
 * Each term is accumulated into the running fp32 sum in member order, as
 * `add_to` adds each delta into `out` in turn.
 */
void oracle_proj_stack(const uint16_t *x, int64_t x_stride, const uint16_t *W, int M, int K, int N,
                       const int32_t *seq_slot, int L, const int32_t *member_off,
                       const uint16_t *const *A, const uint16_t *const *B, const int32_t *rank,
                       const float *scale, const int32_t *rows, int n_rows, const int32_t *cols,
                       int n_cols, float *y)
{
    if (rows == NULL)
        n_rows = M;
    if (cols == NULL)
        n_cols = N;
    if (n_rows <= 0 || n_cols <= 0)
        return;
    int n_members = member_off[L];
    int rmax = 1;
    for (int m = 0; m < n_members; m++)
        if (rank[m] > rmax)
            rmax = rank[m];

#pragma omp parallel for schedule(dynamic, 1)
    for (int j = 0; j < n_rows; j++) {
        int i = rows ? rows[j] : j;
        float *xq = (float *)malloc(sizeof(float) * (size_t)(K > 0 ? K : 1));
        float *h = (float *)malloc(sizeof(float) * (size_t)rmax);
        for (int k = 0; k < K; k++)
            xq[k] = widen(x[(int64_t)i * x_stride + k]);
        int s = seq_slot[i];
        int m0 = 0, m1 = 0;
        if (s >= 0 && s < L) {
            m0 = member_off[s];
            m1 = member_off[s + 1];
        }
        for (int c = 0; c < n_cols; c++) {
            int n = cols ? cols[c] : c;
            const uint16_t *wn = W + (size_t)n * K;
            float base = 0.0f;
            for (int k = 0; k < K; k++)
                base += widen(wn[k]) * xq[k];
            y[(size_t)j * n_cols + c] = base;
        }
        for (int m = m0; m < m1; m++) {
            if (scale[m] == 0.0f || A[m] == NULL || rank[m] <= 0)
                continue;
            /* h = A_m x (ferrox `project`) */
            for (int r = 0; r < rank[m]; r++) {
                const uint16_t *am = A[m] + (size_t)r * K;
                float hv = 0.0f;
                for (int k = 0; k < K; k++)
                    hv += widen(am[k]) * xq[k];
                h[r] = hv;
            }
            /* out[n] += s_m * (b_n . h) (ferrox `accumulate`) */
            for (int c = 0; c < n_cols; c++) {
                int n = cols ? cols[c] : c;
                const uint16_t *bm = B[m] + (size_t)n * rank[m];
                float dm = 0.0f;
                for (int r = 0; r < rank[m]; r++)
                    dm += widen(bm[r]) * h[r];
                y[(size_t)j * n_cols + c] += scale[m] * dm;
            }
        }
        free(xq);
        free(h);
    }
}

/*
 * Embedding row gather through the adapted matrix E + s*B*A (ferrox-core
 * `weight_matrix/lora.rs`, `LoraDelta::add_row_to`: the delta of ONE row r of
 * s*B*A is s * (b_r . A), which is what a token-embedding gather needs):
 *
 *   y[i][e] = E[t][e] + s * sum_r B_s[t][r] * A_s[r][e],    t = tokens[i]
 *
 *   E     [vocab][n_embd] bf16 (the adapted matrix: rows = vocab)
 *   A[s]  [rank[s]][n_embd] bf16, B[s] [vocab][rank[s]] bf16
 * The low-rank term is skipped for rows with no delta, as in oracle_proj; a
 * token outside [0, vocab) gives a zero row. y is [M][n_embd] fp32.
 */
void oracle_embed(const int32_t *tokens, const uint16_t *E, int M, int vocab, int n_embd,
                  const int32_t *seq_slot, int L, const uint16_t *const *A,
                  const uint16_t *const *B, const int32_t *rank, const float *scale, float *y)
{
#pragma omp parallel for schedule(static)
    for (int i = 0; i < M; i++) {
        float *yr = y + (size_t)i * n_embd;
        int t = tokens[i];
        if (t < 0 || t >= vocab) {
            for (int e = 0; e < n_embd; e++)
                yr[e] = 0.0f;
            continue;
        }
        int s = seq_slot[i];
        int on = has_delta(s, L, A, scale);
        for (int e = 0; e < n_embd; e++) {
            float v = widen(E[(size_t)t * n_embd + e]);
            if (on) {
                const uint16_t *b_of_t = B[s] + (size_t)t * rank[s];
                float dsum = 0.0f;
                for (int r = 0; r < rank[s]; r++)
                    dsum += widen(b_of_t[r]) * widen(A[s][(size_t)r * n_embd + e]);
                v += scale[s] * dsum;
            }
            yr[e] = v;
        }
    }
}

/*
 * MoE expert down projection: slot-row j with expert_offsets[e] <= j <
 * expert_offsets[e+1] is the projection above with expert e's base W[e] and
 * expert e's adapters (A[e*L + s], B[e*L + s], rank[e*L + s], scale[e*L + s]).
 * spark_model `lora_delta.rs`, `LoraKernels` (the MoE down_proj fold keyed on
 * the expert through expert_offsets).
 * rows/cols select outputs as in oracle_proj; y is [n_rows][n_cols].
 */
/*
 * Gated MLP input from a fused [gate|up] projection (frink `lora_attach.rs`,
 * `parts_mut`: a fused ffn_up holds the gate rows first, then the up rows, and
 * its adapter's B rows split the same way over one A). y is the projection's
 * output, [M][2I] at row stride y_stride: columns [0, I) are the gate g,
 * [I, 2I) the up u. act[i][n] = silu(g) * u with silu(g) = g / (1 + e^-g),
 * in fp32.
 */
void oracle_silu_mul(const float *y, int M, int I, int64_t y_stride, float *act)
{
    for (int i = 0; i < M; i++) {
        const float *gr = y + (size_t)i * y_stride;
        const float *ur = gr + I;
        for (int n = 0; n < I; n++) {
            float g = gr[n];
            float sg = g / (1.0f + expf(-g));
            act[(size_t)i * I + n] = sg * ur[n];
        }
    }
}

void oracle_moe(const uint16_t *x, int64_t x_stride, const uint16_t *const *W, const int32_t *expert_offsets,
                int E, int T, int K, int N, const int32_t *seq_slot, int L,
                const uint16_t *const *A, const uint16_t *const *B, const int32_t *rank,
                const float *scale, const int32_t *rows, int n_rows, const int32_t *cols,
                int n_cols, float *y)
{
    if (rows == NULL)
        n_rows = T;
    if (cols == NULL)
        n_cols = N;
    for (int j = 0; j < n_rows; j++) {
        int i = rows ? rows[j] : j;
        int e = -1;
        for (int q = 0; q < E; q++)
            if (expert_offsets[q] <= i && i < expert_offsets[q + 1])
                e = q;
        if (e < 0) {
            for (int c = 0; c < n_cols; c++)
                y[(size_t)j * n_cols + c] = NAN;
            continue;
        }
        /* one row through expert e's projection; seq_slot indexed at row i */
        int32_t one = i;
        oracle_proj(x, x_stride, W[e], T, K, N, seq_slot, L, A + (size_t)e * L,
                    B + (size_t)e * L, rank + (size_t)e * L, scale + (size_t)e * L,
                    &one, 1, cols, n_cols, y + (size_t)j * n_cols);
    }
}

/*
 * Decode-path MoE fold keyed on the expert through a per-slot-row index
 * (spark_model `lora_delta.rs`, `LoraKernels`, moe_gather: the unsorted,
 * slot-major analogue of the expert_offsets fold). Slot-row j = token
 * j / top_k, choice j % top_k; its expert is indices[j]. Slot-row value:
 *
 *   v_j = W_e x_j + s B_{e,s} (A_{e,s} x_j),  e = indices[j], s = seq_slot[j]
 *
 * (zero when e is outside [0, E)). Without combine weights y[j] = v_j; with
 * them y[t] = sum_{i < top_k} combine[t*top_k + i] * v_{t*top_k + i}, the
 * weighted sum of a token's expert outputs, accumulated in choice order, fp32.
 * Adapters are indexed e*L + s like oracle_moe.
 */
void oracle_moe_gather(const uint16_t *x, int64_t x_stride, const uint16_t *const *W, const int32_t *indices,
                       int E, int T, int K, int N, const int32_t *seq_slot, int L,
                       const uint16_t *const *A, const uint16_t *const *B, const int32_t *rank,
                       const float *scale, const float *combine, int top_k, float *y)
{
    float *v = (float *)malloc(sizeof(float) * (size_t)N);
    for (int j = 0; j < T; j++) {
        int e = indices[j];
        if (e < 0 || e >= E) {
            for (int n = 0; n < N; n++)
                v[n] = 0.0f;
        } else {
            int32_t one = j;
            oracle_proj(x, x_stride, W[e], T, K, N, seq_slot, L, A + (size_t)e * L, B + (size_t)e * L,
                        rank + (size_t)e * L, scale + (size_t)e * L, &one, 1, NULL, N, v);
        }
        if (combine == NULL) {
            memcpy(y + (size_t)j * N, v, sizeof(float) * (size_t)N);
        } else {
            float *yt = y + (size_t)(j / top_k) * N;
            if (j % top_k == 0)
                for (int n = 0; n < N; n++)
                    yt[n] = 0.0f;
            float w = combine[j];
            for (int n = 0; n < N; n++)
                yt[n] += w * v[n];
        }
    }
    free(v);
}

/* Stable grouping of MoE slot-rows by (expert, slot): for expert e, bucket
 * e*(L+1) holds the segment's rows with no valid slot, bucket e*(L+1)+1+s the
 * rows of slot s. seg_off has E*(L+1)+1 entries. */
void oracle_moe_slot_sort(const int32_t *expert_offsets, int E, const int32_t *seq_slot, int L,
                          int32_t *perm, int32_t *seg_off)
{
    int p = 0;
    for (int e = 0; e < E; e++) {
        for (int b = 0; b <= L; b++) {
            seg_off[e * (L + 1) + b] = p;
            for (int i = expert_offsets[e]; i < expert_offsets[e + 1]; i++) {
                int s = seq_slot[i];
                int key = (s >= 0 && s < L) ? s + 1 : 0;
                if (key == b)
                    perm[p++] = i;
            }
        }
    }
    seg_off[E * (L + 1)] = p;
}
