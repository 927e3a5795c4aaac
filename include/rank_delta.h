/*
 * rank_delta.h -- C ABI of the GB300 multi-adapter LoRA projection.
 *
 * One operation, in two shapes:
 *
 *   y[i,:] = W x_i + s[slot_i] * B[slot_i] (A[slot_i] x_i)        (lora_proj_apply)
 *
 * and the same per slot-row of a mixture-of-experts down projection, with the
 * expert's own base and adapters (lora_moe_down_apply), and as a row gather of
 * the adapted token-embedding matrix (lora_embed_apply):
 *
 *   y[i,:] = E[t_i,:] + s[slot_i] * B[slot_i][t_i,:] A[slot_i]        t_i = tokens[i]
 *
 * Sources (page title, section):
 *   - ferrox-core `weight_matrix/lora.rs`, module doc ("Layouts", "Scale",
 *     "Cost when absent") and `LoraDelta`: the formula, the layouts
 *     W [n_out][n_in], A [rank][n_in], B [n_out][rank], the scale rule and the
 *     rule that a zero scale skips the delta before any arithmetic;
 *   - spark_model `layers/ops/lora_delta.rs`, `LoraRoute`, `LoraPair`,
 *     `apply_lora_bgmv`: per-row routing through an i32 seq_slot buffer
 *     (negative = no delta), [max_loras] device pointer tables a_table/b_table
 *     (NULL = base only) and an f32 scale_table, the pool padded to max_rank
 *     with zeros, row strides in elements, and a graph-safe contract (no
 *     allocation, no synchronisation);
 *   - metrale `lora/slot_math.rs`, `pool_slot_bytes`, `module_slot_offsets`,
 *     `scale_table_values`, `build_seq_slot_host`: the pool byte layout (A then
 *     B per slot, bf16) and the host seq_slot helper.
 *
 * Conventions (all entry points):
 *   - The library allocates nothing. Every buffer is the caller's. Device
 *     pointers are plain CUDA device addresses; "host" arguments are plain
 *     host memory. bf16 values are passed as raw 16-bit storage (`uint16_t`).
 *   - `stream` is a cudaStream_t (NULL = legacy default stream). Work is
 *     enqueued on it; the hot-path calls never synchronise the host.
 *   - Every call returns a lora_status. Host argument errors enqueue
 *     nothing; lora_last_error() then returns a message naming every
 *     dimension involved (thread-local, valid until the next call on that
 *     thread).
 *   - Device-side anomalies (a seq_slot >= max_loras, an in-kernel wait that
 *     gave up) never trap: the row takes the no-delta path and a bit is set in
 *     the workspace status word (lora_status_get).
 *   - Alignment: x, W and the pool must start on a 16-byte boundary, and
 *     n_in, max_rank and every x row stride must be multiples of 8
 *     elements (16 bytes): the kernels stage x and W tiles with the tensor
 *     memory accelerator, which copies 16-byte granules.
 */
#ifndef RANK_DELTA_H
#define RANK_DELTA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* cudaStream_t without requiring the CUDA headers. */
typedef struct CUstream_st *lora_stream_t;

typedef int lora_status;
enum {
    LORA_OK = 0,
    LORA_ERR_NULL = 1,        /* a required pointer is NULL */
    LORA_ERR_SHAPE = 2,       /* a dimension, rank or stride does not fit */
    LORA_ERR_RANGE = 3,       /* a slot or expert index is out of range */
    LORA_ERR_ALIGN = 4,       /* a pointer or stride breaks the 16-byte rule */
    LORA_ERR_WORKSPACE = 5,   /* the workspace is smaller than required */
    LORA_ERR_CUDA = 6,        /* a CUDA runtime call failed (message has the CUDA error) */
    LORA_ERR_UNSUPPORTED = 7, /* a size beyond what the kernels handle (message says which) */
    LORA_ERR_NOT_INIT = 8,    /* the route was not set up by lora_route_init */
    LORA_ERR_POOL_FULL = 9    /* lora_select_victim_slot: every cached slot is in use */
};

/* Bits of the workspace status word (lora_status_get). */
enum {
    LORA_FLAG_SLOT_RANGE = 1u << 0,   /* a seq_slot value >= max_loras was seen; those rows got no delta */
    LORA_FLAG_WAIT_TIMEOUT = 1u << 1, /* an in-kernel wait gave up; that call's output is not valid */
    LORA_FLAG_BAD_OFFSETS = 1u << 2,  /* expert_offsets not non-decreasing within [0, T]; rows outside skipped */
    LORA_FLAG_TOKEN_RANGE = 1u << 3,  /* lora_embed_apply: a token outside [0, vocab); its row is zero */
    LORA_FLAG_EXPERT_RANGE = 1u << 4  /* lora_moe_gather_apply: an expert index outside [0, E); that slot-row adds nothing */
};

/* What a route's pool holds (lora_route.kind). */
enum {
    LORA_ROUTE_PROJ = 0, /* a projection's pairs: A [max_rank][n_in], B [n_out][max_rank] */
    LORA_ROUTE_EMBED = 1 /* a token embedding's pairs: A stored transposed, see lora_embed_route_init */
};

/* Path selection for lora_proj_apply_ex (lora_proj_apply uses LORA_PATH_AUTO). */
enum {
    LORA_PATH_AUTO = 0, /* by row count: CUDA-core GEMV for few rows, tensor cores otherwise */
    LORA_PATH_SIMT = 1, /* CUDA-core GEMV path (any row count; slow for many rows) */
    LORA_PATH_TC = 2,   /* tcgen05 tensor-core path: a routing kernel, then the projection kernel
                           (which also runs the shrink: CUDA-core units below 2048 rows,
                           tensor-core tiles of 128 rows from 2048) */
    LORA_PATH_TC_ONE = 3 /* batches of up to 256 rows in one launch: routing, shrink, base, expand
                            and the split-K sum in a single kernel (other shapes, or a device that
                            cannot hold its grid, take LORA_PATH_TC). Measured slower than
                            LORA_PATH_TC on the decode and fused-QKV shapes; kept for comparison */
};

/*
 * One projection's adapter pool and routing tables (spark_model
 * `lora_delta.rs`, `LoraRoute`). Filled by lora_route_init; the caller owns
 * the struct (host memory) and every buffer it points to (device memory).
 *
 * pool        max_loras slots of slot_bytes = (max_rank*n_in + n_out*max_rank)*2
 *             bytes. Slot s starts at pool + s*slot_bytes and holds A as
 *             [max_rank][n_in] bf16 followed by B as [n_out][max_rank] bf16,
 *             rows and columns past the adapter's rank zero (metrale
 *             `slot_math.rs`, `pool_slot_bytes`).
 * a_table     [max_loras] device pointers to each slot's A, NULL = empty slot.
 * b_table     [max_loras] device pointers to each slot's B, NULL = empty slot.
 * scale_table [max_loras] f32 effective scale, read by the kernels at apply
 *             time; 0 = the delta is skipped.
 * factor_table[max_loras] f32 alpha factor (alpha/rank, alpha/sqrt(rank), or 1
 *             when alpha is 0), so that lora_set_scale can rebuild the scale.
 * rank_table  [max_loras] i32 true rank of each slot (0 = empty).
 * comp_table  [max_loras][LORA_COMP_STRIDE] f32 per-rank factor of each slot:
 *             the delta of slot s is sum_r B[:, r] * (scale_table[s] *
 *             comp_table[s][r]) * (A x)[r]. 1 for every rank of a slot packed
 *             with lora_pool_pack; a slot holding a stack of adapters
 *             (lora_pool_pack_stack) carries each member's own scale on that
 *             member's ranks.
 */
#define LORA_COMP_STRIDE 256

typedef struct lora_route {
    void *pool;
    const void **a_table;
    const void **b_table;
    float *scale_table;
    float *factor_table;
    int32_t *rank_table;
    float *comp_table;
    int32_t n_in;      /* K */
    int32_t n_out;     /* N */
    int32_t max_rank;  /* R: the pool's padded rank */
    int32_t max_loras; /* L: number of slots */
    int32_t kind;      /* LORA_ROUTE_PROJ or LORA_ROUTE_EMBED */
    int32_t reserved;
    uint64_t magic;    /* set by lora_route_init / lora_embed_route_init */
} lora_route;

/* Bytes of one projection's pool: max_loras * (max_rank*n_in + n_out*max_rank) * 2.
 * Returns 0 for a non-positive argument. */
size_t lora_pool_bytes(int max_loras, int max_rank, int n_in, int n_out);

/* Bytes of the device tables of one route (a_table, b_table, scale_table,
 * factor_table, rank_table, comp_table, each 256-byte aligned). 0 for
 * max_loras <= 0. */
size_t lora_route_table_bytes(int max_loras);

/*
 * Fill `rt` and clear its tables on `stream` (every slot empty).
 *   pool    device buffer of at least lora_pool_bytes(...) bytes, 16-byte aligned
 *   tables  device buffer of at least lora_route_table_bytes(max_loras) bytes,
 *           256-byte aligned
 * Errors: NULL pointers, non-positive sizes, n_in not a multiple of 8, buffers
 * too small (message names the sizes), max_loras > 1023, max_rank > 256 or
 * not a multiple of 8.
 */
lora_status lora_route_init(lora_route *rt, void *pool, size_t pool_bytes, void *tables,
                            size_t table_bytes, int max_loras, int max_rank, int n_in,
                            int n_out, lora_stream_t stream);

/*
 * Copy one adapter's pair into `slot` and publish it in the tables
 * (spark_model `lora_delta.rs`, `LoraPair`: PEFT layout, zero padding to the
 * pool rank, scale not folded into B).
 *   A      [rank][n_in] bf16, row-major, host or device memory
 *   B      [n_out][rank] bf16, row-major, host or device memory
 *   alpha  the adapter's alpha; 0 means absent (the scale is then the bare
 *          adapter_scale)
 *   use_rslora  nonzero: factor alpha/sqrt(rank) instead of alpha/rank
 *   adapter_scale  runtime multiplier (1 for a plain adapter)
 * The slot is zeroed first, so pad rows of A and pad columns of B are zero.
 * scale_table[slot] = adapter_scale * factor, computed in f32 on the host
 * (ferrox-core `lora.rs`, `LoraDelta::new` and `effective_scale`).
 * Errors: slot outside [0, max_loras) (message names the range); rank 0 or
 * rank > max_rank (message names [n_out x n_in], the rank, max_rank and the
 * element counts A and B must have); NULL A or B.
 * Stream-ordered: applies enqueued earlier on `stream` see the old contents.
 */
lora_status lora_pool_pack(const lora_route *rt, int slot, const void *A, const void *B,
                           int rank, float alpha, int use_rslora, float adapter_scale,
                           lora_stream_t stream);

/*
 * Several adapters on one matrix, in one slot (ferrox-core `weight_matrix/
 * lora.rs`, `LoraStack`: every adapter attached to a matrix is one term of
 * the sum, y = W x + sum_m s_m B_m (A_m x)). The slot's rows get every
 * member's delta.
 *   n               members (0: the slot becomes empty)
 *   A[m], B[m]      host arrays of n pointers: member m's [ranks[m]][n_in] and
 *                   [n_out][ranks[m]] bf16 pair, host or device memory
 *   ranks, alphas, use_rslora, adapter_scales   host arrays of n entries, each
 *                   member's rank, alpha, rule and runtime scale, with the
 *                   meaning they have in lora_pool_pack
 * Member m's scale s_m = adapter_scales[m] * factor(alphas[m], ranks[m],
 * use_rslora[m]). A member whose s_m is 0 is left out (the delta of a
 * zero-scale adapter is skipped before any arithmetic); the others are laid
 * out one after another along the slot's rank (A rows, B columns), their
 * ranks summing to at most max_rank, and comp_table[slot] holds s_m on member
 * m's ranks. scale_table[slot] = factor_table[slot] = 1, so lora_set_scale /
 * lora_set_scales afterwards multiply the whole stack by the value given. A
 * stack with no member left is an empty slot.
 * Errors: embedding route (LORA_ERR_UNSUPPORTED); slot outside [0, max_loras);
 * n < 0; NULL arrays with n > 0 or a NULL member pointer; a rank < 1; the
 * kept members' ranks summing past max_rank (message names the sum and
 * max_rank). Nothing is written on an error.
 * Stream-ordered like lora_pool_pack.
 */
lora_status lora_pool_pack_stack(const lora_route *rt, int slot, int n, const void *const *A,
                                 const void *const *B, const int32_t *ranks, const float *alphas,
                                 const int32_t *use_rslora, const float *adapter_scales,
                                 lora_stream_t stream);

/* Empty `slot` (table entries NULL / 0): its rows get no delta afterwards. */
lora_status lora_pool_unpack(const lora_route *rt, int slot, lora_stream_t stream);

/*
 * Set the runtime scale of `slot`: scale_table[slot] = adapter_scale *
 * factor_table[slot], written by a one-thread kernel on `stream`, so it takes
 * effect for every apply enqueued after it (ferrox-core `lora.rs`,
 * `LoraScale`; the scale is read at apply time). An empty slot keeps scale 0.
 * Errors: slot outside [0, max_loras); the message names the range (frink
 * `lora_attach.rs`, `set_lora_scales`).
 */
lora_status lora_set_scale(const lora_route *rt, int slot, float adapter_scale,
                           lora_stream_t stream);

/*
 * Set every slot's runtime scale at once (frink `lora_attach.rs`,
 * `set_lora_scales`): slot ids[i] gets scales[i] (the last entry wins when an
 * id is listed twice), every slot not listed gets 0; each entry becomes
 * scale_table[slot] = scale * factor_table[slot]. Written by kernels on
 * `stream` (one launch per 256 slots), so it takes effect for every apply
 * enqueued after it. ids and scales are host arrays of n entries (n >= 0;
 * n = 0 sets every scale to 0).
 * Errors (nothing is written): NULL ids/scales with n > 0; an id outside
 * [0, max_loras) -- the message names the id and the range.
 */
lora_status lora_set_scales(const lora_route *rt, const int32_t *ids, const float *scales, int n,
                            lora_stream_t stream);

/*
 * One cached slot, as the promotion cache sees it (metrale
 * `lora/slot_math.rs`, `select_victim_slot`): whether it holds an adapter, how
 * many in-flight requests use it, and when it was last used (any monotone
 * counter).
 */
typedef struct lora_slot_view {
    int32_t slot;
    int32_t filled;
    int32_t ref_count;
    int32_t pad;
    uint64_t last_used;
} lora_slot_view;

/*
 * The slot a promotion overwrites (host only): the first unfilled slot of
 * `cache` in array order; else, among slots with ref_count == 0, the one with
 * the smallest last_used (the first such in array order on a tie); else
 * LORA_ERR_POOL_FULL. *victim receives the chosen entry's `slot`.
 * Errors: NULL cache with n > 0 or NULL victim; n < 0; LORA_ERR_POOL_FULL
 * (n = 0 included).
 */
lora_status lora_select_victim_slot(const lora_slot_view *cache, int n, int32_t *victim);

/*
 * Workspace of lora_proj_apply for M rows on route `rt` (device scratch the
 * caller provides: the routing sort, the shrink work list, the rank-sized h of
 * every row, split-K partial tiles and handoff counters, and the status
 * words). Its contents need no initialisation: every call tags what it waits
 * on with an epoch kept in the workspace. 256-byte aligned sections; the
 * caller passes a buffer of at least this many bytes, 256-byte aligned.
 * Returns 0 if rt is NULL or not initialised.
 */
size_t lora_proj_workspace_bytes(int M, const lora_route *rt);

/* The workspace a call on an explicit path needs (LORA_PATH_*): for
 * LORA_PATH_TC_ONE and up to 256 rows, the larger of the general workspace
 * and the one-launch kernel's (its h exchange, and the K parts' fp32 tiles
 * for the cooperative launch); otherwise lora_proj_workspace_bytes. With less,
 * LORA_PATH_TC_ONE calls take LORA_PATH_TC. */
size_t lora_proj_workspace_bytes_ex(int M, const lora_route *rt, int path);

/*
 * y[i, :] = W x_i + s * B_s (A_s x_i), s = seq_slot[i], for i in [0, M)
 * (spark_model `lora_delta.rs`, `apply_lora_bgmv`; ferrox-core `lora.rs`,
 * `LoraDelta::add_batch_to`).
 *   x         device, M rows of n_in bf16, row i at x + i*x_stride (elements)
 *   W         device, [N][K] bf16 row-major (the base weight, n_out x n_in)
 *   M, K, N   rows, n_in, n_out; K and N must equal rt->n_in and rt->n_out
 *   seq_slot  device [M] int32: slot in [0, max_loras) or negative for no delta
 *   y         device, M rows of N bf16, row i at y + i*y_stride (elements);
 *             written, not accumulated into
 *   ws        device workspace of lora_proj_workspace_bytes(M, rt) bytes
 * A row gets no delta -- its output is exactly the base product rounded to
 * bf16, byte for byte what an all-(-1) seq_slot gives -- when its slot is
 * negative, >= max_loras (a status bit is also set), empty, or has scale 0.
 * Accumulation is fp32; y is rounded once, to nearest even.
 * M = 0 is a no-op. The call enqueues kernels on `stream` only; it neither
 * allocates nor synchronises, so it can be captured in a CUDA graph.
 * Errors: NULL pointers (M > 0), K or N not matching the route, K or x_stride
 * not a multiple of 8, x_stride < K, y_stride < N, x or W not 16-byte
 * aligned, ws too small.
 */
lora_status lora_proj_apply(const void *x, int64_t x_stride, const void *W, int M, int K, int N,
                            const int32_t *seq_slot, const lora_route *rt, void *y,
                            int64_t y_stride, void *ws, size_t ws_bytes, lora_stream_t stream);

/* lora_proj_apply with an explicit path (LORA_PATH_*); results of the two
 * paths agree within the fp32 accumulation-order tolerance, not bit for bit. */
lora_status lora_proj_apply_ex(const void *x, int64_t x_stride, const void *W, int M, int K,
                               int N, const int32_t *seq_slot, const lora_route *rt, void *y,
                               int64_t y_stride, void *ws, size_t ws_bytes, int path,
                               lora_stream_t stream);

/*
 * Bytes of the scratch array built into the library for
 * lora_proj_apply_static_ws (held on every GPU that loads the library).
 */
#define LORA_STATIC_WS_BYTES (8u << 20)

/*
 * lora_proj_apply for callers that cannot allocate device memory -- for
 * example a plugin whose host framework owns all device memory and offers no
 * allocator, or a service that must not grow device memory after start-up.
 * The pages have no counterpart: it exists for those callers only.
 *
 * Same arguments, results and argument errors as lora_proj_apply, without
 * the workspace: the kernels use a fixed LORA_STATIC_WS_BYTES array compiled
 * into the library instead, and nothing is allocated. Calls whose workspace
 * need (lora_proj_workspace_bytes(M, rt)) exceeds LORA_STATIC_WS_BYTES are
 * refused with LORA_ERR_UNSUPPORTED and a message giving both sizes. The need
 * is the split-K partial tiles of up to 256 rows (K parts x 128 features x
 * rows x 4 bytes per 128 features) or the rank-sized h of larger batches: the
 * tiny, decode (64 x 4096 x 4096, 16 slots, rank 64: 5.2 MB) and prefill
 * (8192 x 4096 x 14336: 5.3 MB) shapes fit; fused QKV at 256 rows (6144
 * outputs: 18.9 MB) and decode rows on 14336 outputs (64 rows: 14.7 MB) do
 * not -- they need a caller workspace.
 * The first call on a device looks up the array's device address with that
 * device current; make that first call before any stream capture. All calls
 * on a device share the array: calls that can overlap on the GPU race, so
 * order them (one stream). Its status word is not readable through
 * lora_status_get.
 */
lora_status lora_proj_apply_static_ws(const void *x, int64_t x_stride, const void *W, int M, int K,
                                      int N, const int32_t *seq_slot, const lora_route *rt,
                                      void *y, int64_t y_stride, lora_stream_t stream);

/*
 * Gated MLP input through a fused [gate|up] projection (frink
 * `lora_attach.rs`, `parts_mut`: a fused ffn_up holds the gate rows first,
 * then the up rows, and its adapter's B rows split the same way over one A):
 *
 *   g = (W x_i + s B (A x_i))[0 .. I),  u = (...)[I .. 2I),
 *   act[i][n] = silu(g[n]) * u[n],  silu(g) = g / (1 + e^-g).
 *
 *   W      device [2I][K] bf16: gate rows, then up rows
 *   rt     a projection route with n_out = 2I (each adapter's B is [2I][rank])
 *   act    device, M rows of I bf16, row i at act + i*act_stride
 *   ws     lora_gate_up_workspace_bytes(M, rt) bytes: the projection's
 *          workspace followed by its [M][2I] bf16 output
 * The projection is lora_proj_apply (every row rule and the status word
 * included: lora_status_get(ws) reads it); the halves are rounded to bf16,
 * then silu(g) * u is formed in fp32 and rounded once to bf16. On the
 * tensor-core path, with K and I multiples of 64 and act rows 16-byte
 * aligned, act is formed inside the projection launch -- in its drain
 * (batches of several token tiles) or its split-K sum (decode sizes) -- and
 * the [M][2I] output is not written; other shapes run the projection, then
 * a separate activation pass. Errors: those of lora_proj_apply, a route
 * whose n_out is not 2I, act_stride < I.
 */
size_t lora_gate_up_workspace_bytes(int M, const lora_route *rt);
/* The workspace of lora_gate_up_apply_ex on `path` (the projection's part
 * sized by lora_proj_workspace_bytes_ex). */
size_t lora_gate_up_workspace_bytes_ex(int M, const lora_route *rt, int path);
lora_status lora_gate_up_apply(const void *x, int64_t x_stride, const void *W, int M, int K, int I,
                               const int32_t *seq_slot, const lora_route *rt, void *act,
                               int64_t act_stride, void *ws, size_t ws_bytes, lora_stream_t stream);

/* lora_gate_up_apply with an explicit path of the projection (LORA_PATH_*).
 * LORA_PATH_TC_ONE takes batches of 17..256 rows with K and I multiples of
 * 64 through the one-launch kernel, whose split-K sum writes act directly
 * (silu(g) * u of the bf16-rounded halves, rounded once: the same rule);
 * LORA_PATH_TC (and AUTO beyond 16 rows) forms act inside the projection
 * launch where lora_gate_up_apply says; every other case runs the projection
 * on that path, then the act pass. */
lora_status lora_gate_up_apply_ex(const void *x, int64_t x_stride, const void *W, int M, int K,
                                  int I, const int32_t *seq_slot, const lora_route *rt, void *act,
                                  int64_t act_stride, void *ws, size_t ws_bytes, int path,
                                  lora_stream_t stream);

/* Largest expert count lora_moe_down_apply takes in one call. */
#define LORA_MAX_EXPERTS 16

/* Workspace of lora_moe_down_apply for T slot-rows over E experts whose
 * routes are rts[0..E-1] (same n_in, n_out, max_rank and max_loras). */
size_t lora_moe_workspace_bytes(int E, int T, const lora_route *rts);

/*
 * Mixture-of-experts down projection with a per-expert LoRA fold
 * (spark_model `lora_delta.rs`, `LoraKernels`: the down_proj fold keyed on the
 * expert through device expert_offsets). Slot-row j with
 * expert_offsets[e] <= j < expert_offsets[e+1] gets
 *   y[j, :] = W_e x_j + s * B_{e,s} (A_{e,s} x_j),  s = seq_slot[j],
 * from expert e's route rts[e].
 *   x               device, T rows of K bf16 grouped by expert, stride x_stride
 *   W_e             host array [E] of device pointers, each [N][K] bf16
 *   expert_offsets  device [E+1] int32, non-decreasing, expert_offsets[E] <= T
 *   seq_slot        device [T] int32
 *   rts             host array [E] of routes (same K, N, max_rank, max_loras)
 *   y               device, T rows of N bf16, stride y_stride; rows outside
 *                   every expert segment are left untouched
 * E must be in [1, LORA_MAX_EXPERTS]. Same conventions and errors as
 * lora_proj_apply.
 */
lora_status lora_moe_down_apply(const void *x, int64_t x_stride, const void *const *W_e,
                                const int32_t *expert_offsets, int E, int T, int K, int N,
                                const int32_t *seq_slot, const lora_route *rts, void *y,
                                int64_t y_stride, void *ws, size_t ws_bytes,
                                lora_stream_t stream);

/*
 * ------------------------------------------------------------------------
 * Token embedding: a row gather of the adapted matrix E + s B A, with E the
 * [vocab][n_embd] embedding table (ferrox-core `weight_matrix/lora.rs`,
 * `LoraDelta::add_row_to`; frink `lora_attach.rs`, `checked_pair`).
 * ------------------------------------------------------------------------
 *
 * An embedding route holds, per slot, A TRANSPOSED as [n_embd][max_rank]
 * followed by B as [vocab][max_rank] (bf16, zero past the adapter's rank;
 * a_table[s] points at the first, b_table[s] at the second). Both are
 * rank-contiguous: a token's B row is one contiguous run, and A^T is the
 * K-major operand of the tensor-core product. Pool bytes: lora_pool_bytes(
 * max_loras, max_rank, n_embd, vocab). Same errors as lora_route_init
 * (n_in there is n_embd here); rt->kind = LORA_ROUTE_EMBED, rt->n_in =
 * n_embd, rt->n_out = vocab.
 */
lora_status lora_embed_route_init(lora_route *rt, void *pool, size_t pool_bytes, void *tables,
                                  size_t table_bytes, int max_loras, int max_rank, int vocab,
                                  int n_embd, lora_stream_t stream);

/*
 * Pack one adapter of an embedding route from the flipped pair the adapter
 * files carry (frink `lora_attach.rs`, `checked_pair`, embedding branch):
 *   rows   [vocab][rank] bf16, row-major: the row a token gathers (the
 *          module layout's B)
 *   cols   [n_embd][rank] bf16, row-major: the module layout's A, transposed
 * host or device memory. Neither is transposed: both are copied into the
 * slot row by row. Scale, slot and rank rules and errors as lora_pool_pack;
 * the route must be an embedding route (LORA_ERR_UNSUPPORTED otherwise).
 * lora_pool_pack on an embedding route takes the module layout instead (A
 * [rank][n_embd], B [vocab][rank]) and transposes A.
 */
lora_status lora_embed_pool_pack(const lora_route *rt, int slot, const void *rows, const void *cols,
                                 int rank, float alpha, int use_rslora, float adapter_scale,
                                 lora_stream_t stream);

/* Workspace of lora_embed_apply for M rows on embedding route `rt` (routing
 * sort and status word; 256-byte aligned). 0 if rt is NULL, not initialised
 * or not an embedding route. */
size_t lora_embed_workspace_bytes(int M, const lora_route *rt);

/*
 * y[i, :] = E[t, :] + s * B_s[t, :] A_s,  t = tokens[i], s = seq_slot[i], for i in [0, M).
 *   tokens    device [M] int32 in [0, vocab)
 *   E         device [vocab][n_embd] bf16 row-major, 16-byte aligned
 *   seq_slot  device [M] int32, as for lora_proj_apply
 *   rt        an embedding route with rt->n_out == vocab, rt->n_in == n_embd
 *   y         device, M rows of n_embd bf16, row i at y + i*y_stride;
 *             16-byte aligned, y_stride a multiple of 8 (rows are written by
 *             16-byte bulk copies)
 *   ws        device workspace of lora_embed_workspace_bytes(M, rt) bytes
 * A row with no delta (slot negative, >= max_loras, empty, scale 0) is
 * E[t, :] byte for byte. A token outside [0, vocab) gives a zero row and
 * sets LORA_FLAG_TOKEN_RANGE. The delta is accumulated in fp32 over the
 * rank and added to E in fp32; y is rounded once, to nearest even.
 * Enqueued on `stream` only (no allocation, no synchronisation; graph-safe).
 * Errors: NULL pointers (M > 0), a projection route, vocab or n_embd not
 * matching the route, E or y not 16-byte aligned, y_stride < n_embd or not a
 * multiple of 8, ws too small.
 */
lora_status lora_embed_apply(const int32_t *tokens, const void *E, int M, int vocab, int n_embd,
                             const int32_t *seq_slot, const lora_route *rt, void *y,
                             int64_t y_stride, void *ws, size_t ws_bytes, lora_stream_t stream);

/*
 * ------------------------------------------------------------------------
 * Decode-path MoE fold keyed on the expert through a per-slot-row index
 * (spark_model `lora_delta.rs`, `LoraKernels`, moe_gather: the unsorted,
 * slot-major analogue of lora_moe_down_apply), with the top-k combine.
 * ------------------------------------------------------------------------
 *
 * Slot-row j (token j / top_k, choice j % top_k) has input x_j and expert
 * e = indices[j]:
 *   v_j = W_e x_j + s B_{e,s} (A_{e,s} x_j),  s = seq_slot[j]
 * (zero when e is outside [0, E): LORA_FLAG_EXPERT_RANGE is set).
 *   combine == NULL   y[j, :] = v_j for j in [0, T), byte for byte what
 *                     lora_moe_down_apply gives for that row
 *   combine != NULL   y[t, :] = sum_i combine[t*top_k + i] * v_{t*top_k + i}
 *                     for t in [0, T / top_k): fp32 sum of the slot-rows (each
 *                     rounded to bf16), rounded once
 *   x          device, T rows of K bf16 in token order, stride x_stride
 *   W_e, rts   as lora_moe_down_apply (host arrays of E device pointers / routes)
 *   indices    device [T] int32
 *   seq_slot   device [T] int32
 *   combine    device [T] f32 or NULL; top_k >= 1 and T a multiple of top_k
 *              when given
 *   y          device, stride y_stride >= N
 *   ws         lora_moe_gather_workspace_bytes(E, T, rts) bytes
 * The rows are sorted by expert on the device (stable), copied into expert
 * order, folded by the grouped path, and combined. T <= LORA_GATHER_MAX_ROWS.
 * Same conventions and errors as lora_moe_down_apply, plus: T above the
 * limit, a top_k that does not divide T.
 */
#define LORA_GATHER_MAX_ROWS 8192
size_t lora_moe_gather_workspace_bytes(int E, int T, const lora_route *rts);
lora_status lora_moe_gather_apply(const void *x, int64_t x_stride, const void *const *W_e,
                                  const int32_t *indices, int E, int T, int K, int N,
                                  const int32_t *seq_slot, const lora_route *rts, const float *combine,
                                  int top_k, void *y, int64_t y_stride, void *ws, size_t ws_bytes,
                                  lora_stream_t stream);

/* Read the status word (LORA_FLAG_* bits) of the most recent call that used
 * workspace `ws`. Synchronises `stream` (diagnostic, not a hot-path call).
 * The first 16 bytes of a workspace hold the bits, the tag of the call that
 * set them and an epoch that every call advances by one; the bits count when
 * the tag is the last call's (epoch - 1), so a call that sets no bit needs no
 * clearing pass and reads as 0. */
lora_status lora_status_get(const void *ws, uint32_t *flags, lora_stream_t stream);

/* Which kernels a projection call of M rows on `rt` takes on the current
 * device (lora_proj_plan; the pages have no counterpart: a diagnostic). */
enum {
    LORA_PLAN_SIMT = 1,        /* <= 16 rows: CUDA-core GEMV (routing, shrink, GEMV launches) */
    LORA_PLAN_TC = 2,          /* routing launch, then one tensor-core launch (and the act pass
                                  of gated shapes that cannot form act in it) */
    LORA_PLAN_ONE_LAUNCH = 3   /* <= 256 rows: everything in one clustered tensor-core launch */
};
typedef struct lora_plan_info {
    int32_t path;              /* LORA_PLAN_* */
    int32_t kernels;           /* kernel launches of one call */
    int32_t cluster_size;      /* one-launch kernel: CTAs per cluster (the K parts) */
    int32_t clusters_needed;   /* one-launch kernel: clusters of the grid (feature tiles) */
    int32_t clusters_resident; /* clusters of that size the device can hold at once */
    int32_t smem_per_cta;      /* bytes of shared memory of one CTA of the one-launch kernel */
} lora_plan_info;

/*
 * Fill `info` for a lora_proj_apply_ex of M rows on projection route `rt`
 * and `path` (LORA_PATH_*; gated = 1: lora_gate_up_apply_ex with I = n_out /
 * 2). The one-launch kernel (LORA_PATH_TC_ONE only) needs its whole grid
 * resident at once (its CTAs exchange h through the workspace); a shape whose
 * clusters do not all fit, or that needs more CTAs than the device has SMs,
 * takes LORA_PLAN_TC. Calls whose shapes take different plans (a fused q/k/v
 * call on one, its split calls on the other) are not byte-identical to each
 * other. Errors: NULL info, a route that is not a projection route, M < 0, a
 * path out of range.
 */
lora_status lora_proj_plan(int M, const lora_route *rt, int gated, int path, lora_plan_info *info);

/*
 * Test hook for the bounded device waits of the one-launch kernel of up to
 * 256 rows (the pages have no counterpart). With wait_ns > 0, later calls
 * give up their exchange wait after wait_ns nanoseconds instead of about a
 * second, and wait for extra_flags flags that no CTA ever writes, so the
 * wait runs out: the call then returns with LORA_FLAG_WAIT_TIMEOUT in its
 * status word and y holding the base product without the delta. The same
 * setting covers the tensor-core kernel's split-K wait (LORA_PATH_TC with K
 * parts) and, from 2048 rows, its wait for the launch's shrink tiles: those
 * waits run out, the call returns with LORA_FLAG_WAIT_TIMEOUT and y is not
 * (fully) written. Nothing faults or hangs.
 * wait_ns = 0 restores normal operation. Process-wide; for tests only.
 */
void lora_test_wait_hook(uint64_t wait_ns, int extra_flags);

/*
 * Copy the routing sort of the most recent lora_proj_apply on `ws` to host
 * memory: perm [M] (row ids grouped by slot, stable: bucket 0 = rows with no
 * valid slot, then slot 0, 1, ...) and seg_off [max_loras + 2] (bucket starts,
 * last entry M). Synchronises `stream`. For tests and diagnostics.
 */
lora_status lora_proj_routing(const void *ws, int M, int max_loras, int32_t *perm,
                              int32_t *seg_off, lora_stream_t stream);

/* Message of the last error on this thread ("" after a successful call). */
const char *lora_last_error(void);

/*
 * Host helper (metrale `lora/slot_math.rs`, `build_seq_slot_host`): out[i] =
 * adapter_slots[i] for i < n when it is >= 0, `active` when it is negative;
 * out[i] = -1 for the padding rows n <= i < padded_n. Requires n <= padded_n.
 */
lora_status lora_build_seq_slot(const int32_t *adapter_slots, int n, int padded_n, int active,
                                int32_t *out);

#ifdef __cplusplus
}
#endif

#endif /* RANK_DELTA_H */
