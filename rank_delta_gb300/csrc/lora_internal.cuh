// Internal definitions shared by the host ABI (lora_api.cu) and the kernels.
#pragma once
#include <atomic>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/rank_delta.h"

namespace rd {

constexpr int MAX_E = LORA_MAX_EXPERTS;
constexpr int MAX_BUCKETS = 1024;   // experts * (max_loras + 1)
constexpr int SHRINK_RG = 8;        // ranks per shrink work unit (one warp each)
constexpr int SHRINK_TC = 4;        // rows per shrink work unit (one pass)
constexpr int PREP_THREADS = 1024;

// Device routing tables of one expert's route.
struct Tables {
    const uint16_t *const *a_table;
    const uint16_t *const *b_table;
    const float *scale_table;
    const int32_t *rank_table;
    const float *comp_table; // [L][LORA_COMP_STRIDE] per-rank factors
};

// What the expand needs for a row routed to slot s of table t. A row gets no
// delta when its slot is negative or >= L, the slot is empty, or its scale
// is 0 (the delta is then skipped, not multiplied by zero).
struct SlotInfo {
    const uint16_t *a; // A of the slot, [R][K]
    const uint16_t *b; // B of the slot, [N][R]
    float scale;
    int rank;
    int on;
};

__device__ __forceinline__ SlotInfo slot_info(const Tables &t, int s, int L)
{
    SlotInfo si{nullptr, nullptr, 0.0f, 0, 0};
    if (s < 0 || s >= L)
        return si;
    si.a = t.a_table[s];
    si.b = t.b_table[s];
    si.scale = t.scale_table[s];
    si.rank = t.rank_table[s];
    si.on = (si.a != nullptr && si.b != nullptr && si.scale != 0.0f && si.rank > 0) ? 1 : 0;
    return si;
}

// Workspace sections (device pointers carved from the caller's buffer).
struct Ws {
    uint32_t *status;   // [1] LORA_FLAG_* bits of the last call
    int32_t *perm;      // [rows] row ids grouped by (expert, slot bucket)
    int32_t *seg_off;   // [nb + 1] bucket starts in perm
    int32_t *unit_off;  // [nb + 1] first shrink unit of each bucket
    int32_t *done;      // [nb] finished shrink units per bucket
    float *h;           // [kp][rows][R] partial A_s x_i of every adapted row (fp32)
    uint16_t *hs;       // [rows][R] bf16 of (s * comp[r]) * h, written by the tensor-core shrink tiles
    int32_t *tiles;     // [1 + 3*max_tiles]: count, then (expert, first row, rows) per token tile
    float *part;        // [tiles][csplit][tn][128] split-K partial tiles (fp32)
    int32_t *tile_cnt;  // [tiles] split-K parts written so far (zeroed by prep)
    int32_t *stile;     // [ceil(rows / 128)] shrink tiles of the projection launch published (zeroed by prep)
};

// Everything a launch needs except tensor maps.
// A plain projection is the one-expert case with segment [0, rows).
struct Params {
    const uint16_t *x;
    int64_t x_stride;
    uint16_t *y;
    int64_t y_stride;
    const int32_t *seq_slot;
    const int32_t *expert_offsets; // device [E+1], or nullptr for one segment [0, rows)
    int E;
    int rows; // M (projection) or T (slot-rows)
    int K, N, L, R;
    int tn;   // token tile of the tensor-core path (rows per tile)
    int kp;   // K parts of a shrink unit (h is summed over them)
    int ncnt; // split-K tile counters the prep kernel clears
    int no_units; // 1: h comes from the tensor-core shrink tiles (no shrink work units)
    int max_tiles; // token tiles the routing kernel may list (0: the workspace bound)
    int ystore_ok; // 1: maps.y is encoded (y 16-byte aligned, y_stride a multiple of 8)
    const void *pool;  // the route's pool (A of slot s at pool + s * slot_bytes when packed there)
    size_t slot_bytes;
    int gated, I;  // 1: W is the fused [gate I | up I] (N = 2I) read as tiles of 64 gate + 64 up rows,
                   // and y receives act = silu(g) * u, [rows][I] (one K part, TMA stores only)
    const uint16_t *W[MAX_E];
    Tables tab[MAX_E];
    Ws ws;
    int stc_tiles; // shrink tiles (128 rows) the projection launch runs itself (no_units), else 0
    int stc_rs;    // their max rank rounded up to 16
    int stc_amap;  // 1: the shrink's A map covers the route's pool (A rows by TMA)
};

struct WsLayout {
    size_t status, perm, seg_off, unit_off, done, h, hs, tiles, part, tile_cnt, stile, total;
};

// Status words at the start of a workspace: [0] LORA_FLAG_* bits, [1] the
// tag of the call that set them, [2] the epoch, which every call advances by
// one. The tag of the call with epoch e is status_tag(e), so the bits belong
// to the last call when [1] == status_tag([2] - 1); whatever else a fresh
// workspace holds there (zeros, leftover integers) does not pass for a tag.
__host__ __device__ inline uint32_t status_tag(uint32_t e) { return e ^ 0x6A09E667u; }

// One thread of a call's first kernel opens the call's status this way.
__device__ __forceinline__ void status_begin(uint32_t *st, uint32_t flags)
{
    volatile uint32_t *v = st;
    const uint32_t e = v[2];
    v[0] = flags;
    v[1] = status_tag(e);
    v[2] = e + 1;
}

// Upper bound on token tiles: each expert adds at most one partial tile.
__host__ __device__ inline int max_token_tiles(int rows, int E) { return rows / 16 + E + 1; }

inline size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

// K parts of a shrink unit: about 2048 of K each, at most 4 (enough units to
// spread over the SMs for a decode batch, few enough to keep each one busy).
inline int shrink_kparts(int K)
{
    int kp = K / 2048;
    return kp < 1 ? 1 : (kp > 4 ? 4 : kp);
}

inline WsLayout ws_layout(int rows, int nb, int R, int kp, size_t part_elems = 0, int ncnt = 0)
{
    WsLayout l;
    size_t o = 0;
    l.status = o;   o = align256(o + 256);
    l.perm = o;     o = align256(o + sizeof(int32_t) * (size_t)rows);
    l.seg_off = o;  o = align256(o + sizeof(int32_t) * (size_t)(nb + 1));
    l.unit_off = o; o = align256(o + sizeof(int32_t) * (size_t)(nb + 1));
    l.done = o;     o = align256(o + sizeof(int32_t) * (size_t)nb);
    l.h = o;        o = align256(o + sizeof(float) * (size_t)kp * (size_t)rows * (size_t)R);
    l.hs = o;       o = align256(o + sizeof(uint16_t) * (size_t)rows * (size_t)R);
    l.tiles = o;    o = align256(o + sizeof(int32_t) * (1 + 3 * (size_t)max_token_tiles(rows, nb)));
    l.part = o;     o = align256(o + sizeof(float) * part_elems);
    l.tile_cnt = o; o = align256(o + sizeof(int32_t) * (size_t)ncnt);
    l.stile = o;    o = align256(o + sizeof(int32_t) * (size_t)((rows + 127) / 128));
    l.total = o;
    return l;
}

// Tensor maps of one launch of the tensor-core kernel.
struct TmapSet {
    CUtensorMap x;
    CUtensorMap w[MAX_E];
    CUtensorMap y;  // boxes of 128 features x YSTORE_ROWS rows of y, no swizzle (when ystore_ok)
};

// Tensor maps of the shrink tiles of a launch (stc_tiles > 0), passed only to
// the kernel instantiation that runs them.
struct StcMaps {
    CUtensorMap sx; // x: boxes of 64 x 128 rows
    CUtensorMap sa; // the pool's A rows: boxes of 64 x Rs rows x one slot (when stc_amap)
};
// Rows of one TMA store of the tensor-core epilogue.
constexpr int YSTORE_ROWS = 64;

// Raise a kernel's dynamic shared-memory limit on the current device. The
// attribute belongs to the device's context, so a process driving several
// GPUs raises it on each: `done` keeps one bit per device already raised.
template <typename F>
inline cudaError_t raise_smem_limit(std::atomic<uint64_t> &done, F *fn, int bytes)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= 64)
        return cudaErrorInvalidDevice;
    const uint64_t bit = 1ull << dev;
    if (done.load(std::memory_order_acquire) & bit)
        return cudaSuccess;
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess)
        done.fetch_or(bit, std::memory_order_release);
    return e;
}

// Launchers (each defined next to its kernel). They return the launch error.
cudaError_t launch_prep(const Params &p, cudaStream_t st);
cudaError_t launch_shrink(const Params &p, int num_sms, cudaStream_t st);
cudaError_t launch_simt(const Params &p, int num_sms, cudaStream_t st);
// Rows from which a projection call computes h with tensor-core shrink tiles
// of 128 rows inside the projection launch (enough tiles to spread over the
// SMs; below, CUDA-core shrink units).
constexpr int TC_SHRINK_MIN_ROWS = 2048;
// Shape of one tensor-core launch: token tile, 64-wide K chunks per pipeline
// stage, stages, K parts, whether the 3D tensor-map view (K a multiple of 64)
// is used, and the expand's staging buffers.
struct TcPlan {
    int tn, kc, stages, csplit, use3d;
    int pair; // 1: two adjacent feature tiles per x box (per-expert tiles)
    int xblk; // 64-wide k blocks of one tensor-core expand round
    int hl;   // planes of the staged s * h: 1 (bf16) or 2 (bf16 hi + lo)
};
TcPlan plan_tc(const Params &p, bool per_expert_tiles);
cudaError_t launch_tc(const Params &p, const TmapSet &maps, const StcMaps &sm, const TcPlan &plan, int num_sms,
                      cudaStream_t st);
cudaError_t launch_table_set(const lora_route &rt, int slot, const void *a, const void *b,
                             int rank, float factor, float scale, cudaStream_t st);
cudaError_t launch_scale_set(const lora_route &rt, int slot, float adapter_scale, cudaStream_t st);
// The per-rank factors of one slot, passed by value.
struct CompRow {
    float v[LORA_COMP_STRIDE];
};
cudaError_t launch_comp_set(const lora_route &rt, int slot, const CompRow &row, cudaStream_t st);
// A^T [n][R] of a device A [rank][n], into a zeroed slot.
cudaError_t launch_transpose_pack(uint16_t *At, int R, const uint16_t *A, int rank, int n, cudaStream_t st);
// Runtime scales of up to SCALE_CHUNK consecutive slots, passed by value.
constexpr int SCALE_CHUNK = 256;
struct ScaleChunk {
    int first, count;
    float s[SCALE_CHUNK];
};
cudaError_t launch_scales_set(const lora_route &rt, const ScaleChunk &c, cudaStream_t st);

// Embedding row gather with the adapted rows (lora_embed.cu):
//   y[i, :] = E[t_i, :] + s * B[t_i, :] A,  t_i = tokens[i], s = the scale of seq_slot[i].
// The pool of an embedding route stores A transposed, [n_embd][max_rank]
// (rank contiguous: the K-major operand of the tensor-core product), then B
// as [vocab][max_rank].
struct EmbedParams {
    const uint16_t *E;      // [vocab][n_embd]
    const int32_t *tokens;  // [M]
    const int32_t *seq_slot; // [M]
    uint16_t *y;
    int64_t y_stride;
    int M, vocab, n_embd, L, R;
    int ft;  // embedding features per work item (the UMMA N), a multiple of 32
    int nft; // feature tiles: n_embd / ft rounded up
    int local; // 1: every CTA sorts the rows itself (no routing kernel); M <= EMBED_LOCAL_ROWS
    Tables tab;
    Ws ws;
};
// Rows per chunk of the embedding gather: the UMMA M.
constexpr int EMBED_CHUNK_ROWS = 128;
// Features per work item for pool rank R: the widest of 128 / 64 / 32 whose
// double-buffered operands and E rows fit in shared memory.
int embed_tile_features(int R);
// Rows and buckets (max_loras + 1) up to which each CTA of the gather sorts
// the batch by slot itself.
constexpr int EMBED_LOCAL_ROWS = 4096;
constexpr int EMBED_LOCAL_BUCKETS = 64;
// Whether the sorted rows of an M-row batch fit in shared memory beside the buffers.
bool embed_local_fits(int M, int ft, int R, int L);
cudaError_t launch_embed(const EmbedParams &p, int num_sms, cudaStream_t st);

// Decode-path MoE fold with per-slot-row expert indices (lora_gather.cu).
struct GatherParams {
    const uint16_t *x;
    int64_t x_stride;
    const int32_t *indices;  // [T] expert of each slot-row
    const int32_t *seq_slot; // [T]
    int E, T, K, N;
    uint16_t *x_sorted;      // [T][K] rows in expert order (workspace)
    int32_t *perm;           // [T] sorted position -> slot-row
    int32_t *inv;            // [T] slot-row -> sorted position
    int32_t *slots_sorted;   // [T]
    int32_t *offsets;        // [E+2] expert starts in the sorted order; [E] = rows with an expert
    const uint16_t *y_sorted; // [T][N] the grouped fold's output (workspace)
    const float *combine;    // [T] weights, or nullptr
    int top_k;
    uint16_t *y;
    int64_t y_stride;
    uint32_t *status;
};
size_t gather_sort_smem(int T, int E);
cudaError_t launch_gather_sort(const GatherParams &p, int num_sms, cudaStream_t st);
cudaError_t launch_gather_combine(const GatherParams &p, int num_sms, cudaStream_t st);

// act[i][n] = silu(y[i][n]) * y[i][I + n] (lora_act.cu).
cudaError_t launch_silu_mul(const uint16_t *y, int64_t y_stride, int M, int I, uint16_t *act,
                            int64_t act_stride, int num_sms, cudaStream_t st);

// One-launch projection of up to 256 rows (lora_dec.cu): the routing, the
// tensor-core shrink inside the base K loop, the h exchange through the
// workspace, the expand and the split-K sum over a thread-block cluster.
struct DecLaunch {
    TmapSet maps;            // x: boxes [kc][tn][64] (3D) or [tn][64]; W: [kc][128][64], or the gated 4D view
    const uint16_t *x;
    int64_t x_stride;
    uint16_t *y;             // y [M][N], or act [M][I] when gated
    int64_t y_stride;
    const int32_t *seq_slot;
    int M, K, N, L, R;
    int gated, I;            // gated: W is [gate I | up I] and y receives act = silu(g) * u
    int yvec;                // y / act 8-byte aligned with y_stride a multiple of 4
    Tables tab;
    uint32_t *status;        // [0] flags, [1] tag, [2] epoch, u64 [8] h arrival counter (workspace)
    int32_t *perm, *seg_off; // routing export
    float *hpart;            // dec_hpart_floats(...) floats
    float *gpart;            // dec_flag_count(...) * M * 128 floats, or null (the workspace sum then cannot run)
    unsigned long long *pflags; // dec_flag_count(...) words
    CUtensorMap amap;        // the pool's A rows: [L slots][R rank rows][K], boxes of 8 rows x 64 k
    CUtensorMap amap5[5];    // the same, boxes of 2^lg 8-row groups over a whole K part (bit lg of gb_mask: encoded)
    int gb_mask;
    const void *pool;        // the route's pool and its bytes per slot (where the A rows of slot s lie)
    size_t slot_bytes;
};
// K chunks per pipeline stage the kernel would take (0: the shape does not fit it).
int dec_plan_kc(int M, int K, int N, int L, int R, int gated, int I);
size_t dec_hpart_floats(int M, int K, int N, int L, int R, int gated);
// 1 when a call of this shape takes the one-launch kernel on the current
// device: the clusters it needs, how many can be resident at once, their
// size (the K parts) and the shared memory of one CTA.
int dec_plan_info(int M, int K, int N, int L, int R, int gated, int I, int num_sms, int *clusters_needed,
                  int *clusters_resident, int *cluster_size, uint32_t *smem);
int dec_flag_count(int M, int K, int N, int gated);
// cudaErrorNotSupported: the shape or the device does not take this kernel.
cudaError_t launch_dec(const DecLaunch &d, int num_sms, cudaStream_t st);
// The test hook's setting (lora_test_wait_hook): a wait limit in ns (0 = the
// normal one) and arrivals that never come added to the waits it covers.
void test_hook_get(uint64_t &wait_ns, int &extra);
// 1 when the tensor-core kernel can take this gated call (W the fused
// [gate | up], act written from its drain): see launch_tc.
bool tc_gated_ok(const Params &p);
// Test hook: the exchange wait gives up after wait_ns and waits for
// extra_flags flags that no CTA writes (0, 0: normal operation).
void dec_test_hook(uint64_t wait_ns, int extra_flags);

// Record `msg` as the thread's last error and return `code` (lora_api.cu).
lora_status api_fail(lora_status code, const char *msg);

// Token tile of the tensor-core path: the rows of one segment rounded up to
// 16 (the UMMA N granularity), at most 256 (the largest UMMA N and TMA box).
inline int tc_token_tile(int rows_per_segment)
{
    int t = (rows_per_segment + 15) / 16 * 16;
    if (t < 16) t = 16;
    return t > 256 ? 256 : t;
}

// CTAs splitting K for one tile, from the row count and K only -- never from
// N -- so a fused q/k/v call and its split calls compute every element
// identically. Several token tiles (rows > 256) or expert tiles: no split.
// Per-expert tiles (MoE): one K part (a split leaves the in-launch shrink
// longer than the first item's W stream).
inline int tc_csplit(int rows, int K, bool per_expert_tiles)
{
    if (per_expert_tiles)
        return 1;
    if (rows > 256)
        return 1;
    const int cap = rows <= 64 ? 4 : 3;
    const int c = ((K + 63) / 64) / 16;
    return c < 1 ? 1 : (c > cap ? cap : c);
}

// Token tile of a MoE call: the mean expert segment with 1/8 headroom, so a
// typical expert is one tile.
inline int moe_token_tile(int T, int E)
{
    const int mean = (T + E - 1) / E;
    return tc_token_tile(mean + mean / 8);
}

// Token tiles of a MoE call at most: each expert segment adds at most one
// partial tile (the routing kernel never lists more).
inline int moe_max_tiles(int T, int E) { return (T + moe_token_tile(T, E) - 1) / moe_token_tile(T, E) + E; }

// Split-K scratch of a MoE call: partial tiles and tile counters.
inline void moe_split_scratch(int T, int E, int K, int N, size_t &part_elems, int &ncnt)
{
    const int cs = tc_csplit(T, K, true);
    const int tiles = ((N + 127) / 128) * moe_max_tiles(T, E);
    part_elems = cs > 1 ? (size_t)tiles * cs * 128 * moe_token_tile(T, E) : 0;
    ncnt = cs > 1 ? tiles : 0;
}

// Split-K scratch of a projection call: partial tiles and tile counters.
inline void split_scratch(int M, int K, int N, size_t &part_elems, int &ncnt)
{
    const int tn = tc_token_tile(M);
    const int cs = tc_csplit(M, K, false);
    const int tiles = ((N + 127) / 128) * ((M + tn - 1) / tn);
    part_elems = cs > 1 ? (size_t)tiles * cs * 128 * tn : 0;
    ncnt = cs > 1 ? tiles : 0;
}

} // namespace rd
