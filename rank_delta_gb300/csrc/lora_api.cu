// Host side of the C ABI declared in include/rank_delta.h: argument checks,
// pool packing, workspace carving, tensor-map encoding and kernel launches.
// No allocation and no host synchronisation on the apply path.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include <cudaTypedefs.h>

#include "lora_internal.cuh"

using namespace rd;

namespace {

constexpr uint64_t ROUTE_MAGIC = 0x6c6f72615f727431ull; // "lora_rt1"
constexpr int MAX_LORAS = MAX_BUCKETS - 1;
constexpr int MAX_RANK = 256;
constexpr int SIMT_MAX_ROWS = 16; // LORA_PATH_AUTO: at most this many rows per segment -> GEMV

thread_local std::string g_err;

lora_status fail(lora_status code, const char *fmt, ...)
{
    char buf[1024];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_err = buf;
    return code;
}

lora_status ok()
{
    g_err.clear();
    return LORA_OK;
}

lora_status cuda_fail(cudaError_t e, const char *what)
{
    return fail(LORA_ERR_CUDA, "%s: CUDA error %d (%s)", what, (int)e, cudaGetErrorString(e));
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t slot_bytes(int R, int K, int N) { return ((size_t)R * K + (size_t)N * R) * 2; }

struct TableLayout {
    size_t a, b, scale, factor, rank, comp, total;
};

TableLayout table_layout(int L)
{
    TableLayout t;
    size_t o = 0;
    t.a = o;      o = align256(o + sizeof(void *) * (size_t)L);
    t.b = o;      o = align256(o + sizeof(void *) * (size_t)L);
    t.scale = o;  o = align256(o + sizeof(float) * (size_t)L);
    t.factor = o; o = align256(o + sizeof(float) * (size_t)L);
    t.rank = o;   o = align256(o + sizeof(int32_t) * (size_t)L);
    t.comp = o;   o = align256(o + sizeof(float) * LORA_COMP_STRIDE * (size_t)L);
    t.total = o;
    return t;
}

lora_status check_route(const lora_route *rt, const char *who)
{
    if (rt == nullptr)
        return fail(LORA_ERR_NULL, "%s: route is NULL", who);
    if (rt->magic != ROUTE_MAGIC)
        return fail(LORA_ERR_NOT_INIT, "%s: route was not set up by lora_route_init", who);
    return LORA_OK;
}

// A set-up route of the given kind.
lora_status check_route_kind(const lora_route *rt, int kind, const char *who)
{
    lora_status s = check_route(rt, who);
    if (s != LORA_OK)
        return s;
    if (rt->kind != kind)
        return fail(LORA_ERR_UNSUPPORTED,
                    kind == LORA_ROUTE_EMBED
                        ? "%s: the route holds projection adapters; this call takes a token-embedding "
                          "route (lora_embed_route_init)"
                        : "%s: the route holds token-embedding adapters (A stored transposed); this "
                          "call takes a projection route (lora_route_init)",
                    who);
    return LORA_OK;
}

// The alpha factor of one adapter, in f32: alpha/rank, alpha/sqrt(rank)
// under rsLoRA, 1 when alpha is 0 (ferrox-core `weight_matrix/lora.rs`,
// `LoraDelta::new`; spark_model `lora_delta.rs`, `LoraPair`).
float alpha_factor(float alpha, int rank, int use_rslora)
{
    if (alpha == 0.0f)
        return 1.0f;
    return use_rslora ? alpha / sqrtf((float)rank) : alpha / (float)rank;
}

struct DevInfo {
    int num_sms = 0;
};

bool device_info(DevInfo &out)
{
    static std::mutex mu;
    static DevInfo cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return false;
    std::lock_guard<std::mutex> g(mu);
    if (cache[dev].num_sms == 0) {
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return false;
        cache[dev].num_sms = sms;
    }
    out = cache[dev];
    return true;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

// 2D bf16 map over [rows][inner] (row stride in elements), box inner x box_rows,
// 128-byte swizzle, zero fill out of bounds.
bool make_map(CUtensorMap *m, const void *base, uint64_t inner, uint64_t rows, uint64_t stride_elems,
              uint32_t box_inner, uint32_t box_rows)
{
    auto fn = encode_fn();
    if (!fn)
        return false;
    cuuint64_t dims[2] = {inner, rows};
    cuuint64_t strides[1] = {stride_elems * 2};
    cuuint32_t box[2] = {box_inner, box_rows};
    cuuint32_t es[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides,
                    box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Row-major bf16 [rows][inner] (row stride stride_elems) without swizzle,
// for TMA stores of row-major boxes.
bool make_map_plain(CUtensorMap *m, const void *base, uint64_t inner, uint64_t rows, uint64_t stride_elems,
                    uint32_t box_inner, uint32_t box_rows)
{
    auto fn = encode_fn();
    if (!fn)
        return false;
    cuuint64_t dims[2] = {inner, rows};
    cuuint64_t strides[1] = {stride_elems * 2};
    cuuint32_t box[2] = {box_inner, box_rows};
    cuuint32_t es[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides,
                    box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 3D view [K/64 chunks][rows][64] of a K-major bf16 matrix (K a multiple of
// 64): one box of box_chunks x box_rows x 64 brings several 64-wide K slices
// of the same rows in one copy, each slice laid out as a 2D 128-byte-swizzled
// tile.
bool make_map_3d(CUtensorMap *m, const void *base, uint64_t K, uint64_t rows, uint64_t stride_elems,
                 uint32_t box_rows, uint32_t box_chunks)
{
    auto fn = encode_fn();
    if (!fn)
        return false;
    cuuint64_t dims[3] = {64, rows, K / 64};
    cuuint64_t strides[2] = {stride_elems * 2, 128};
    cuuint32_t box[3] = {64, box_rows, box_chunks};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides,
                    box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// The fused [gate | up] weight W [2I][K] (K a multiple of 64) as a 4D view
// [K/64 chunks][2 halves][I rows][64]: one box of kc x 2 x 64 x 64 brings, per
// 64-wide K slice, gate rows f..f+63 then up rows I+f..I+f+63 -- 128 rows in
// the layout of a plain 128-row box.
bool make_map_gated(CUtensorMap *m, const void *W, uint64_t K, uint64_t I, uint32_t box_chunks)
{
    auto fn = encode_fn();
    if (!fn)
        return false;
    cuuint64_t dims[4] = {64, I, 2, K / 64};
    cuuint64_t strides[3] = {K * 2, I * K * 2, 128};
    cuuint32_t box[4] = {64, 64, 2, box_chunks};
    cuuint32_t es[4] = {1, 1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(W), dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// The A rows of every slot of a projection pool as a 3D bf16 view
// [L slots][R rank rows][K] (slot stride = the pool's bytes per slot), boxes
// of 8 rank rows x 64 k with the 128-byte swizzle: the shrink operand layout.
bool make_map_pool_a(CUtensorMap *m, const void *pool, uint64_t K, uint64_t R, uint64_t L, uint64_t slot_bytes)
{
    auto fn = encode_fn();
    if (!fn)
        return false;
    cuuint64_t dims[3] = {K, R, L};
    cuuint64_t strides[2] = {K * 2, slot_bytes};
    cuuint32_t box[3] = {64, 8, 1};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(pool), dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// The same pool in boxes of `rows` rank rows (from row 0) x 64 k of one slot.
bool make_map_pool_rows(CUtensorMap *m, const void *pool, uint64_t K, uint64_t R, uint64_t L, uint64_t slot_bytes,
                        uint32_t rows)
{
    auto fn = encode_fn();
    if (!fn)
        return false;
    cuuint64_t dims[3] = {K, R, L};
    cuuint64_t strides[2] = {K * 2, slot_bytes};
    cuuint32_t box[3] = {64, rows, 1};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(pool), dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// The same pool (R a multiple of 8, K of 64) as a 5D view [L slots][K/64
// chunks][R/8 groups][8 rows][64 k]: one box of 2^lg groups x nch chunks of
// one slot lands chunk by chunk, each chunk's groups 1 KB apart, as the
// shrink reads its A rows.
bool make_map_pool_a5(CUtensorMap *m, const void *pool, uint64_t K, uint64_t R, uint64_t L, uint64_t slot_bytes,
                      uint32_t groups, uint32_t nch)
{
    auto fn = encode_fn();
    if (!fn)
        return false;
    cuuint64_t dims[5] = {64, 8, R / 8, K / 64, L};
    cuuint64_t strides[4] = {K * 2, K * 16, 128, slot_bytes};
    cuuint32_t box[5] = {64, 8, groups, nch, 1};
    cuuint32_t es[5] = {1, 1, 1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void *>(pool), dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Workspace of the one-launch kernel of up to 256 rows: the status words (and
// the h arrival counter, in the same 256-byte block) and the routing export
// where the general layout has them, then the partial h of every CTA and,
// for the workspace sum, the K parts' tile flags and tiles.
struct DecWs {
    size_t perm, seg_off, hpart, pflags, gpart, core, total;
};

// `core` bytes serve the cluster-sum mode; `total` adds the K parts' fp32
// tiles of the workspace-sum mode.
DecWs dec_ws_layout(int M, int K, int N, int L, int R, int gated)
{
    DecWs l;
    const size_t nf = (size_t)dec_flag_count(M, K, N, gated);
    size_t o = 256;
    l.perm = o;    o = align256(o + sizeof(int32_t) * (size_t)M);
    l.seg_off = o; o = align256(o + sizeof(int32_t) * (size_t)(L + 2));
    l.hpart = o;   o = align256(o + sizeof(float) * dec_hpart_floats(M, K, N, L, R, gated));
    l.pflags = o;  o = align256(o + sizeof(unsigned long long) * nf);
    l.core = o;
    l.gpart = o;   o = align256(o + sizeof(float) * nf * (size_t)M * 128);
    l.total = o;
    return l;
}

constexpr int DEC_MAX_ROWS = 256;

} // namespace

namespace rd {
lora_status api_fail(lora_status code, const char *msg) { return fail(code, "%s", msg); }
} // namespace rd

extern "C" {

const char *lora_last_error(void) { return g_err.c_str(); }

size_t lora_pool_bytes(int max_loras, int max_rank, int n_in, int n_out)
{
    if (max_loras <= 0 || max_rank <= 0 || n_in <= 0 || n_out <= 0)
        return 0;
    return (size_t)max_loras * slot_bytes(max_rank, n_in, n_out);
}

size_t lora_route_table_bytes(int max_loras)
{
    if (max_loras <= 0)
        return 0;
    return table_layout(max_loras).total;
}

} // extern "C"

namespace {

lora_status route_setup(lora_route *rt, void *pool, size_t pool_bytes, void *tables, size_t table_bytes,
                        int max_loras, int max_rank, int n_in, int n_out, int kind, const char *who, lora_stream_t stream)
{
    if (rt == nullptr || pool == nullptr || tables == nullptr)
        return fail(LORA_ERR_NULL, "%s: route, pool and tables must be non-NULL", who);
    if (max_loras <= 0 || max_rank <= 0 || n_in <= 0 || n_out <= 0)
        return fail(LORA_ERR_SHAPE,
                    "%s: sizes must be positive (max_loras %d, max_rank %d, n_in %d, "
                    "n_out %d)",
                    who, max_loras, max_rank, n_in, n_out);
    if (max_loras > MAX_LORAS)
        return fail(LORA_ERR_UNSUPPORTED, "%s: max_loras %d exceeds %d", who, max_loras,
                    MAX_LORAS);
    if (max_rank > MAX_RANK || max_rank % 8 != 0)
        return fail(LORA_ERR_UNSUPPORTED,
                    "%s: max_rank %d must be a multiple of 8 and at most %d", who, max_rank,
                    MAX_RANK);
    if (n_in % 8 != 0)
        return fail(LORA_ERR_ALIGN, "%s: n_in %d must be a multiple of 8", who, n_in);
    if (!aligned16(pool))
        return fail(LORA_ERR_ALIGN, "%s: pool must be 16-byte aligned", who);
    if ((reinterpret_cast<uintptr_t>(tables) & 255u) != 0)
        return fail(LORA_ERR_ALIGN, "%s: tables must be 256-byte aligned", who);
    const size_t need_pool = lora_pool_bytes(max_loras, max_rank, n_in, n_out);
    const size_t need_tab = lora_route_table_bytes(max_loras);
    if (pool_bytes < need_pool || table_bytes < need_tab)
        return fail(LORA_ERR_WORKSPACE,
                    "%s: pool has %zu bytes (needs %zu for %d slots of [%d x %d] at "
                    "max_rank %d), tables have %zu bytes (needs %zu)",
                    who, pool_bytes, need_pool, max_loras, n_out, n_in, max_rank, table_bytes, need_tab);
    const TableLayout tl = table_layout(max_loras);
    uint8_t *tb = static_cast<uint8_t *>(tables);
    cudaError_t e = cudaMemsetAsync(tables, 0, tl.total, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e, who);
    rt->pool = pool;
    rt->a_table = reinterpret_cast<const void **>(tb + tl.a);
    rt->b_table = reinterpret_cast<const void **>(tb + tl.b);
    rt->scale_table = reinterpret_cast<float *>(tb + tl.scale);
    rt->factor_table = reinterpret_cast<float *>(tb + tl.factor);
    rt->rank_table = reinterpret_cast<int32_t *>(tb + tl.rank);
    rt->comp_table = reinterpret_cast<float *>(tb + tl.comp);
    rt->n_in = n_in;
    rt->n_out = n_out;
    rt->max_rank = max_rank;
    rt->max_loras = max_loras;
    rt->kind = kind;
    rt->reserved = 0;
    rt->magic = ROUTE_MAGIC;
    return ok();
}

// A^T [n][R] (rows R apart) of A [rank][n] held in host memory: transposed on
// the host, then one 2D copy. Pageable sources are staged before the copy
// call returns, so the temporary may go when it does.
cudaError_t copy_transposed_from_host(uint16_t *At, int R, const uint16_t *A, int rank, int n,
                                      cudaStream_t st)
{
    std::vector<uint16_t> t((size_t)n * rank);
    for (int k = 0; k < rank; ++k)
        for (int e = 0; e < n; ++e)
            t[(size_t)e * rank + k] = A[(size_t)k * n + e];
    cudaError_t e = cudaMemcpy2DAsync(At, (size_t)R * 2, t.data(), (size_t)rank * 2, (size_t)rank * 2,
                                      (size_t)n, cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess)
        e = cudaStreamSynchronize(st); // the temporary is read before it is freed, pinned or not
    return e;
}

bool device_readable(const void *p)
{
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        (void)cudaGetLastError();
        return false;
    }
    return a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged;
}

// Copy one adapter into `slot` and publish it (spark_model `lora_delta.rs`,
// `LoraPair`: zero padding to the pool rank, scale not folded into B).
// Projection route: A [rank][n_in] and B [n_out][rank], both as given.
// Embedding route: B [vocab][rank] as given; A^T [n_embd][rank] as given when
// `a_is_transposed` (the flipped pair), else A [rank][n_embd] is transposed.
lora_status pack_slot(const lora_route *rt, int slot, const void *A, const void *B, int rank, float alpha,
                      int use_rslora, float adapter_scale, lora_stream_t stream, bool a_is_transposed)
{
    const char *who = a_is_transposed ? "lora_embed_pool_pack" : "lora_pool_pack";
    lora_status s = a_is_transposed ? check_route_kind(rt, LORA_ROUTE_EMBED, who) : check_route(rt, who);
    if (s != LORA_OK)
        return s;
    if (slot < 0 || slot >= rt->max_loras)
        return fail(LORA_ERR_RANGE, "%s: slot %d is out of range: pool has %d slot(s)", who, slot,
                    rt->max_loras);
    if (rank <= 0 || rank > rt->max_rank)
        return fail(LORA_ERR_SHAPE,
                    "%s: rank %d does not fit route [n_out %d x n_in %d] with "
                    "max_rank %d (need 1 <= rank <= max_rank; A holds rank*n_in = %lld values, "
                    "B n_out*rank = %lld)",
                    who, rank, rt->n_out, rt->n_in, rt->max_rank, (long long)rank * rt->n_in,
                    (long long)rt->n_out * rank);
    if (A == nullptr || B == nullptr)
        return fail(LORA_ERR_NULL, a_is_transposed ? "%s: rows and cols must be non-NULL"
                                                   : "%s: A and B must be non-NULL", who);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const int R = rt->max_rank, K = rt->n_in, N = rt->n_out;
    const bool embed = rt->kind == LORA_ROUTE_EMBED;
    uint8_t *base = static_cast<uint8_t *>(rt->pool) + (size_t)slot * slot_bytes(R, K, N);
    uint16_t *dA = reinterpret_cast<uint16_t *>(base); // A [R][K], or A^T [K][R] for an embedding
    uint16_t *dB = reinterpret_cast<uint16_t *>(base + (size_t)R * K * 2);
    // Unpublish first so no apply ordered after this call sees a half-written slot.
    cudaError_t e = launch_table_set(*rt, slot, nullptr, nullptr, 0, 0.0f, 0.0f, st);
    if (e == cudaSuccess)
        e = cudaMemsetAsync(base, 0, slot_bytes(R, K, N), st);
    if (e == cudaSuccess) {
        if (!embed)
            e = cudaMemcpyAsync(dA, A, (size_t)rank * K * 2, cudaMemcpyDefault, st);
        else if (a_is_transposed)
            e = cudaMemcpy2DAsync(dA, (size_t)R * 2, A, (size_t)rank * 2, (size_t)rank * 2, (size_t)K,
                                  cudaMemcpyDefault, st);
        else if (device_readable(A))
            e = launch_transpose_pack(dA, R, static_cast<const uint16_t *>(A), rank, K, st);
        else
            e = copy_transposed_from_host(dA, R, static_cast<const uint16_t *>(A), rank, K, st);
    }
    if (e == cudaSuccess)
        e = cudaMemcpy2DAsync(dB, (size_t)R * 2, B, (size_t)rank * 2, (size_t)rank * 2, (size_t)N,
                              cudaMemcpyDefault, st);
    const float factor = alpha_factor(alpha, rank, use_rslora);
    if (e == cudaSuccess && !embed) {
        CompRow ones;
        for (int k = 0; k < LORA_COMP_STRIDE; ++k)
            ones.v[k] = 1.0f; // s * 1 == s: the slot's delta is its scale times B (A x)
        e = launch_comp_set(*rt, slot, ones, st);
    }
    if (e == cudaSuccess)
        e = launch_table_set(*rt, slot, dA, dB, rank, factor, adapter_scale * factor, st);
    if (e != cudaSuccess)
        return cuda_fail(e, who);
    return ok();
}

} // namespace

extern "C" {

lora_status lora_route_init(lora_route *rt, void *pool, size_t pool_bytes, void *tables,
                            size_t table_bytes, int max_loras, int max_rank, int n_in, int n_out,
                            lora_stream_t stream)
{
    return route_setup(rt, pool, pool_bytes, tables, table_bytes, max_loras, max_rank, n_in, n_out,
                       LORA_ROUTE_PROJ, "lora_route_init", stream);
}

lora_status lora_embed_route_init(lora_route *rt, void *pool, size_t pool_bytes, void *tables,
                                  size_t table_bytes, int max_loras, int max_rank, int vocab,
                                  int n_embd, lora_stream_t stream)
{
    // the adapted matrix is [vocab][n_embd]: n_in = n_embd, n_out = vocab
    return route_setup(rt, pool, pool_bytes, tables, table_bytes, max_loras, max_rank, n_embd, vocab,
                       LORA_ROUTE_EMBED, "lora_embed_route_init", stream);
}

lora_status lora_pool_pack(const lora_route *rt, int slot, const void *A, const void *B, int rank,
                           float alpha, int use_rslora, float adapter_scale, lora_stream_t stream)
{
    return pack_slot(rt, slot, A, B, rank, alpha, use_rslora, adapter_scale, stream, false);
}

lora_status lora_pool_pack_stack(const lora_route *rt, int slot, int n, const void *const *A,
                                 const void *const *B, const int32_t *ranks, const float *alphas,
                                 const int32_t *use_rslora, const float *adapter_scales,
                                 lora_stream_t stream)
{
    const char *who = "lora_pool_pack_stack";
    lora_status s = check_route_kind(rt, LORA_ROUTE_PROJ, who);
    if (s != LORA_OK)
        return s;
    if (slot < 0 || slot >= rt->max_loras)
        return fail(LORA_ERR_RANGE, "%s: slot %d is out of range: pool has %d slot(s)", who, slot,
                    rt->max_loras);
    if (n < 0)
        return fail(LORA_ERR_SHAPE, "%s: n %d is negative", who, n);
    if (n > 0 && (A == nullptr || B == nullptr || ranks == nullptr || alphas == nullptr ||
                  use_rslora == nullptr || adapter_scales == nullptr))
        return fail(LORA_ERR_NULL, "%s: the member arrays must be non-NULL when n > 0", who);
    const int R = rt->max_rank, K = rt->n_in, N = rt->n_out;
    // members kept (nonzero scale), their scales and rank offsets
    CompRow comp;
    for (int k = 0; k < LORA_COMP_STRIDE; ++k)
        comp.v[k] = 0.0f;
    int total = 0;
    for (int m = 0; m < n; ++m) {
        if (ranks[m] < 1)
            return fail(LORA_ERR_SHAPE, "%s: member %d has rank %d (need >= 1)", who, m, ranks[m]);
        if (A[m] == nullptr || B[m] == nullptr)
            return fail(LORA_ERR_NULL, "%s: member %d has a NULL A or B", who, m);
        const float sm = adapter_scales[m] * alpha_factor(alphas[m], ranks[m], use_rslora[m]);
        if (sm == 0.0f)
            continue;
        if (total + ranks[m] > R) {
            int sum = 0;
            for (int q = 0; q < n; ++q)
                if (adapter_scales[q] * alpha_factor(alphas[q], ranks[q], use_rslora[q]) != 0.0f)
                    sum += ranks[q];
            return fail(LORA_ERR_SHAPE,
                        "%s: the members' ranks sum to %d, past max_rank %d of route [n_out %d x n_in %d]",
                        who, sum, R, N, K);
        }
        for (int k = total; k < total + ranks[m]; ++k)
            comp.v[k] = sm;
        total += ranks[m];
    }
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    uint8_t *base = static_cast<uint8_t *>(rt->pool) + (size_t)slot * slot_bytes(R, K, N);
    uint16_t *dA = reinterpret_cast<uint16_t *>(base);
    uint16_t *dB = reinterpret_cast<uint16_t *>(base + (size_t)R * K * 2);
    // unpublish first, as lora_pool_pack does
    cudaError_t e = launch_table_set(*rt, slot, nullptr, nullptr, 0, 0.0f, 0.0f, st);
    if (e == cudaSuccess && total > 0)
        e = cudaMemsetAsync(base, 0, slot_bytes(R, K, N), st);
    int off = 0;
    for (int m = 0; m < n && e == cudaSuccess && total > 0; ++m) {
        const int r = ranks[m];
        if (adapter_scales[m] * alpha_factor(alphas[m], r, use_rslora[m]) == 0.0f)
            continue;
        e = cudaMemcpyAsync(dA + (size_t)off * K, A[m], (size_t)r * K * 2, cudaMemcpyDefault, st);
        if (e == cudaSuccess)
            e = cudaMemcpy2DAsync(dB + off, (size_t)R * 2, B[m], (size_t)r * 2, (size_t)r * 2, (size_t)N,
                                  cudaMemcpyDefault, st);
        off += r;
    }
    if (e == cudaSuccess && total > 0)
        e = launch_comp_set(*rt, slot, comp, st);
    if (e == cudaSuccess && total > 0)
        e = launch_table_set(*rt, slot, dA, dB, total, 1.0f, 1.0f, st);
    if (e != cudaSuccess)
        return cuda_fail(e, who);
    return ok();
}

lora_status lora_embed_pool_pack(const lora_route *rt, int slot, const void *rows, const void *cols,
                                 int rank, float alpha, int use_rslora, float adapter_scale,
                                 lora_stream_t stream)
{
    // the flipped pair: `cols` is A^T as the slot stores it, `rows` is B
    return pack_slot(rt, slot, cols, rows, rank, alpha, use_rslora, adapter_scale, stream, true);
}

lora_status lora_pool_unpack(const lora_route *rt, int slot, lora_stream_t stream)
{
    lora_status s = check_route(rt, "lora_pool_unpack");
    if (s != LORA_OK)
        return s;
    if (slot < 0 || slot >= rt->max_loras)
        return fail(LORA_ERR_RANGE, "lora_pool_unpack: slot %d is out of range: pool has %d slot(s)",
                    slot, rt->max_loras);
    cudaError_t e = launch_table_set(*rt, slot, nullptr, nullptr, 0, 0.0f, 0.0f,
                                     reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e, "lora_pool_unpack");
    return ok();
}

lora_status lora_set_scale(const lora_route *rt, int slot, float adapter_scale, lora_stream_t stream)
{
    lora_status s = check_route(rt, "lora_set_scale");
    if (s != LORA_OK)
        return s;
    if (slot < 0 || slot >= rt->max_loras)
        return fail(LORA_ERR_RANGE, "lora_set_scale: slot %d is outside [0, %d)", slot,
                    rt->max_loras);
    cudaError_t e = launch_scale_set(*rt, slot, adapter_scale, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e, "lora_set_scale");
    return ok();
}

lora_status lora_set_scales(const lora_route *rt, const int32_t *ids, const float *scales, int n,
                            lora_stream_t stream)
{
    const char *who = "lora_set_scales";
    lora_status s = check_route(rt, who);
    if (s != LORA_OK)
        return s;
    if (n < 0)
        return fail(LORA_ERR_SHAPE, "%s: n %d is negative", who, n);
    if (n > 0 && (ids == nullptr || scales == nullptr))
        return fail(LORA_ERR_NULL, "%s: ids and scales must be non-NULL when n > 0", who);
    for (int i = 0; i < n; ++i)
        if (ids[i] < 0 || ids[i] >= rt->max_loras)
            return fail(LORA_ERR_RANGE, "%s: lora adapter id %d is out of range: %d slot(s) in the route (ids 0..%d)",
                        who, ids[i], rt->max_loras, rt->max_loras - 1);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    for (int first = 0; first < rt->max_loras; first += SCALE_CHUNK) {
        ScaleChunk c;
        c.first = first;
        c.count = rt->max_loras - first < SCALE_CHUNK ? rt->max_loras - first : SCALE_CHUNK;
        for (int i = 0; i < SCALE_CHUNK; ++i)
            c.s[i] = 0.0f; // not listed: scale 0
        for (int i = 0; i < n; ++i) // in order, so the last entry of an id wins
            if (ids[i] >= first && ids[i] < first + c.count)
                c.s[ids[i] - first] = scales[i];
        cudaError_t e = launch_scales_set(*rt, c, st);
        if (e != cudaSuccess)
            return cuda_fail(e, who);
    }
    return ok();
}

lora_status lora_select_victim_slot(const lora_slot_view *cache, int n, int32_t *victim)
{
    const char *who = "lora_select_victim_slot";
    if (n < 0)
        return fail(LORA_ERR_SHAPE, "%s: n %d is negative", who, n);
    if ((n > 0 && cache == nullptr) || victim == nullptr)
        return fail(LORA_ERR_NULL, "%s: cache and victim must be non-NULL", who);
    for (int i = 0; i < n; ++i)
        if (!cache[i].filled) {
            *victim = cache[i].slot;
            return ok();
        }
    int best = -1;
    for (int i = 0; i < n; ++i)
        if (cache[i].ref_count == 0 && (best < 0 || cache[i].last_used < cache[best].last_used))
            best = i; // strict <: the first of equal last_used values is kept
    if (best < 0)
        return fail(LORA_ERR_POOL_FULL, "%s: all %d cached slots are filled and in use", who, n);
    *victim = cache[best].slot;
    return ok();
}

lora_status lora_build_seq_slot(const int32_t *adapter_slots, int n, int padded_n, int active,
                                int32_t *out)
{
    if (n < 0 || padded_n < n)
        return fail(LORA_ERR_SHAPE, "lora_build_seq_slot: need 0 <= n (%d) <= padded_n (%d)", n,
                    padded_n);
    if ((n > 0 && adapter_slots == nullptr) || (padded_n > 0 && out == nullptr))
        return fail(LORA_ERR_NULL, "lora_build_seq_slot: NULL buffer");
    for (int i = 0; i < padded_n; ++i)
        out[i] = i < n ? (adapter_slots[i] >= 0 ? adapter_slots[i] : active) : -1;
    return ok();
}

} // extern "C"

namespace {

lora_status carve_ws(void *ws, size_t ws_bytes, int rows, int nb, int R, int kp, size_t part_elems,
                     int ncnt, Ws &out, const char *who)
{
    const WsLayout l = ws_layout(rows, nb, R, kp, part_elems, ncnt);
    if (ws == nullptr)
        return fail(LORA_ERR_NULL, "%s: workspace is NULL", who);
    if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0)
        return fail(LORA_ERR_ALIGN, "%s: workspace must be 256-byte aligned", who);
    if (ws_bytes < l.total)
        return fail(LORA_ERR_WORKSPACE,
                    "%s: workspace has %zu bytes, needs %zu (%d rows, %d buckets, max_rank %d)", who,
                    ws_bytes, l.total, rows, nb, R);
    uint8_t *b = static_cast<uint8_t *>(ws);
    out.status = reinterpret_cast<uint32_t *>(b + l.status);
    out.perm = reinterpret_cast<int32_t *>(b + l.perm);
    out.seg_off = reinterpret_cast<int32_t *>(b + l.seg_off);
    out.unit_off = reinterpret_cast<int32_t *>(b + l.unit_off);
    out.done = reinterpret_cast<int32_t *>(b + l.done);
    out.h = reinterpret_cast<float *>(b + l.h);
    out.hs = reinterpret_cast<uint16_t *>(b + l.hs);
    out.tiles = reinterpret_cast<int32_t *>(b + l.tiles);
    out.part = reinterpret_cast<float *>(b + l.part);
    out.tile_cnt = reinterpret_cast<int32_t *>(b + l.tile_cnt);
    out.stile = reinterpret_cast<int32_t *>(b + l.stile);
    return LORA_OK;
}

Tables tables_of(const lora_route &rt)
{
    Tables t;
    t.a_table = reinterpret_cast<const uint16_t *const *>(rt.a_table);
    t.b_table = reinterpret_cast<const uint16_t *const *>(rt.b_table);
    t.scale_table = rt.scale_table;
    t.rank_table = rt.rank_table;
    t.comp_table = rt.comp_table;
    return t;
}

lora_status check_io(const char *who, const void *x, int64_t x_stride, int rows, int K, int N,
                     const int32_t *seq_slot, void *y, int64_t y_stride)
{
    if (x == nullptr || seq_slot == nullptr || y == nullptr)
        return fail(LORA_ERR_NULL, "%s: x, seq_slot and y must be non-NULL", who);
    if (K % 8 != 0)
        return fail(LORA_ERR_ALIGN, "%s: K %d must be a multiple of 8", who, K);
    if (x_stride < K || x_stride % 8 != 0)
        return fail(LORA_ERR_ALIGN, "%s: x_stride %lld must be >= K %d and a multiple of 8", who,
                    (long long)x_stride, K);
    if (y_stride < N)
        return fail(LORA_ERR_SHAPE, "%s: y_stride %lld must be >= N %d", who, (long long)y_stride, N);
    if (!aligned16(x))
        return fail(LORA_ERR_ALIGN, "%s: x must be 16-byte aligned", who);
    (void)rows;
    return LORA_OK;
}

// Tensor-core path: prep (routing sort, work lists) then one fused launch
// (shrink, base product, expand-fold); from TC_SHRINK_MIN_ROWS rows the
// shrink is a tensor-core launch of its own between the two. CUDA-core
// path: prep, shrink, GEMV.
lora_status run(Params &p, int path, cudaStream_t st, const char *who)
{
    DevInfo di;
    if (!device_info(di))
        return fail(LORA_ERR_CUDA, "%s: no CUDA device", who);
    cudaError_t e = launch_prep(p, st);
    if (e != cudaSuccess)
        return cuda_fail(e, who);
    if (path == LORA_PATH_SIMT) {
        e = launch_shrink(p, di.num_sms, st);
        if (e == cudaSuccess)
            e = launch_simt(p, di.num_sms, st);
    } else {
        const bool moe = p.expert_offsets != nullptr;
        const TcPlan plan = plan_tc(p, moe);
        TmapSet maps;
        memset(&maps, 0, sizeof maps);
        StcMaps sm;
        memset(&sm, 0, sizeof sm);
        bool ok;
        if (plan.use3d)
            ok = make_map_3d(&maps.x, p.x, (uint64_t)p.K, (uint64_t)p.rows, (uint64_t)p.x_stride,
                             (uint32_t)plan.tn, (uint32_t)plan.kc);
        else
            ok = make_map(&maps.x, p.x, (uint64_t)p.K, (uint64_t)p.rows, (uint64_t)p.x_stride, 64,
                          (uint32_t)plan.tn);
        if (!ok)
            return fail(LORA_ERR_CUDA, "%s: encoding the x tensor map failed", who);
        if (p.stc_tiles > 0) {
            // h from the launch's own tensor-core shrink tiles: whole K, one
            // part, no work units; x in 128-row boxes
            if (!make_map(&sm.sx, p.x, (uint64_t)p.K, (uint64_t)p.rows, (uint64_t)p.x_stride, 64, 128))
                return fail(LORA_ERR_CUDA, "%s: encoding the x tensor map of the shrink failed", who);
            // the pool's A rows by TMA (one box of R rows per slot and chunk) when
            // R is a multiple of 16 (the shrink's rows per slot)
            p.stc_rs = (p.R + 15) & ~15;
            p.stc_amap = (p.pool != nullptr && p.R % 16 == 0 && p.R <= 256 &&
                          make_map_pool_rows(&sm.sa, p.pool, (uint64_t)p.K, (uint64_t)p.R, (uint64_t)p.L,
                                             (uint64_t)p.slot_bytes, (uint32_t)p.R))
                             ? 1
                             : 0;
        }
        for (int q = 0; q < p.E; ++q) {
            if (p.gated)
                ok = make_map_gated(&maps.w[q], p.W[q], (uint64_t)p.K, (uint64_t)p.I, (uint32_t)plan.kc);
            else if (plan.use3d)
                ok = make_map_3d(&maps.w[q], p.W[q], (uint64_t)p.K, (uint64_t)p.N, (uint64_t)p.K, 128,
                                 (uint32_t)plan.kc);
            else
                ok = make_map(&maps.w[q], p.W[q], (uint64_t)p.K, (uint64_t)p.N, (uint64_t)p.K, 64, 128);
            if (!ok)
                return fail(LORA_ERR_CUDA, "%s: encoding the W tensor map of expert %d failed", who, q);
        }
        // y by TMA stores where its layout allows (16-byte aligned rows);
        // otherwise the epilogue stores y element by element
        if (p.gated) // act [rows][I], boxes of 64 act features x 64 rows (the one-part drain)
            p.ystore_ok = (aligned16(p.y) && p.y_stride % 8 == 0 &&
                           make_map_plain(&maps.y, p.y, (uint64_t)p.I, (uint64_t)p.rows, (uint64_t)p.y_stride, 64,
                                          (uint32_t)YSTORE_ROWS))
                              ? 1
                              : 0;
        else
            p.ystore_ok = (aligned16(p.y) && p.y_stride % 8 == 0 &&
                           make_map_plain(&maps.y, p.y, (uint64_t)p.N, (uint64_t)p.rows, (uint64_t)p.y_stride,
                                          128, (uint32_t)YSTORE_ROWS))
                              ? 1
                              : 0;
        // with one K part the gated drain writes act only through these boxes
        if (p.gated && !p.ystore_ok && plan.csplit == 1)
            return fail(LORA_ERR_CUDA, "%s: encoding the act tensor map failed", who);
        e = launch_tc(p, maps, sm, plan, di.num_sms, st);
    }
    if (e != cudaSuccess)
        return cuda_fail(e, who);
    return ok();
}

// One-launch path of up to 256 rows (routing, shrink, base, expand and the
// split-K sum in one kernel). `taken` stays false when the shape, the
// workspace or the device does not suit it; the caller then takes the
// general path.
lora_status run_dec(const Params &p, const void *rt_pool, void *ws, size_t ws_bytes, int gated, int I,
                    cudaStream_t st, const char *who, bool &taken)
{
    taken = false;
    if (p.rows > DEC_MAX_ROWS || p.E != 1)
        return LORA_OK;
    // the gated weight view takes whole 64-row halves of each tile
    if (gated && (p.K % 64 != 0 || I % 64 != 0))
        return LORA_OK;
    const int kc = dec_plan_kc(p.rows, p.K, p.N, p.L, p.R, gated, I);
    if (kc == 0)
        return LORA_OK;
    const DecWs l = dec_ws_layout(p.rows, p.K, p.N, p.L, p.R, gated);
    if (ws_bytes < l.core)
        return LORA_OK;
    DevInfo di;
    if (!device_info(di))
        return fail(LORA_ERR_CUDA, "%s: no CUDA device", who);
    DecLaunch d;
    memset(&d, 0, sizeof d);
    const int tn = tc_token_tile(p.rows);
    const bool use3d = p.K % 64 == 0;
    bool okm = use3d ? make_map_3d(&d.maps.x, p.x, (uint64_t)p.K, (uint64_t)p.rows, (uint64_t)p.x_stride,
                                   (uint32_t)tn, (uint32_t)kc)
                     : make_map(&d.maps.x, p.x, (uint64_t)p.K, (uint64_t)p.rows, (uint64_t)p.x_stride, 64,
                                (uint32_t)tn);
    if (okm)
        okm = gated ? make_map_gated(&d.maps.w[0], p.W[0], (uint64_t)p.K, (uint64_t)I, (uint32_t)kc)
                    : (use3d ? make_map_3d(&d.maps.w[0], p.W[0], (uint64_t)p.K, (uint64_t)p.N, (uint64_t)p.K, 128,
                                           (uint32_t)kc)
                             : make_map(&d.maps.w[0], p.W[0], (uint64_t)p.K, (uint64_t)p.N, (uint64_t)p.K, 64, 128));
    if (!okm)
        return fail(LORA_ERR_CUDA, "%s: encoding the tensor maps failed", who);
    d.pool = rt_pool;
    d.slot_bytes = slot_bytes(p.R, p.K, p.N);
    if (!make_map_pool_a(&d.amap, rt_pool, (uint64_t)p.K, (uint64_t)p.R, (uint64_t)p.L, (uint64_t)d.slot_bytes))
        return fail(LORA_ERR_CUDA, "%s: encoding the A-row tensor map failed", who);
    // one-copy A rows: boxes of 1..16 groups over the largest K part
    d.gb_mask = 0;
    if (use3d && p.R % 8 == 0) {
        const int kch = p.K / 64, C = tc_csplit(p.rows, p.K, false);
        const uint32_t nchb = (uint32_t)((kch + C - 1) / C);
        for (int lg = 0; lg <= 4 && (8 << lg) <= p.R && nchb <= 256; ++lg)
            if (make_map_pool_a5(&d.amap5[lg], rt_pool, (uint64_t)p.K, (uint64_t)p.R, (uint64_t)p.L,
                                 (uint64_t)d.slot_bytes, 1u << lg, nchb))
                d.gb_mask |= 1 << lg;
    }
    uint8_t *b = static_cast<uint8_t *>(ws);
    d.x = p.x;
    d.x_stride = p.x_stride;
    d.y = p.y;
    d.y_stride = p.y_stride;
    d.seq_slot = p.seq_slot;
    d.M = p.rows;
    d.K = p.K;
    d.N = p.N;
    d.L = p.L;
    d.R = p.R;
    d.gated = gated;
    d.I = I;
    d.yvec = ((reinterpret_cast<uintptr_t>(p.y) & 7u) == 0 && p.y_stride % 4 == 0) ? 1 : 0;
    d.tab = p.tab[0];
    d.status = reinterpret_cast<uint32_t *>(b);
    d.perm = reinterpret_cast<int32_t *>(b + l.perm);
    d.seg_off = reinterpret_cast<int32_t *>(b + l.seg_off);
    d.hpart = reinterpret_cast<float *>(b + l.hpart);
    d.pflags = reinterpret_cast<unsigned long long *>(b + l.pflags);
    d.gpart = ws_bytes >= l.total ? reinterpret_cast<float *>(b + l.gpart) : nullptr;
    cudaError_t e = launch_dec(d, di.num_sms, st);
    if (e == cudaErrorNotSupported)
        return LORA_OK;
    taken = true;
    if (e != cudaSuccess)
        return cuda_fail(e, who);
    return ok();
}

// gated_I > 0: W is the fused [gate I | up I] (N = 2I) and y receives act
// [M][gated_I] from the tensor-core kernel's drain (the caller has checked
// that the shape takes it: tc_gated_ok).
lora_status proj_apply(const void *x, int64_t x_stride, const void *W, int M, int K, int N,
                       const int32_t *seq_slot, const lora_route *rt, void *y, int64_t y_stride,
                       void *ws, size_t ws_bytes, int path, lora_stream_t stream, int gated_I = 0)
{
    const char *who = "lora_proj_apply";
    lora_status s = check_route_kind(rt, LORA_ROUTE_PROJ, who);
    if (s != LORA_OK)
        return s;
    if (M < 0)
        return fail(LORA_ERR_SHAPE, "%s: M %d is negative", who, M);
    if (path < LORA_PATH_AUTO || path > LORA_PATH_TC_ONE)
        return fail(LORA_ERR_RANGE, "%s: path %d is not one of LORA_PATH_*", who, path);
    if (K != rt->n_in || N != rt->n_out)
        return fail(LORA_ERR_SHAPE,
                    "%s: x is [M %d][K %d] and W [N %d][K %d], but the route is [n_out %d x n_in %d]",
                    who, M, K, N, K, rt->n_out, rt->n_in);
    if (M == 0)
        return ok();
    if (W == nullptr)
        return fail(LORA_ERR_NULL, "%s: W is NULL", who);
    if (!aligned16(W))
        return fail(LORA_ERR_ALIGN, "%s: W must be 16-byte aligned", who);
    if ((s = check_io(who, x, x_stride, M, K, gated_I > 0 ? gated_I : N, seq_slot, y, y_stride)) != LORA_OK)
        return s;
    Params p;
    memset(&p, 0, sizeof p);
    p.x = static_cast<const uint16_t *>(x);
    p.x_stride = x_stride;
    p.y = static_cast<uint16_t *>(y);
    p.y_stride = y_stride;
    p.gated = gated_I > 0 ? 1 : 0;
    p.I = gated_I;
    p.pool = rt->pool;
    p.slot_bytes = slot_bytes(rt->max_rank, rt->n_in, rt->n_out);
    p.seq_slot = seq_slot;
    p.expert_offsets = nullptr;
    p.E = 1;
    p.rows = M;
    p.K = K;
    p.N = N;
    p.L = rt->max_loras;
    p.R = rt->max_rank;
    p.W[0] = static_cast<const uint16_t *>(W);
    p.tab[0] = tables_of(*rt);
    p.kp = shrink_kparts(K);
    size_t part_elems = 0;
    split_scratch(M, K, N, part_elems, p.ncnt);
    if ((s = carve_ws(ws, ws_bytes, M, p.L + 1, p.R, p.kp, part_elems, p.ncnt, p.ws, who)) != LORA_OK)
        return s;
    if (path == LORA_PATH_AUTO)
        path = M <= SIMT_MAX_ROWS ? LORA_PATH_SIMT : LORA_PATH_TC;
    p.tn = tc_token_tile(M);
    if (path == LORA_PATH_TC_ONE) {
        bool taken = false;
        s = run_dec(p, rt->pool, ws, ws_bytes, 0, 0, reinterpret_cast<cudaStream_t>(stream), who, taken);
        if (taken || s != LORA_OK)
            return s;
        path = LORA_PATH_TC;
    }
    if (path == LORA_PATH_TC && M >= TC_SHRINK_MIN_ROWS) {
        p.kp = 1; // the tensor-core shrink tiles write h over the whole K
        p.no_units = 1;
        p.stc_tiles = (M + 127) / 128;
    }
    return run(p, path, reinterpret_cast<cudaStream_t>(stream), who);
}

} // namespace

extern "C" {

size_t lora_proj_workspace_bytes(int M, const lora_route *rt)
{
    if (rt == nullptr || rt->magic != ROUTE_MAGIC || M < 0)
        return 0;
    size_t part_elems = 0;
    int ncnt = 0;
    split_scratch(M, rt->n_in, rt->n_out, part_elems, ncnt);
    return ws_layout(M, rt->max_loras + 1, rt->max_rank, shrink_kparts(rt->n_in), part_elems, ncnt).total;
}

size_t lora_proj_workspace_bytes_ex(int M, const lora_route *rt, int path)
{
    size_t need = lora_proj_workspace_bytes(M, rt);
    if (need > 0 && path == LORA_PATH_TC_ONE && M <= DEC_MAX_ROWS) {
        const size_t d = dec_ws_layout(M, rt->n_in, rt->n_out, rt->max_loras, rt->max_rank, 0).total;
        need = d > need ? d : need;
    }
    return need;
}

lora_status lora_proj_apply(const void *x, int64_t x_stride, const void *W, int M, int K, int N,
                            const int32_t *seq_slot, const lora_route *rt, void *y, int64_t y_stride,
                            void *ws, size_t ws_bytes, lora_stream_t stream)
{
    return proj_apply(x, x_stride, W, M, K, N, seq_slot, rt, y, y_stride, ws, ws_bytes,
                      LORA_PATH_AUTO, stream);
}

lora_status lora_proj_apply_ex(const void *x, int64_t x_stride, const void *W, int M, int K, int N,
                               const int32_t *seq_slot, const lora_route *rt, void *y,
                               int64_t y_stride, void *ws, size_t ws_bytes, int path,
                               lora_stream_t stream)
{
    return proj_apply(x, x_stride, W, M, K, N, seq_slot, rt, y, y_stride, ws, ws_bytes, path, stream);
}

size_t lora_gate_up_workspace_bytes(int M, const lora_route *rt)
{
    if (rt == nullptr || rt->magic != ROUTE_MAGIC || rt->kind != LORA_ROUTE_PROJ || M < 0 || rt->n_out % 2 != 0)
        return 0;
    // the projection's workspace, then its [M][2I] bf16 output
    return align256(lora_proj_workspace_bytes(M, rt)) + align256((size_t)M * (size_t)rt->n_out * 2);
}

size_t lora_gate_up_workspace_bytes_ex(int M, const lora_route *rt, int path)
{
    const size_t base = lora_gate_up_workspace_bytes(M, rt);
    if (base == 0)
        return 0;
    return align256(lora_proj_workspace_bytes_ex(M, rt, path)) + align256((size_t)M * (size_t)rt->n_out * 2);
}

lora_status lora_gate_up_apply(const void *x, int64_t x_stride, const void *W, int M, int K, int I,
                               const int32_t *seq_slot, const lora_route *rt, void *act, int64_t act_stride,
                               void *ws, size_t ws_bytes, lora_stream_t stream)
{
    return lora_gate_up_apply_ex(x, x_stride, W, M, K, I, seq_slot, rt, act, act_stride, ws, ws_bytes,
                                 LORA_PATH_AUTO, stream);
}

lora_status lora_gate_up_apply_ex(const void *x, int64_t x_stride, const void *W, int M, int K, int I,
                                  const int32_t *seq_slot, const lora_route *rt, void *act, int64_t act_stride,
                                  void *ws, size_t ws_bytes, int path, lora_stream_t stream)
{
    const char *who = "lora_gate_up_apply";
    lora_status s = check_route_kind(rt, LORA_ROUTE_PROJ, who);
    if (s != LORA_OK)
        return s;
    if (M < 0)
        return fail(LORA_ERR_SHAPE, "%s: M %d is negative", who, M);
    if (I <= 0 || (int64_t)rt->n_out != 2 * (int64_t)I || K != rt->n_in)
        return fail(LORA_ERR_SHAPE,
                    "%s: a fused [gate|up] of I %d over K %d needs a route of [n_out 2I = %lld x n_in %d], "
                    "the route is [n_out %d x n_in %d]",
                    who, I, K, 2 * (long long)I, K, rt->n_out, rt->n_in);
    if (M == 0)
        return ok();
    if (act == nullptr)
        return fail(LORA_ERR_NULL, "%s: act is NULL", who);
    if (act_stride < I)
        return fail(LORA_ERR_SHAPE, "%s: act_stride %lld must be >= I %d", who, (long long)act_stride, I);
    const size_t need = lora_gate_up_workspace_bytes(M, rt);
    if (ws == nullptr)
        return fail(LORA_ERR_NULL, "%s: workspace is NULL", who);
    if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0)
        return fail(LORA_ERR_ALIGN, "%s: workspace must be 256-byte aligned", who);
    if (ws_bytes < need)
        return fail(LORA_ERR_WORKSPACE, "%s: workspace has %zu bytes, needs %zu (%d rows, 2I = %d)", who,
                    ws_bytes, need, M, 2 * I);
    if (path < LORA_PATH_AUTO || path > LORA_PATH_TC_ONE)
        return fail(LORA_ERR_RANGE, "%s: path %d is not one of LORA_PATH_*", who, path);
    // the one-launch kernel needs its own workspace ahead of the act scratch;
    // with less, the call takes the tensor-core path
    if (path == LORA_PATH_TC_ONE && ws_bytes < lora_gate_up_workspace_bytes_ex(M, rt, path))
        path = LORA_PATH_TC;
    DevInfo di;
    if (!device_info(di))
        return fail(LORA_ERR_CUDA, "%s: no CUDA device", who);
    const size_t proj_ws = align256(lora_proj_workspace_bytes_ex(M, rt, path));
    if (path == LORA_PATH_TC_ONE && M > SIMT_MAX_ROWS && M <= DEC_MAX_ROWS) {
        // one launch: the sum of the K parts rounds both halves and writes act
        if (W == nullptr || x == nullptr || seq_slot == nullptr)
            return fail(LORA_ERR_NULL, "%s: x, W and seq_slot must be non-NULL", who);
        if (!aligned16(W))
            return fail(LORA_ERR_ALIGN, "%s: W must be 16-byte aligned", who);
        if ((s = check_io(who, x, x_stride, M, K, I, seq_slot, act, act_stride)) != LORA_OK)
            return s;
        Params p;
        memset(&p, 0, sizeof p);
        p.x = static_cast<const uint16_t *>(x);
        p.x_stride = x_stride;
        p.y = static_cast<uint16_t *>(act);
        p.y_stride = act_stride;
        p.seq_slot = seq_slot;
        p.E = 1;
        p.rows = M;
        p.K = K;
        p.N = 2 * I;
        p.L = rt->max_loras;
        p.R = rt->max_rank;
        p.W[0] = static_cast<const uint16_t *>(W);
        p.tab[0] = tables_of(*rt);
        bool taken = false;
        s = run_dec(p, rt->pool, ws, proj_ws, 1, I, reinterpret_cast<cudaStream_t>(stream), who, taken);
        if (taken || s != LORA_OK)
            return s;
    }
    // the tensor-core kernel reads W as 64 gate + 64 up rows per tile and
    // writes act from its drain (one K part) or from its split-K sum
    if (path != LORA_PATH_SIMT && !(path == LORA_PATH_AUTO && M <= SIMT_MAX_ROWS)) {
        Params q;
        memset(&q, 0, sizeof q);
        q.rows = M;
        q.K = K;
        q.N = 2 * I;
        q.I = I;
        q.gated = 1;
        q.E = 1;
        q.L = rt->max_loras;
        q.R = rt->max_rank;
        q.tn = tc_token_tile(M);
        q.ystore_ok = aligned16(act) && act_stride % 8 == 0 ? 1 : 0;
        if (tc_gated_ok(q))
            return proj_apply(x, x_stride, W, M, K, 2 * I, seq_slot, rt, act, act_stride, ws, proj_ws,
                              LORA_PATH_TC, stream, I);
    }
    uint16_t *gu = reinterpret_cast<uint16_t *>(static_cast<uint8_t *>(ws) + proj_ws);
    s = proj_apply(x, x_stride, W, M, K, 2 * I, seq_slot, rt, gu, 2 * (int64_t)I, ws, proj_ws,
                   path == LORA_PATH_TC_ONE ? LORA_PATH_TC : path, stream);
    if (s != LORA_OK)
        return s;
    cudaError_t e = launch_silu_mul(gu, 2 * (int64_t)I, M, I, static_cast<uint16_t *>(act), act_stride,
                                    di.num_sms, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e, who);
    return ok();
}

size_t lora_moe_workspace_bytes(int E, int T, const lora_route *rts)
{
    if (rts == nullptr || E < 1 || E > MAX_E || T < 0 || rts[0].magic != ROUTE_MAGIC)
        return 0;
    size_t part_elems = 0;
    int ncnt = 0;
    moe_split_scratch(T, E, rts[0].n_in, rts[0].n_out, part_elems, ncnt);
    return ws_layout(T, E * (rts[0].max_loras + 1), rts[0].max_rank, shrink_kparts(rts[0].n_in), part_elems,
                     ncnt)
        .total;
}

lora_status lora_moe_down_apply(const void *x, int64_t x_stride, const void *const *W_e,
                                const int32_t *expert_offsets, int E, int T, int K, int N,
                                const int32_t *seq_slot, const lora_route *rts, void *y,
                                int64_t y_stride, void *ws, size_t ws_bytes, lora_stream_t stream)
{
    const char *who = "lora_moe_down_apply";
    if (E < 1 || E > MAX_E)
        return fail(LORA_ERR_UNSUPPORTED, "%s: E %d must be in [1, %d]", who, E, MAX_E);
    if (rts == nullptr || W_e == nullptr || expert_offsets == nullptr)
        return fail(LORA_ERR_NULL, "%s: rts, W_e and expert_offsets must be non-NULL", who);
    for (int q = 0; q < E; ++q) {
        lora_status s = check_route_kind(&rts[q], LORA_ROUTE_PROJ, who);
        if (s != LORA_OK)
            return s;
        if (rts[q].n_in != K || rts[q].n_out != N || rts[q].max_rank != rts[0].max_rank ||
            rts[q].max_loras != rts[0].max_loras)
            return fail(LORA_ERR_SHAPE,
                        "%s: route of expert %d is [n_out %d x n_in %d] rank %d with %d slots; "
                        "expected [%d x %d] rank %d with %d slots",
                        who, q, rts[q].n_out, rts[q].n_in, rts[q].max_rank, rts[q].max_loras, N, K,
                        rts[0].max_rank, rts[0].max_loras);
        if (W_e[q] == nullptr)
            return fail(LORA_ERR_NULL, "%s: W_e[%d] is NULL", who, q);
        if (!aligned16(W_e[q]))
            return fail(LORA_ERR_ALIGN, "%s: W_e[%d] must be 16-byte aligned", who, q);
    }
    if (T < 0)
        return fail(LORA_ERR_SHAPE, "%s: T %d is negative", who, T);
    if (T == 0)
        return ok();
    lora_status s = check_io(who, x, x_stride, T, K, N, seq_slot, y, y_stride);
    if (s != LORA_OK)
        return s;
    const int L = rts[0].max_loras, R = rts[0].max_rank;
    if (E * (L + 1) > MAX_BUCKETS)
        return fail(LORA_ERR_UNSUPPORTED, "%s: E * (max_loras + 1) = %d exceeds %d", who, E * (L + 1),
                    MAX_BUCKETS);
    Params p;
    memset(&p, 0, sizeof p);
    p.x = static_cast<const uint16_t *>(x);
    p.x_stride = x_stride;
    p.y = static_cast<uint16_t *>(y);
    p.y_stride = y_stride;
    p.seq_slot = seq_slot;
    p.expert_offsets = expert_offsets;
    p.E = E;
    p.rows = T;
    p.K = K;
    p.N = N;
    p.L = L;
    p.R = R;
    for (int q = 0; q < E; ++q) {
        p.W[q] = static_cast<const uint16_t *>(W_e[q]);
        p.tab[q] = tables_of(rts[q]);
    }
    p.kp = shrink_kparts(K);
    size_t part_elems = 0;
    moe_split_scratch(T, E, K, N, part_elems, p.ncnt);
    if ((s = carve_ws(ws, ws_bytes, T, E * (L + 1), R, p.kp, part_elems, p.ncnt, p.ws, who)) != LORA_OK)
        return s;
    p.tn = moe_token_tile(T, E);
    p.max_tiles = moe_max_tiles(T, E);
    return run(p, LORA_PATH_TC, reinterpret_cast<cudaStream_t>(stream), who);
}

size_t lora_embed_workspace_bytes(int M, const lora_route *rt)
{
    if (rt == nullptr || rt->magic != ROUTE_MAGIC || rt->kind != LORA_ROUTE_EMBED || M < 0)
        return 0;
    return ws_layout(M, rt->max_loras + 1, 0, 1).total; // routing sort and status only
}

lora_status lora_embed_apply(const int32_t *tokens, const void *E, int M, int vocab, int n_embd,
                             const int32_t *seq_slot, const lora_route *rt, void *y, int64_t y_stride,
                             void *ws, size_t ws_bytes, lora_stream_t stream)
{
    const char *who = "lora_embed_apply";
    lora_status s = check_route_kind(rt, LORA_ROUTE_EMBED, who);
    if (s != LORA_OK)
        return s;
    if (M < 0)
        return fail(LORA_ERR_SHAPE, "%s: M %d is negative", who, M);
    if (vocab != rt->n_out || n_embd != rt->n_in)
        return fail(LORA_ERR_SHAPE, "%s: E is [vocab %d][n_embd %d], but the route is [vocab %d x n_embd %d]",
                    who, vocab, n_embd, rt->n_out, rt->n_in);
    if (M == 0)
        return ok();
    if (tokens == nullptr || E == nullptr || seq_slot == nullptr || y == nullptr)
        return fail(LORA_ERR_NULL, "%s: tokens, E, seq_slot and y must be non-NULL", who);
    if (!aligned16(E) || !aligned16(y))
        return fail(LORA_ERR_ALIGN, "%s: E and y must be 16-byte aligned", who);
    if (y_stride < n_embd || y_stride % 8 != 0)
        return fail(LORA_ERR_ALIGN, "%s: y_stride %lld must be >= n_embd %d and a multiple of 8", who,
                    (long long)y_stride, n_embd);
    DevInfo di;
    if (!device_info(di))
        return fail(LORA_ERR_CUDA, "%s: no CUDA device", who);
    // the routing kernel: one expert segment, no shrink work units
    Params p;
    memset(&p, 0, sizeof p);
    p.seq_slot = seq_slot;
    p.expert_offsets = nullptr;
    p.E = 1;
    p.rows = M;
    p.K = n_embd;
    p.N = vocab;
    p.L = rt->max_loras;
    p.R = rt->max_rank;
    p.tab[0] = tables_of(*rt);
    p.kp = 1;
    p.no_units = 1;
    if ((s = carve_ws(ws, ws_bytes, M, p.L + 1, 0, 1, 0, 0, p.ws, who)) != LORA_OK)
        return s;
    EmbedParams ep;
    memset(&ep, 0, sizeof ep);
    ep.E = static_cast<const uint16_t *>(E);
    ep.tokens = tokens;
    ep.seq_slot = seq_slot;
    ep.y = static_cast<uint16_t *>(y);
    ep.y_stride = y_stride;
    ep.M = M;
    ep.vocab = vocab;
    ep.n_embd = n_embd;
    ep.L = rt->max_loras;
    ep.R = rt->max_rank;
    ep.ft = embed_tile_features(ep.R);
    ep.nft = (n_embd + ep.ft - 1) / ep.ft;
    ep.tab = p.tab[0];
    ep.ws = p.ws;
    p.tn = EMBED_CHUNK_ROWS;
    // up to EMBED_LOCAL_ROWS rows every CTA sorts the batch itself: one launch
    ep.local = embed_local_fits(M, ep.ft, ep.R, ep.L) ? 1 : 0;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = ep.local ? cudaSuccess : launch_prep(p, st);
    if (e == cudaSuccess)
        e = launch_embed(ep, di.num_sms, st);
    if (e != cudaSuccess)
        return cuda_fail(e, who);
    return ok();
}

namespace {

struct GatherWs {
    size_t moe, x_sorted, y_sorted, perm, inv, slots, offsets, total;
};

GatherWs gather_ws(int E, int T, const lora_route *rts)
{
    GatherWs l;
    const int K = rts[0].n_in, N = rts[0].n_out;
    size_t o = align256(lora_moe_workspace_bytes(E, T, rts));
    l.moe = o;
    l.x_sorted = o; o = align256(o + (size_t)T * K * 2);
    l.y_sorted = o; o = align256(o + (size_t)T * N * 2);
    l.perm = o;     o = align256(o + (size_t)T * 4);
    l.inv = o;      o = align256(o + (size_t)T * 4);
    l.slots = o;    o = align256(o + (size_t)T * 4);
    l.offsets = o;  o = align256(o + (size_t)(E + 2) * 4);
    l.total = o;
    return l;
}

} // namespace

size_t lora_moe_gather_workspace_bytes(int E, int T, const lora_route *rts)
{
    if (rts == nullptr || E < 1 || E > MAX_E || T < 0 || rts[0].magic != ROUTE_MAGIC ||
        rts[0].kind != LORA_ROUTE_PROJ)
        return 0;
    return gather_ws(E, T, rts).total;
}

lora_status lora_moe_gather_apply(const void *x, int64_t x_stride, const void *const *W_e,
                                  const int32_t *indices, int E, int T, int K, int N,
                                  const int32_t *seq_slot, const lora_route *rts, const float *combine,
                                  int top_k, void *y, int64_t y_stride, void *ws, size_t ws_bytes,
                                  lora_stream_t stream)
{
    const char *who = "lora_moe_gather_apply";
    if (E < 1 || E > MAX_E)
        return fail(LORA_ERR_UNSUPPORTED, "%s: E %d must be in [1, %d]", who, E, MAX_E);
    if (rts == nullptr || W_e == nullptr)
        return fail(LORA_ERR_NULL, "%s: rts and W_e must be non-NULL", who);
    for (int q = 0; q < E; ++q) {
        lora_status s = check_route_kind(&rts[q], LORA_ROUTE_PROJ, who);
        if (s != LORA_OK)
            return s;
        if (rts[q].n_in != K || rts[q].n_out != N)
            return fail(LORA_ERR_SHAPE, "%s: route of expert %d is [n_out %d x n_in %d]; expected [%d x %d]",
                        who, q, rts[q].n_out, rts[q].n_in, N, K);
    }
    if (T < 0)
        return fail(LORA_ERR_SHAPE, "%s: T %d is negative", who, T);
    if (T > LORA_GATHER_MAX_ROWS)
        return fail(LORA_ERR_UNSUPPORTED, "%s: T %d exceeds %d slot-rows (group the rows by expert and use "
                    "lora_moe_down_apply)", who, T, LORA_GATHER_MAX_ROWS);
    if (combine != nullptr && (top_k < 1 || T % top_k != 0))
        return fail(LORA_ERR_SHAPE, "%s: with combine weights top_k %d must be >= 1 and divide T %d", who,
                    top_k, T);
    if (T == 0)
        return ok();
    if (indices == nullptr)
        return fail(LORA_ERR_NULL, "%s: indices is NULL", who);
    lora_status s = check_io(who, x, x_stride, T, K, N, seq_slot, y, y_stride);
    if (s != LORA_OK)
        return s;
    const GatherWs l = gather_ws(E, T, rts);
    if (ws == nullptr)
        return fail(LORA_ERR_NULL, "%s: workspace is NULL", who);
    if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0)
        return fail(LORA_ERR_ALIGN, "%s: workspace must be 256-byte aligned", who);
    if (ws_bytes < l.total)
        return fail(LORA_ERR_WORKSPACE, "%s: workspace has %zu bytes, needs %zu (%d slot-rows, %d experts)",
                    who, ws_bytes, l.total, T, E);
    DevInfo di;
    if (!device_info(di))
        return fail(LORA_ERR_CUDA, "%s: no CUDA device", who);
    uint8_t *b = static_cast<uint8_t *>(ws);
    GatherParams g;
    memset(&g, 0, sizeof g);
    g.x = static_cast<const uint16_t *>(x);
    g.x_stride = x_stride;
    g.indices = indices;
    g.seq_slot = seq_slot;
    g.E = E;
    g.T = T;
    g.K = K;
    g.N = N;
    g.x_sorted = reinterpret_cast<uint16_t *>(b + l.x_sorted);
    g.perm = reinterpret_cast<int32_t *>(b + l.perm);
    g.inv = reinterpret_cast<int32_t *>(b + l.inv);
    g.slots_sorted = reinterpret_cast<int32_t *>(b + l.slots);
    g.offsets = reinterpret_cast<int32_t *>(b + l.offsets);
    g.y_sorted = reinterpret_cast<const uint16_t *>(b + l.y_sorted);
    g.combine = combine;
    g.top_k = combine ? top_k : 1;
    g.y = static_cast<uint16_t *>(y);
    g.y_stride = y_stride;
    g.status = static_cast<uint32_t *>(ws); // the grouped fold's status word
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = launch_gather_sort(g, di.num_sms, st);
    if (e != cudaSuccess)
        return cuda_fail(e, who);
    s = lora_moe_down_apply(g.x_sorted, K, W_e, g.offsets, E, T, K, N, g.slots_sorted, rts, b + l.y_sorted, N,
                            ws, l.moe, stream);
    if (s != LORA_OK)
        return s;
    e = launch_gather_combine(g, di.num_sms, st);
    if (e != cudaSuccess)
        return cuda_fail(e, who);
    return ok();
}

lora_status lora_proj_plan(int M, const lora_route *rt, int gated, int path, lora_plan_info *info)
{
    const char *who = "lora_proj_plan";
    if (info == nullptr)
        return fail(LORA_ERR_NULL, "%s: info is NULL", who);
    memset(info, 0, sizeof *info);
    lora_status s = check_route_kind(rt, LORA_ROUTE_PROJ, who);
    if (s != LORA_OK)
        return s;
    if (M < 0)
        return fail(LORA_ERR_SHAPE, "%s: M %d is negative", who, M);
    if (gated && rt->n_out % 2 != 0)
        return fail(LORA_ERR_SHAPE, "%s: a gated plan needs an even n_out (%d)", who, rt->n_out);
    if (path < LORA_PATH_AUTO || path > LORA_PATH_TC_ONE)
        return fail(LORA_ERR_RANGE, "%s: path %d is not one of LORA_PATH_*", who, path);
    if (M == 0)
        return ok();
    DevInfo di;
    if (!device_info(di))
        return fail(LORA_ERR_CUDA, "%s: no CUDA device", who);
    const int K = rt->n_in, N = rt->n_out, I = gated ? N / 2 : 0;
    if (path == LORA_PATH_SIMT || (path == LORA_PATH_AUTO && M <= SIMT_MAX_ROWS)) {
        info->path = LORA_PLAN_SIMT;
        info->kernels = gated ? 4 : 3;
        return ok();
    }
    // the gated call writes act from the tensor-core drain or split-K sum
    // (act rows taken as 16-byte aligned)
    bool fused_act = false;
    if (gated) {
        Params q;
        memset(&q, 0, sizeof q);
        q.rows = M;
        q.K = K;
        q.N = N;
        q.I = I;
        q.gated = 1;
        q.E = 1;
        q.L = rt->max_loras;
        q.R = rt->max_rank;
        q.tn = tc_token_tile(M);
        q.ystore_ok = 1;
        fused_act = tc_gated_ok(q);
    }
    uint32_t smem = 0;
    const bool one = path == LORA_PATH_TC_ONE && M <= DEC_MAX_ROWS && (!gated || M > SIMT_MAX_ROWS) &&
                     (!gated || (K % 64 == 0 && I % 64 == 0)) &&
                     dec_plan_info(M, K, N, rt->max_loras, rt->max_rank, gated, I, di.num_sms,
                                   &info->clusters_needed, &info->clusters_resident, &info->cluster_size,
                                   &smem) == 1;
    info->smem_per_cta = (int)smem;
    if (one) {
        info->path = LORA_PLAN_ONE_LAUNCH;
        info->kernels = 1;
    } else {
        info->path = LORA_PLAN_TC;
        info->kernels = 2 + (gated && !fused_act ? 1 : 0);
    }
    return ok();
}

void lora_test_wait_hook(uint64_t wait_ns, int extra_flags)
{
    dec_test_hook(wait_ns, extra_flags < 0 ? 0 : extra_flags);
}

lora_status lora_status_get(const void *ws, uint32_t *flags, lora_stream_t stream)
{
    if (ws == nullptr || flags == nullptr)
        return fail(LORA_ERR_NULL, "lora_status_get: ws and flags must be non-NULL");
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    uint32_t w[3] = {0, 0, 0}; // flags, tag of the call that set them, epoch
    cudaError_t e = cudaMemcpyAsync(w, ws, sizeof w, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess)
        e = cudaStreamSynchronize(st);
    if (e != cudaSuccess)
        return cuda_fail(e, "lora_status_get");
    *flags = w[1] == status_tag(w[2] - 1u) ? w[0] : 0u;
    return ok();
}

lora_status lora_proj_routing(const void *ws, int M, int max_loras, int32_t *perm, int32_t *seg_off,
                              lora_stream_t stream)
{
    if (ws == nullptr || perm == nullptr || seg_off == nullptr)
        return fail(LORA_ERR_NULL, "lora_proj_routing: ws, perm and seg_off must be non-NULL");
    if (M < 0 || max_loras <= 0 || max_loras > MAX_LORAS)
        return fail(LORA_ERR_SHAPE, "lora_proj_routing: M %d / max_loras %d out of range", M,
                    max_loras);
    const WsLayout l = ws_layout(M, max_loras + 1, 8, 1); // perm / seg_off do not depend on R or kp
    const uint8_t *b = static_cast<const uint8_t *>(ws);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaSuccess;
    if (M > 0)
        e = cudaMemcpyAsync(perm, b + l.perm, sizeof(int32_t) * (size_t)M, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(seg_off, b + l.seg_off, sizeof(int32_t) * (size_t)(max_loras + 2),
                            cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess)
        e = cudaStreamSynchronize(st);
    if (e != cudaSuccess)
        return cuda_fail(e, "lora_proj_routing");
    return ok();
}

} // extern "C"
