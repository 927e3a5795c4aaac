// Internal definitions shared by the host ABI (lora_api.cu) and the kernels.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/rank_delta.h"

namespace rd {

constexpr int MAX_E = LORA_MAX_EXPERTS;
constexpr int MAX_BUCKETS = 1024;   // experts * (max_loras + 1)
constexpr int SHRINK_RG = 8;        // ranks per shrink work unit (one warp each)
constexpr int SHRINK_TC = 16;       // rows per shrink work unit
constexpr int PREP_THREADS = 1024;

// Device routing tables of one expert's route.
struct Tables {
    const uint16_t *const *a_table;
    const uint16_t *const *b_table;
    const float *scale_table;
    const int32_t *rank_table;
};

// What the expand needs for a row routed to slot s of table t. A row gets no
// delta when its slot is negative or >= L, the slot is empty, or its scale
// is 0 (the delta is then skipped, not multiplied by zero).
struct SlotInfo {
    const uint16_t *b; // B of the slot, [N][R]
    float scale;
    int rank;
    int on;
};

__device__ __forceinline__ SlotInfo slot_info(const Tables &t, int s, int L)
{
    SlotInfo si{nullptr, 0.0f, 0, 0};
    if (s < 0 || s >= L)
        return si;
    const uint16_t *a = t.a_table[s];
    si.b = t.b_table[s];
    si.scale = t.scale_table[s];
    si.rank = t.rank_table[s];
    si.on = (a != nullptr && si.b != nullptr && si.scale != 0.0f && si.rank > 0) ? 1 : 0;
    return si;
}

// Workspace sections (device pointers carved from the caller's buffer).
struct Ws {
    uint32_t *status;   // [1] LORA_FLAG_* bits of the last call
    int32_t *perm;      // [rows] row ids grouped by (expert, slot bucket)
    int32_t *seg_off;   // [nb + 1] bucket starts in perm
    int32_t *unit_off;  // [nb + 1] first shrink unit of each bucket
    int32_t *done;      // [nb] finished shrink units per bucket
    float *h;           // [rows][R] A_s x_i of every adapted row (fp32)
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
    const uint16_t *W[MAX_E];
    Tables tab[MAX_E];
    Ws ws;
};

struct WsLayout {
    size_t status, perm, seg_off, unit_off, done, h, total;
};

inline size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

inline WsLayout ws_layout(int rows, int nb, int R)
{
    WsLayout l;
    size_t o = 0;
    l.status = o;   o = align256(o + 256);
    l.perm = o;     o = align256(o + sizeof(int32_t) * (size_t)rows);
    l.seg_off = o;  o = align256(o + sizeof(int32_t) * (size_t)(nb + 1));
    l.unit_off = o; o = align256(o + sizeof(int32_t) * (size_t)(nb + 1));
    l.done = o;     o = align256(o + sizeof(int32_t) * (size_t)nb);
    l.h = o;        o = align256(o + sizeof(float) * (size_t)rows * (size_t)R);
    l.total = o;
    return l;
}

// Tensor maps of one launch of the tensor-core kernel.
struct TmapSet {
    CUtensorMap x;
    CUtensorMap w[MAX_E];
};

// Launchers (each defined next to its kernel). They return the launch error.
cudaError_t launch_prep(const Params &p, cudaStream_t st);
cudaError_t launch_shrink(const Params &p, int num_sms, cudaStream_t st);
cudaError_t launch_simt(const Params &p, int num_sms, cudaStream_t st);
cudaError_t launch_tc(const Params &p, const TmapSet &maps, int token_tile, cudaStream_t st);
cudaError_t launch_table_set(const lora_route &rt, int slot, const void *a, const void *b,
                             int rank, float factor, float scale, cudaStream_t st);
cudaError_t launch_scale_set(const lora_route &rt, int slot, float adapter_scale, cudaStream_t st);

// Record `msg` as the thread's last error and return `code` (lora_api.cu).
lora_status api_fail(lora_status code, const char *msg);

// The token-tile sizes the tensor-core kernel is built for.
inline int tc_token_tile(int rows_per_segment)
{
    if (rows_per_segment <= 64) return 64;
    if (rows_per_segment <= 128) return 128;
    return 256;
}

} // namespace rd
