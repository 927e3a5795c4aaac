// Routing and shrink kernels of the LoRA projection.
//
// prep_kernel   -- one CTA: stable counting sort of rows into (expert, slot)
//                  buckets (perm / seg_off), the shrink work list (unit_off),
//                  handoff counters cleared, the token tiles of each expert
//                  segment, status word of this call. It lets the dependent
//                  projection kernel launch at once (programmatic dependent
//                  launch); that kernel waits for this one only where it reads
//                  these results.
// shrink_kernel -- the shrink units (shrink.cuh) as a kernel of their own, for
//                  the CUDA-core GEMV path.
// table kernels -- stream-ordered writes of one slot's table entries.
#include "lora_internal.cuh"
#include "shrink.cuh"
#include "vec.cuh"

namespace rd {

// Exclusive scan of one value per thread across the 1024-thread block.
__device__ __forceinline__ int block_exclusive_scan(int v, int *warp_tot, int &total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o)
            incl += t;
    }
    if (lane == 31)
        warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int w = warp_tot[lane];
        int wi = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int t = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o)
                wi += t;
        }
        warp_tot[lane] = wi - w; // exclusive prefix of warp totals
        if (lane == 31)
            warp_tot[32] = wi;
    }
    __syncthreads();
    int r = warp_tot[warp] + incl - v;
    total = warp_tot[32];
    __syncthreads();
    return r;
}

// Bucket of row i given the expert segment bounds and its slot value.
__device__ __forceinline__ int bucket_of(const Params &p, const int *offs, int i, int s)
{
    int e = -1;
    for (int q = 0; q < p.E; ++q)
        if (offs[q] <= i && i < offs[q + 1]) {
            e = q;
            break;
        }
    if (e < 0)
        return -1;
    const int key = (s >= 0 && s < p.L) ? s + 1 : 0;
    return e * (p.L + 1) + key;
}

// Every global read the kernel needs is issued up front (the first 1024
// slots, the expert offsets, the slot tables); later passes work from
// registers and shared memory.
__global__ void __launch_bounds__(PREP_THREADS, 1) prep_kernel(Params p)
{
    extern __shared__ int4 prep_smem4[];
    int *sm = reinterpret_cast<int *>(prep_smem4);
    const int nb = p.E * (p.L + 1);
    int *cnt = sm;                                            // [nb] rows per bucket (pass 1)
    int *base = sm + nb;                                      // [nb] next free position
    int *brank = sm + 2 * nb;                                 // [nb] rank of an active slot's bucket, else 0
    int *ccnt = sm + 3 * nb;                                  // [nb] rows per bucket in this chunk
    uint16_t *wc = reinterpret_cast<uint16_t *>(sm + 4 * nb); // [32][nb]
    __shared__ int offs[MAX_E + 1];
    __shared__ int warp_tot[33];
    __shared__ int etiles[MAX_E + 1];
    __shared__ uint32_t flags;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    // Launched early (programmatic dependent launch) behind whatever the
    // stream ran before; nothing is read until that work is complete, and only
    // then may the projection kernel launch.
    grid_dependency_wait();
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int slot0 = tid < p.rows ? p.seq_slot[tid] : -1;
    if (tid == 0)
        flags = 0;
    if (tid <= p.E)
        offs[tid] = p.expert_offsets ? p.expert_offsets[tid] : (tid == 0 ? 0 : p.rows);
    for (int b = tid; b < nb; b += PREP_THREADS) {
        cnt[b] = 0;
        const int e = b / (p.L + 1), key = b % (p.L + 1);
        int rk = 0;
        if (key > 0) {
            const Tables &t = p.tab[e];
            const int s = key - 1;
            const int r = t.rank_table[s];
            const bool active = t.a_table[s] != nullptr && t.b_table[s] != nullptr &&
                                t.scale_table[s] != 0.0f && r > 0;
            rk = active ? r : 0;
        }
        brank[b] = rk;
        p.ws.done[b] = 0;
    }
    for (int q = tid; q < p.stc_tiles; q += PREP_THREADS)
        p.ws.stile[q] = 0;
    for (int q = tid; q < p.ncnt; q += PREP_THREADS)
        p.ws.tile_cnt[q] = 0;
    __syncthreads();
    if (tid == 0) {
        bool ok = offs[0] >= 0 && offs[p.E] <= p.rows;
        for (int q = 0; q < p.E; ++q)
            ok = ok && offs[q] <= offs[q + 1];
        if (!ok)
            atomicOr(&flags, (uint32_t)LORA_FLAG_BAD_OFFSETS); // pass 1 may already be setting bits
    }

    // Pass 1: bucket sizes.
    for (int i = tid; i < p.rows; i += PREP_THREADS) {
        const int s = i < PREP_THREADS ? slot0 : p.seq_slot[i];
        const int b = bucket_of(p, offs, i, s);
        if (b >= 0) {
            atomicAdd(&cnt[b], 1);
            if (s >= p.L)
                atomicOr(&flags, (uint32_t)LORA_FLAG_SLOT_RANGE);
        }
    }
    __syncthreads();
    {
        int v = tid < nb ? cnt[tid] : 0, total;
        int ex = block_exclusive_scan(v, warp_tot, total);
        if (tid < nb) {
            base[tid] = ex;
            p.ws.seg_off[tid] = ex;
        }
        if (tid == 0)
            p.ws.seg_off[nb] = total;
    }
    // Shrink work list from the bucket sizes (shared memory only).
    {
        int units = 0;
        if (tid < nb && brank[tid] > 0 && cnt[tid] > 0 && !p.no_units)
            units = bucket_units(brank[tid], cnt[tid], p.kp);
        int total;
        int ex = block_exclusive_scan(units, warp_tot, total);
        if (tid < nb)
            p.ws.unit_off[tid] = ex;
        if (tid == 0)
            p.ws.unit_off[nb] = total;
    }
    __syncthreads();

    // Pass 2: stable placement, 1024 rows at a time in input order. Inside a
    // chunk, a row's position among equal keys = (rows of earlier warps with
    // that key) + (earlier lanes of its own warp with that key).
    for (int c0 = 0; c0 < p.rows; c0 += PREP_THREADS) {
        for (int q = tid; q < 32 * nb; q += PREP_THREADS)
            wc[q] = 0;
        __syncthreads();
        const int i = c0 + tid;
        const int s = c0 == 0 ? slot0 : (i < p.rows ? p.seq_slot[i] : -1);
        const int b = i < p.rows ? bucket_of(p, offs, i, s) : -1;
        const unsigned peers = __match_any_sync(0xffffffffu, b);
        const int rank_in_warp = __popc(peers & ((1u << lane) - 1u));
        if (b >= 0 && rank_in_warp == 0)
            wc[warp * nb + b] = (uint16_t)__popc(peers);
        __syncthreads();
        for (int bb = tid; bb < nb; bb += PREP_THREADS) {
            int run = 0;
            for (int w = 0; w < 32; ++w) {
                const int v = wc[w * nb + bb];
                wc[w * nb + bb] = (uint16_t)run;
                run += v;
            }
            ccnt[bb] = run;
        }
        __syncthreads();
        if (b >= 0)
            p.ws.perm[base[b] + wc[warp * nb + b] + rank_in_warp] = i;
        __syncthreads();
        for (int bb = tid; bb < nb; bb += PREP_THREADS)
            base[bb] += ccnt[bb];
        __syncthreads();
    }

    // Token tiles: each expert segment cut into tiles of at most tn rows,
    // expert by expert (thread e counts expert e's tiles; a scan places them).
    const int tn = p.tn > 0 ? p.tn : 256;
    const int cap = p.max_tiles > 0 ? min(p.max_tiles, max_token_tiles(p.rows, nb)) : max_token_tiles(p.rows, nb);
    if (tid < p.E) {
        const int a = max(offs[tid], 0), b = min(offs[tid + 1], p.rows);
        etiles[tid + 1] = b > a ? (b - a + tn - 1) / tn : 0;
    }
    __syncthreads();
    if (tid == 0) {
        etiles[0] = 0;
        for (int e = 0; e < p.E; ++e)
            etiles[e + 1] += etiles[e];
        p.ws.tiles[0] = min(etiles[p.E], cap);
        status_begin(p.ws.status, flags);
    }
    __syncthreads();
    if (tid < p.E) {
        const int a = max(offs[tid], 0), b = min(offs[tid + 1], p.rows);
        int k = etiles[tid];
        for (int r0 = a; r0 < b && k < cap; r0 += tn, ++k) {
            p.ws.tiles[1 + 3 * k] = tid;
            p.ws.tiles[2 + 3 * k] = r0;
            p.ws.tiles[3 + 3 * k] = min(tn, b - r0);
        }
    }
}

__global__ void __launch_bounds__(SHRINK_WARPS * 32) shrink_kernel(Params p)
{
    __shared__ float red[SHRINK_WARPS * 32];
    const int total = p.ws.unit_off[p.E * (p.L + 1)];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int u = blockIdx.x; u < total; u += gridDim.x) {
        const UnitMeta m = unit_meta(p, u, p.ws.unit_off, p.ws.seg_off);
        shrink_unit(p, m, warp, lane, red, 1);
        if (threadIdx.x == 0)
            shrink_unit_done(p, m.b);
    }
}

cudaError_t launch_prep(const Params &p, cudaStream_t st)
{
    const int nb = p.E * (p.L + 1);
    const size_t smem = (size_t)nb * 16 + (size_t)32 * nb * 2;
    static std::atomic<uint64_t> raised{0};
    cudaError_t ea = raise_smem_limit(raised, prep_kernel, (int)((size_t)MAX_BUCKETS * 16 + (size_t)32 * MAX_BUCKETS * 2));
    if (ea != cudaSuccess)
        return ea;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1);
    cfg.blockDim = dim3(PREP_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, prep_kernel, p);
}

cudaError_t launch_shrink(const Params &p, int num_sms, cudaStream_t st)
{
    shrink_kernel<<<4 * num_sms, SHRINK_WARPS * 32, 0, st>>>(p);
    return cudaGetLastError();
}

// ------------------------------------------------------------- table writes
__global__ void table_set_kernel(const void **a_table, const void **b_table, float *scale_table,
                                 float *factor_table, int32_t *rank_table, int slot, const void *a,
                                 const void *b, int rank, float factor, float scale)
{
    a_table[slot] = a;
    b_table[slot] = b;
    rank_table[slot] = rank;
    factor_table[slot] = factor;
    scale_table[slot] = scale;
}

__global__ void scale_set_kernel(float *scale_table, const float *factor_table, int slot,
                                 float adapter_scale)
{
    scale_table[slot] = adapter_scale * factor_table[slot];
}

cudaError_t launch_table_set(const lora_route &rt, int slot, const void *a, const void *b, int rank,
                             float factor, float scale, cudaStream_t st)
{
    table_set_kernel<<<1, 1, 0, st>>>(rt.a_table, rt.b_table, rt.scale_table, rt.factor_table,
                                      rt.rank_table, slot, a, b, rank, factor, scale);
    return cudaGetLastError();
}

// scale_table[first + i] = s[i] * factor_table[first + i] for i < count.
__global__ void scales_set_kernel(float *scale_table, const float *factor_table, ScaleChunk c)
{
    const int i = threadIdx.x;
    if (i < c.count)
        scale_table[c.first + i] = c.s[i] * factor_table[c.first + i];
}

cudaError_t launch_scales_set(const lora_route &rt, const ScaleChunk &c, cudaStream_t st)
{
    scales_set_kernel<<<1, SCALE_CHUNK, 0, st>>>(rt.scale_table, rt.factor_table, c);
    return cudaGetLastError();
}

// At[e][k] = A[k][e] for k < rank, e < n (rows of At are R apart; the rest of
// the slot was zeroed before). 32 x 32 tiles through shared memory, so both
// the reads and the writes are row runs.
__global__ void transpose_pack_kernel(uint16_t *At, int R, const uint16_t *A, int rank, int n)
{
    __shared__ uint16_t tile[32][33];
    const int e0 = blockIdx.x * 32, k0 = blockIdx.y * 32;
    for (int r = threadIdx.y; r < 32; r += 8) {
        const int k = k0 + r, e = e0 + threadIdx.x;
        if (k < rank && e < n)
            tile[r][threadIdx.x] = A[(size_t)k * n + e];
    }
    __syncthreads();
    for (int r = threadIdx.y; r < 32; r += 8) {
        const int e = e0 + r, k = k0 + threadIdx.x;
        if (e < n && k < rank)
            At[(size_t)e * R + k] = tile[threadIdx.x][r];
    }
}

cudaError_t launch_transpose_pack(uint16_t *At, int R, const uint16_t *A, int rank, int n, cudaStream_t st)
{
    transpose_pack_kernel<<<dim3((unsigned)((n + 31) / 32), (unsigned)((rank + 31) / 32)), dim3(32, 8), 0, st>>>(
        At, R, A, rank, n);
    return cudaGetLastError();
}

__global__ void comp_set_kernel(float *comp_row, CompRow row)
{
    comp_row[threadIdx.x] = row.v[threadIdx.x];
}

cudaError_t launch_comp_set(const lora_route &rt, int slot, const CompRow &row, cudaStream_t st)
{
    comp_set_kernel<<<1, LORA_COMP_STRIDE, 0, st>>>(rt.comp_table + (size_t)slot * LORA_COMP_STRIDE, row);
    return cudaGetLastError();
}

cudaError_t launch_scale_set(const lora_route &rt, int slot, float adapter_scale, cudaStream_t st)
{
    scale_set_kernel<<<1, 1, 0, st>>>(rt.scale_table, rt.factor_table, slot, adapter_scale);
    return cudaGetLastError();
}

} // namespace rd
