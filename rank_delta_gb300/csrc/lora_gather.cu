// Decode-path MoE fold keyed on the expert through a per-slot-row index
// (spark_model `lora_delta.rs`, `LoraKernels`: the moe_gather shrink /
// expand-fold, the unsorted slot-major analogue of the expert_offsets fold),
// with the top-k combine weights.
//
// The slot-rows arrive in token order, each naming its expert. Around the
// grouped fold (lora_moe_down_apply) two kernels:
//   gather_sort_kernel   every CTA sorts the slot-rows by expert (stable
//                        counting sort, rows past the E experts last); CTA 0
//                        publishes the order, its inverse, the expert offsets
//                        and the sorted slots; each CTA copies its share of x
//                        rows into expert order (16-byte vectors).
//   gather_combine_kernel y[t] = sum_i w[t*k+i] * v[inv[t*k+i]] in fp32 with one
//                        rounding (or, without weights, y[j] = v[inv[j]]
//                        byte for byte); a slot-row whose index is outside
//                        [0, E) contributes nothing and sets
//                        LORA_FLAG_EXPERT_RANGE.
#include "lora_internal.cuh"

namespace rd {

namespace {

constexpr int GS_THREADS = 256;

__device__ __forceinline__ int bucket_of_expert(int e, int E) { return (e >= 0 && e < E) ? e : E; }

// Stable counting sort of T slot-rows by expert into sperm (shared memory);
// thread t owns rows [t*RT, (t+1)*RT) and counts them in its own column of
// cnt[E+1][256]. Returns through seg[0..E+1] the bucket starts.
__device__ void sort_by_expert(const GatherParams &p, uint16_t *cnt, int *seg, int32_t *sperm)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nb = p.E + 1;
    const int RT = (p.T + GS_THREADS - 1) / GS_THREADS;
    for (int q = tid; q < nb * GS_THREADS; q += GS_THREADS)
        cnt[q] = 0;
    __syncthreads();
    for (int k = 0; k < RT; ++k) {
        const int j = tid * RT + k;
        if (j < p.T)
            ++cnt[bucket_of_expert(p.indices[j], p.E) * GS_THREADS + tid];
    }
    __syncthreads();
    __shared__ int tot[LORA_MAX_EXPERTS + 1];
    for (int b = warp; b < nb; b += GS_THREADS / 32) { // counts of bucket b -> exclusive starts
        uint16_t *row = cnt + b * GS_THREADS + lane * 8;
        int v[8], sum = 0;
#pragma unroll
        for (int h = 0; h < 8; ++h) {
            v[h] = row[h];
            sum += v[h];
        }
        int incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t2 = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o)
                incl += t2;
        }
        int run = incl - sum;
#pragma unroll
        for (int h = 0; h < 8; ++h) {
            row[h] = (uint16_t)run;
            run += v[h];
        }
        if (lane == 31)
            tot[b] = incl;
    }
    __syncthreads();
    if (tid == 0) {
        int run = 0;
        for (int b = 0; b < nb; ++b) {
            seg[b] = run;
            run += tot[b];
        }
        seg[nb] = run;
    }
    __syncthreads();
    for (int k = 0; k < RT; ++k) {
        const int j = tid * RT + k;
        if (j < p.T) {
            const int b = bucket_of_expert(p.indices[j], p.E);
            uint16_t &c = cnt[b * GS_THREADS + tid];
            sperm[seg[b] + c] = j;
            c = (uint16_t)(c + 1);
        }
    }
    __syncthreads();
}

__global__ void __launch_bounds__(GS_THREADS) gather_sort_kernel(GatherParams p)
{
    extern __shared__ int4 gs_smem4[];
    int32_t *sperm = reinterpret_cast<int32_t *>(gs_smem4);                      // [T]
    uint16_t *cnt = reinterpret_cast<uint16_t *>(sperm + ((p.T + 3) & ~3));      // [E+1][256]
    __shared__ int seg[LORA_MAX_EXPERTS + 2];
    sort_by_expert(p, cnt, seg, sperm);
    if (blockIdx.x == 0) {
        for (int q = threadIdx.x; q < p.T; q += GS_THREADS) {
            const int j = sperm[q];
            p.perm[q] = j;
            p.inv[j] = q;
            p.slots_sorted[q] = p.seq_slot[j];
        }
        if (threadIdx.x <= p.E)
            p.offsets[threadIdx.x] = seg[threadIdx.x];
    }
    // rows of the E experts into expert order, one row per CTA at a time
    const int valid = seg[p.E];
    const int chunks = p.K >> 3;
    for (int q = blockIdx.x; q < valid; q += gridDim.x) {
        const uint4 *src = reinterpret_cast<const uint4 *>(p.x + (size_t)sperm[q] * p.x_stride);
        uint4 *dst = reinterpret_cast<uint4 *>(p.x_sorted + (size_t)q * p.K);
        for (int c = threadIdx.x; c < chunks; c += GS_THREADS)
            dst[c] = src[c];
    }
}

__device__ __forceinline__ float lo_f(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float hi_f(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ uint32_t pack2(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// One output row per CTA step; eight columns per thread and step when the
// shapes allow 16-byte access, else one.
template <bool VEC>
__global__ void __launch_bounds__(GS_THREADS) gather_combine_kernel(GatherParams p)
{
    const int valid = p.offsets[p.E]; // sorted positions past this are rows of no expert
    const int rows_out = p.combine ? p.T / p.top_k : p.T;
    const int per = p.combine ? p.top_k : 1;
    const int step = VEC ? 8 : 1;
    bool bad = false;
    for (int r = blockIdx.x; r < rows_out; r += gridDim.x) {
        uint16_t *yr = p.y + (size_t)r * p.y_stride;
        for (int n = threadIdx.x * step; n < p.N; n += GS_THREADS * step) {
            float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            uint4 raw = make_uint4(0u, 0u, 0u, 0u);
            uint16_t raw1 = 0;
            for (int i = 0; i < per; ++i) {
                const int j = r * per + i;
                const int q = p.inv[j];
                if (q >= valid) {
                    bad = true;
                    continue;
                }
                const uint16_t *v = p.y_sorted + (size_t)q * p.N + n;
                if (!p.combine) { // a copy of the slot-row, bit for bit
                    if (VEC)
                        raw = *reinterpret_cast<const uint4 *>(v);
                    else
                        raw1 = *v;
                    continue;
                }
                const float w = p.combine[j];
                if (VEC) {
                    const uint4 u = *reinterpret_cast<const uint4 *>(v);
                    const uint32_t e[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        acc[2 * h] += w * lo_f(e[h]);
                        acc[2 * h + 1] += w * hi_f(e[h]);
                    }
                } else {
                    acc[0] += w * __uint_as_float((uint32_t)*v << 16);
                }
            }
            if (VEC) {
                if (p.combine)
                    raw = make_uint4(pack2(acc[0], acc[1]), pack2(acc[2], acc[3]), pack2(acc[4], acc[5]),
                                     pack2(acc[6], acc[7]));
                *reinterpret_cast<uint4 *>(yr + n) = raw;
            } else {
                yr[n] = p.combine ? (uint16_t)(pack2(acc[0], 0.f) & 0xffffu) : raw1;
            }
        }
    }
    if (bad)
        atomicOr(p.status, (uint32_t)LORA_FLAG_EXPERT_RANGE);
}

} // namespace

size_t gather_sort_smem(int T, int E) { return (size_t)((T + 3) & ~3) * 4 + (size_t)(E + 1) * GS_THREADS * 2; }

cudaError_t launch_gather_sort(const GatherParams &p, int num_sms, cudaStream_t st)
{
    const size_t smem = gather_sort_smem(p.T, p.E);
    static std::atomic<uint64_t> raised{0};
    cudaError_t ea = raise_smem_limit(raised, gather_sort_kernel, (int)gather_sort_smem(LORA_GATHER_MAX_ROWS, LORA_MAX_EXPERTS));
    if (ea != cudaSuccess)
        return ea;
    int grid = p.T < 2 * num_sms ? p.T : 2 * num_sms;
    if (grid < 1)
        grid = 1;
    gather_sort_kernel<<<grid, GS_THREADS, smem, st>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_gather_combine(const GatherParams &p, int num_sms, cudaStream_t st)
{
    const int rows_out = p.combine ? p.T / p.top_k : p.T;
    int grid = rows_out < 4 * num_sms ? rows_out : 4 * num_sms;
    if (grid < 1)
        grid = 1;
    const bool vec = p.N % 8 == 0 && p.y_stride % 8 == 0 && (reinterpret_cast<uintptr_t>(p.y) & 15u) == 0;
    if (vec)
        gather_combine_kernel<true><<<grid, GS_THREADS, 0, st>>>(p);
    else
        gather_combine_kernel<false><<<grid, GS_THREADS, 0, st>>>(p);
    return cudaGetLastError();
}

} // namespace rd
