// Tensor-core path of the LoRA projection (tcgen05 / TMEM / TMA, sm_103a).
//
// The base product is computed transposed: each CTA owns 128 output features
// n (the UMMA M dimension) and a tile of TN rows of x (the UMMA N dimension),
//   D[n, t] = sum_k W[n, k] x[t, k],
// so that a decode batch of 64..256 rows is one UMMA N extent and W -- the
// bytes that bound the decode shapes -- streams through shared memory once.
// Both operands are K-major in global memory (W [N][K], x [rows][K]) and are
// staged by TMA with the 128-byte swizzle in 64-element K slices; one
// elected thread issues the UMMAs (M=128, N=TN, K=16, bf16 in, f32 out) into
// a TMEM accumulator; a multi-stage mbarrier pipeline keeps TMA and UMMA
// overlapped.
//
// Epilogue (all four warps, warp w reading TMEM lanes 32w..32w+31): the
// expand-fold y = base + s * (B_s[n, :] . h_t) for adapted rows, the base
// alone -- byte for byte -- for the others, then one round-to-nearest-even to
// bf16 (spark_model `layers/ops/lora_delta.rs`: the fold fused with the base
// instead of a separate scaled-add pass over an [m, n_out] scratch).
//
// MoE: blockIdx.z is the expert; its token tiles start at expert_offsets[e]
// and W comes from that expert's tensor map (spark_model `lora_delta.rs`,
// `LoraKernels`, grouped down_proj keyed on expert_offsets).
//
// Every wait is bounded; on a timeout the CTA flags LORA_FLAG_WAIT_TIMEOUT,
// stops issuing, waits (bounded) for its own copies in flight, frees TMEM
// and returns.
#include "lora_internal.cuh"
#include "ptx.cuh"
#include "vec.cuh"

namespace rd {

constexpr int TC_BM = 128;      // output features per CTA (UMMA M)
constexpr int TC_BK = 64;       // K per pipeline stage (one 128-byte swizzle row)
constexpr int TC_THREADS = 128; // 4 warps: TMA producer, UMMA issuer, then all four drain TMEM

template <int TN>
struct TcCfg {
    static constexpr int W_BYTES = TC_BM * TC_BK * 2;
    static constexpr int X_BYTES = TN * TC_BK * 2;
    static constexpr int STAGE_BYTES = W_BYTES + X_BYTES;
    static constexpr int STAGES = TN == 64 ? 8 : (TN == 128 ? 6 : 4);
    static constexpr int TMEM_COLS = TN < 32 ? 32 : TN;
    static constexpr int CTRL_BYTES = 1024; // barriers, TMEM address, flags
    static constexpr size_t SMEM =
        1024 + (size_t)STAGES * STAGE_BYTES + CTRL_BYTES + (size_t)TN * sizeof(SlotInfo);
};

__device__ __forceinline__ uint8_t *align1024(uint8_t *p)
{
    uintptr_t a = reinterpret_cast<uintptr_t>(p);
    return reinterpret_cast<uint8_t *>((a + 1023) & ~uintptr_t(1023));
}

template <int TN>
__global__ void __launch_bounds__(TC_THREADS, 1)
    tc_kernel(const __grid_constant__ TmapSet maps, const __grid_constant__ Params p)
{
    using C = TcCfg<TN>;
    extern __shared__ uint8_t tc_smem_raw[];
    uint8_t *smem = align1024(tc_smem_raw);
    uint8_t *tiles = smem;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::STAGES * C::STAGE_BYTES);
    uint64_t *empty = full + C::STAGES;
    uint64_t *done = empty + C::STAGES;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(done + 1);
    int *abort_flag = reinterpret_cast<int *>(tmem_slot + 1);
    SlotInfo *sinfo = reinterpret_cast<SlotInfo *>(smem + C::STAGES * C::STAGE_BYTES + C::CTRL_BYTES);

    const int e = blockIdx.z;
    int s0 = 0, s1 = p.rows;
    if (p.expert_offsets) {
        s0 = max(p.expert_offsets[e], 0);
        s1 = min(p.expert_offsets[e + 1], p.rows);
    }
    const int t0 = s0 + (int)blockIdx.y * TN;
    if (t0 >= s1)
        return; // uniform: nothing of this expert in this tile
    const int n0 = blockIdx.x * TC_BM;
    const int nkb = (p.K + TC_BK - 1) / TC_BK;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < C::STAGES; ++i) {
            mbar_init(full + i, 1);
            mbar_init(empty + i, 1);
        }
        mbar_init(done, 1);
        *abort_flag = 0;
        fence_barrier_init();
        fence_proxy_async_smem();
        prefetch_tmap(&maps.x);
        prefetch_tmap(&maps.w[e]);
    }
    if (warp == 0)
        tmem_alloc(tmem_slot, C::TMEM_COLS);
    for (int j = threadIdx.x; j < TN; j += TC_THREADS) {
        const int t = t0 + j;
        SlotInfo si{nullptr, 0.0f, 0, 0};
        if (t < s1)
            si = slot_info(p.tab[e], p.seq_slot[t], p.L);
        sinfo[j] = si;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0 && lane == 0) {
        // ---- TMA producer
        int last_parity[C::STAGES];
        for (int i = 0; i < C::STAGES; ++i)
            last_parity[i] = -1;
        for (int kb = 0; kb < nkb; ++kb) {
            const int st = kb % C::STAGES;
            const uint32_t ph = (uint32_t)(kb / C::STAGES) & 1u;
            if (*(volatile int *)abort_flag || !mbar_wait(empty + st, ph ^ 1u)) {
                *(volatile int *)abort_flag = 1;
                break;
            }
            uint8_t *dst = tiles + st * C::STAGE_BYTES;
            mbar_arrive_expect_tx(full + st, C::STAGE_BYTES);
            tma_load_2d(dst, &maps.w[e], kb * TC_BK, n0, full + st);
            tma_load_2d(dst + C::W_BYTES, &maps.x, kb * TC_BK, t0, full + st);
            last_parity[st] = (int)ph;
        }
        if (*(volatile int *)abort_flag) {
            // let our own copies land before the CTA's shared memory goes away
            for (int i = 0; i < C::STAGES; ++i)
                if (last_parity[i] >= 0)
                    mbar_wait(full + i, (uint32_t)last_parity[i]);
        }
    } else if (warp == 1 && lane == 0) {
        // ---- UMMA issuer
        const uint32_t idesc = idesc_bf16_f32(TC_BM, TN);
        for (int kb = 0; kb < nkb; ++kb) {
            const int st = kb % C::STAGES;
            const uint32_t ph = (uint32_t)(kb / C::STAGES) & 1u;
            if (*(volatile int *)abort_flag || !mbar_wait(full + st, ph)) {
                *(volatile int *)abort_flag = 1;
                break;
            }
            tc_fence_after();
            const uint32_t a = smem_u32(tiles + st * C::STAGE_BYTES);
            const uint32_t b = a + C::W_BYTES;
#pragma unroll
            for (int j = 0; j < TC_BK / 16; ++j)
                umma_bf16(tmem, sw128_kmajor_desc(a + j * 32), sw128_kmajor_desc(b + j * 32), idesc,
                          (kb | j) != 0 ? 1u : 0u);
            umma_commit(empty + st);
        }
        umma_commit(done); // always: arrives once every issued UMMA has finished
    }
    __syncwarp();

    // ---- epilogue
    bool ok = mbar_wait(done, 0);
    tc_fence_after();
    ok = __syncthreads_and(ok && !*(volatile int *)abort_flag) != 0;
    if (!ok) {
        if (threadIdx.x == 0)
            atomicOr(p.ws.status, (uint32_t)LORA_FLAG_WAIT_TIMEOUT);
    } else {
        const int n = n0 + warp * 32 + lane;
        const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);
        const bool n_ok = n < p.N;
        for (int c = 0; c < TN; c += 16) {
            float v[16];
            tmem_ld16(trow + (uint32_t)c, v);
#pragma unroll 4
            for (int j = 0; j < 16; ++j) {
                const int jj = c + j;
                const int t = t0 + jj;
                if (t >= s1 || !n_ok)
                    continue;
                float out = v[j];
                const SlotInfo si = sinfo[jj];
                if (si.on) {
                    const uint16_t *brow = si.b + (size_t)n * p.R;
                    const float *hrow = p.ws.h + (size_t)t * p.R;
                    float d = 0.0f;
                    for (int q = 0; q < si.rank; q += 8) {
                        const float4 h0 = *reinterpret_cast<const float4 *>(hrow + q);
                        const float4 h1 = *reinterpret_cast<const float4 *>(hrow + q + 4);
                        d = dot8_bf_f32(d, ld_nc_16(brow + q), h0, h1);
                    }
                    out = out + si.scale * d;
                }
                p.y[(int64_t)t * p.y_stride + n] = f32_to_bf16_bits(out);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

template <int TN>
static cudaError_t launch_tc_t(const Params &p, const TmapSet &maps, cudaStream_t st)
{
    using C = TcCfg<TN>;
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(tc_kernel<TN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)C::SMEM);
        if (e != cudaSuccess)
            return e;
        attr_set = true;
    }
    dim3 grid((p.N + TC_BM - 1) / TC_BM, (p.rows + TN - 1) / TN, p.E);
    tc_kernel<TN><<<grid, TC_THREADS, C::SMEM, st>>>(maps, p);
    return cudaGetLastError();
}

cudaError_t launch_tc(const Params &p, const TmapSet &maps, int token_tile, cudaStream_t st)
{
    switch (token_tile) {
    case 64: return launch_tc_t<64>(p, maps, st);
    case 128: return launch_tc_t<128>(p, maps, st);
    default: return launch_tc_t<256>(p, maps, st);
    }
}

} // namespace rd
