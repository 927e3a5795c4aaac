// Tensor-core shrink h_t = A_{s_t} x_t for batches of many rows (ferrox-core
// `weight_matrix/lora.rs`, `LoraDelta::project`: the rank-sized projection of
// each row through its own adapter's A), run inside the projection launch.
//
// The work is cut into shrink tiles of 128 rows of x (UMMA M = 128: TMEM lane
// t is row t of the tile). The adapted slots present in a tile are stacked
// along UMMA N, Rs = max_rank rounded up to 16 columns each, up to 256 columns
// per group:
//   D[t, i*Rs + r] = sum_k x[t, k] A_{slot_i}[r, k]
// so a tile whose rows share one adapter (a prefill sequence) costs one
// 128 x Rs x K product. x tiles arrive by TMA, and so do the A rows when
// every slot of a group lies in the route's pool (one box of Rs rows per slot
// and K chunk, pad rows zero by the pack); otherwise they are copied with
// cp.async through the slot pointer table (a_table), into the same 128-byte
// swizzled K-major layout. The drain keeps, for row t, the Rs columns of its
// own slot and writes h[t][0..R) in fp32 and the expand's operand
// (s * comp[r]) * h rounded to bf16 -- with K unsplit, so h has one part.
//
// The projection kernel's CTAs run the shrink tiles before their projection
// items, the last CTAs first (CTA gridDim - 1 takes tile 0): when the items
// do not divide evenly over the CTAs, those are the ones with one item fewer.
// A finished tile is published by a counter in the workspace (ws.stile,
// cleared by the routing kernel); the projection epilogue waits for the
// counters of its rows before it stages s * h, long after they are set.
//
// Roles (warps 0..5 of the projection kernel's CTA; the other warps only join
// the CTA barriers): warp 0 issues the x copies, warp 1 issues the UMMAs into
// TMEM columns 0..255 of the CTA's allocation, warps 2..5 copy A rows and then
// drain TMEM (warp w reads lanes 32 (w % 4)..+31). Every wait is bounded
// (LORA_FLAG_WAIT_TIMEOUT).
#pragma once

#include "lora_internal.cuh"
#include "ptx.cuh"
#include "shrink.cuh"
#include "vec.cuh"

namespace rd {

constexpr int STC_M = 128;
constexpr int STC_THREADS = 192;  // the phase's threads: warps 0..5
constexpr int STC_LOADERS = 128;  // warps 2..5
constexpr int STC_MAX_N = 256;
constexpr int STC_MAX_STAGES = 4;
constexpr uint32_t STC_X_BYTES = STC_M * 128u;     // 128 rows x 64 bf16
constexpr uint32_t STC_A_BYTES = STC_MAX_N * 128u; // up to 256 A rows x 64 bf16
constexpr uint32_t STC_STAGE_BYTES = STC_X_BYTES + STC_A_BYTES;

struct StcShared {
    uint64_t full[STC_MAX_STAGES];
    uint64_t empty[STC_MAX_STAGES];
    uint64_t acc_full;
    uint64_t acc_empty;
    int abort_flag;
    int nslots;
    int16_t tslot[STC_M];     // slot of row t when it takes a delta, else -1
    int16_t slot_list[STC_M]; // the tile's adapted slots, ascending
    int16_t slot_rank[STC_M];
    const uint16_t *slot_a[STC_M];
    int32_t used[1024];       // per slot: row count in this tile, then its list index
    int32_t wsum[STC_THREADS / 32];
};

// Shared memory of the phase with `stages` stages, from a 1024-aligned base.
__host__ __device__ constexpr uint32_t stc_smem_bytes(int stages)
{
    return (uint32_t)stages * STC_STAGE_BYTES + (uint32_t)sizeof(StcShared);
}

// The shrink tiles' launch arguments (tensor maps of x in 128-row boxes and of
// the pool's A rows, the rank padded to 16, whether the A map may be used).
struct StcArgs {
    int tiles;  // shrink tiles of the launch (0: none)
    int Rs;     // max rank rounded up to 16
    int a_map;  // 1: amap covers the route's pool
    int stages; // pipeline stages (fit below the projection kernel's own state)
};

__device__ __forceinline__ void stc_abort(const Params &p, StcShared *sh)
{
    *(volatile int *)&sh->abort_flag = 1;
    atomicOr(p.ws.status, (uint32_t)LORA_FLAG_WAIT_TIMEOUT);
}

__device__ __forceinline__ bool stc_aborted(StcShared *sh) { return *(volatile int *)&sh->abort_flag != 0; }

// This CTA's shrink tiles. Called by every thread of the CTA (blockDim >=
// STC_THREADS); smem is 1024-aligned and free for stc_smem_bytes(a.stages)
// bytes; tmem is the CTA's TMEM allocation (at least 256 columns), free.
// Returns true when the CTA wrote its tiles' h (then stc_publish makes them
// visible); false when it has no tile, or a wait gave up (flagged).
__device__ bool stc_phase(const CUtensorMap &xmap, const CUtensorMap &amap, const Params &p, const StcArgs &a,
                          uint8_t *smem, uint32_t tmem)
{
    const int first = (int)gridDim.x - 1 - (int)blockIdx.x;
    if (first >= a.tiles)
        return false; // uniform over the CTA
    StcShared *sh = reinterpret_cast<StcShared *>(smem + (size_t)a.stages * STC_STAGE_BYTES);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int S = a.stages, Rs = a.Rs;
    const int G = STC_MAX_N / Rs; // slots per UMMA group
    const int kchunks = (p.K + 63) / 64;
    if (tid == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(sh->full + i, 1 + STC_LOADERS); // the x copy + every A loader
            mbar_init(sh->empty + i, 1);
        }
        mbar_init(&sh->acc_full, 1);
        mbar_init(&sh->acc_empty, STC_LOADERS);
        sh->abort_flag = 0;
        fence_barrier_init();
        prefetch_tmap(&xmap);
        if (a.a_map)
            prefetch_tmap(&amap);
    }
    __syncthreads();

    // pipeline positions, carried across groups and tiles by each role
    int gx = 0, gm = 0, ga = 0, groups_done = 0;
    for (int tile = first; tile < a.tiles; tile += gridDim.x) {
        const int r0 = tile * STC_M;
        // (1) the tile's adapted slots, ascending (the phase's threads)
        for (int s = tid; s < p.L && tid < STC_THREADS; s += STC_THREADS)
            sh->used[s] = 0;
        __syncthreads();
        if (tid < STC_M) {
            int sl = -1;
            if (r0 + tid < p.rows) {
                const int s = p.seq_slot[r0 + tid];
                const SlotInfo si = slot_info(p.tab[0], s, p.L);
                if (si.on) {
                    sl = s;
                    sh->used[s] = 1;
                }
            }
            sh->tslot[tid] = (int16_t)sl;
        }
        __syncthreads();
        {
            const int per = (p.L + STC_THREADS - 1) / STC_THREADS;
            const int s0 = tid < STC_THREADS ? min(p.L, tid * per) : p.L, s1 = min(p.L, s0 + per);
            int cnt = 0;
            for (int s = s0; s < s1; ++s)
                cnt += sh->used[s];
            int incl = cnt;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o)
                    incl += v;
            }
            if (lane == 31 && warp < STC_THREADS / 32)
                sh->wsum[warp] = incl;
            __syncthreads();
            int ex = incl - cnt, total = 0;
            for (int q = 0; q < STC_THREADS / 32; ++q) {
                if (q < warp)
                    ex += sh->wsum[q];
                total += sh->wsum[q];
            }
            for (int s = s0; s < s1; ++s)
                if (sh->used[s]) {
                    sh->slot_list[ex] = (int16_t)s;
                    sh->slot_a[ex] = p.tab[0].a_table[s];
                    sh->slot_rank[ex] = (int16_t)p.tab[0].rank_table[s];
                    sh->used[s] = ex;
                    ++ex;
                }
            if (tid == 0)
                sh->nslots = total;
        }
        __syncthreads();
        const int nslots = sh->nslots;
        const int ngroups = (nslots + G - 1) / G;

        for (int grp = 0; grp < ngroups; ++grp, ++groups_done) {
            const int gs = min(G, nslots - grp * G);
            const int N = gs * Rs;
            // A rows by TMA when every slot of the group lies in the pool
            bool a_tma = a.a_map != 0;
            for (int i = 0; i < gs && a_tma; ++i) {
                const int li = grp * G + i;
                a_tma = reinterpret_cast<const uint8_t *>(sh->slot_a[li]) ==
                        static_cast<const uint8_t *>(p.pool) + (size_t)sh->slot_list[li] * p.slot_bytes;
            }
            if (warp == 0) {
                if (lane == 0) { // x copies
                    for (int kc = 0; kc < kchunks; ++kc, ++gx) {
                        const int st = gx % S;
                        if (stc_aborted(sh) || !mbar_wait(sh->empty + st, ((uint32_t)(gx / S) & 1u) ^ 1u)) {
                            stc_abort(p, sh);
                            break;
                        }
                        uint8_t *xs = smem + (size_t)st * STC_STAGE_BYTES;
                        if (a_tma) {
                            // x and every slot's Rs A rows of the chunk on one arrival, and
                            // the loaders' arrivals given at once (they copy nothing)
                            mbar_arrive_expect_tx(sh->full + st, STC_X_BYTES + (uint32_t)N * 128u);
                            tma_load_2d(xs, &xmap, kc * 64, r0, sh->full + st);
                            for (int i = 0; i < gs; ++i)
                                tma_load_3d(xs + STC_X_BYTES + (size_t)i * Rs * 128, &amap, kc * 64, 0,
                                            sh->slot_list[grp * G + i], sh->full + st);
                            mbar_arrive_count(sh->full + st, STC_LOADERS);
                        } else {
                            mbar_arrive_expect_tx(sh->full + st, STC_X_BYTES);
                            tma_load_2d(xs, &xmap, kc * 64, r0, sh->full + st);
                        }
                    }
                }
            } else if (warp == 1) {
                if (lane == 0) { // UMMAs
                    const uint32_t idesc = idesc_bf16_f32(STC_M, (uint32_t)N);
                    bool ok = mbar_wait(&sh->acc_empty, ((uint32_t)groups_done & 1u) ^ 1u);
                    if (!ok)
                        stc_abort(p, sh);
                    tc_fence_after();
                    uint32_t acc = 0;
                    for (int kc = 0; ok && kc < kchunks; ++kc, ++gm) {
                        const int st = gm % S;
                        if (stc_aborted(sh) || !mbar_wait(sh->full + st, (uint32_t)(gm / S) & 1u)) {
                            stc_abort(p, sh);
                            break;
                        }
                        tc_fence_after();
                        const uint32_t xs = smem_u32(smem + (size_t)st * STC_STAGE_BYTES);
                        const uint32_t as = xs + STC_X_BYTES;
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            umma_bf16(tmem, sw128_kmajor_desc(xs + j * 32), sw128_kmajor_desc(as + j * 32), idesc, acc);
                            acc = 1;
                        }
                        umma_commit(sh->empty + st);
                    }
                    umma_commit(&sh->acc_full);
                }
            } else if (warp < STC_THREADS / 32) {
                // A rows of the group's slots: row n = i * Rs + rr of the stage is
                // row rr of A of slot (grp * G + i); rows past the rank, and K past
                // the end, are zero-filled. Each stage's copies form one cp.async
                // group; a stage is signalled (after a proxy fence) once S - 1
                // later groups have been issued, so that many stages stay in flight.
                const int et = tid - 64;
                const int LAG = S - 1;
                const int ga0 = ga;
                int kc = a_tma ? kchunks : 0; // by TMA: nothing to copy here
                ga += kc;
                for (; kc < kchunks; ++kc, ++ga) {
                    const int st = ga % S;
                    if (stc_aborted(sh) || !mbar_wait(sh->empty + st, ((uint32_t)(ga / S) & 1u) ^ 1u)) {
                        stc_abort(p, sh);
                        break;
                    }
                    uint8_t *as = smem + (size_t)st * STC_STAGE_BYTES + STC_X_BYTES;
                    for (int idx = et; idx < N * 8; idx += STC_LOADERS) {
                        const int n = idx >> 3, c = idx & 7;
                        const int i = n / Rs, rr = n - i * Rs;
                        const int li = grp * G + i;
                        const int k = kc * 64 + c * 8;
                        const bool has = rr < sh->slot_rank[li] && k < p.K;
                        const uint16_t *src = sh->slot_a[li] + (has ? (size_t)rr * p.K + k : 0);
                        cp_async_16(as + n * 128 + ((c ^ (n & 7)) << 4), src, has ? 16u : 0u);
                    }
                    cp_async_commit();
                    if (kc >= LAG) {
                        // at most S - 1 younger groups pending: the one LAG back has landed
                        if (LAG >= 3)
                            cp_async_wait_group<3>();
                        else if (LAG == 2)
                            cp_async_wait_group<2>();
                        else
                            cp_async_wait_group<1>();
                        fence_proxy_async_smem(); // generic-proxy copies, read by the UMMAs
                        mbar_arrive(sh->full + (ga - LAG) % S);
                    }
                }
                // the last (up to LAG) stages issued
                cp_async_wait_all();
                fence_proxy_async_smem();
                if (!a_tma)
                    for (int q = max(0, kc - LAG); q < kc; ++q)
                        mbar_arrive(sh->full + (ga0 + q) % S);
                // drain: row t keeps the columns of its own slot
                const bool got = mbar_wait(&sh->acc_full, (uint32_t)groups_done & 1u);
                tc_fence_after();
                if (!got)
                    stc_abort(p, sh);
                const int t = 32 * (warp & 3) + lane;
                const uint32_t taddr = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
                const int sl = sh->tslot[t];
                const int li = sl >= 0 ? sh->used[sl] : -1;
                const int i = li - grp * G; // this row's slot block in the group, if any
                const int rank = li >= 0 ? sh->slot_rank[li] : 0;
                float *hrow = p.ws.h + (size_t)(r0 + t) * p.R;
                // the expand's bf16 operand (s * comp[r]) * h, rounded as the
                // epilogue would round it from h
                uint16_t *hsrow = p.ws.hs + (size_t)(r0 + t) * p.R;
                const float sc = sl >= 0 ? p.tab[0].scale_table[sl] : 0.0f;
                const float *crow = p.tab[0].comp_table + (size_t)(sl >= 0 ? sl : 0) * LORA_COMP_STRIDE;
                const bool skip = __any_sync(0xffffffffu, stc_aborted(sh)); // warp-uniform: the loads are collective
                for (int c0 = 0; c0 < N && !skip; c0 += 16) {
                    float v[16];
                    tmem_ld16(taddr + (uint32_t)c0, v);
                    const int r = c0 - i * Rs; // rank of column c0 for this row's slot
                    if (i >= 0 && i < gs && r >= 0 && r < Rs && r0 + t < p.rows) {
#pragma unroll
                        for (int q = 0; q < 16; q += 4)
                            if (r + q < p.R)
                                *reinterpret_cast<float4 *>(hrow + r + q) =
                                    make_float4(r + q + 0 < rank ? v[q + 0] : 0.0f, r + q + 1 < rank ? v[q + 1] : 0.0f,
                                                r + q + 2 < rank ? v[q + 2] : 0.0f, r + q + 3 < rank ? v[q + 3] : 0.0f);
#pragma unroll
                        for (int q = 0; q < 16; q += 8)
                            if (r + q < p.R) {
                                uint32_t w[4];
#pragma unroll
                                for (int e = 0; e < 8; e += 2) {
                                    const float a0 = r + q + e < rank ? v[q + e] : 0.0f;
                                    const float b0 = r + q + e + 1 < rank ? v[q + e + 1] : 0.0f;
                                    w[e / 2] = (uint32_t)f32_to_bf16_bits(a0 * (sc * crow[r + q + e])) |
                                               ((uint32_t)f32_to_bf16_bits(b0 * (sc * crow[r + q + e + 1])) << 16);
                                }
                                *reinterpret_cast<uint4 *>(hsrow + r + q) = make_uint4(w[0], w[1], w[2], w[3]);
                            }
                    }
                }
                __threadfence(); // this row's h and s * h, before the tile's counter
                tc_fence_before();
                mbar_arrive(&sh->acc_empty);
            }
        }
        __syncthreads(); // the tile's h rows are written; its slot lists are rewritten by the next tile
    }
    // every copy has landed and every UMMA has been drained: the stages and
    // TMEM go back to the projection
    tc_fence_before();
    __syncthreads();
    const bool ok = !stc_aborted(sh);
    if (tid == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_inval(sh->full + i);
            mbar_inval(sh->empty + i);
        }
        mbar_inval(&sh->acc_full);
        mbar_inval(&sh->acc_empty);
    }
    __syncthreads();
    tc_fence_after();
    return ok;
}

// Publish this CTA's shrink tiles (one thread, after stc_phase returned true):
// the routing kernel clears the counters, so this waits for it to complete --
// off the CTA's critical path, on a warp the projection items leave idle.
__device__ __forceinline__ void stc_publish(const Params &p, const StcArgs &a)
{
    grid_dependency_wait();
    for (int tile = (int)gridDim.x - 1 - (int)blockIdx.x; tile < a.tiles; tile += gridDim.x)
        atomicAdd(p.ws.stile + tile, 1);
}

// Wait until shrink tile t has been published (its counter reaches target,
// 1 but under the test hook); false after wait_ns.
__device__ __forceinline__ bool stc_wait_tile(const Params &p, int t, int target, uint64_t wait_ns)
{
    const int32_t *cnt = p.ws.stile + t;
    if (ld_acquire_gpu(cnt) >= target)
        return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        if (ld_acquire_gpu(cnt) >= target)
            return true;
        if (globaltimer_ns() - t0 > wait_ns)
            return false;
    }
}

} // namespace rd
