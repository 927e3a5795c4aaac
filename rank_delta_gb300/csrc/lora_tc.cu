// Tensor-core path of the LoRA projection (tcgen05 / TMEM / TMA, sm_103a).
//
// The base product is computed transposed, D[n, t] = sum_k W[n, k] x[t, k]:
// a CTA owns 128 output features n (UMMA M) and a token tile of up to 256
// rows of x (UMMA N), so a decode batch is one UMMA N extent and W -- the
// bytes that bound these shapes -- streams through shared memory once.
//
// Work: items = (token tile, 128-feature tile, K part), spread over a grid
// that never exceeds the SMs (every CTA resident). With csplit K parts, each
// part writes its fp32 partial tile to the workspace (coalesced, L2-resident)
// and bumps the tile's counter; once all parts are in, each part's CTA sums a
// contiguous third (quarter) of the columns in part order -- so every output
// element is computed the same way whatever N is. With csplit = 1 the CTA
// keeps two TMEM accumulators, draining one while the next tile accumulates.
//
// Warp roles (256 threads):
//   warps 0, 1   TMA producers of W (even / odd pipeline stages): 3D boxes
//                [kc chunks][128 rows][64] so one copy brings kc K-slices;
//   warp  2      allocates TMEM and issues the UMMAs (M=128, N=tokens, K=16,
//                bf16 in, f32 accumulate) from one elected thread;
//   warp  3      TMA producer of x;
//   warps 4..7   first run their share of the shrink work units (h = A_s x,
//                shrink.cuh), then drain TMEM (warp w reads TMEM lanes
//                32(w-4)..+31) and apply the expand-fold s * (B_s[n, :] . h_t)
//                to the rows of the slots this K part owns (slot % csplit), the
//                B rows of those slots staged in shared memory while the
//                mainloop runs; rows with no delta get nothing added. The sum
//                is rounded once to bf16 (spark_model `layers/ops/lora_delta.rs`:
//                the fold fused with the base product instead of a scaled-add
//                pass over an [m, n_out] scratch).
// The shrink is handed over inside the launch: a unit bumps its bucket's
// counter after writing h; the epilogue waits (bounded) for the counters of
// the buckets its tokens use. The grid never exceeds the SM count (one CTA
// per SM), so every unit and every K part runs while others wait.
//
// The kernel starts before the routing/prep kernel has finished (programmatic
// dependent launch); only the roles that read its results wait for it.
//
// MoE (spark_model `lora_delta.rs`, `LoraKernels`: the down_proj fold keyed on
// expert_offsets): token tiles come from the prep kernel's per-expert list and
// W from that expert's tensor map.
//
// Every wait is bounded; on a timeout the CTA records LORA_FLAG_WAIT_TIMEOUT,
// stops issuing work, lets its own copies land, frees TMEM and exits.
#include "lora_internal.cuh"
#include "ptx.cuh"
#include "shrink.cuh"
#include "vec.cuh"

namespace rd {

constexpr int TC_BM = 128;
constexpr int TC_THREADS = 256;
constexpr int EPI_THREADS = 128;
constexpr int MAX_TN = 256;
constexpr int MAX_STAGES = 8;
constexpr uint32_t W_CHUNK_BYTES = TC_BM * 64 * 2;

struct TcCfg {
    int tn, kc, stages, csplit;
    int n_tiles;      // ceil(N / 128)
    int static_tiles; // total tiles when the host knows them, -1 when the prep kernel lists them
    int kchunks, kstages;
    int use3d;
    int sb;           // B slices (one slot x 128 rows each) the expand keeps in shared memory
    uint32_t x_chunk, stage_bytes;
    uint32_t brow;    // bytes per staged B row (R * 2 + 16: padded against bank conflicts)
    uint32_t s_off, aux_off, b_off, h_off, meta_off, x_off, bar_off, smem_bytes;
    uint32_t tmem_cols;
};

// Per-tile bookkeeping of the epilogue warps (shared memory at aux_off).
struct EpiAux {
    int16_t hidx[MAX_TN];    // row of the staged h for column j, or -1
    int16_t entry[MAX_TN];   // staged B slice of column j's slot, or -1
    int32_t slot_entry_n;    // staged B slices in use
    int32_t slot_of_entry[64];
    int32_t n_h;             // staged h rows in use
    int32_t eslot[1024];     // staged B slice of slot s (-1 none yet, -2 claimed, -3 no room)
};

struct Bars {
    uint64_t full[MAX_STAGES];
    uint64_t empty[MAX_STAGES];
    uint64_t acc_full[2];
    uint64_t acc_empty[2];
    uint64_t epi_done; // every epilogue thread has finished reading TMEM
    uint32_t tmem_base;
    int abort_flag;
};

struct TileInfo {
    int e, r0, cnt, n0;
};

__device__ __forceinline__ uint8_t *align1024(uint8_t *ptr)
{
    uintptr_t a = reinterpret_cast<uintptr_t>(ptr);
    return reinterpret_cast<uint8_t *>((a + 1023) & ~uintptr_t(1023));
}

// Work items: tile * csplit + K part.
__device__ __forceinline__ int item_total(const Params &p, const TcCfg &c)
{
    return (c.static_tiles >= 0 ? c.static_tiles : p.ws.tiles[0] * c.n_tiles) * c.csplit;
}

__device__ __forceinline__ bool get_tile(const Params &p, const TcCfg &c, int tile, int total, TileInfo &ti)
{
    if (tile >= total)
        return false;
    const int tt = tile / c.n_tiles, nt = tile % c.n_tiles;
    ti.n0 = nt * TC_BM;
    if (c.static_tiles >= 0) {
        ti.e = 0;
        ti.r0 = tt * c.tn;
        ti.cnt = min(c.tn, p.rows - ti.r0);
    } else {
        ti.e = p.ws.tiles[1 + 3 * tt];
        ti.r0 = p.ws.tiles[2 + 3 * tt];
        ti.cnt = p.ws.tiles[3 + 3 * tt];
    }
    return true;
}

__device__ __forceinline__ void flag_abort(const Params &p, Bars *bars)
{
    *(volatile int *)&bars->abort_flag = 1;
    atomicOr(p.ws.status, (uint32_t)LORA_FLAG_WAIT_TIMEOUT);
}

__device__ __forceinline__ bool aborted(Bars *bars) { return *(volatile int *)&bars->abort_flag != 0; }

// TMA producer of W (par = 0 / 1: even / odd pipeline stages) or of x (par = -1).
__device__ __forceinline__ void produce(const TmapSet &maps, const Params &p, const TcCfg &c, Bars *bars,
                                        uint8_t *smem, int par)
{
    const bool is_x = par < 0;
    if (c.static_tiles < 0)
        grid_dependency_wait();
    const int total = item_total(p, c);
    int last_parity[MAX_STAGES];
    for (int i = 0; i < MAX_STAGES; ++i)
        last_parity[i] = -1;
    int g = 0;
    TileInfo ti;
    for (int w = blockIdx.x; w < total && get_tile(p, c, w / c.csplit, total, ti); w += gridDim.x) {
        const int part = w % c.csplit;
        const int ks0 = part * c.kstages / c.csplit, ks1 = (part + 1) * c.kstages / c.csplit;
        for (int ks = ks0; ks < ks1; ++ks, ++g) {
            if (!is_x && (g & 1) != par)
                continue;
            const int slot = g % c.stages;
            const uint32_t ph = (uint32_t)(g / c.stages) & 1u;
            if (aborted(bars) || !mbar_wait(bars->empty + slot, ph ^ 1u)) {
                flag_abort(p, bars);
                goto drain;
            }
            uint8_t *stage = smem + (size_t)slot * c.stage_bytes;
            if (is_x) {
                mbar_arrive_expect_tx(bars->full + slot, (uint32_t)c.kc * c.x_chunk);
                uint8_t *dst = stage + (size_t)c.kc * W_CHUNK_BYTES;
                if (c.use3d)
                    tma_load_3d(dst, &maps.x, 0, ti.r0, ks * c.kc, bars->full + slot);
                else
                    tma_load_2d(dst, &maps.x, ks * 64, ti.r0, bars->full + slot);
            } else {
                mbar_arrive_expect_tx(bars->full + slot, (uint32_t)c.kc * W_CHUNK_BYTES);
                if (c.use3d)
                    tma_load_3d(stage, &maps.w[ti.e], 0, ti.n0, ks * c.kc, bars->full + slot);
                else
                    tma_load_2d(stage, &maps.w[ti.e], ks * 64, ti.n0, bars->full + slot);
            }
            last_parity[slot] = (int)ph;
        }
    }
    return;
drain:
    // let this thread's copies land before the CTA's shared memory goes away
    for (int i = 0; i < c.stages; ++i)
        if (last_parity[i] >= 0)
            mbar_wait(bars->full + i, (uint32_t)last_parity[i]);
}

__device__ __forceinline__ void issue_mma(const Params &p, const TcCfg &c, Bars *bars, uint8_t *smem,
                                          uint32_t tmem)
{
    if (c.static_tiles < 0)
        grid_dependency_wait();
    const int total = item_total(p, c);
    int g = 0, it = 0;
    TileInfo ti;
    for (int w = blockIdx.x; w < total && get_tile(p, c, w / c.csplit, total, ti); w += gridDim.x, ++it) {
        const int part = w % c.csplit;
        const int ks0 = part * c.kstages / c.csplit, ks1 = (part + 1) * c.kstages / c.csplit;
        const int buf = it & 1;
        const uint32_t use = (uint32_t)(it >> 1);
        if (aborted(bars) || !mbar_wait(bars->acc_empty + buf, (use & 1u) ^ 1u)) {
            flag_abort(p, bars);
            break;
        }
        tc_fence_after();
        const uint32_t acc = tmem + (uint32_t)(buf * c.tn);
        const int nmma = (ti.cnt + 15) & ~15;
        const uint32_t idesc = idesc_bf16_f32(TC_BM, (uint32_t)nmma);
        uint32_t accumulate = 0;
        bool ok = true;
        for (int ks = ks0; ks < ks1; ++ks, ++g) {
            const int slot = g % c.stages;
            const uint32_t ph = (uint32_t)(g / c.stages) & 1u;
            if (aborted(bars) || !mbar_wait(bars->full + slot, ph)) {
                flag_abort(p, bars);
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t wb = smem_u32(smem + (size_t)slot * c.stage_bytes);
            const uint32_t xb = wb + (uint32_t)c.kc * W_CHUNK_BYTES;
            for (int q = 0; q < c.kc; ++q) {
                if (ks * c.kc + q >= c.kchunks)
                    break;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    umma_bf16(acc, sw128_kmajor_desc(wb + q * W_CHUNK_BYTES + j * 32),
                              sw128_kmajor_desc(xb + q * c.x_chunk + j * 32), idesc, accumulate);
                    accumulate = 1;
                }
            }
            umma_commit(bars->empty + slot);
        }
        umma_commit(bars->acc_full + buf); // arrives once every UMMA above has finished
        if (!ok)
            break;
    }
}

// Deltas s * (B_s[n, :] . h_t) of four columns at once (so the loads of the
// four are in flight together), h_t staged (row k of Hs), B_s[n, :] staged
// (slice e of Bs) or, when the slot did not fit, read from the pool. Column
// i takes part when on[i]; d[i] receives its delta.
__device__ __forceinline__ void lora_delta4(const Params &p, const TcCfg &c, const SlotInfo *const (&si)[4],
                                            const uint8_t *Bs, const float *Hs, const int (&e)[4],
                                            const int (&k)[4], const bool (&on)[4], int et, int n,
                                            float (&d)[4])
{
    int rk[4], rmax = 0;
    const float *hrow[4];
    const uint8_t *bst[4];
    const uint16_t *bgl[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        d[i] = 0.0f;
        rk[i] = on[i] ? si[i]->rank : 0;
        rmax = max(rmax, rk[i]);
        hrow[i] = Hs + (size_t)(on[i] ? k[i] : 0) * p.R;
        bst[i] = Bs + ((size_t)(e[i] >= 0 ? e[i] : 0) * TC_BM + et) * c.brow;
        bgl[i] = on[i] ? si[i]->b + (size_t)n * p.R : nullptr;
    }
#pragma unroll 2
    for (int q = 0; q < rmax; q += 8) {
        uint4 bv[4];
        float4 h0[4], h1[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const bool use = q < rk[i];
            bv[i] = !use ? make_uint4(0, 0, 0, 0)
                         : (e[i] >= 0 ? *reinterpret_cast<const uint4 *>(bst[i] + q * 2) : ld_nc_16(bgl[i] + q));
            h0[i] = use ? *reinterpret_cast<const float4 *>(hrow[i] + q) : make_float4(0, 0, 0, 0);
            h1[i] = use ? *reinterpret_cast<const float4 *>(hrow[i] + q + 4) : make_float4(0, 0, 0, 0);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
            d[i] = dot8_bf_f32(d[i], bv[i], h0[i], h1[i]);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
        d[i] *= on[i] ? si[i]->scale : 0.0f;
}

__device__ __forceinline__ bool wait_count(const int32_t *cnt, int target)
{
    if (ld_acquire_gpu(cnt) >= target)
        return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        if (ld_acquire_gpu(cnt) >= target)
            return true;
        if (globaltimer_ns() - t0 > WAIT_NS)
            return false;
    }
}

// Per item: which columns get their delta here (adapted rows whose slot is
// this K part's: slot % csplit), stage those slots' B rows and the summed h
// of those columns in shared memory, then add the deltas to this part's
// accumulator; with csplit > 1 write the partial tile and, once every part
// is in, sum this part's share of the columns in part order.
__device__ __forceinline__ void epilogue(const Params &p, const TcCfg &c, Bars *bars, uint8_t *smem,
                                         uint32_t tmem)
{
    const int et = threadIdx.x - (TC_THREADS - EPI_THREADS); // TMEM lane 0..127
    const int ew = et >> 5, lane = et & 31;
    SlotInfo *sinfo = reinterpret_cast<SlotInfo *>(smem + c.s_off);
    EpiAux *aux = reinterpret_cast<EpiAux *>(smem + c.aux_off);
    uint8_t *Bs = smem + c.b_off;
    float *Hs = reinterpret_cast<float *>(smem + c.h_off);
    const int C = c.csplit;
    const int nb = p.E * (p.L + 1);
    int32_t *unit_off = reinterpret_cast<int32_t *>(smem + c.meta_off); // copies of the routing
    int32_t *seg_off = unit_off + nb + 1;                                 // results, in shared memory

    grid_dependency_wait();
    for (int q = et; q <= nb; q += EPI_THREADS) {
        unit_off[q] = p.ws.unit_off[q];
        seg_off[q] = p.ws.seg_off[q];
    }
    named_bar_sync(1, EPI_THREADS);
    // this CTA's share of the shrink work units; one fence publishes them all
    const int total_units = unit_off[nb];
    float *scratch = reinterpret_cast<float *>(smem + c.x_off); // [16][128] fp32
    for (int u = blockIdx.x; u < total_units; u += gridDim.x)
        shrink_unit(p, locate_unit(p, u, unit_off, seg_off), ew, lane, scratch, 1);
    if (blockIdx.x < total_units) {
        __threadfence();
        named_bar_sync(1, EPI_THREADS);
        for (int u = blockIdx.x + et * gridDim.x; u < total_units; u += EPI_THREADS * gridDim.x)
            atomicAdd(p.ws.done + locate_unit(p, u, unit_off, seg_off).b, 1);
    }

    const int total = item_total(p, c);
    int it = 0;
    TileInfo ti;
    for (int w = blockIdx.x; w < total && get_tile(p, c, w / c.csplit, total, ti); w += gridDim.x, ++it) {
        const int tile = w / c.csplit, part = w % c.csplit;
        const int buf = it & 1;
        const uint32_t use = (uint32_t)(it >> 1);
        const int n = ti.n0 + ew * 32 + lane;
        const Tables &tab = p.tab[ti.e];

        // (1) slot of every column; staged-h row and staged B slice of the
        // columns whose delta this part adds
        if (et == 0) {
            aux->slot_entry_n = 0;
            aux->n_h = 0;
        }
        for (int q = et; q < p.L; q += EPI_THREADS)
            aux->eslot[q] = -1;
        named_bar_sync(1, EPI_THREADS);
        for (int j = et; j < ti.cnt; j += EPI_THREADS) {
            const int sl = p.seq_slot[ti.r0 + j];
            const SlotInfo si = slot_info(tab, sl, p.L);
            sinfo[j] = si;
            aux->hidx[j] = -1;
            if (si.on && sl % C == part) {
                aux->hidx[j] = (int16_t)atomicAdd(&aux->n_h, 1);
                if (atomicCAS(&aux->eslot[sl], -1, -2) == -1) {
                    const int e = atomicAdd(&aux->slot_entry_n, 1);
                    if (e < c.sb) {
                        aux->slot_of_entry[e] = sl;
                        aux->eslot[sl] = e;
                    } else {
                        aux->eslot[sl] = -3;
                    }
                }
            }
        }
        named_bar_sync(1, EPI_THREADS);
        for (int j = et; j < ti.cnt; j += EPI_THREADS) {
            int e = -1;
            if (aux->hidx[j] >= 0) {
                e = aux->eslot[p.seq_slot[ti.r0 + j]];
                e = e >= 0 ? e : -1;
            }
            aux->entry[j] = (int16_t)e;
        }
        // (2) B rows of the staged slots: thread et copies row n0 + et of each
        const int nent = min(aux->slot_entry_n, c.sb);
        for (int e = 0; e < nent; ++e) {
            const int sl = aux->slot_of_entry[e];
            const int rk = tab.rank_table[sl];
            const uint16_t *src = tab.b_table[sl] + (size_t)n * p.R;
            uint8_t *dst = Bs + ((size_t)e * TC_BM + et) * c.brow;
#pragma unroll 4
            for (int q = 0; q < rk; q += 8)
                *reinterpret_cast<uint4 *>(dst + q * 2) = n < p.N ? ld_nc_16(src + q) : make_uint4(0, 0, 0, 0);
        }
        // (3) wait for the shrink of those columns, stage their h
        for (int j = et; j < ti.cnt; j += EPI_THREADS) {
            if (aux->hidx[j] < 0)
                continue;
            const int b = ti.e * (p.L + 1) + p.seq_slot[ti.r0 + j] + 1;
            if (!wait_bucket(p, b, unit_off))
                flag_abort(p, bars);
        }
        named_bar_sync(1, EPI_THREADS);
        const int rv = p.R / 8;
        for (int idx = et; idx < ti.cnt * rv; idx += EPI_THREADS) {
            const int j = idx / rv, q = (idx % rv) * 8;
            const int k = aux->hidx[j];
            if (k < 0 || q >= sinfo[j].rank)
                continue;
            float4 a, b2;
            h_sum8(p, ti.r0 + j, q, a, b2);
            float *dst = Hs + (size_t)k * p.R + q;
            *reinterpret_cast<float4 *>(dst) = a;
            *reinterpret_cast<float4 *>(dst + 4) = b2;
        }
        // (4) accumulator of this item
        const bool got = mbar_wait(bars->acc_full + buf, use & 1u);
        tc_fence_after();
        if (!got)
            flag_abort(p, bars);
        named_bar_sync(1, EPI_THREADS);
        if (aborted(bars))
            break;
        const uint32_t tl = tmem + (uint32_t)(buf * c.tn) + ((uint32_t)(ew * 32) << 16);
        float *my_part = p.ws.part + ((size_t)tile * C + part) * (size_t)c.tn * EPI_THREADS;
        uint32_t raw[16];
        tmem_ld16_nowait(tl, raw);
        for (int c0 = 0; c0 < ti.cnt; c0 += 16) {
            tmem_wait_ld();
            float v[16];
#pragma unroll
            for (int j = 0; j < 16; ++j)
                v[j] = __uint_as_float(raw[j]);
            if (c0 + 16 < ti.cnt) // next chunk's accumulator load overlaps this chunk's work
                tmem_ld16_nowait(tl + (uint32_t)(c0 + 16), raw);
            bool any = false;
#pragma unroll
            for (int j = 0; j < 16; ++j)
                any |= c0 + j < ti.cnt && aux->hidx[c0 + j] >= 0;
            if (any && n < p.N) { // columns to adapt: deltas four at a time, values via scratch
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    scratch[j * EPI_THREADS + et] = v[j];
#pragma unroll 1
                for (int j4 = 0; j4 < 16; j4 += 4) {
                    const SlotInfo *si[4];
                    int e[4], k[4];
                    bool on[4], any4 = false;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int col = c0 + j4 + i;
                        k[i] = col < ti.cnt ? aux->hidx[col] : -1;
                        on[i] = k[i] >= 0;
                        any4 |= on[i];
                        e[i] = on[i] ? aux->entry[col] : -1;
                        si[i] = sinfo + (col < ti.cnt ? col : 0);
                    }
                    if (!any4)
                        continue;
                    float d[4];
                    lora_delta4(p, c, si, Bs, Hs, e, k, on, et, n, d);
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        if (on[i])
                            scratch[(j4 + i) * EPI_THREADS + et] += d[i];
                }
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    v[j] = scratch[j * EPI_THREADS + et];
            }
            if (C == 1) {
                if (n < p.N) {
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        if (c0 + j < ti.cnt)
                            p.y[(int64_t)(ti.r0 + c0 + j) * p.y_stride + n] = f32_to_bf16_bits(v[j]);
                }
            } else {
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    if (c0 + j < ti.cnt)
                        my_part[(size_t)(c0 + j) * EPI_THREADS + et] = v[j];
            }
        }
        tc_fence_before();
        if (C > 1)
            __threadfence();
        named_bar_sync(1, EPI_THREADS);
        if (et == 0) {
            mbar_arrive(bars->acc_empty + buf);
            if (C > 1)
                atomicAdd(p.ws.tile_cnt + tile, 1);
        }
        if (C > 1) {
            // every part of the tile written: sum this part's share of the columns
            if (et == 0 && !wait_count(p.ws.tile_cnt + tile, C))
                flag_abort(p, bars);
            named_bar_sync(1, EPI_THREADS);
            if (aborted(bars))
                break;
            const float *parts = p.ws.part + (size_t)tile * C * c.tn * EPI_THREADS;
            const size_t pstride = (size_t)c.tn * EPI_THREADS;
            const int cb = part * ti.cnt / C, ce = (part + 1) * ti.cnt / C;
            for (int col = cb; col < ce; col += 16) {
                float acc[16][4];
#pragma unroll
                for (int jj = 0; jj < 16; ++jj)
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        if (q < C && col + jj < ce)
                            acc[jj][q] = __ldcg(parts + q * pstride + (size_t)(col + jj) * EPI_THREADS + et);
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) {
                    if (col + jj >= ce || n >= p.N)
                        continue;
                    float y = acc[jj][0];
#pragma unroll
                    for (int q = 1; q < 4; ++q)
                        if (q < C)
                            y += acc[jj][q];
                    p.y[(int64_t)(ti.r0 + col + jj) * p.y_stride + n] = f32_to_bf16_bits(y);
                }
            }
        }
        named_bar_sync(1, EPI_THREADS); // staged rows are rewritten by the next item
    }
}

__global__ void __launch_bounds__(TC_THREADS, 1)
    tc_kernel(const __grid_constant__ TmapSet maps, const __grid_constant__ Params p,
              const __grid_constant__ TcCfg c)
{
    extern __shared__ uint8_t tc_smem_raw[];
    uint8_t *smem = align1024(tc_smem_raw);
    Bars *bars = reinterpret_cast<Bars *>(smem + c.bar_off);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < c.stages; ++i) {
            mbar_init(bars->full + i, 2); // the W copy and the x copy of a stage
            mbar_init(bars->empty + i, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bars->acc_full + b, 1);
            mbar_init(bars->acc_empty + b, 1);
        }
        mbar_init(&bars->epi_done, EPI_THREADS);
        bars->abort_flag = 0;
        fence_barrier_init();
        fence_proxy_async_smem();
        prefetch_tmap(&maps.x);
        for (int e = 0; e < p.E; ++e)
            prefetch_tmap(&maps.w[e]);
    }
    if (warp == 2)
        tmem_alloc(&bars->tmem_base, c.tmem_cols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;

    if (warp < 2) {
        if (lane == 0)
            produce(maps, p, c, bars, smem, warp);
    } else if (warp == 3) {
        if (lane == 0)
            produce(maps, p, c, bars, smem, -1);
    } else if (warp == 2) {
        if (lane == 0)
            issue_mma(p, c, bars, smem, tmem);
    } else {
        epilogue(p, c, bars, smem, tmem);
        tc_fence_before();
        mbar_arrive(&bars->epi_done);
    }
    __syncwarp();
    if (warp == 2) {
        // TMEM is freed only once the epilogue warps are done reading it
        mbar_wait(&bars->epi_done, 0);
        tc_fence_after();
        tmem_dealloc(tmem, c.tmem_cols);
    }
    __syncthreads();
}

// ----------------------------------------------------------------- host side

static uint32_t pow2_at_least(uint32_t v)
{
    uint32_t r = 32;
    while (r < v)
        r <<= 1;
    return r;
}

static uint32_t align_up(uint32_t v, uint32_t a) { return (v + a - 1) / a * a; }

// Bytes per staged B row: R bf16, plus 16 when the row length is a multiple
// of 64 bytes (rows that would otherwise put a warp's 16-byte reads in the
// same shared-memory banks).
static uint32_t staged_brow(int R)
{
    const uint32_t b = (uint32_t)R * 2u;
    return (b % 64u) == 0 ? b + 16u : b;
}

// Shared-memory layout of one launch for a given plan.
static TcCfg make_cfg(const Params &p, const TcPlan &plan, bool dyn)
{
    TcCfg c;
    memset(&c, 0, sizeof c);
    c.tn = plan.tn;
    c.kc = plan.kc;
    c.csplit = plan.csplit;
    c.use3d = plan.use3d;
    c.sb = plan.sb;
    c.n_tiles = (p.N + TC_BM - 1) / TC_BM;
    c.kchunks = (p.K + 63) / 64;
    c.kstages = (c.kchunks + c.kc - 1) / c.kc;
    c.x_chunk = (uint32_t)c.tn * 128u;
    c.stage_bytes = (uint32_t)c.kc * (W_CHUNK_BYTES + c.x_chunk);
    c.stages = plan.stages;
    c.brow = staged_brow(p.R);
    uint32_t o = (uint32_t)c.stages * c.stage_bytes;
    c.s_off = align_up(o, 16);
    o = c.s_off + (uint32_t)(c.tn * sizeof(SlotInfo));
    c.aux_off = align_up(o, 16);
    o = c.aux_off + (uint32_t)sizeof(EpiAux);
    c.b_off = align_up(o, 16);
    o = c.b_off + (uint32_t)c.sb * TC_BM * c.brow;
    c.h_off = align_up(o, 16);
    o = c.h_off + (uint32_t)c.tn * (uint32_t)p.R * 4u;
    c.meta_off = align_up(o, 16);
    o = c.meta_off + 2u * (uint32_t)(p.E * (p.L + 1) + 1) * 4u;
    c.x_off = align_up(o, 16);
    o = c.x_off + 16u * EPI_THREADS * 4u;
    c.bar_off = align_up(o, 16);
    c.smem_bytes = 1024u + c.bar_off + (uint32_t)sizeof(Bars);
    c.tmem_cols = pow2_at_least(2u * (uint32_t)c.tn);
    const int tt = (p.rows + c.tn - 1) / c.tn;
    c.static_tiles = dyn ? -1 : tt * c.n_tiles;
    return c;
}

static constexpr uint32_t SMEM_LIMIT = 232448; // 227 KB per CTA

// Choose K chunks per stage, stages, reduction width and staged B slices:
// keep at least 3 stages for tiles of 128+ rows (2 for the small decode
// tile), then give the rest of shared memory to the B rows of the slots this
// CTA finishes (up to every such slot).
TcPlan plan_tc(const Params &p, bool dyn)
{
    TcPlan plan;
    memset(&plan, 0, sizeof plan);
    plan.tn = p.tn;
    plan.use3d = (p.K % 64) == 0 ? 1 : 0;
    const int kchunks = (p.K + 63) / 64;
    plan.csplit = tc_csplit(p.rows, p.K, dyn);
    const int need_sb = min(64, min(p.tn, (p.L + plan.csplit - 1) / plan.csplit));
    const int min_stages = p.tn <= 64 ? 2 : 3;
    int best = -1;
    TcPlan cand = plan;
    const int kcs[3] = {4, 2, 1};
    {
        for (int ik = 0; ik < 3; ++ik) {
            const int kc = kcs[ik];
            if (kc > 1 && !plan.use3d)
                continue;
            if ((kchunks + kc - 1) / kc < plan.csplit)
                continue;
            for (int st = MAX_STAGES; st >= 2; --st) {
                cand.kc = kc;
                cand.stages = st;
                cand.sb = 0;
                const TcCfg c0 = make_cfg(p, cand, dyn);
                if (c0.smem_bytes > SMEM_LIMIT)
                    continue;
                const uint32_t slice = (uint32_t)TC_BM * staged_brow(p.R);
                cand.sb = (int)min((uint32_t)need_sb, (SMEM_LIMIT - c0.smem_bytes) / slice);
                const int score = (st >= min_stages ? 100000 : 0) + (cand.sb >= need_sb ? 10000 : 0) +
                                  cand.sb * 100 + min(st, 4) * 10 + kc * 2;
                if (score > best) {
                    best = score;
                    plan = cand;
                }
            }
        }
    }
    if (best < 0) {
        plan.kc = 1;
        plan.stages = 2;
        plan.sb = 0;
    }
    return plan;
}

cudaError_t launch_tc(const Params &p, const TmapSet &maps, const TcPlan &plan, cudaStream_t st)
{
    const bool dyn = p.expert_offsets != nullptr;
    const TcCfg c = make_cfg(p, plan, dyn);
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)SMEM_LIMIT);
        if (e != cudaSuccess)
            return e;
        attr_set = true;
    }
    if (c.smem_bytes > SMEM_LIMIT)
        return cudaErrorInvalidConfiguration;
    // One CTA per SM at most, so every CTA is resident (the in-launch waits
    // rely on it); never more CTAs than work items.
    static int sms_cache[64];
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64)
        return cudaErrorInvalidDevice;
    if (sms_cache[dev] == 0) {
        int sms = 0;
        cudaError_t e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess)
            return e;
        sms_cache[dev] = sms;
    }
    int grid = sms_cache[dev];
    if (c.static_tiles >= 0 && c.static_tiles * c.csplit < grid)
        grid = c.static_tiles * c.csplit;
    grid = grid / c.csplit * c.csplit;

    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(TC_THREADS);
    cfg.dynamicSmemBytes = c.smem_bytes;
    cfg.stream = st;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, tc_kernel, maps, p, c);
}

} // namespace rd
