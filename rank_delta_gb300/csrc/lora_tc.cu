// Tensor-core path of the LoRA projection (tcgen05 / TMEM / TMA, sm_103a).
//
// The base product is computed transposed, D[n, t] = sum_k W[n, k] x[t, k]:
// a CTA owns 128 output features n (UMMA M) and a token tile of up to 256
// rows of x (UMMA N), so a decode batch is one UMMA N extent and W -- the
// bytes that bound these shapes -- streams through shared memory once.
//
// Work: items = (token tile, 128-feature tile, K part), spread over a grid
// that never exceeds the SMs (every CTA resident); several token tiles are
// walked in groups of 16 per feature tile so a wave shares W tiles in L2.
// With csplit K parts, each part writes its fp32 partial tile to the
// workspace (coalesced, L2-resident) and bumps the tile's counter; once all
// parts are in, each part's CTA sums a contiguous share of the columns in
// part order -- so every output element is computed the same way whatever N
// is. With one part, y leaves in 64-row bf16 boxes staged in the free XH
// buffers and written by TMA stores. Two TMEM accumulators let the epilogue
// drain one item while the next accumulates.
//
// The expand-fold runs on the tensor cores too. Each adapted slot of a tile
// is owned by one K part (slots sorted by padded rank, largest first, dealt
// to the parts in snake order). For the slots an item owns, the
// epilogue warps stage in shared memory, in the same 128-byte swizzled
// K-major layout TMA writes:
//   XB[n, k]  the B rows n0..n0+127 of those slots, concatenated along k (each
//             slot's rank padded to 16, slots in ascending order),
//   XH[t, k]  s_t * h_t placed in its slot's k range, zero elsewhere (bf16;
//             with two planes, hi + lo, so that h keeps 16 significant bits),
// and the MMA warp issues D'[n, t] = sum_k XB[n, k] XH[t, k] (UMMA M=128,
// N=tokens, K=16 per instruction). D' goes to its own TMEM columns and the
// epilogue adds it only to the columns that take a delta, so a row with no
// delta is the base product byte for byte. D' has TMEM columns of its own
// when three token tiles fit in the 512 columns. Otherwise (tiles of more
// than 170 rows): when every row of the tile takes its delta here, D'
// accumulates straight into the base accumulator; else it borrows the other
// accumulator and the next item waits for this one's drain. When the staged
// k range exceeds the buffers, the expand runs in several rounds.
//
// Warp roles (256 threads):
//   warp  0      TMA producer of W and x (3D boxes [kc chunks][128 rows][64],
//                so one copy brings kc K-slices);
//   warp  1      allocates TMEM and issues the UMMAs from one elected thread;
//   warps 2, 3   one-tile launches: run this CTA's shrink work units (h = A_s x,
//                shrink.cuh, two warps per unit) once the epilogue has sorted
//                the rows, while the epilogue goes on;
//   warps 4..7   (other launches: first run their share of the shrink units),
//                then per item stage the expand operands and
//                drain TMEM (warp w reads TMEM lanes 32(w-4)..+31), rounding
//                once to bf16 (spark_model `layers/ops/lora_delta.rs`: the fold
//                fused with the base product instead of a scaled-add pass over
//                an [m, n_out] scratch).
// The shrink is handed over inside the launch: a unit bumps its bucket's
// counter after writing h; the epilogue waits (bounded) for the counters of
// the slots it stages. From 2048 rows the shrink runs on the tensor cores in
// tiles of 128 rows (shrink_tc.cuh), as the first work of the CTAs that have
// one item fewer; a tile bumps its own counter once h and s * h are written,
// and the epilogue waits for the tiles of its rows. The grid never exceeds
// the SM count (one CTA per SM) and launches with such waits are
// cooperative, so every unit, tile and K part runs while others wait (a grid
// that cannot be resident at once fails to launch).
//
// The kernel starts before the routing/prep kernel has finished (programmatic
// dependent launch); only the roles that read its results wait for it.
//
// MoE (spark_model `lora_delta.rs`, `LoraKernels`: the down_proj fold keyed on
// expert_offsets): token tiles come from the prep kernel's per-expert list and
// W from that expert's tensor map; tiles of at least 128 rows run as pairs of
// adjacent feature tiles (two W boxes per x box, one K loop into both
// accumulators).
//
// Every wait is bounded; on a timeout the CTA records LORA_FLAG_WAIT_TIMEOUT,
// stops issuing work, lets its own copies land, frees TMEM and exits.
#include "lora_internal.cuh"
#include "ptx.cuh"
#include "shrink.cuh"
#include "shrink_tc.cuh"
#include "vec.cuh"

namespace rd {

constexpr int TC_BM = 128;
constexpr int TC_THREADS = 256;
constexpr int EPI_THREADS = 128;
constexpr int MAX_TN = 256;
constexpr int MAX_STAGES = 8;
constexpr uint32_t W_CHUNK_BYTES = TC_BM * 64 * 2;
constexpr uint32_t XB_BLOCK = TC_BM * 128; // 64 k of 128 B rows, 128 rows
constexpr int LR_MAX_L = 64;               // slots a launch may have for local routing
constexpr int TC_TGROUP = 16;              // token tiles per group of the grouped tile order

struct TcCfg {
    int tn, kc, stages, csplit;
    int n_tiles;      // ceil(N / 128)
    int static_tiles; // total tiles when the host knows them, -1 when the prep kernel lists them
    int tgroup;       // token tiles walked together per feature tile (L2 reuse of W), 1 = row-major
    int kchunks, kstages;
    int use3d;
    int xblk;         // 64-wide k blocks of one expand round (dedicated buffers, region 0)
    int xblk_b;       // k blocks that fit in the pipeline stages (region 1, a CTA's last item)
    int hl;           // XH planes: 1 (bf16) or 2 (hi + lo)
    int borrow;       // 1: no room for D' beside two accumulators; D' borrows the other one
    int local_route;  // 1: one token tile holds every row; each CTA sorts them itself for the shrink
    int ystore;       // y boxes staged in the XH buffers: 0 = per-thread stores, else 1 or 2 buffers
    uint64_t wait_ns; // limit of the split-K and shrink-tile waits (the test hook shortens it)
    int extra_parts;  // test hook: parts (or tile publications) those waits also wait for, that never come
    uint32_t x_chunk, stage_bytes;
    int pair;         // 1: a CTA takes items in pairs (adjacent feature tiles of one token tile),
                      //    both W boxes and one x box per stage, one K loop into both accumulators
    uint32_t xb_off, xh_off, aux_off, meta_off, red_off, umeta_off, bar_off, smem_bytes;
    uint32_t tmem_cols;
    int stc_stages;   // pipeline stages of the launch's shrink tiles (below bar_off), 0: none
};

// Per-item state of the epilogue warps (shared memory at aux_off) and the
// expand round the MMA issuer reads. Offsets fit 16 bits: at most 256 slots
// per tile, ranks at most 256, so every k offset is below 65536.
struct EpiAux {
    int32_t koff[MAX_TN];            // k offset of column j's slot in the expand, -1: no delta here
    float cscale[MAX_TN];            // scale of column j's slot
    int16_t crank[MAX_TN];           // rank of column j's slot
    int16_t cslot[MAX_TN];           // column j's slot (per-rank factors)
    uint16_t soff[1024];             // per slot: padded rank if used (0 if not), then its k offset
    int8_t part_of[1024];            // per used slot: the K part that adds its delta
    int16_t entry_slot[MAX_TN];      // the expand's slots, ascending
    int32_t ent_off[MAX_TN];         // k offset of entry e
    int16_t ent_rank[MAX_TN];        // rank of entry e
    const uint16_t *ent_b[MAX_TN];   // B of entry e
    uint32_t onbits[MAX_TN / 32];    // bit j: column j takes its delta here
    int32_t wsum[2][4];              // scan scratch: per-warp totals
    // local routing (local_route): per slot s < L of the launch's one token tile
    int32_t lr_cnt[LR_MAX_L];        // adapted rows of slot s
    int16_t lr_rank[LR_MAX_L];
    int16_t lr_seg[LR_MAX_L];        // first position of slot s in lr_perm
    int16_t lr_run[LR_MAX_L];        // placement cursor
    int32_t lr_uoff[LR_MAX_L + 1];   // first shrink unit of slot s
    const uint16_t *lr_a[LR_MAX_L];
    const uint16_t *lr_b[LR_MAX_L];
    int16_t lr_wcnt[4][LR_MAX_L];    // rows of slot s in each warp's 32 (stable placement)
    int16_t lr_perm[MAX_TN];         // tile rows grouped by slot, in row order within a slot
    int32_t n_on;
    int32_t xr_mode[2];              // per staging region: 0 no expand, 1 into D', 2 into the base accumulator
    int32_t xr_nk16[2], xr_last[2];  // K=16 steps of the region's round; last round of the item
};

struct Bars {
    uint64_t full[MAX_STAGES];
    uint64_t empty[MAX_STAGES];
    uint64_t acc_full[2];
    uint64_t acc_empty[2];
    uint64_t x_full[2];  // an expand round is staged in region 0 / 1
    uint64_t x_empty[2]; // the UMMAs of that region's last round have finished reading it
    uint64_t base_done;  // the base UMMAs of an item have finished (its stages are free)
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
    int tt = tile / c.n_tiles, nt = tile % c.n_tiles;
    if (c.static_tiles >= 0 && c.tgroup > 1) {
        // grouped order: consecutive tiles cycle over tgroup token tiles for
        // one feature tile, then move to the next feature tile, so the CTAs
        // of one wave share each W tile among several token tiles in L2
        const int ntt = c.static_tiles / c.n_tiles;
        const int span = c.tgroup * c.n_tiles;
        const int g = tile / span, within = tile - g * span;
        const int gt = min(c.tgroup, ntt - g * c.tgroup);
        tt = g * c.tgroup + within % gt;
        nt = within / gt;
    }
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

// The j-th item of this CTA: blockIdx.x + j * gridDim.x, or with feature-tile
// pairs the pairs in that order, each pair as two consecutive items (its even
// item the first feature tile).
__device__ __forceinline__ int cta_item(const TcCfg &c, int j)
{
    return c.pair ? 2 * ((int)blockIdx.x + (j >> 1) * (int)gridDim.x) + (j & 1)
                  : (int)blockIdx.x + j * (int)gridDim.x;
}

__device__ __forceinline__ void flag_abort(const Params &p, Bars *bars)
{
    *(volatile int *)&bars->abort_flag = 1;
    atomicOr(p.ws.status, (uint32_t)LORA_FLAG_WAIT_TIMEOUT);
}

__device__ __forceinline__ bool aborted(Bars *bars) { return *(volatile int *)&bars->abort_flag != 0; }

// TMA producer of the pipeline: for every stage, the W box and the x box of
// its K chunks, both counted on the stage's full barrier.
__device__ __forceinline__ void produce(const TmapSet &maps, const Params &p, const TcCfg &c, Bars *bars,
                                        uint8_t *smem)
{
    if (c.static_tiles < 0)
        grid_dependency_wait();
    const int total = item_total(p, c);
    int last_parity[MAX_STAGES];
    for (int i = 0; i < MAX_STAGES; ++i)
        last_parity[i] = -1;
    int g = 0, j = 0;
    TileInfo ti;
    for (int w = cta_item(c, 0); w < total && get_tile(p, c, w / c.csplit, total, ti); w = cta_item(c, ++j)) {
        if (c.pair && (j & 1))
            continue; // the pair's second feature tile came with its first
        const int part = w % c.csplit;
        const int ks0 = part * c.kstages / c.csplit, ks1 = (part + 1) * c.kstages / c.csplit;
        for (int ks = ks0; ks < ks1; ++ks, ++g) {
            const int slot = g % c.stages;
            const uint32_t ph = (uint32_t)(g / c.stages) & 1u;
            if (aborted(bars) || !mbar_wait(bars->empty + slot, ph ^ 1u)) {
                flag_abort(p, bars);
                goto drain;
            }
            uint8_t *stage = smem + (size_t)slot * c.stage_bytes;
            if (c.pair) { // [W tile n0][W tile n0 + 128][x], kc chunks each
                mbar_arrive_expect_tx(bars->full + slot, c.stage_bytes);
                tma_load_3d(stage, &maps.w[ti.e], 0, ti.n0, ks * c.kc, bars->full + slot);
                tma_load_3d(stage + (size_t)c.kc * W_CHUNK_BYTES, &maps.w[ti.e], 0, ti.n0 + TC_BM, ks * c.kc,
                            bars->full + slot);
                tma_load_3d(stage + (size_t)2 * c.kc * W_CHUNK_BYTES, &maps.x, 0, ti.r0, ks * c.kc, bars->full + slot);
                last_parity[slot] = (int)ph;
                continue;
            }
            mbar_arrive_expect_tx(bars->full + slot, (uint32_t)c.kc * (W_CHUNK_BYTES + c.x_chunk));
            uint8_t *xdst = stage + (size_t)c.kc * W_CHUNK_BYTES;
            if (p.gated) {
                // [chunks][2 halves][I rows][64]: gate rows n0/2.. then up rows I + n0/2..
                tma_load_4d(stage, &maps.w[0], 0, ti.n0 >> 1, 0, ks * c.kc, bars->full + slot);
                tma_load_3d(xdst, &maps.x, 0, ti.r0, ks * c.kc, bars->full + slot);
            } else if (c.use3d) {
                tma_load_3d(stage, &maps.w[ti.e], 0, ti.n0, ks * c.kc, bars->full + slot);
                tma_load_3d(xdst, &maps.x, 0, ti.r0, ks * c.kc, bars->full + slot);
            } else {
                tma_load_2d(stage, &maps.w[ti.e], ks * 64, ti.n0, bars->full + slot);
                tma_load_2d(xdst, &maps.x, ks * 64, ti.r0, bars->full + slot);
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


// UMMAs of every item: the base product into accumulator it & 1, then the
// expand rounds the epilogue stages (into D', or into the base accumulator).
// Accumulator acquisitions are counted per buffer (acq), matching the
// epilogue's releases in order: item i takes buffer i & 1 and, when its D'
// borrows the other buffer, that one too.
__device__ __forceinline__ void issue_mma(const Params &p, const TcCfg &c, Bars *bars, uint8_t *smem,
                                          uint32_t tmem)
{
    if (c.static_tiles < 0)
        grid_dependency_wait();
    const EpiAux *aux = reinterpret_cast<const EpiAux *>(smem + c.aux_off);
    const uint32_t xh_blk = (uint32_t)c.tn * 128u;
    // staging regions: 0 = dedicated buffers, 1 = the pipeline stages
    const uint32_t rxb[2] = {smem_u32(smem + c.xb_off), smem_u32(smem)};
    const uint32_t rxh[2] = {smem_u32(smem + c.xh_off), smem_u32(smem) + (uint32_t)c.xblk_b * XB_BLOCK};
    const uint32_t rplane[2] = {(uint32_t)c.xblk * xh_blk, (uint32_t)c.xblk_b * xh_blk};
    const int total = item_total(p, c);
    int g = 0, it = 0, xg[2] = {0, 0};
    uint32_t acq[2] = {0u, 0u};
    TileInfo ti;
    for (int w = cta_item(c, 0); w < total && get_tile(p, c, w / c.csplit, total, ti); w = cta_item(c, ++it)) {
        const int part = w % c.csplit;
        const int ks0 = part * c.kstages / c.csplit, ks1 = (part + 1) * c.kstages / c.csplit;
        const int buf = it & 1;
        // a pair's first item takes both accumulators, its second none
        const int nacq = c.pair ? ((it & 1) ? 0 : 2) : 1;
        bool got = true;
        for (int b = buf; b < buf + nacq; ++b)
            if (aborted(bars) || !mbar_wait(bars->acc_empty + b, (acq[b] & 1u) ^ 1u)) {
                got = false;
                break;
            } else {
                ++acq[b];
            }
        if (!got) {
            flag_abort(p, bars);
            break;
        }
        tc_fence_after();
        const uint32_t acc = tmem + (uint32_t)(buf * c.tn);
        const int nmma = (ti.cnt + 15) & ~15;
        const uint32_t idesc = idesc_bf16_f32(TC_BM, (uint32_t)nmma);
        uint32_t accumulate = 0;
        bool ok = true;
        // the pair's K loop ran with its first item
        for (int ks = ks0; ks < ks1 && !(c.pair && (it & 1)); ++ks, ++g) {
            const int slot = g % c.stages;
            const uint32_t ph = (uint32_t)(g / c.stages) & 1u;
            if (aborted(bars) || !mbar_wait(bars->full + slot, ph)) {
                flag_abort(p, bars);
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t wb = smem_u32(smem + (size_t)slot * c.stage_bytes);
            const uint32_t xsb = wb + (uint32_t)c.kc * W_CHUNK_BYTES;
            if (c.pair) { // accumulator 0: W tile n0, accumulator 1: W tile n0 + 128
                const uint32_t xpb = wb + (uint32_t)(2 * c.kc) * W_CHUNK_BYTES;
                for (int q = 0; q < c.kc; ++q) {
                    if (ks * c.kc + q >= c.kchunks)
                        break;
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const uint64_t xd = sw128_kmajor_desc(xpb + q * c.x_chunk + j * 32);
                        umma_bf16(acc, sw128_kmajor_desc(wb + q * W_CHUNK_BYTES + j * 32), xd, idesc, accumulate);
                        umma_bf16(acc + (uint32_t)c.tn,
                                  sw128_kmajor_desc(wb + (c.kc + q) * W_CHUNK_BYTES + j * 32), xd, idesc,
                                  accumulate);
                        accumulate = 1;
                    }
                }
            } else {
                for (int q = 0; q < c.kc; ++q) {
                    if (ks * c.kc + q >= c.kchunks)
                        break;
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        umma_bf16(acc, sw128_kmajor_desc(wb + q * W_CHUNK_BYTES + j * 32),
                                  sw128_kmajor_desc(xsb + q * c.x_chunk + j * 32), idesc, accumulate);
                        accumulate = 1;
                    }
                }
            }
            umma_commit(bars->empty + slot);
        }
        umma_commit(&bars->base_done);
        // expand rounds of this item: round 1 of a CTA's last item is staged in
        // the pipeline stages (region 1), every other round in region 0
        const bool last_item = cta_item(c, it + 1) >= total;
        bool first = true;
        uint32_t dacc = 0;
        for (int round = 0; ok; ++round) {
            const int rg = (round == 1 && last_item && c.xblk_b > 0) ? 1 : 0;
            if (aborted(bars) || !mbar_wait(bars->x_full + rg, (uint32_t)xg[rg] & 1u)) {
                flag_abort(p, bars);
                ok = false;
                break;
            }
            ++xg[rg];
            tc_fence_after();
            const int mode = *(volatile const int32_t *)&aux->xr_mode[rg];
            const int nk16 = *(volatile const int32_t *)&aux->xr_nk16[rg];
            const int last = *(volatile const int32_t *)&aux->xr_last[rg];
            if (mode == 1 && first && c.borrow) {
                const int ob = buf ^ 1;
                if (aborted(bars) || !mbar_wait(bars->acc_empty + ob, (acq[ob] & 1u) ^ 1u)) {
                    flag_abort(p, bars);
                    ok = false;
                    break;
                }
                ++acq[ob];
                tc_fence_after();
            }
            if (first)
                dacc = mode == 2 ? acc : tmem + (uint32_t)((c.borrow ? (buf ^ 1) : 2) * c.tn);
            uint32_t dacc_on = (mode == 2 || !first) ? 1u : 0u;
            for (int k = 0; k < nk16; ++k) {
                const uint32_t koff = (uint32_t)(k >> 2) * XB_BLOCK + (uint32_t)(k & 3) * 32u;
                const uint32_t hoff = (uint32_t)(k >> 2) * xh_blk + (uint32_t)(k & 3) * 32u;
                for (int h = 0; h < c.hl; ++h) {
                    umma_bf16(dacc, sw128_kmajor_desc(rxb[rg] + koff),
                              sw128_kmajor_desc(rxh[rg] + h * rplane[rg] + hoff), idesc, dacc_on);
                    dacc_on = 1;
                }
            }
            umma_commit(bars->x_empty + rg);
            first = false;
            if (last)
                break;
        }
        umma_commit(bars->acc_full + buf); // arrives once every UMMA above has finished
        if (!ok)
            break;
    }
}

__device__ __forceinline__ bool wait_count(const int32_t *cnt, int target, uint64_t wait_ns)
{
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

// Exclusive scan of two values over the 128 epilogue threads (ea, eb), and
// their totals (ta, tb).
__device__ __forceinline__ void epi_scan2(int a, int b, int &ea, int &eb, int &ta, int &tb, EpiAux *aux,
                                          int et)
{
    const int lane = et & 31, w = et >> 5;
    int ia = a, ib = b;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int xa = __shfl_up_sync(0xffffffffu, ia, o);
        const int xb = __shfl_up_sync(0xffffffffu, ib, o);
        if (lane >= o) {
            ia += xa;
            ib += xb;
        }
    }
    if (lane == 31) {
        aux->wsum[0][w] = ia;
        aux->wsum[1][w] = ib;
    }
    named_bar_sync(1, EPI_THREADS);
    int pa = 0, pb = 0;
    ta = 0;
    tb = 0;
#pragma unroll
    for (int q = 0; q < EPI_THREADS / 32; ++q) {
        const int va = aux->wsum[0][q], vb = aux->wsum[1][q];
        if (q < w) {
            pa += va;
            pb += vb;
        }
        ta += va;
        tb += vb;
    }
    ea = pa + ia - a;
    eb = pb + ib - b;
    named_bar_sync(1, EPI_THREADS); // wsum is free again
}

// bf16 bits of v, and of the remainder v - bf16(v).
__device__ __forceinline__ void split_hi_lo(float v, uint32_t &hi, uint32_t &lo)
{
    const uint16_t h = f32_to_bf16_bits(v);
    hi = h;
    lo = f32_to_bf16_bits(v - __uint_as_float((uint32_t)h << 16));
}

constexpr int UNIT_BATCH = 64; // shrink units whose metadata is built at once
constexpr int SHRINK_GROUP_THREADS = 64; // warps 2 and 3

// This CTA's share of the shrink work units (h = A_s x, shrink.cuh): the
// metadata of up to UNIT_BATCH units is built in parallel (one thread each:
// bucket search, table and perm reads) into shared memory, then the units run
// back to back. One fence publishes them all, then each unit's bucket counter
// is bumped.
__device__ __forceinline__ void epi_shrink(const Params &p, const int32_t *unit_off, const int32_t *seg_off,
                                           float *red, UnitMeta *um, int et)
{
    const int nb = p.E * (p.L + 1);
    const int total_units = unit_off[nb];
    const int mine = total_units > (int)blockIdx.x ? (total_units - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x : 0;
    for (int k0 = 0; k0 < mine; k0 += UNIT_BATCH) {
        const int nk = min(UNIT_BATCH, mine - k0);
        if (et < nk)
            um[et] = unit_meta(p, (int)blockIdx.x + (k0 + et) * (int)gridDim.x, unit_off, seg_off);
        named_bar_sync(1, EPI_THREADS);
        for (int k = 0; k < nk; ++k)
            shrink_unit(p, um[k], et >> 5, et & 31, red, 1);
        __threadfence();
        named_bar_sync(1, EPI_THREADS);
        if (et < nk)
            atomicAdd(p.ws.done + um[et].b, 1);
        named_bar_sync(1, EPI_THREADS); // um is rewritten by the next batch
    }
}

// Metadata of shrink unit u from the local routing of a one-tile launch:
// units are numbered as the routing kernel numbers them (slot by slot, then
// rank group, row chunk, K part), over the tile's rows grouped by slot.
__device__ __forceinline__ UnitMeta lr_unit_meta(const Params &p, const EpiAux *aux, int u, int r0)
{
    int lo = 0, hi = p.L;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (aux->lr_uoff[mid] <= u)
            lo = mid;
        else
            hi = mid;
    }
    const int s = lo, rank = aux->lr_rank[s];
    const int nrg = (rank + SHRINK_RG - 1) / SHRINK_RG;
    int local = u - aux->lr_uoff[s];
    UnitMeta m;
    m.kpart = (int16_t)(local % p.kp);
    local /= p.kp;
    m.rg = (int16_t)(local % nrg);
    const int c0 = aux->lr_seg[s] + (local / nrg) * SHRINK_TC;
    const int nrows = min(SHRINK_TC, aux->lr_seg[s] + aux->lr_cnt[s] - c0);
#pragma unroll
    for (int j = 0; j < SHRINK_TC; ++j)
        m.row[j] = r0 + aux->lr_perm[c0 + min(j, nrows - 1)];
    m.A = aux->lr_a[s];
    m.b = (int16_t)(s + 1);
    m.rank = (int16_t)rank;
    m.nrows = (int16_t)nrows;
    m.pad = 0;
    return m;
}

// Where one staging pass writes: relative k in [0, kr0) goes to region 0,
// [kr0, kr0 + kr1) to region 1 (kr1 = 0: one region).
struct XDst {
    uint8_t *xb[2];
    uint8_t *xh[2];
    uint32_t plane[2]; // bytes between the hi and lo planes of XH
    int kr0, kr1;
};

// B rows n0 + et of the expand's slots, the part whose k relative to r0k lies
// in [klo, khi), copied into XB (128-byte swizzle) of the region that k maps
// to, without passing through registers; pad columns of the padded rank and
// rows past N are zero-filled.
__device__ __forceinline__ void stage_b(const Params &p, const EpiAux *aux, const XDst &d, int klo, int khi,
                                        int nent, int r0k, int n, int et)
{
    const bool row_ok = n < p.N;
    for (int e = 0; e < nent; ++e) {
        const int so = aux->ent_off[e] - r0k;
        const int rk = aux->ent_rank[e];
        const int pk = (rk + 15) & ~15;
        if (so + pk <= klo || so >= khi)
            continue;
        const uint16_t *src = aux->ent_b[e] + (size_t)(row_ok ? n : 0) * p.R;
        for (int q = max(0, klo - so); q < pk && so + q < khi; q += 8) {
            const int k = so + q, rg = k >= d.kr0 ? 1 : 0, kl = k - (rg ? d.kr0 : 0);
            const int cq = kl >> 3;
            const bool has = row_ok && q < rk;
            cp_async_16(d.xb[rg] + (cq >> 3) * XB_BLOCK + et * 128 + (((cq & 7) ^ (et & 7)) << 4),
                        src + (has ? q : 0), has ? 16u : 0u);
        }
    }
}

// XH rows 0..nmma-1 of the pass [r0k, r0k + kr0 + kr1): s_t * h_t in column
// t's slot range (hi, and lo = the bf16 remainder when hl = 2), zero
// elsewhere (zero_xh has zeroed every chunk of the pass before). Each
// column's data chunks are split over 128 / nmma threads, each issuing the
// loads of up to four chunks (every K part of h) before converting any.
// Zero the XH chunks of one staging region of the pass (rows 0..nmma-1,
// every plane), before any of s * h is written: it needs nothing but the
// region being free, so region 0 is zeroed while the shrink is still running.
__device__ __forceinline__ void zero_xh(const TcCfg &c, const XDst &d, int rg, int nmma, int et)
{
    const uint32_t xh_block = (uint32_t)c.tn * 128u;
    const int nch = (((rg ? d.kr1 : d.kr0) + 63) >> 6) * 8;
    const uint4 z = make_uint4(0, 0, 0, 0);
    for (int idx = et; idx < nmma * nch; idx += EPI_THREADS) {
        const int j = idx / nch, cl = idx - j * nch;
        uint8_t *dst = d.xh[rg] + (uint32_t)(cl >> 3) * xh_block + j * 128 + (((cl & 7) ^ (j & 7)) << 4);
        *reinterpret_cast<uint4 *>(dst) = z;
        if (c.hl == 2)
            *reinterpret_cast<uint4 *>(dst + d.plane[rg]) = z;
    }
}

__device__ __forceinline__ void stage_h(const Params &p, const TcCfg &c, const EpiAux *aux, const XDst &d,
                                        const TileInfo &ti, int nmma, int r0k, int et)
{
    const uint32_t xh_block = (uint32_t)c.tn * 128u;
    named_bar_sync(1, EPI_THREADS); // the zeroed chunks (zero_xh, any thread) before the data
    const int kt = d.kr0 + d.kr1;
    const size_t part_stride = (size_t)p.rows * p.R;
    // tpc threads per column (a power of two), each taking every tpc-th chunk
    const int tpc = nmma >= EPI_THREADS ? 1 : EPI_THREADS / nmma;
    const int sub = et % tpc;
    for (int j = et / tpc; j < ti.cnt; j += EPI_THREADS / tpc) {
        const int ko = aux->koff[j];
        if (ko < 0)
            continue;
        const int rk = aux->crank[j];
        const float s = aux->cscale[j];
        const float *cr = p.tab[ti.e].comp_table + (size_t)aux->cslot[j] * LORA_COMP_STRIDE;
        // ranks r (multiples of 8, r < rank) of this slot that fall in the pass
        const int rlo = max(0, r0k - ko), rhi = min(rk, r0k + kt - ko);
        if (c.hl == 1 && p.no_units) {
            // the tensor-core shrink tiles wrote this operand already rounded to
            // bf16 (ws.hs, zero past the rank): copy it in 16-byte chunks
            const uint16_t *hsrow = p.ws.hs + (size_t)(ti.r0 + j) * p.R;
            for (int r = rlo + 8 * sub; r < rhi; r += 8 * tpc) {
                const int k = ko + r - r0k, rg = k >= d.kr0 ? 1 : 0, kl = k - (rg ? d.kr0 : 0);
                const int cq = kl >> 3;
                cp_async_16(d.xh[rg] + (uint32_t)(cq >> 3) * xh_block + j * 128 + (((cq & 7) ^ (j & 7)) << 4),
                            hsrow + r, 16u);
            }
            continue;
        }
        const float *hrow = p.ws.h + (size_t)(ti.r0 + j) * p.R;
        for (int r = rlo + 8 * sub; r < rhi; r += 32 * tpc) {
            float4 a[4], b[4], ca[4], cb[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int rr = r + 8 * tpc * u;
                a[u] = make_float4(0.f, 0.f, 0.f, 0.f);
                b[u] = a[u];
                ca[u] = a[u];
                cb[u] = a[u];
                if (rr < rhi) {
                    ca[u] = __ldg(reinterpret_cast<const float4 *>(cr + rr));
                    cb[u] = __ldg(reinterpret_cast<const float4 *>(cr + rr + 4));
#pragma unroll
                    for (int kq = 0; kq < 4; ++kq) {
                        if (kq < p.kp) { // parts summed in part order
                            const float *h = hrow + (size_t)kq * part_stride + rr;
                            const float4 c4 = __ldcg(reinterpret_cast<const float4 *>(h));
                            const float4 d4 = __ldcg(reinterpret_cast<const float4 *>(h + 4));
                            a[u].x += c4.x; a[u].y += c4.y; a[u].z += c4.z; a[u].w += c4.w;
                            b[u].x += d4.x; b[u].y += d4.y; b[u].z += d4.z; b[u].w += d4.w;
                        }
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int rr = r + 8 * tpc * u;
                if (rr >= rhi)
                    break;
                // s * comp: the slot's scale times the rank's factor (1 unless the
                // slot holds a stack of adapters)
                const float v[8] = {a[u].x * (s * ca[u].x), a[u].y * (s * ca[u].y), a[u].z * (s * ca[u].z),
                                    a[u].w * (s * ca[u].w), b[u].x * (s * cb[u].x), b[u].y * (s * cb[u].y),
                                    b[u].z * (s * cb[u].z), b[u].w * (s * cb[u].w)};
                uint32_t h8[8], l8[8];
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    split_hi_lo(v[i], h8[i], l8[i]);
                const int k = ko + rr - r0k, rg = k >= d.kr0 ? 1 : 0, kl = k - (rg ? d.kr0 : 0);
                const int cq = kl >> 3;
                uint8_t *dst = d.xh[rg] + (uint32_t)(cq >> 3) * xh_block + j * 128 + (((cq & 7) ^ (j & 7)) << 4);
                *reinterpret_cast<uint4 *>(dst) = make_uint4(h8[0] | (h8[1] << 16), h8[2] | (h8[3] << 16),
                                                             h8[4] | (h8[5] << 16), h8[6] | (h8[7] << 16));
                if (c.hl == 2)
                    *reinterpret_cast<uint4 *>(dst + d.plane[rg]) =
                        make_uint4(l8[0] | (l8[1] << 16), l8[2] | (l8[3] << 16), l8[4] | (l8[5] << 16),
                                   l8[6] | (l8[7] << 16));
            }
        }
    }
}

// Shrink warps (warps 2 and 3) of one-tile launches: once the epilogue has
// sorted the tile's rows by slot (named barrier 3), they run this CTA's
// shrink units -- two warps per unit splitting its K part -- while the
// epilogue assigns slots to K parts and stages the B rows; after the routing
// kernel has finished (it clears the counters) each unit's bucket counter is
// bumped. Named barrier 4 tells the epilogue the sort tables are free again.
__device__ __forceinline__ void shrink_warps(const Params &p, const TcCfg &c, uint8_t *smem)
{
    const int st = threadIdx.x - 64; // 0..63
    const EpiAux *aux = reinterpret_cast<const EpiAux *>(smem + c.aux_off);
    float *red = reinterpret_cast<float *>(smem + c.red_off);
    UnitMeta *um = reinterpret_cast<UnitMeta *>(smem + c.umeta_off);
    named_bar_sync(3, SHRINK_GROUP_THREADS + EPI_THREADS);
    const int tu = aux->lr_uoff[p.L];
    const int mine = tu > (int)blockIdx.x ? (tu - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x : 0;
    bool routed = false;
    for (int k0 = 0; k0 < mine; k0 += UNIT_BATCH) {
        const int nk = min(UNIT_BATCH, mine - k0);
        if (st < nk)
            um[st] = lr_unit_meta(p, aux, (int)blockIdx.x + (k0 + st) * (int)gridDim.x, 0);
        named_bar_sync(2, SHRINK_GROUP_THREADS);
        for (int k = 0; k < nk; ++k)
            shrink_unit<2>(p, um[k], st >> 5, st & 31, red, 2);
        __threadfence();
        named_bar_sync(2, SHRINK_GROUP_THREADS);
        if (!routed) {
            grid_dependency_wait();
            routed = true;
        }
        if (st < nk)
            atomicAdd(p.ws.done + um[st].b, 1);
        named_bar_sync(2, SHRINK_GROUP_THREADS); // um is rewritten by the next batch
    }
    named_bar_arrive(4, SHRINK_GROUP_THREADS + EPI_THREADS);
}

// Per item: which columns take their delta here (adapted rows whose slot the
// rank-balanced assignment gives to this K part) and the k offset of each such
// slot; stage the
// expand operands round by round for the MMA warp (the first round of the
// first item is issued before this CTA's shrink units, so its B copies overlap
// them); then drain the accumulator (adding D' to those columns only), and
// with csplit > 1 write the partial tile and, once every part is in, sum this
// part's share of the columns in part order.
template <bool kStc>
__device__ __forceinline__ void epilogue(const TmapSet &maps, const Params &p, const TcCfg &c, Bars *bars,
                                         uint8_t *smem, uint32_t tmem)
{
    const int et = threadIdx.x - (TC_THREADS - EPI_THREADS); // TMEM lane 0..127
    const int ew = et >> 5;
    EpiAux *aux = reinterpret_cast<EpiAux *>(smem + c.aux_off);
    uint8_t *XB = smem + c.xb_off;
    uint8_t *XH = smem + c.xh_off;
    const int C = c.csplit;
    const int nb = p.E * (p.L + 1);
    int32_t *unit_off = reinterpret_cast<int32_t *>(smem + c.meta_off); // copies of the routing
    int32_t *seg_off = unit_off + nb + 1;                                 // results, in shared memory
    float *red = reinterpret_cast<float *>(smem + c.red_off);
    UnitMeta *um = reinterpret_cast<UnitMeta *>(smem + c.umeta_off);

    // With token tiles known on the host, the first item's column scan and B
    // copies need nothing from the routing kernel: the wait for it (and the
    // copy of its bucket tables) comes just before this CTA's shrink units.
    bool routed = false;
    auto route_wait = [&]() {
        grid_dependency_wait();
        for (int q = et; q <= nb; q += EPI_THREADS) {
            unit_off[q] = p.ws.unit_off[q];
            seg_off[q] = p.ws.seg_off[q];
        }
        named_bar_sync(1, EPI_THREADS);
        routed = true;
    };
    if (c.static_tiles < 0)
        route_wait();

    const int total = item_total(p, c);
    bool shrink_done = false, grp_joined = false;
    int it = 0, xg[2] = {0, 0};
    // an item's expand extent, slot entries and mode (kept for a pair's second item)
    int kx = 0, nent = 0, mode = 0;
    bool pair_reuse = false; // the pair's first item staged its one expand round in region 0
    TileInfo ti;
    for (int w = cta_item(c, 0); w < total && get_tile(p, c, w / c.csplit, total, ti); w = cta_item(c, ++it)) {
        const int tile = w / c.csplit, part = w % c.csplit;
        const int buf = it & 1;
        const uint32_t use = (uint32_t)(it >> 1);
        // this thread's row of W and B: feature n0 + et, or for the gated view
        // gate row n0/2 + et (et < 64) and up row I + n0/2 + et - 64
        const int n = p.gated ? (et < 64 ? (ti.n0 >> 1) + et : p.I + (ti.n0 >> 1) + et - 64) : ti.n0 + et;
        const Tables &tab = p.tab[ti.e];
        const int nmma = (ti.cnt + 15) & ~15;

        if (c.local_route && it == 1) {
            named_bar_sync(4, SHRINK_GROUP_THREADS + EPI_THREADS); // the shrink warps are done with lr_*
            grp_joined = true;
        }
        // The second item of a pair (same token tile, the next 128 features)
        // has the first one's slot lists, and, when the first staged its one
        // expand round in region 0, the same s * h operand there.
        const bool reuse = c.pair && (it & 1) && pair_reuse;
        if (!reuse) {
            // (1) the columns whose delta this part adds, and the slots they use
            for (int q = et; q < p.L; q += EPI_THREADS)
                aux->soff[q] = 0;
            if (c.local_route && et < p.L)
                aux->lr_cnt[et] = 0;
            if (et < MAX_TN / 32)
                aux->onbits[et] = 0;
            if (et == 0)
                aux->n_on = 0;
            named_bar_sync(1, EPI_THREADS);
            for (int j = et; j < ti.cnt; j += EPI_THREADS) {
                const int sl = p.seq_slot[ti.r0 + j];
                const SlotInfo si = slot_info(tab, sl, p.L);
                aux->koff[j] = si.on ? sl : -1;
                aux->cscale[j] = si.scale;
                aux->crank[j] = (int16_t)si.rank;
                aux->cslot[j] = (int16_t)(si.on ? sl : 0);
                if (si.on) {
                    aux->soff[sl] = (uint16_t)((si.rank + 15) & ~15); // same value from every writer
                    if (c.local_route) {
                        atomicAdd(&aux->lr_cnt[sl], 1);
                        aux->lr_rank[sl] = (int16_t)si.rank;
                        aux->lr_a[sl] = si.a;
                        aux->lr_b[sl] = si.b;
                    }
                }
            }
            named_bar_sync(1, EPI_THREADS);
            if (c.local_route && !shrink_done) {
                // (1a) every row of the launch is in this tile: sort them by slot
                // here (stable, so every CTA builds the same shrink work list); the
                // shrink warps run this CTA's units from this sort without waiting
                // for the routing kernel (only their counter updates wait for it:
                // it clears the counters).
                int u_s = 0, c_s = 0;
                if (et < p.L) {
                    c_s = aux->lr_cnt[et];
                    u_s = c_s > 0 ? bucket_units(aux->lr_rank[et], c_s, p.kp) : 0;
                }
                int eu, ecn, tu, tcn;
                epi_scan2(u_s, c_s, eu, ecn, tu, tcn, aux, et);
                if (et < p.L) {
                    aux->lr_uoff[et] = eu;
                    aux->lr_seg[et] = (int16_t)ecn;
                    aux->lr_run[et] = (int16_t)ecn;
                }
                if (et == 0)
                    aux->lr_uoff[p.L] = tu;
                for (int c0 = 0; c0 < ti.cnt; c0 += EPI_THREADS) {
                    for (int q = et; q < 4 * LR_MAX_L; q += EPI_THREADS)
                        (&aux->lr_wcnt[0][0])[q] = 0;
                    named_bar_sync(1, EPI_THREADS);
                    const int j = c0 + et, lane = et & 31;
                    const int sl = j < ti.cnt ? aux->koff[j] : -1;
                    const unsigned peers = __match_any_sync(0xffffffffu, sl);
                    const int r = __popc(peers & ((1u << lane) - 1u));
                    if (sl >= 0 && r == 0)
                        aux->lr_wcnt[ew][sl] = (int16_t)__popc(peers);
                    named_bar_sync(1, EPI_THREADS);
                    if (sl >= 0) {
                        int pre = 0;
                        for (int q = 0; q < ew; ++q)
                            pre += aux->lr_wcnt[q][sl];
                        aux->lr_perm[aux->lr_run[sl] + pre + r] = (int16_t)j;
                    }
                    named_bar_sync(1, EPI_THREADS);
                    if (et < p.L)
                        aux->lr_run[et] = (int16_t)(aux->lr_run[et] + aux->lr_wcnt[0][et] + aux->lr_wcnt[1][et] +
                                                    aux->lr_wcnt[2][et] + aux->lr_wcnt[3][et]);
                    named_bar_sync(1, EPI_THREADS);
                }
                // the sort is done: the shrink warps run this CTA's units from here
                named_bar_arrive(3, SHRINK_GROUP_THREADS + EPI_THREADS);
                shrink_done = true;
            }
            const int per = (p.L + EPI_THREADS - 1) / EPI_THREADS;
            const int s0 = min(p.L, et * per), s1 = min(p.L, s0 + per);
            if (C > 1) {
                // (1b) the tile's adapted slots shared among the K parts: sorted by
                // padded rank, largest first (ties: lower slot), and dealt in snake
                // order 0, 1, .., C-1, C-1, .., 0, 0, 1, .. so the parts' k extents
                // stay close. Every CTA of the tile derives the same assignment.
                int cnt = 0;
                for (int s = s0; s < s1; ++s)
                    cnt += aux->soff[s] != 0;
                int ec0, dummy, nu, dummy2;
                epi_scan2(cnt, 0, ec0, dummy, nu, dummy2, aux, et);
                for (int s = s0; s < s1; ++s)
                    if (aux->soff[s]) {
                        aux->entry_slot[ec0] = (int16_t)s;
                        aux->ent_off[ec0] = aux->soff[s]; // padded rank, by list position
                        ++ec0;
                    }
                named_bar_sync(1, EPI_THREADS);
                for (int i = et; i < nu; i += EPI_THREADS) {
                    const int ci = aux->ent_off[i];
                    int pos = 0;
                    for (int j = 0; j < nu; ++j) {
                        const int cj = aux->ent_off[j];
                        pos += (cj > ci) | ((cj == ci) & (j < i));
                    }
                    const int r = pos % (2 * C);
                    aux->part_of[aux->entry_slot[i]] = (int8_t)(r < C ? r : 2 * C - 1 - r);
                }
                named_bar_sync(1, EPI_THREADS);
            }
            int my_on = 0;
            for (int j = et; j < ti.cnt; j += EPI_THREADS) {
                const int sl = aux->koff[j];
                const bool on = sl >= 0 && (C == 1 || aux->part_of[sl] == part);
                if (on) {
                    atomicOr(&aux->onbits[j >> 5], 1u << (j & 31));
                    ++my_on;
                } else {
                    aux->koff[j] = -1;
                }
            }
            if (my_on)
                atomicAdd(&aux->n_on, my_on);
            named_bar_sync(1, EPI_THREADS);
            // (2) k offsets of this part's slots in ascending order, each rank padded to 16
            int ksum = 0, scount = 0;
            for (int s = s0; s < s1; ++s) {
                const int v = (C == 1 || aux->part_of[s] == part) ? aux->soff[s] : 0;
                ksum += v;
                scount += v != 0;
            }
            int ek, ec;
            epi_scan2(ksum, scount, ek, ec, kx, nent, aux, et);
            for (int s = s0; s < s1; ++s) {
                const int v = (C == 1 || aux->part_of[s] == part) ? aux->soff[s] : 0;
                if (v) {
                    aux->soff[s] = (uint16_t)ek;
                    aux->entry_slot[ec] = (int16_t)s;
                    aux->ent_off[ec] = ek;
                    ek += v;
                    ++ec;
                }
            }
            named_bar_sync(1, EPI_THREADS);
            for (int e = et; e < nent; e += EPI_THREADS) {
                const int s = aux->entry_slot[e];
                aux->ent_b[e] = c.local_route ? aux->lr_b[s] : tab.b_table[s];
                aux->ent_rank[e] = c.local_route ? aux->lr_rank[s] : (int16_t)tab.rank_table[s];
            }
            for (int j = et; j < ti.cnt; j += EPI_THREADS) {
                const int sl = aux->koff[j];
                if (sl >= 0)
                    aux->koff[j] = aux->soff[sl];
            }
            named_bar_sync(1, EPI_THREADS);
            const int n_on = aux->n_on;
            mode = n_on == 0 ? 0 : (c.borrow && n_on == ti.cnt ? 2 : 1);
            if (kx > c.xblk * 64 && n < p.N) {
                // B rows of the later rounds: warm them in L2 now
                for (int e = 0; e < nent; ++e)
                    if (aux->ent_off[e] + aux->ent_rank[e] > c.xblk * 64)
                        prefetch_l2(aux->ent_b[e] + (size_t)n * p.R);
            }
        }
        if (c.pair && !(it & 1))
            pair_reuse = kx <= c.xblk * 64;

        // (3) expand rounds: k range [r0k, r0k + kr) of the concatenated slots.
        // The first pass stages round 0 in the dedicated buffers (region 0)
        // and, on this CTA's last item, round 1 in the pipeline stages (region
        // 1, free once the item's base UMMAs are done); each later pass stages
        // one round in region 0.
        const bool last_item = cta_item(c, it + 1) >= total;
        int r0k = 0;
        bool stop = false;
        if (reuse) {
            // only B's rows for these features change: restage XB
            if (et == 0 && !mbar_wait(bars->x_empty, (uint32_t)(xg[0] - 1) & 1u))
                flag_abort(p, bars);
            named_bar_sync(1, EPI_THREADS);
            XDst d;
            d.xb[0] = d.xb[1] = XB;
            d.xh[0] = d.xh[1] = XH;
            d.plane[0] = d.plane[1] = (uint32_t)c.xblk * (uint32_t)c.tn * 128u;
            d.kr0 = kx;
            d.kr1 = 0;
            if (kx > 0)
                stage_b(p, aux, d, 0, kx, nent, 0, n, et);
            cp_async_wait_all();
            fence_proxy_async_smem(); // generic-proxy writes, read by the UMMAs
            named_bar_sync(1, EPI_THREADS);
            if (et == 0) {
                aux->xr_mode[0] = mode;
                aux->xr_nk16[0] = kx / 16;
                aux->xr_last[0] = 1;
                mbar_arrive(bars->x_full);
            }
            ++xg[0];
        }
        for (int pass = 0; !reuse && (pass == 0 || r0k < kx); ++pass) {
            XDst d;
            d.xb[0] = XB;
            d.xh[0] = XH;
            d.plane[0] = (uint32_t)c.xblk * (uint32_t)c.tn * 128u;
            d.xb[1] = smem;
            d.xh[1] = smem + (size_t)c.xblk_b * XB_BLOCK;
            d.plane[1] = (uint32_t)c.xblk_b * (uint32_t)c.tn * 128u;
            d.kr0 = min(kx - r0k, c.xblk * 64);
            d.kr1 = (pass == 0 && last_item && c.xblk_b > 0) ? min(kx - r0k - d.kr0, c.xblk_b * 64) : 0;
            if (xg[0] > 0) { // the UMMAs of region 0's previous round have read it
                if (et == 0 && !mbar_wait(bars->x_empty, (uint32_t)(xg[0] - 1) & 1u))
                    flag_abort(p, bars);
                named_bar_sync(1, EPI_THREADS);
            }
            if (d.kr0 > 0) {
                stage_b(p, aux, d, 0, d.kr0, nent, r0k, n, et);
                zero_xh(c, d, 0, nmma, et);
            }
            if (!shrink_done) {
                if (!routed)
                    route_wait();
                epi_shrink(p, unit_off, seg_off, red, um, et);
                shrink_done = true;
            }
            if (!routed)
                route_wait(); // the counters below are the routing kernel's
            if (d.kr1 > 0) { // region 1: the stages are free once the base UMMAs are done
                if (et == 0 && !mbar_wait(&bars->base_done, (uint32_t)it & 1u))
                    flag_abort(p, bars);
                named_bar_sync(1, EPI_THREADS);
                stage_b(p, aux, d, d.kr0, d.kr0 + d.kr1, nent, r0k, n, et);
                zero_xh(c, d, 1, nmma, et);
            }
            if (pass == 0 && nent > 0) { // the shrink of the staged slots has finished
                for (int e = et; e < nent; e += EPI_THREADS) {
                    const int b = ti.e * (p.L + 1) + aux->entry_slot[e] + 1;
                    if (!wait_bucket(p, b, unit_off))
                        flag_abort(p, bars);
                }
                // or the launch's shrink tiles of these rows
                if (kStc && p.stc_tiles > 0)
                    for (int t = ti.r0 / STC_M + et; t <= (ti.r0 + ti.cnt - 1) / STC_M; t += EPI_THREADS)
                        if (!stc_wait_tile(p, t, 1 + c.extra_parts, c.wait_ns))
                            flag_abort(p, bars);
                named_bar_sync(1, EPI_THREADS);
                if (aborted(bars)) {
                    cp_async_wait_all();
                    stop = true;
                    break;
                }
            }
            if (d.kr0 + d.kr1 > 0)
                stage_h(p, c, aux, d, ti, nmma, r0k, et);
            cp_async_wait_all();
            fence_proxy_async_smem(); // generic-proxy writes, read by the UMMAs
            named_bar_sync(1, EPI_THREADS);
            if (et == 0) {
                aux->xr_mode[0] = mode;
                aux->xr_nk16[0] = d.kr0 / 16;
                aux->xr_last[0] = (d.kr1 == 0 && r0k + d.kr0 >= kx) ? 1 : 0;
                mbar_arrive(bars->x_full);
                if (d.kr1 > 0) {
                    aux->xr_mode[1] = mode;
                    aux->xr_nk16[1] = d.kr1 / 16;
                    aux->xr_last[1] = r0k + d.kr0 + d.kr1 >= kx ? 1 : 0;
                    mbar_arrive(bars->x_full + 1);
                }
            }
            ++xg[0];
            if (d.kr1 > 0)
                ++xg[1];
            r0k += d.kr0 + d.kr1;
        }
        if (stop)
            break;

        // (4) accumulator of this item
        const bool got = mbar_wait(bars->acc_full + buf, use & 1u);
        tc_fence_after();
        if (!got)
            flag_abort(p, bars);
        named_bar_sync(1, EPI_THREADS);
        if (aborted(bars))
            break;
        const uint32_t lane_off = (uint32_t)(ew * 32) << 16;
        const uint32_t tb = tmem + (uint32_t)(buf * c.tn) + lane_off;
        const uint32_t td = tmem + (uint32_t)((c.borrow ? (buf ^ 1) : 2) * c.tn) + lane_off;
        float *my_part = p.ws.part + ((size_t)tile * C + part) * (size_t)c.tn * EPI_THREADS;
        // y boxes: in XH, or for a pair's first item that leaves XH to the
        // second, in XB (one box; its expand round has been read)
        const bool y_in_xb = c.pair && !(it & 1) && pair_reuse;
        uint8_t *ybuf = y_in_xb ? XB : XH;
        const int nys = y_in_xb ? 1 : c.ystore;
        for (int c0 = 0; c0 < ti.cnt; c0 += 16) {
            uint32_t rb[16], rdl[16];
            tmem_ld16_nowait(tb + (uint32_t)c0, rb);
            if (mode == 1)
                tmem_ld16_nowait(td + (uint32_t)c0, rdl);
            const uint32_t on16 = mode == 1 ? (aux->onbits[c0 >> 5] >> (c0 & 16)) & 0xFFFFu : 0u;
            tmem_wait_ld();
            float v[16];
#pragma unroll
            for (int j = 0; j < 16; ++j)
                v[j] = (on16 >> j) & 1u ? __uint_as_float(rb[j]) + __uint_as_float(rdl[j])
                                        : __uint_as_float(rb[j]);
            if (p.gated && C == 1) {
                // act = silu(g) * u of the bf16-rounded halves, rounded once: each
                // thread's 16 values (gate or up of one feature) go through shared
                // memory [16 rows][128] to the thread forming them; thread et then
                // forms feature et % 64 for rows 8 (et / 64).. +7 into the staging
                // box [row][64 act] bf16, and a full box goes out as one TMA store
                const int sub = c0 % YSTORE_ROWS, bi = (c0 / YSTORE_ROWS) % c.ystore;
                uint16_t *box = reinterpret_cast<uint16_t *>(XH) + (size_t)bi * YSTORE_ROWS * 64;
                uint16_t *xs = reinterpret_cast<uint16_t *>(XH) + (size_t)c.ystore * YSTORE_ROWS * 64;
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    xs[j * EPI_THREADS + et] = f32_to_bf16_bits(v[j]);
                named_bar_sync(1, EPI_THREADS);
                const int fe = et & 63, j0 = (et >> 6) * 8;
#pragma unroll
                for (int jj = 0; jj < 8; ++jj) {
                    const int j = j0 + jj;
                    const float g = bf_lo(xs[j * EPI_THREADS + fe]), u = bf_lo(xs[j * EPI_THREADS + 64 + fe]);
                    box[(sub + j) * 64 + fe] = f32_to_bf16_bits(g / (1.0f + expf(-g)) * u);
                }
                if (sub + 16 == YSTORE_ROWS || c0 + 16 >= ti.cnt) {
                    fence_proxy_async_smem(); // generic-proxy writes, read by the TMA
                    named_bar_sync(1, EPI_THREADS);
                    if (et == 0) {
                        tma_store_2d(&maps.y, box, ti.n0 >> 1, ti.r0 + c0 - sub);
                        bulk_commit();
                        if (c.ystore == 1)
                            bulk_wait_read<0>();
                        else
                            bulk_wait_read<1>(); // the other buffer is free again
                    }
                }
                named_bar_sync(1, EPI_THREADS); // xs is written again by the next rows
            } else if (C == 1 && c.ystore) {
                // rows c0..c0+15 into the staging box (row-major [row][128
                // features] bf16); a full box (or the tile's last rows) goes out
                // as one TMA store, rows past the tensor clipped
                const int sub = c0 % YSTORE_ROWS, bi = (c0 / YSTORE_ROWS) % nys;
                uint16_t *box = reinterpret_cast<uint16_t *>(ybuf) + (size_t)bi * YSTORE_ROWS * TC_BM;
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    box[(sub + j) * TC_BM + et] = f32_to_bf16_bits(v[j]);
                if (sub + 16 == YSTORE_ROWS || c0 + 16 >= ti.cnt) {
                    const int brows = min(YSTORE_ROWS, ti.cnt - (c0 - sub));
                    if (brows < YSTORE_ROWS && c.static_tiles < 0) {
                        // a tile of an expert segment: the rows past it belong to
                        // the next segment, so this last box goes out element-wise
                        // (each thread its own feature column)
                        if (n < p.N)
                            for (int rr = 0; rr < brows; ++rr)
                                p.y[(int64_t)(ti.r0 + c0 - sub + rr) * p.y_stride + n] = box[rr * TC_BM + et];
                    } else {
                        fence_proxy_async_smem(); // generic-proxy writes, read by the TMA
                        named_bar_sync(1, EPI_THREADS);
                        if (et == 0) {
                            tma_store_2d(&maps.y, box, ti.n0, ti.r0 + c0 - sub);
                            bulk_commit();
                            if (nys == 1)
                                bulk_wait_read<0>();
                            else
                                bulk_wait_read<1>(); // the other buffer is free again
                        }
                        named_bar_sync(1, EPI_THREADS);
                    }
                }
            } else if (C == 1) {
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
        if (C == 1 && c.ystore && et == 0)
            bulk_wait_read<0>(); // the XH buffers are staged again by the next item
        named_bar_sync(1, EPI_THREADS);
        if (et == 0) {
            mbar_arrive(bars->acc_empty + buf);
            if (mode == 1 && c.borrow)
                mbar_arrive(bars->acc_empty + (buf ^ 1));
            if (C > 1)
                atomicAdd(p.ws.tile_cnt + tile, 1);
        }
        if (C > 1) {
            // every part of the tile written: sum this part's share of the columns
            if (et == 0 && !wait_count(p.ws.tile_cnt + tile, C + c.extra_parts, c.wait_ns))
                flag_abort(p, bars);
            named_bar_sync(1, EPI_THREADS);
            if (aborted(bars))
                break;
            const float *parts = p.ws.part + (size_t)tile * C * c.tn * EPI_THREADS;
            const size_t pstride = (size_t)c.tn * EPI_THREADS;
            const int cb = part * ti.cnt / C, ce = (part + 1) * ti.cnt / C;
            if (p.gated) {
                // act of 4 consecutive features (fq) x every 8th column of the
                // share: gate rows 4 fq.. and up rows 64 + 4 fq.. of the tile,
                // each summed in part order and rounded to bf16, then silu(g) * u
                // rounded once
                const int fq = et & 15, cg8 = et >> 4;
                const int fa = (ti.n0 >> 1) + 4 * fq;
                for (int cc = cb + cg8; cc < ce; cc += 8) {
                    float4 g = make_float4(0.f, 0.f, 0.f, 0.f), u = g;
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        if (q < C) {
                            const float *pc = parts + q * pstride + (size_t)cc * EPI_THREADS;
                            const float4 gq = __ldcg(reinterpret_cast<const float4 *>(pc) + fq);
                            const float4 uq = __ldcg(reinterpret_cast<const float4 *>(pc + 64) + fq);
                            if (q == 0) {
                                g = gq;
                                u = uq;
                            } else {
                                g.x += gq.x; g.y += gq.y; g.z += gq.z; g.w += gq.w;
                                u.x += uq.x; u.y += uq.y; u.z += uq.z; u.w += uq.w;
                            }
                        }
                    const float gv[4] = {g.x, g.y, g.z, g.w}, uv[4] = {u.x, u.y, u.z, u.w};
                    uint16_t *ar = p.y + (int64_t)(ti.r0 + cc) * p.y_stride;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float gb = bf_lo(f32_to_bf16_bits(gv[i])), ub = bf_lo(f32_to_bf16_bits(uv[i]));
                        if (fa + i < p.I)
                            ar[fa + i] = f32_to_bf16_bits(gb / (1.0f + expf(-gb)) * ub);
                    }
                }
                named_bar_sync(1, EPI_THREADS); // per-item state is rewritten by the next item
                continue;
            }
            // thread = 4 consecutive features (quad) x every 4th column of the
            // share: 16-byte loads, each warp reading whole 512-byte column rows
            const int quad = et & 31, cg = et >> 5;
            const int nq = ti.n0 + 4 * quad;
            for (int col0 = cb + cg; col0 < ce; col0 += 4 * 8) {
                float4 acc[8][4];
#pragma unroll
                for (int jj = 0; jj < 8; ++jj)
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        // only the parts and columns that exist are loaded
                        const int cc = col0 + 4 * jj;
                        acc[jj][q] = (q < C && cc < ce)
                                         ? __ldcg(reinterpret_cast<const float4 *>(parts + q * pstride +
                                                                                   (size_t)cc * EPI_THREADS) +
                                                  quad)
                                         : make_float4(0.f, 0.f, 0.f, 0.f);
                    }
#pragma unroll
                for (int jj = 0; jj < 8; ++jj) {
                    const int cc = col0 + 4 * jj;
                    if (cc >= ce)
                        continue;
                    float4 y = acc[jj][0];
#pragma unroll
                    for (int q = 1; q < 4; ++q)
                        if (q < C) {
                            y.x += acc[jj][q].x;
                            y.y += acc[jj][q].y;
                            y.z += acc[jj][q].z;
                            y.w += acc[jj][q].w;
                        }
                    uint16_t *yr = p.y + (int64_t)(ti.r0 + cc) * p.y_stride;
                    if (nq + 0 < p.N) yr[nq + 0] = f32_to_bf16_bits(y.x);
                    if (nq + 1 < p.N) yr[nq + 1] = f32_to_bf16_bits(y.y);
                    if (nq + 2 < p.N) yr[nq + 2] = f32_to_bf16_bits(y.z);
                    if (nq + 3 < p.N) yr[nq + 3] = f32_to_bf16_bits(y.w);
                }
            }
        }
        named_bar_sync(1, EPI_THREADS); // per-item state is rewritten by the next item
    }
    if (!shrink_done) { // a CTA without items still runs its shrink units
        if (!routed)
            route_wait();
        epi_shrink(p, unit_off, seg_off, red, um, et);
    }
    if (c.local_route && !grp_joined && shrink_done)
        named_bar_sync(4, SHRINK_GROUP_THREADS + EPI_THREADS);
    if (c.ystore && et == 0)
        bulk_wait_all(); // the y stores have landed
}

// The shrink tiles' maps as a kernel argument: present only in the
// instantiation that runs them.
template <bool kStc> struct StcMapsArg {
    StcMaps m;
};
template <> struct StcMapsArg<false> {
    int none;
};

// kStc: the launch runs shrink tiles (a separate instantiation, so the
// launches without them keep the smaller code and arguments of the other).
template <bool kStc>
__global__ void __launch_bounds__(TC_THREADS, 1)
    tc_kernel(const __grid_constant__ TmapSet maps, const __grid_constant__ Params p,
              const __grid_constant__ TcCfg c, const __grid_constant__ StcMapsArg<kStc> sm)
{
    extern __shared__ uint8_t tc_smem_raw[];
    uint8_t *smem = align1024(tc_smem_raw);
    Bars *bars = reinterpret_cast<Bars *>(smem + c.bar_off);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // The next call's routing kernel may launch now and wait in place (it
    // reads nothing before this kernel has completed), so its launch latency
    // is hidden behind this one.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (threadIdx.x == 0) {
        for (int i = 0; i < c.stages; ++i) {
            mbar_init(bars->full + i, 1); // one arrival; the W and x copies are counted in bytes
            mbar_init(bars->empty + i, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bars->acc_full + b, 1);
            mbar_init(bars->acc_empty + b, 1);
        }
        for (int r = 0; r < 2; ++r) {
            mbar_init(bars->x_full + r, 1);
            mbar_init(bars->x_empty + r, 1);
        }
        mbar_init(&bars->base_done, 1);
        mbar_init(&bars->epi_done, EPI_THREADS);
        bars->abort_flag = 0;
        fence_barrier_init();
        fence_proxy_async_smem();
        prefetch_tmap(&maps.x);
        for (int e = 0; e < p.E; ++e)
            prefetch_tmap(&maps.w[e]);
    }
    if (warp == 1)
        tmem_alloc(&bars->tmem_base, c.tmem_cols);
    if (warp >= 4 && c.static_tiles >= 0) {
        // warm L2 with what the epilogue reads first: its first tile's slots
        // and the slot tables (one line of 32 entries per thread)
        const int et = threadIdx.x - (TC_THREADS - EPI_THREADS);
        TileInfo t0;
        const int r0 = get_tile(p, c, blockIdx.x / c.csplit, c.static_tiles, t0) ? t0.r0 : 0;
        if (et < c.tn && r0 + et < p.rows && (et & 31) == 0)
            prefetch_l2(p.seq_slot + r0 + et);
        for (int s = et * 32; s < p.L; s += EPI_THREADS * 32) {
            prefetch_l2(p.tab[0].a_table + s);
            prefetch_l2(p.tab[0].b_table + s);
            prefetch_l2(p.tab[0].scale_table + s);
            prefetch_l2(p.tab[0].rank_table + s);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;

    // the shrink tiles of this CTA (batches from 2048 rows), before its items:
    // they publish h for the epilogues of every CTA
    const StcArgs sa{p.stc_tiles, p.stc_rs, p.stc_amap, c.stc_stages};
    bool stc_wrote = false;
    if constexpr (kStc)
        stc_wrote = p.stc_tiles > 0 && stc_phase(sm.m.sx, sm.m.sa, p, sa, smem, tmem);

    if (warp == 0) {
        if (lane == 0)
            produce(maps, p, c, bars, smem);
    } else if (warp == 1) {
        if (lane == 0)
            issue_mma(p, c, bars, smem, tmem);
    } else if (warp < 4) {
        if (c.local_route)
            shrink_warps(p, c, smem);
        else if (stc_wrote && warp == 2 && lane == 0)
            stc_publish(p, sa);
    } else {
        epilogue<kStc>(maps, p, c, bars, smem, tmem);
        tc_fence_before();
        mbar_arrive(&bars->epi_done);
    }
    __syncwarp();
    if (warp == 1) {
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

// Shared-memory layout of one launch for a given plan. The pipeline stages,
// XB and XH start on 1024-byte boundaries (the 128-byte swizzle repeats every
// 8 rows of 128 B): stage_bytes, XB_BLOCK and tn * 128 are multiples of 1024.
static TcCfg make_cfg(const Params &p, const TcPlan &plan, bool dyn)
{
    TcCfg c;
    memset(&c, 0, sizeof c);
    c.tn = plan.tn;
    c.kc = plan.kc;
    c.csplit = plan.csplit;
    c.use3d = plan.use3d;
    c.xblk = plan.xblk;
    c.hl = plan.hl;
    c.borrow = 3 * c.tn > 512 ? 1 : 0;
    c.local_route = (!dyn && p.E == 1 && p.rows <= c.tn && p.L <= LR_MAX_L && !p.no_units) ? 1 : 0;
    c.n_tiles = (p.N + TC_BM - 1) / TC_BM;
    c.kchunks = (p.K + 63) / 64;
    c.kstages = (c.kchunks + c.kc - 1) / c.kc;
    c.x_chunk = (uint32_t)c.tn * 128u;
    c.pair = plan.pair;
    c.stage_bytes = (uint32_t)c.kc * ((c.pair ? 2u : 1u) * W_CHUNK_BYTES + c.x_chunk);
    c.stages = plan.stages;
    uint32_t o = (uint32_t)c.stages * c.stage_bytes;
    c.xb_off = o;
    o += (uint32_t)c.xblk * XB_BLOCK;
    c.xh_off = o;
    o += (uint32_t)c.hl * (uint32_t)c.xblk * (uint32_t)c.tn * 128u;
    c.aux_off = align_up(o, 16);
    o = c.aux_off + (uint32_t)sizeof(EpiAux);
    c.meta_off = align_up(o, 16);
    o = c.meta_off + 2u * (uint32_t)(p.E * (p.L + 1) + 1) * 4u;
    c.red_off = align_up(o, 16);
    o = c.red_off + (uint32_t)(SHRINK_WARPS * 32 * 4);
    c.umeta_off = align_up(o, 16);
    o = c.umeta_off + (uint32_t)(UNIT_BATCH * sizeof(UnitMeta));
    c.bar_off = align_up(o, 16);
    c.smem_bytes = 1024u + c.bar_off + (uint32_t)sizeof(Bars);
    c.tmem_cols = c.borrow ? 512u : pow2_at_least(3u * (uint32_t)c.tn);
    // the launch's shrink tiles: stages below this kernel's barriers, 256 TMEM columns
    c.stc_stages = 0;
    if (p.stc_tiles > 0) {
        int s = STC_MAX_STAGES;
        while (s > 2 && stc_smem_bytes(s) > c.bar_off)
            --s;
        c.stc_stages = s;
        if (c.tmem_cols < (uint32_t)STC_MAX_N)
            c.tmem_cols = STC_MAX_N;
    }
    // region 1: XB blocks then XH blocks (hl planes) carved from the stages
    c.xblk_b = (int)min(8u, (uint32_t)c.stages * c.stage_bytes / (XB_BLOCK + (uint32_t)c.hl * (uint32_t)c.tn * 128u));
    const int tt = (p.rows + c.tn - 1) / c.tn;
    c.static_tiles = dyn ? -1 : tt * c.n_tiles;
    c.tgroup = (!dyn && tt > 1) ? (tt < TC_TGROUP ? tt : TC_TGROUP) : 1;
    // y through TMA stores from the XH buffers (free while an item drains):
    // one K part and room for a box (expert tiles write a last partial box
    // element-wise)
    const uint32_t xh_bytes = (uint32_t)c.hl * (uint32_t)c.xblk * (uint32_t)c.tn * 128u;
    const uint32_t box_bytes = (uint32_t)YSTORE_ROWS * TC_BM * 2u;
    c.ystore = (p.ystore_ok && c.csplit == 1 && xh_bytes >= box_bytes) ? (xh_bytes >= 2 * box_bytes ? 2 : 1) : 0;
    return c;
}

static constexpr uint32_t SMEM_LIMIT = 232448; // 227 KB per CTA

// Choose K chunks per stage, stages, expand k blocks and XH planes. In order:
// at least 3 stages; W bytes in flight up to 6 chunks (96 KB); an expand round
// of at least min(2, worst case) k blocks; two XH planes; more k blocks (up to
// every slot of a K part at the pool rank); then larger copies. Per-expert
// tiles (MoE) take the widest K chunk that leaves two stages first, or
// feature-tile pairs (below).
TcPlan plan_tc(const Params &p, bool dyn)
{
    TcPlan plan;
    memset(&plan, 0, sizeof plan);
    plan.tn = p.tn;
    plan.use3d = (p.K % 64) == 0 ? 1 : 0;
    const int kchunks = (p.K + 63) / 64;
    plan.csplit = tc_csplit(p.rows, p.K, dyn);
    const int slots = min(p.tn, (p.L + plan.csplit - 1) / plan.csplit);
    const int need_blk = max(1, min(8, (slots * ((p.R + 15) & ~15) + 63) / 64));
    long best = -1;
    TcPlan cand = plan;
    const int kcs[3] = {4, 2, 1};
    for (int ik = 0; ik < 3; ++ik) {
        const int kc = kcs[ik];
        if (kc > 1 && !plan.use3d)
            continue;
        if ((kchunks + kc - 1) / kc < plan.csplit)
            continue;
        for (int st = MAX_STAGES; st >= 2; --st)
            for (int xb = need_blk; xb >= 1; --xb)
                for (int hl = 2; hl >= 1; --hl) {
                    cand.kc = kc;
                    cand.stages = st;
                    cand.xblk = xb;
                    cand.hl = hl;
                    const TcCfg c0 = make_cfg(p, cand, dyn);
                    if (c0.smem_bytes > SMEM_LIMIT)
                        continue;
                    // expert weights (per-expert tiles, long rows): the widest K
                    // chunk per row with two stages first -- each W row then comes in
                    // kc * 128 contiguous bytes (measured: MoE 240 -> 222 us at kc 2,
                    // the decode gather 190 -> 183 us at kc 4); otherwise three
                    // stages first, then W bytes in flight
                    const long score = dyn ? (st >= 2 ? 100000000L : 0L) + kc * 10000000L +
                                                 min(st * kc, 8) * 1000000L +
                                                 min(xb, min(need_blk, 2)) * 100000L + hl * 10000L +
                                                 xb * 1000L + st
                                           : (st >= 3 ? 10000000L : 0L) + min(st * kc, 6) * 1000000L +
                                                 min(xb, min(need_blk, 2)) * 100000L + hl * 10000L +
                                                 xb * 1000L + kc * 10L + st;
                    if (score > best) {
                        best = score;
                        plan = cand;
                    }
                }
    }
    if (best < 0) {
        plan.kc = 1;
        plan.stages = 2;
        plan.xblk = 1;
        plan.hl = 1;
    }
    // Per-expert tiles of at least 128 token rows: feature-tile pairs. Each
    // stage then carries two W boxes for one x box, so the shared memory of a
    // stage buys more W in flight (x, an L2 hit, is as large as W at these
    // tiles), and a CTA's pair shares its slot lists and staged s * h.
    // Measured on the MoE down projection (tn 144): 235 -> 207 us per call with
    // three stages of one K chunk; two stages 246 us. Small tiles (the decode
    // gather, tn 32) measured slower paired (192 -> 205 us).
    if (dyn && plan.use3d && !p.gated && plan.csplit == 1 && p.tn >= TC_BM && 3 * p.tn <= 512 &&
        ((p.N + TC_BM - 1) / TC_BM) % 2 == 0) {
        TcPlan pp = plan, pb = plan;
        long pbest = -1;
        pp.pair = 1;
        for (int kc = 2; kc >= 1; --kc)
            for (int st = MAX_STAGES; st >= 3; --st)
                for (int xb = need_blk; xb >= 1; --xb)
                    for (int hl = 2; hl >= 1; --hl) {
                        pp.kc = kc;
                        pp.stages = st;
                        pp.xblk = xb;
                        pp.hl = hl;
                        if (make_cfg(p, pp, dyn).smem_bytes > SMEM_LIMIT)
                            continue;
                        const long score = min(st * kc, 6) * 1000000L + min(xb, min(need_blk, 2)) * 100000L +
                                           hl * 10000L + xb * 1000L + kc * 10L + st;
                        if (score > pbest) {
                            pbest = score;
                            pb = pp;
                        }
                    }
        if (pbest >= 0)
            plan = pb;
    }
    return plan;
}

// The gated view needs 64-wide K chunks and, with one K part, the TMA-store
// drain (p.ystore_ok: act 16-byte aligned rows): the plan of these rows must
// give them. With several K parts the split-K sum forms act.
bool tc_gated_ok(const Params &p)
{
    if (p.expert_offsets != nullptr || p.K % 64 != 0 || p.I % 64 != 0 || p.N != 2 * p.I)
        return false;
    const Params &q = p;
    const TcPlan plan = plan_tc(q, false);
    const TcCfg c = make_cfg(q, plan, false);
    const uint32_t xh_bytes = (uint32_t)c.hl * (uint32_t)c.xblk * (uint32_t)c.tn * 128u;
    // act boxes [64 rows][64] bf16, then the [16][128] bf16 exchange rows
    // one K part: the drain writes act through TMA boxes; several: the split-K
    // sum forms it
    if (c.csplit > 1)
        return plan.use3d && c.smem_bytes <= SMEM_LIMIT;
    return plan.use3d && c.ystore > 0 && c.smem_bytes <= SMEM_LIMIT &&
           xh_bytes >= (uint32_t)c.ystore * YSTORE_ROWS * 64u * 2u + 16u * EPI_THREADS * 2u;
}

cudaError_t launch_tc(const Params &p, const TmapSet &maps, const StcMaps &stc_maps, const TcPlan &plan, int num_sms,
                      cudaStream_t st)
{
    const bool dyn = p.expert_offsets != nullptr;
    TcCfg c = make_cfg(p, plan, dyn);
    uint64_t tw = 0;
    test_hook_get(tw, c.extra_parts);
    c.wait_ns = tw ? tw : WAIT_NS;
    static std::atomic<uint64_t> raised{0}, raised_stc{0};
    const bool stc = p.stc_tiles > 0;
    cudaError_t ea = stc ? raise_smem_limit(raised_stc, tc_kernel<true>, (int)SMEM_LIMIT)
                         : raise_smem_limit(raised, tc_kernel<false>, (int)SMEM_LIMIT);
    if (ea != cudaSuccess)
        return ea;
    if (c.smem_bytes > SMEM_LIMIT || (stc && stc_smem_bytes(c.stc_stages) > c.bar_off))
        return cudaErrorInvalidConfiguration;
    // One CTA per SM at most (the in-launch waits need every CTA resident; the
    // cooperative launch below makes sure they are); never more CTAs than work
    // items.
    int grid = num_sms;
    if (c.static_tiles >= 0 && c.static_tiles * c.csplit < grid)
        grid = c.static_tiles * c.csplit;
    grid = grid / c.csplit * c.csplit;

    // Where CTAs wait on counters other CTAs write (split-K parts, in-launch
    // shrink units) the launch is cooperative, so the whole grid is resident
    // at once or the launch fails -- never a wait on a CTA that has not
    // started. Launches without such waits (one K part, h from the shrink
    // kernel) stay plain, so they start beside the kernel before them.
    const bool waits = c.csplit > 1 || !p.no_units || p.stc_tiles > 0;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeCooperative;
    attr[1].val.cooperative = waits ? 1 : 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(TC_THREADS);
    cfg.dynamicSmemBytes = c.smem_bytes;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    if (stc) {
        StcMapsArg<true> a;
        a.m = stc_maps;
        return cudaLaunchKernelEx(&cfg, tc_kernel<true>, maps, p, c, a);
    }
    return cudaLaunchKernelEx(&cfg, tc_kernel<false>, maps, p, c, StcMapsArg<false>{0});
}

} // namespace rd
