// Embedding row gather with the adapted rows:
//
//   y[i, :] = E[t_i, :] + s * B[t_i, :] A      t_i = tokens[i], s = scale of slot seq_slot[i]
//
// ferrox-core `weight_matrix/lora.rs`, `LoraDelta::add_row_to`: the delta of one
// row of the adapted matrix s B A is what a token-embedding gather needs; frink
// `lora_attach.rs`, `checked_pair`: the adapted matrix of an embedding is
// [n_vocab][n_embd], its pair arrives flipped (a row of [n_vocab][rank] per token
// times [n_embd][rank]).
//
// Rows arrive grouped by slot (the routing kernel's stable sort). Each bucket
// of rows is cut into balanced chunks of at most 128 rows; a work item is one
// chunk x one tile of ft embedding features (f0 .. f0 + ft - 1).
//   delta chunk (an active slot): D[j][e] = sum_r B[t_j][r] * At[f0 + e][r] on the
//     tensor cores (UMMA M = 128 chunk rows, N = ft features, K = the slot's rank
//     rounded up to 16), fp32 in TMEM (lane = row, column = feature);
//     y = bf16(E + s * D), one rounding.
//   copy chunk (no delta): y = the E row's bytes, copied global to global.
// A delta item's E rows come into shared memory by 16-byte cp.async copies
// (chunk c of row j at position c ^ (j & 7): the epilogue's row-per-thread
// reads are free of bank conflicts); the epilogue thread of row j reads its D
// row from TMEM 16 columns at a time, adds, rounds and stores 32 bytes of y.
//
// Warps 0-3 (loader): per delta item the B rows of the chunk, the A^T tile
// (cp.async into the 128-byte-swizzled K-major layout) and the E rows, without
// waiting for any of them: the copies' completion is counted on mbarriers.
// Warp 8 (one thread) issues the UMMAs once an item's operands have landed.
// Warps 4-7 (epilogue): TMEM -> scale -> add -> store, and the copy chunks.
// Two buffers of each kind: the loader runs up to two items ahead. Every wait
// is bounded; a wait that gives up sets LORA_FLAG_WAIT_TIMEOUT and the CTA
// unwinds (its copies and UMMAs in flight are waited for first).
#include <cstring>

#include "lora_internal.cuh"
#include "ptx.cuh"

namespace rd {

namespace {

constexpr int LOADERS = 256;                 // warps 0-7: the loader group
constexpr int EPIS = 128;                    // warps 8-11: the epilogue group
constexpr int EPI0 = LOADERS;                // first epilogue thread
constexpr int MMA_WARP = (LOADERS + EPIS) / 32; // warp 12: the UMMA issuer
constexpr int COL_SPLIT = EPIS / EMBED_CHUNK_ROWS; // epilogue threads per chunk row (each a share of the columns)
constexpr int EMB_THREADS = LOADERS + EPIS + 32;
constexpr int SORTERS = 256;                 // threads of the in-kernel routing sort
constexpr int CH = EMBED_CHUNK_ROWS;         // rows per chunk (UMMA M)
constexpr uint32_t KB_BYTES_G = CH * 128;    // one 64-wide k block of the chunk's B rows
constexpr int BAR_LOAD = 1, BAR_EPI = 2;     // named barriers of the two groups

struct EmbBars {
    uint64_t op_full[2];   // operands of buffer b have landed (one arrival per loader thread)
    uint64_t op_empty[2];  // the UMMAs that read operand buffer b are done
    uint64_t acc_full[2];  // accumulator b holds an item's D
    uint64_t acc_empty[2]; // the epilogue has read accumulator b
    uint64_t e_full[2];    // E rows of row buffer b have landed (one arrival per loader thread)
    uint64_t e_empty[2];   // the epilogue has read row buffer b
    uint64_t fin;          // every UMMA of this CTA is done
    uint32_t tmem_base;
    int abort_flag;
    int go[2];             // a group leader's wait result, broadcast to its group
};

struct EmbCfg {
    uint32_t g_bytes, a_bytes, e_bytes; // one buffer of B rows / of the A^T tile / of E rows
    uint32_t g_off[2], a_off[2], e_off[2];
    uint32_t seg_off, cpre_off, act_off, cbase_off, crem_off, ltok_off, crow_off, sperm_off, stok_off, slot_off,
        bar_off;
    uint32_t smem_bytes, tmem_cols;
};

struct Item {
    int delta; // 1: an active slot's chunk
    int slot;
    int lo, n; // rows perm[lo .. lo + n) of the sorted order
    int f0, fw;
};

__device__ __forceinline__ uint8_t *align1024(uint8_t *ptr)
{
    uintptr_t a = reinterpret_cast<uintptr_t>(ptr);
    return reinterpret_cast<uint8_t *>((a + 1023) & ~uintptr_t(1023));
}

__device__ __forceinline__ bool aborted(EmbBars *b) { return *(volatile int *)&b->abort_flag != 0; }

__device__ __forceinline__ void flag_abort(const EmbedParams &p, EmbBars *b)
{
    *(volatile int *)&b->abort_flag = 1;
    atomicOr(p.ws.status, (uint32_t)LORA_FLAG_WAIT_TIMEOUT);
}

// The bucket list: bucket b holds seg[b+1] - seg[b] rows in
// cpre[b+1] - cpre[b] chunks, balanced: chunk q has cbase[b] rows, plus one
// for q < crem[b].
struct Buckets {
    const int *seg, *cpre, *cbase, *crem;
    const uint8_t *act;
};

// A CTA's work items in order: item w = chunk w / nft x feature tile w % nft,
// for w = blockIdx.x, + gridDim.x, ... Stepped without dividing; the bucket of
// the current chunk is a cursor that only moves forward.
struct ItemIter {
    int c, f, b;
    int dc, df; // gridDim.x / nft, gridDim.x % nft
};

__device__ __forceinline__ ItemIter iter_begin(int nft)
{
    ItemIter r;
    r.c = (int)blockIdx.x / nft;
    r.f = (int)blockIdx.x - r.c * nft;
    r.dc = (int)gridDim.x / nft;
    r.df = (int)gridDim.x - r.dc * nft;
    r.b = 0;
    return r;
}

__device__ __forceinline__ void iter_next(ItemIter &r, int nft)
{
    r.c += r.dc;
    r.f += r.df;
    if (r.f >= nft) {
        r.f -= nft;
        ++r.c;
    }
}

// The item at the iterator (chunk c < the chunk count).
__device__ __forceinline__ Item iter_item(const EmbedParams &p, const Buckets &bk, ItemIter &r)
{
    while (bk.cpre[r.b + 1] <= r.c)
        ++r.b;
    const int b = r.b, q = r.c - bk.cpre[b];
    const int base = bk.cbase[b], rem = bk.crem[b];
    Item it;
    it.delta = bk.act[b];
    it.slot = b - 1;
    it.lo = bk.seg[b] + q * base + min(q, rem);
    it.n = base + (q < rem ? 1 : 0);
    it.f0 = r.f * p.ft;
    it.fw = min(p.ft, p.n_embd - it.f0);
    return it;
}

// What a delta chunk needs of its slot, read once per CTA from the tables
// (bucket b = slot b - 1).
struct SlotRec {
    const uint16_t *at; // A^T [n_embd][R]
    const uint16_t *b;  // B [vocab][R]
    float scale;
    int rank;
};

// Exclusive scan of one value per thread over the block.
__device__ __forceinline__ int block_scan(int v, int *tmp, int &total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o)
            incl += t;
    }
    if (lane == 31)
        tmp[warp] = incl;
    __syncthreads();
    int wex = 0;
    total = 0;
#pragma unroll
    for (int q = 0; q < EMB_THREADS / 32; ++q) {
        const int t = tmp[q];
        if (q < warp)
            wex += t;
        total += t;
    }
    __syncthreads();
    return wex + incl - v;
}

// Byte offset of 16-byte chunk c of row j in a row buffer with `cpr` chunks
// per row (4, 8 or 16): chunks permuted within each group of up to eight by
// the row's low bits, so eight consecutive rows read at one chunk index hit
// distinct banks.
__device__ __forceinline__ uint32_t erow_chunk(int j, int c, int cpr)
{
    const int m = cpr >= 8 ? 7 : cpr - 1;
    return (uint32_t)(j * cpr + (c ^ (j & m))) << 4;
}

// Where a chunk's rows come from: the sorted order kept in shared memory by
// this CTA's own routing pass (perm and tokens), or the routing kernel's perm
// in global memory with the tokens looked up per row.
struct RowView {
    const int32_t *perm; // sorted position -> row
    const int32_t *stok; // sorted position -> token, -1 = out of range; nullptr: look it up
};

__device__ __forceinline__ void row_at(const EmbedParams &p, const RowView &v, int pos, int &row, int &tk)
{
    row = v.perm[pos];
    if (v.stok != nullptr) {
        tk = v.stok[pos];
        return;
    }
    tk = p.tokens[row];
    if (tk < 0 || tk >= p.vocab) {
        tk = -1;
        atomicOr(p.ws.status, (uint32_t)LORA_FLAG_TOKEN_RANGE);
    }
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Two floats -> packed bf16 pair (lo in the low half), each rounded to
// nearest even.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

} // namespace

namespace {

// Loader group (threads 0 .. 255) over the delta chunks. Per item the leader
// waits until buffer b is free (its UMMAs done, its E rows read); the group
// reads the chunk's tokens (one row per thread), then issues the operand
// copies (B rows, A^T tile; their landing counted on op_full[b]) and the E row
// copies (counted on e_full[b]), and moves on without waiting for them.
__device__ void embed_loader(const EmbedParams &p, const EmbCfg &c, EmbBars *bars, uint8_t *smem,
                             const SlotRec *srec, const Buckets &bk, int chunks, const RowView rv)
{
    const int t = threadIdx.x;
    int32_t *tok = reinterpret_cast<int32_t *>(smem + c.ltok_off); // [128]: token of each chunk row, -1 = out of range
    const int ecpr = p.ft >> 3;                                    // 16-byte chunks of a row in the row buffer
    const uint32_t a_kb = (uint32_t)p.ft * 128u;                   // one 64-wide k block of the A^T tile
    // the E-row copy of thread t: chunk eq of rows ej0 + estep * i (estep a
    // multiple of the swizzle period, so the chunk's place is fixed)
    const int lg = 31 - __clz(ecpr);
    const int eq = t & (ecpr - 1), ej0 = t >> lg, estep = LOADERS >> lg;
    const uint32_t erow_bytes = (uint32_t)ecpr * 16u;
    const uint32_t eswz = erow_chunk(ej0, eq, ecpr) - (uint32_t)ej0 * erow_bytes;
    int u[2] = {0, 0};
    int d = 0;
    for (ItemIter r = iter_begin(p.nft); r.c < chunks; iter_next(r, p.nft)) {
        const Item it = iter_item(p, bk, r);
        if (!it.delta)
            continue; // copy chunks are the epilogue's alone
        const int b = d & 1;
        if (t == 0) {
            const uint32_t par = ((uint32_t)u[b] & 1u) ^ 1u;
            const bool ok = !aborted(bars) && mbar_wait(&bars->e_empty[b], par) &&
                            mbar_wait(&bars->op_empty[b], par);
            if (!ok && !aborted(bars))
                flag_abort(p, bars);
            *(volatile int *)&bars->go[0] = ok ? 1 : 0;
        }
        named_bar_sync(BAR_LOAD, LOADERS);
        if (*(volatile int *)&bars->go[0] == 0)
            break;
        if (t < it.n) {
            int row, tk;
            row_at(p, rv, it.lo + t, row, tk);
            tok[t] = tk;
        }
        named_bar_sync(BAR_LOAD, LOADERS); // tok[] complete

        const SlotRec sr = srec[it.slot + 1];
        const int pk = (sr.rank + 15) & ~15; // UMMA K granularity; k >= rank is zero-filled
        const int cpr = pk >> 3;             // 16-byte chunks of a staged operand row
        uint8_t *gbuf = smem + c.g_off[b], *abuf = smem + c.a_off[b], *eb = smem + c.e_off[b];
        // Operands: thread t copies 16-byte chunk t & 7 of each 64-wide k block
        // of rows t / 8, t / 8 + 32, ... (a row's eight chunks on consecutive
        // threads; the swizzle term (chunk ^ row) & 7 is the same for all of a
        // thread's rows). B rows of the chunk are the UMMA's A operand, A^T
        // rows f0 .. f0 + fw - 1 its B operand; rows past n and past fw are not
        // staged: the D rows and columns they feed are never read.
        const int q8 = t & 7, r16 = t >> 3;
        const uint32_t swz = (uint32_t)((q8 ^ (r16 & 7)) << 4);
        for (int kb = 0; kb * 8 < cpr; ++kb) {
            const int q = kb * 8 + q8; // 16-byte chunk along k
            if (q >= cpr)
                break;
            const bool kin = q * 8 < sr.rank;
            uint8_t *gdst = gbuf + kb * KB_BYTES_G + swz;
            for (int j = r16; j < it.n; j += LOADERS / 8) {
                const int tk = tok[j];
                const bool has = kin && tk >= 0;
                cp_async_16(gdst + j * 128, sr.b + (has ? (size_t)tk * p.R + q * 8 : 0), has ? 16u : 0u);
            }
            uint8_t *adst = abuf + kb * a_kb + swz;
            const uint16_t *asrc = sr.at + (size_t)it.f0 * p.R + q * 8;
            for (int e = r16; e < it.fw; e += LOADERS / 8)
                cp_async_16(adst + e * 128, kin ? asrc + (size_t)e * p.R : sr.at, kin ? 16u : 0u);
        }
        cp_async_mbar_arrive_noinc(&bars->op_full[b]);
        // E rows: thread t copies chunk t % ecpr of rows t / ecpr, + 256 / ecpr, ...
        if (eq < (it.fw >> 3)) {
            const uint16_t *esrc = p.E + it.f0 + eq * 8;
            for (int j = ej0; j < it.n; j += estep) {
                const int tk = tok[j];
                if (tk >= 0)
                    cp_async_16(eb + (uint32_t)j * erow_bytes + eswz, esrc + (size_t)tk * p.n_embd, 16u);
            }
        }
        cp_async_mbar_arrive_noinc(&bars->e_full[b]);
        ++u[b];
        ++d;
    }
    cp_async_wait_all(); // nothing of this CTA may be in flight when it exits
}

// UMMA issuer (one thread of warp 8): per delta item, once its operands have
// landed and its accumulator is free, D = B rows x A^T^T over the slot's rank.
__device__ void embed_mma(const EmbedParams &p, const EmbCfg &c, EmbBars *bars, uint8_t *smem, uint32_t tmem,
                          const SlotRec *srec, const Buckets &bk, int chunks)
{
    const uint32_t a_kb = (uint32_t)p.ft * 128u;
    const uint32_t idesc = idesc_bf16_f32(CH, (uint32_t)p.ft);
    int u[2] = {0, 0};
    int d = 0;
    bool issued = false;
    for (ItemIter r = iter_begin(p.nft); r.c < chunks; iter_next(r, p.nft)) {
        const Item it = iter_item(p, bk, r);
        if (!it.delta)
            continue;
        const int b = d & 1;
        const uint32_t par = (uint32_t)u[b] & 1u;
        if (aborted(bars) || !mbar_wait(&bars->op_full[b], par) || !mbar_wait(&bars->acc_empty[b], par ^ 1u)) {
            if (!aborted(bars))
                flag_abort(p, bars);
            break;
        }
        fence_proxy_async_smem(); // the copies landed through the generic proxy; the UMMAs read through the async one
        tc_fence_after();
        const int pk = (srec[it.slot + 1].rank + 15) & ~15;
        const uint32_t acc = tmem + (uint32_t)(b * p.ft);
        const uint32_t gb = smem_u32(smem + c.g_off[b]), ab = smem_u32(smem + c.a_off[b]);
        for (int k16 = 0; k16 < pk / 16; ++k16) {
            const uint32_t kb = (uint32_t)k16 >> 2, kk = ((uint32_t)k16 & 3u) * 32u;
            umma_bf16(acc, sw128_kmajor_desc(gb + kb * KB_BYTES_G + kk), sw128_kmajor_desc(ab + kb * a_kb + kk),
                      idesc, k16 > 0 ? 1u : 0u);
        }
        umma_commit(&bars->op_empty[b]);
        umma_commit(&bars->acc_full[b]);
        issued = true;
        ++u[b];
        ++d;
    }
    if (issued) { // every UMMA done before the CTA frees TMEM and exits
        umma_commit(&bars->fin);
        if (!mbar_wait(&bars->fin, 0))
            flag_abort(p, bars);
    }
}

// y = bf16(e + sc * d) for eight features: e packed bf16 pairs, d fp32.
__device__ __forceinline__ uint4 add_scaled8(uint4 e, const uint32_t *d, float sc)
{
    uint4 o;
    o.x = pack_bf16x2(bf16_lo(e.x) + sc * __uint_as_float(d[0]), bf16_hi(e.x) + sc * __uint_as_float(d[1]));
    o.y = pack_bf16x2(bf16_lo(e.y) + sc * __uint_as_float(d[2]), bf16_hi(e.y) + sc * __uint_as_float(d[3]));
    o.z = pack_bf16x2(bf16_lo(e.z) + sc * __uint_as_float(d[4]), bf16_hi(e.z) + sc * __uint_as_float(d[5]));
    o.w = pack_bf16x2(bf16_lo(e.w) + sc * __uint_as_float(d[6]), bf16_hi(e.w) + sc * __uint_as_float(d[7]));
    return o;
}

// Epilogue group (threads 256 .. 383). Thread et owns row et % 128 of a delta
// chunk, its columns' share et / 128 (warp 8 + q reads TMEM lanes 32q ..
// 32q + 31): D row from TMEM 32 columns at
// a time, E row from the row buffer, 16-byte stores of y. Copy chunks: the
// group copies the E rows to y, 16 bytes per thread, a row's chunks on
// consecutive threads.
__device__ void embed_epilogue(const EmbedParams &p, const EmbCfg &c, EmbBars *bars, uint8_t *smem,
                               uint32_t tmem, const SlotRec *srec, const Buckets &bk, int chunks,
                               const RowView rv)
{
    const int et = threadIdx.x - EPI0;
    const int wq = (threadIdx.x >> 5) & 3; // TMEM lane quarter of this warp
    const int er = et & (CH - 1);          // chunk row of this thread in a delta item
    const int hh = et / CH;                // which share of the item's columns
    const int half = p.ft / COL_SPLIT;     // columns per share, a multiple of 16
    int32_t *crow = reinterpret_cast<int32_t *>(smem + c.crow_off); // [128] y row of each chunk row
    int32_t *ctok = crow + CH;                                      // [128] its token, -1 = out of range
    const int ecpr = p.ft >> 3;
    // copying rows out, thread et takes 16-byte chunk cq of rows cj0, + cstep, ...
    // (cstep a multiple of the swizzle period: the chunk's place in a row is fixed)
    const int cq = et & (ecpr - 1), cj0 = et >> (31 - __clz(ecpr)), cstep = EPIS / ecpr;
    const uint32_t erow_bytes = (uint32_t)ecpr * 16u;
    const uint32_t cswz = erow_chunk(cj0, cq, ecpr) - (uint32_t)cj0 * erow_bytes;
    const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
    int u[2] = {0, 0};
    int d = 0;
    for (ItemIter r = iter_begin(p.nft); r.c < chunks; iter_next(r, p.nft)) {
        const Item it = iter_item(p, bk, r);
        if (!it.delta) {
            if (et < it.n) {
                int i, tk;
                row_at(p, rv, it.lo + et, i, tk);
                crow[et] = i;
                ctok[et] = tk;
            }
            named_bar_sync(BAR_EPI, EPIS);
            // thread et copies chunk cq of rows cj0, cj0 + cstep, ...; four
            // loads in flight before their stores
            if (cq < (it.fw >> 3)) {
                const uint16_t *src = p.E + it.f0 + cq * 8;
                uint16_t *dst = p.y + it.f0 + cq * 8;
                for (int j0 = cj0; j0 < it.n; j0 += 4 * cstep) {
                    uint4 v[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int j = j0 + k * cstep;
                        const int tk = j < it.n ? ctok[j] : -1;
                        v[k] = tk >= 0 ? __ldg(reinterpret_cast<const uint4 *>(src + (size_t)tk * p.n_embd)) : zero;
                    }
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int j = j0 + k * cstep;
                        if (j < it.n)
                            *reinterpret_cast<uint4 *>(dst + (size_t)crow[j] * p.y_stride) = v[k];
                    }
                }
            }
            named_bar_sync(BAR_EPI, EPIS); // crow / ctok are rewritten by the next copy chunk
            continue;
        }
        const int b = d & 1;
        bool tvalid = false;
        if (er < it.n) {
            int yrow, tk;
            row_at(p, rv, it.lo + er, yrow, tk);
            tvalid = tk >= 0;
            if (hh == 0)
                crow[er] = yrow;
        }
        const float sc = srec[it.slot + 1].scale;
        if (et == 0) {
            const uint32_t par = (uint32_t)u[b] & 1u;
            const bool ok = !aborted(bars) && mbar_wait(&bars->e_full[b], par) &&
                            mbar_wait(&bars->acc_full[b], par);
            if (!ok && !aborted(bars))
                flag_abort(p, bars);
            *(volatile int *)&bars->go[1] = ok ? 1 : 0;
        }
        named_bar_sync(BAR_EPI, EPIS);
        if (*(volatile int *)&bars->go[1] == 0)
            break;
        mbar_wait(&bars->e_full[b], (uint32_t)u[b] & 1u); // complete: the copied rows are visible here
        tc_fence_after();
        uint8_t *eb = smem + c.e_off[b];
        if (wq * 32 < it.n) { // TMEM loads are per warp: a warp with no row of the chunk skips them
            const uint32_t tb = tmem + ((uint32_t)(wq * 32) << 16) + (uint32_t)(b * p.ft);
            const bool mine = er < it.n;
            const int cend = min(it.fw, (hh + 1) * half);
            for (int c0 = hh * half; c0 < cend; c0 += 64) {
                // up to four 16-column loads in flight per wait (half is a
                // multiple of 16, so column c0 + 16g below the half's end is a
                // whole load)
                uint32_t r[4][16];
#pragma unroll
                for (int g = 0; g < 4; ++g)
                    if (c0 + 16 * g < (hh + 1) * half)
                        tmem_ld16_nowait(tb + (uint32_t)(c0 + 16 * g), r[g]);
                tmem_wait_ld();
                if (mine) {
#pragma unroll
                    for (int h = 0; h < 8; ++h) {
                        const int col = c0 + 8 * h;
                        if (col < cend) {
                            uint4 *ep = reinterpret_cast<uint4 *>(eb + erow_chunk(er, col >> 3, ecpr));
                            *ep = add_scaled8(tvalid ? *ep : zero, &r[h >> 1][(h & 1) * 8], sc);
                        }
                    }
                }
            }
        }
        tc_fence_before();
        named_bar_sync(BAR_EPI, EPIS); // accumulator b is read; the y rows are final in row buffer b
        if (et == 0)
            mbar_arrive(&bars->acc_empty[b]);
        // y rows out with 16 threads (or fewer) per row: whole rows per store
        if (cq < (it.fw >> 3)) {
            uint16_t *dst = p.y + it.f0 + cq * 8;
            for (int j = cj0; j < it.n; j += cstep)
                *reinterpret_cast<uint4 *>(dst + (size_t)crow[j] * p.y_stride) =
                    *reinterpret_cast<const uint4 *>(eb + (uint32_t)j * erow_bytes + cswz);
        }
        named_bar_sync(BAR_EPI, EPIS); // row buffer b is read; crow is rewritten by the next item
        if (et == 0)
            mbar_arrive(&bars->e_empty[b]);
        ++u[b];
        ++d;
    }
}

// This CTA's own routing pass over a batch of at most EMBED_LOCAL_ROWS rows
// and EMBED_LOCAL_BUCKETS buckets: a counting sort of the rows by
// bucket (0 = no valid slot, s + 1 = slot s) into sperm / stok, bucket starts
// into seg. Deterministic, so every CTA cuts a bucket into the same chunks
// (a chunk's feature tiles run on different CTAs): thread t of the first 256
// owns rows t, t + 256, ... (coalesced loads); it counts its keys in its own
// column of cnt[nb][256] (no atomics), one warp per bucket turns the bucket's
// counts into exclusive starts, warp 0 scans the bucket totals, and each
// thread places its rows in its own order, so a bucket lists thread 0's rows,
// then thread 1's, and so on. CTA 0 writes the call's status word (there is no
// routing kernel). cnt: [nb][256] and tot: [nb] scratch; sflags: a word.
__device__ void local_route(const EmbedParams &p, int *seg, uint16_t *cnt, int *tot, int32_t *sperm,
                            int32_t *stok, int nb, uint32_t *sflags)
{
    constexpr int LR = EMBED_LOCAL_ROWS / SORTERS;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const bool sorter = tid < SORTERS;
    uint32_t *cnt32 = reinterpret_cast<uint32_t *>(cnt);
    for (int q = tid; q < nb * SORTERS / 2; q += EMB_THREADS)
        cnt32[q] = 0;
    if (tid == 0)
        *sflags = 0;
    int key[LR], tok[LR];
#pragma unroll
    for (int k = 0; k < LR; ++k) { // every load issued before any is used
        const int i = tid + k * SORTERS;
        const bool in = sorter && i < p.M;
        key[k] = in ? p.seq_slot[i] : -1;
        tok[k] = in ? p.tokens[i] : 0;
    }
    uint32_t fl = 0;
#pragma unroll
    for (int k = 0; k < LR; ++k) {
        const int i = tid + k * SORTERS;
        if (sorter && i < p.M) {
            const int sl = key[k];
            if (sl >= p.L)
                fl |= LORA_FLAG_SLOT_RANGE;
            key[k] = (sl >= 0 && sl < p.L) ? sl + 1 : 0;
            if (tok[k] < 0 || tok[k] >= p.vocab) {
                fl |= LORA_FLAG_TOKEN_RANGE;
                tok[k] = -1;
            }
        } else {
            key[k] = -1;
        }
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < LR; ++k)
        if (key[k] >= 0)
            ++cnt[key[k] * SORTERS + tid];
    __syncthreads();
    // bucket b's counts -> exclusive starts, one warp per bucket (lane: 8 entries)
    for (int b = warp; b < nb; b += EMB_THREADS / 32) {
        uint4 *rowv = reinterpret_cast<uint4 *>(cnt + b * SORTERS) + lane;
        const uint4 v = *rowv;
        uint32_t e[4] = {v.x, v.y, v.z, v.w};
        int sum = 0;
#pragma unroll
        for (int h = 0; h < 4; ++h)
            sum += (int)(e[h] & 0xffffu) + (int)(e[h] >> 16);
        int incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t2 = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o)
                incl += t2;
        }
        int run = incl - sum;
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            const int lo = (int)(e[h] & 0xffffu), hi = (int)(e[h] >> 16);
            e[h] = (uint32_t)run | ((uint32_t)(run + lo) << 16);
            run += lo + hi;
        }
        *rowv = make_uint4(e[0], e[1], e[2], e[3]);
        if (lane == 31)
            tot[b] = incl;
    }
    __syncthreads();
    if (warp == 0) { // bucket starts (two buckets per lane: nb <= 64)
        const int b0 = lane * 2;
        const int t0 = b0 < nb ? tot[b0] : 0, t1 = b0 + 1 < nb ? tot[b0 + 1] : 0;
        int incl = t0 + t1;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t2 = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o)
                incl += t2;
        }
        const int ex = incl - t0 - t1;
        if (b0 < nb)
            seg[b0] = ex;
        if (b0 + 1 < nb)
            seg[b0 + 1] = ex + t0;
        if (lane == 31)
            seg[nb] = incl;
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < LR; ++k) {
        if (key[k] >= 0) {
            uint16_t &c = cnt[key[k] * SORTERS + tid];
            const int pos = seg[key[k]] + (int)c;
            c = (uint16_t)(c + 1);
            sperm[pos] = tid + k * SORTERS;
            stok[pos] = tok[k];
        }
    }
    if (fl != 0)
        atomicOr(sflags, fl);
    __syncthreads();
    if (blockIdx.x == 0 && tid == 0)
        status_begin(p.ws.status, *sflags);
}

} // namespace

__global__ void __launch_bounds__(EMB_THREADS, 1)
    embed_kernel(const __grid_constant__ EmbedParams p, const __grid_constant__ EmbCfg c)
{
    extern __shared__ uint8_t emb_smem_raw[];
    __shared__ int scan_tmp[EMB_THREADS / 32];
    uint8_t *smem = align1024(emb_smem_raw);
    EmbBars *bars = reinterpret_cast<EmbBars *>(smem + c.bar_off);
    int *seg = reinterpret_cast<int *>(smem + c.seg_off);
    int *cpre = reinterpret_cast<int *>(smem + c.cpre_off);
    uint8_t *act = smem + c.act_off;
    SlotRec *srec = reinterpret_cast<SlotRec *>(smem + c.slot_off);
    const int warp = threadIdx.x >> 5;

    // The next call's routing kernel may launch now; it reads nothing before
    // this kernel has completed.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (threadIdx.x == 0) {
        for (int b = 0; b < 2; ++b) {
            mbar_init(&bars->op_full[b], LOADERS); // one cp.async arrival per loader thread
            mbar_init(&bars->op_empty[b], 1);
            mbar_init(&bars->acc_full[b], 1);
            mbar_init(&bars->acc_empty[b], 1);
            mbar_init(&bars->e_full[b], LOADERS);
            mbar_init(&bars->e_empty[b], 1);
        }
        mbar_init(&bars->fin, 1);
        bars->abort_flag = 0;
        bars->go[0] = bars->go[1] = 0;
        fence_barrier_init();
    }
    if (warp == 0)
        tmem_alloc(&bars->tmem_base, c.tmem_cols);

    grid_dependency_wait();
    const int nb = p.L + 1;
    // Each bucket's slot record (the tables are read here once), loads issued
    // before the routing sort so their latency overlaps it.
    for (int b = threadIdx.x; b < nb; b += EMB_THREADS) {
        SlotRec r{nullptr, nullptr, 0.0f, 0};
        if (b > 0) {
            r.at = p.tab.a_table[b - 1];
            r.b = p.tab.b_table[b - 1];
            r.scale = p.tab.scale_table[b - 1];
            r.rank = p.tab.rank_table[b - 1];
        }
        srec[b] = r;
    }
    // The routing sort: this CTA's own pass over the batch (up to
    // EMBED_LOCAL_ROWS rows), or the routing kernel's result.
    RowView rv;
    if (p.local) {
        int32_t *sperm = reinterpret_cast<int32_t *>(smem + c.sperm_off);
        int32_t *stok = reinterpret_cast<int32_t *>(smem + c.stok_off);
        // scratch: the operand buffers hold nothing yet
        uint16_t *cnt = reinterpret_cast<uint16_t *>(smem + c.g_off[0]);
        __shared__ uint32_t s_flags;
        local_route(p, seg, cnt, reinterpret_cast<int *>(cnt + (size_t)nb * SORTERS), sperm, stok, nb, &s_flags);
        rv.perm = sperm;
        rv.stok = stok;
    } else {
        for (int b = threadIdx.x; b <= nb; b += EMB_THREADS)
            seg[b] = p.ws.seg_off[b];
        rv.perm = p.ws.perm;
        rv.stok = nullptr;
        __syncthreads();
    }
    // active flag, chunk count and chunk size of each bucket, then the chunk
    // starts: warp 0 alone for up to 64 buckets (two per lane), else four
    // buckets per thread and a block scan
    int *cbase = reinterpret_cast<int *>(smem + c.cbase_off);
    int *crem = reinterpret_cast<int *>(smem + c.crem_off);
    __shared__ int s_chunks;
    auto bucket_chunks = [&](int b) {
        const int cnt = seg[b + 1] - seg[b];
        const SlotRec r = srec[b];
        act[b] = (b > 0 && r.at != nullptr && r.b != nullptr && r.scale != 0.0f && r.rank > 0) ? 1 : 0;
        const int n = cnt > 0 ? (cnt + CH - 1) / CH : 0;
        cbase[b] = n > 0 ? cnt / n : 0;
        crem[b] = n > 0 ? cnt - cbase[b] * n : 0;
        return n;
    };
    if (nb <= 64) {
        if (warp == 0) {
            const int lane = threadIdx.x & 31, b0 = 2 * lane;
            const int n0 = b0 < nb ? bucket_chunks(b0) : 0, n1 = b0 + 1 < nb ? bucket_chunks(b0 + 1) : 0;
            int incl = n0 + n1;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int t2 = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o)
                    incl += t2;
            }
            const int ex = incl - n0 - n1;
            if (b0 < nb)
                cpre[b0] = ex;
            if (b0 + 1 < nb)
                cpre[b0 + 1] = ex + n0;
            if (lane == 31) {
                cpre[nb] = incl;
                s_chunks = incl;
            }
        }
    } else {
        int nch[4], sum = 0;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int b = threadIdx.x * 4 + q;
            nch[q] = b < nb ? bucket_chunks(b) : 0;
            sum += nch[q];
        }
        int total;
        int ex = block_scan(sum, scan_tmp, total);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int b = threadIdx.x * 4 + q;
            if (b < nb) {
                cpre[b] = ex;
                ex += nch[q];
            }
        }
        if (threadIdx.x == 0) {
            cpre[nb] = total;
            s_chunks = total;
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;
    const Buckets bk{seg, cpre, cbase, crem, act};
    const int chunks = s_chunks;

    if (threadIdx.x < LOADERS)
        embed_loader(p, c, bars, smem, srec, bk, chunks, rv);
    else if (warp < MMA_WARP)
        embed_epilogue(p, c, bars, smem, tmem, srec, bk, chunks, rv);
    else if (threadIdx.x == MMA_WARP * 32)
        embed_mma(p, c, bars, smem, tmem, srec, bk, chunks);
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, c.tmem_cols);
    }
}

// ----------------------------------------------------------------- host side

namespace {

constexpr uint32_t SMEM_LIMIT = 232448 - 256; // opt-in shared memory per block (227 KB), less the static part

uint32_t au(uint32_t v, uint32_t a) { return (v + a - 1) / a * a; }

uint32_t pow2_cols(uint32_t v)
{
    uint32_t r = 32;
    while (r < v)
        r <<= 1;
    return r;
}

EmbCfg make_embed_cfg(int ft, int R, int L, int local_rows)
{
    EmbCfg c;
    memset(&c, 0, sizeof c);
    const uint32_t nkb = (uint32_t)(R + 63) / 64;
    c.g_bytes = nkb * KB_BYTES_G;
    c.a_bytes = nkb * (uint32_t)ft * 128u;
    c.e_bytes = (uint32_t)CH * (uint32_t)ft * 2u;
    uint32_t o = 0; // every buffer a multiple of 1024 bytes: the swizzled operands stay aligned
    for (int b = 0; b < 2; ++b) {
        c.g_off[b] = o;
        o += c.g_bytes;
    }
    for (int b = 0; b < 2; ++b) {
        c.a_off[b] = o;
        o += c.a_bytes;
    }
    for (int b = 0; b < 2; ++b) {
        c.e_off[b] = o;
        o += c.e_bytes;
    }
    const uint32_t nb = (uint32_t)L + 1;
    c.slot_off = o; o = au(o + (uint32_t)sizeof(SlotRec) * nb, 16);
    c.seg_off = o;  o = au(o + 4u * (nb + 1), 16);
    c.cpre_off = o; o = au(o + 4u * (nb + 1), 16);
    c.act_off = o;  o = au(o + nb, 16);
    c.cbase_off = o; o = au(o + 4u * nb, 16);
    c.crem_off = o;  o = au(o + 4u * nb, 16);
    c.ltok_off = o; o = au(o + 4u * CH, 16);
    c.crow_off = o; o = au(o + 8u * CH, 16);
    c.sperm_off = o; o = au(o + 4u * (uint32_t)local_rows, 16);
    c.stok_off = o;  o = au(o + 4u * (uint32_t)local_rows, 16);
    c.bar_off = o;  o = au(o + (uint32_t)sizeof(EmbBars), 16);
    c.smem_bytes = o + 1024; // slack to align the base to 1024
    c.tmem_cols = pow2_cols(2u * (uint32_t)ft);
    return c;
}

} // namespace

int embed_tile_features(int R)
{
    // sized for the largest slot count, so the choice depends on R only
    for (int ft = 128; ft > 32; ft >>= 1)
        if (make_embed_cfg(ft, R, MAX_BUCKETS - 1, 0).smem_bytes <= SMEM_LIMIT)
            return ft;
    return 32;
}

bool embed_local_fits(int M, int ft, int R, int L)
{
    // the sort's scratch ([L + 1][256] counts and L + 1 totals) lives in the buffers
    const EmbCfg c = make_embed_cfg(ft, R, L, M);
    return M <= EMBED_LOCAL_ROWS && L + 1 <= EMBED_LOCAL_BUCKETS && c.smem_bytes <= SMEM_LIMIT &&
           (uint32_t)(L + 1) * (SORTERS * 2u + 4u) <= c.e_off[0];
}

cudaError_t launch_embed(const EmbedParams &p, int num_sms, cudaStream_t st)
{
    const EmbCfg c = make_embed_cfg(p.ft, p.R, p.L, p.local ? p.M : 0);
    static std::atomic<uint64_t> raised{0};
    cudaError_t ea = raise_smem_limit(raised, embed_kernel, (int)SMEM_LIMIT);
    if (ea != cudaSuccess)
        return ea;
    // chunks at most: every non-empty bucket adds at most one partial chunk
    const long long nb = p.L + 1;
    const long long chunks = p.M / CH + (p.M < nb ? p.M : nb);
    const long long items = chunks * p.nft;
    const int grid = (int)(items < num_sms ? (items > 0 ? items : 1) : num_sms);
    // CTAs wait on counters other CTAs write: cooperative, so the whole grid
    // is resident at once or the launch fails
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeCooperative;
    attr[1].val.cooperative = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(EMB_THREADS);
    cfg.dynamicSmemBytes = c.smem_bytes;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, embed_kernel, p, c);
}

} // namespace rd
