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
// (cp.async into the 128-byte-swizzled K-major layout) and the E rows; thread
// 0 issues the UMMAs. Warps 4-7 (epilogue): TMEM -> scale -> add -> store, and
// the copy chunks. Two buffers of each kind: one item loads while the previous
// one drains. Every wait is bounded; a wait that gives up sets
// LORA_FLAG_WAIT_TIMEOUT and the CTA unwinds (its copies and UMMAs in flight
// are waited for first).
#include <cstring>

#include "lora_internal.cuh"
#include "ptx.cuh"

namespace rd {

namespace {

constexpr int EMB_THREADS = 256;
constexpr int GRP = 128;                     // threads of the loader and of the epilogue group
constexpr int CH = EMBED_CHUNK_ROWS;         // rows per chunk (UMMA M)
constexpr uint32_t KB_BYTES_G = CH * 128;    // one 64-wide k block of the chunk's B rows
constexpr int BAR_LOAD = 1, BAR_EPI = 2;     // named barriers of the two groups

struct EmbBars {
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
    uint32_t seg_off, cpre_off, act_off, ltok_off, crow_off, sperm_off, stok_off, bar_off;
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

// Item w: chunk w / nft of the bucket list, feature tile w % nft. Bucket b
// holds cpre[b+1] - cpre[b] chunks of its seg[b+1] - seg[b] rows, balanced
// (chunk q gets rows [q*cnt/nch, (q+1)*cnt/nch) of the bucket).
__device__ __forceinline__ Item get_item(const EmbedParams &p, const int *seg, const int *cpre,
                                         const uint8_t *act, int nb, int w)
{
    Item it;
    const int c = w / p.nft, f = w % p.nft;
    int lo = 0, hi = nb; // largest b with cpre[b] <= c (cpre non-decreasing, cpre[0] = 0)
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (cpre[mid] <= c)
            lo = mid;
        else
            hi = mid;
    }
    const int b = lo;
    const int q = c - cpre[b], nch = cpre[b + 1] - cpre[b];
    const long long cnt = seg[b + 1] - seg[b];
    const int r0 = seg[b] + (int)(q * cnt / nch), r1 = seg[b] + (int)((q + 1) * cnt / nch);
    it.delta = act[b];
    it.slot = b - 1;
    it.lo = r0;
    it.n = r1 - r0;
    it.f0 = f * p.ft;
    it.fw = min(p.ft, p.n_embd - it.f0);
    return it;
}

// Exclusive scan of one value per thread over the 256-thread block.
__device__ __forceinline__ int block_scan_256(int v, int *tmp, int &total)
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

// Loader group (threads 0 .. 127) over the delta chunks: the leader waits
// until buffer b is free (its UMMAs done, its E rows read); the group reads
// the chunk's tokens (one row per thread), stages the B rows and the A^T tile
// (one cp.async group, waited for before the UMMAs) and the E rows (a second
// group, whose landing the epilogue waits for on e_full); thread 0 issues the
// UMMAs.
__device__ void embed_loader(const EmbedParams &p, const EmbCfg &c, EmbBars *bars, uint8_t *smem,
                             uint32_t tmem, const int *seg, const int *cpre, const uint8_t *act, int nb,
                             int total, const RowView rv)
{
    const int t = threadIdx.x;
    int32_t *tok = reinterpret_cast<int32_t *>(smem + c.ltok_off); // [128]: token of each chunk row, -1 = out of range
    const int ecpr = p.ft >> 3;                                    // 16-byte chunks of a row in the row buffer
    const uint32_t a_kb = (uint32_t)p.ft * 128u;                   // one 64-wide k block of the A^T tile
    int u[2] = {0, 0};
    int d = 0;
    bool issued = false;
    for (int w = blockIdx.x; w < total; w += gridDim.x) {
        const Item it = get_item(p, seg, cpre, act, nb, w);
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
        named_bar_sync(BAR_LOAD, GRP);
        if (*(volatile int *)&bars->go[0] == 0)
            break;
        if (t < it.n) {
            int row, tk;
            row_at(p, rv, it.lo + t, row, tk);
            tok[t] = tk;
        }
        named_bar_sync(BAR_LOAD, GRP); // tok[] complete

        const int rank = p.tab.rank_table[it.slot];
        const int pk = (rank + 15) & ~15; // UMMA K granularity; k >= rank is zero-filled
        const int cpr = pk >> 3;          // 16-byte chunks of a staged operand row
        const uint16_t *At = p.tab.a_table[it.slot];
        const uint16_t *Bt = p.tab.b_table[it.slot];
        uint8_t *gbuf = smem + c.g_off[b], *abuf = smem + c.a_off[b], *eb = smem + c.e_off[b];
        // B rows of the chunk (the UMMA's A operand). Rows past n are not
        // staged: the D rows they feed are never read.
        for (int f = t; f < it.n * cpr; f += GRP) {
            const int j = f / cpr, q = f - j * cpr;
            const int tk = tok[j];
            const bool has = tk >= 0 && q * 8 < rank;
            cp_async_16(gbuf + (q >> 3) * KB_BYTES_G + j * 128 + (((q & 7) ^ (j & 7)) << 4),
                        Bt + (has ? (size_t)tk * p.R + q * 8 : 0), has ? 16u : 0u);
        }
        // A^T rows f0 .. f0 + fw - 1 (the UMMA's B operand); columns past fw
        // of D are never read either.
        for (int f = t; f < it.fw * cpr; f += GRP) {
            const int e = f / cpr, q = f - e * cpr;
            const bool has = q * 8 < rank;
            cp_async_16(abuf + (q >> 3) * a_kb + e * 128 + (((q & 7) ^ (e & 7)) << 4),
                        At + (has ? (size_t)(it.f0 + e) * p.R + q * 8 : 0), has ? 16u : 0u);
        }
        cp_async_commit();
        const int epr = it.fw >> 3;
        for (int f = t; f < it.n * ecpr; f += GRP) {
            const int j = f / ecpr, q = f - j * ecpr;
            const int tk = tok[j];
            if (q < epr && tk >= 0)
                cp_async_16(eb + erow_chunk(j, q, ecpr), p.E + (size_t)tk * p.n_embd + it.f0 + q * 8, 16u);
        }
        cp_async_commit();
        cp_async_mbar_arrive_noinc(&bars->e_full[b]);
        cp_async_wait_group<1>(); // the operand group (the E rows may still be in flight)
        fence_proxy_async_smem();  // generic-proxy copies, read by the UMMAs
        named_bar_sync(BAR_LOAD, GRP);
        if (t == 0) {
            // A failed wait only skips the issue: the group learns of the abort
            // at the next item's leader wait, so no thread leaves a barrier early.
            if (!aborted(bars) && mbar_wait(&bars->acc_empty[b], ((uint32_t)u[b] & 1u) ^ 1u)) {
                tc_fence_after();
                const uint32_t acc = tmem + (uint32_t)(b * p.ft);
                const uint32_t idesc = idesc_bf16_f32(CH, (uint32_t)p.ft);
                const uint32_t gb = smem_u32(gbuf), ab = smem_u32(abuf);
                for (int k16 = 0; k16 < pk / 16; ++k16) {
                    const uint32_t kb = (uint32_t)k16 >> 2, kk = ((uint32_t)k16 & 3u) * 32u;
                    umma_bf16(acc, sw128_kmajor_desc(gb + kb * KB_BYTES_G + kk),
                              sw128_kmajor_desc(ab + kb * a_kb + kk), idesc, k16 > 0 ? 1u : 0u);
                }
                umma_commit(&bars->op_empty[b]);
                umma_commit(&bars->acc_full[b]);
                issued = true;
            } else if (!aborted(bars)) {
                flag_abort(p, bars);
            }
        }
        ++u[b];
        ++d;
    }
    // Nothing of this CTA may still be in flight when it exits: the cp.async
    // copies, the UMMAs.
    cp_async_wait_all();
    if (t == 0 && issued) {
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

// Epilogue group (threads 128 .. 255). Thread et owns row et of a delta chunk
// (warp 4 + q reads TMEM lanes 32q .. 32q + 31): D row from TMEM 32 columns at
// a time, E row from the row buffer, 16-byte stores of y. Copy chunks: the
// group copies the E rows to y, 16 bytes per thread, a row's chunks on
// consecutive threads.
__device__ void embed_epilogue(const EmbedParams &p, const EmbCfg &c, EmbBars *bars, uint8_t *smem,
                               uint32_t tmem, const int *seg, const int *cpre, const uint8_t *act, int nb,
                               int total, const RowView rv)
{
    const int et = threadIdx.x - GRP;
    const int wq = (threadIdx.x >> 5) & 3;
    int32_t *crow = reinterpret_cast<int32_t *>(smem + c.crow_off); // [128] y row of a copy chunk's row
    int32_t *ctok = crow + CH;                                      // [128] its token, -1 = out of range
    const int ecpr = p.ft >> 3;
    const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
    int u[2] = {0, 0};
    int d = 0;
    for (int w = blockIdx.x; w < total; w += gridDim.x) {
        const Item it = get_item(p, seg, cpre, act, nb, w);
        if (!it.delta) {
            if (et < it.n) {
                int i, tk;
                row_at(p, rv, it.lo + et, i, tk);
                crow[et] = i;
                ctok[et] = tk;
            }
            named_bar_sync(BAR_EPI, GRP);
            const int epr = it.fw >> 3;
            for (int f = et; f < it.n * epr; f += GRP) {
                const int j = f / epr, q = f - j * epr;
                const int tk = ctok[j];
                const uint4 v = tk >= 0 ? __ldg(reinterpret_cast<const uint4 *>(
                                              p.E + (size_t)tk * p.n_embd + it.f0 + q * 8))
                                        : zero;
                *reinterpret_cast<uint4 *>(p.y + (size_t)crow[j] * p.y_stride + it.f0 + q * 8) = v;
            }
            named_bar_sync(BAR_EPI, GRP); // crow / ctok are rewritten by the next copy chunk
            continue;
        }
        const int b = d & 1;
        int yrow = 0;
        bool tvalid = false;
        if (et < it.n) {
            int tk;
            row_at(p, rv, it.lo + et, yrow, tk);
            tvalid = tk >= 0;
        }
        if (et == 0) {
            const uint32_t par = (uint32_t)u[b] & 1u;
            const bool ok = !aborted(bars) && mbar_wait(&bars->e_full[b], par) &&
                            mbar_wait(&bars->acc_full[b], par);
            if (!ok && !aborted(bars))
                flag_abort(p, bars);
            *(volatile int *)&bars->go[1] = ok ? 1 : 0;
        }
        named_bar_sync(BAR_EPI, GRP);
        if (*(volatile int *)&bars->go[1] == 0)
            break;
        mbar_wait(&bars->e_full[b], (uint32_t)u[b] & 1u); // complete: the copied rows are visible here
        tc_fence_after();
        if (wq * 32 < it.n) { // TMEM loads are per warp: a warp with no row of the chunk skips them
            const float sc = p.tab.scale_table[it.slot];
            const uint32_t tb = tmem + ((uint32_t)(wq * 32) << 16) + (uint32_t)(b * p.ft);
            const uint8_t *eb = smem + c.e_off[b];
            uint16_t *yr = p.y + (size_t)yrow * p.y_stride + it.f0;
            const bool mine = et < it.n;
            for (int c0 = 0; c0 < it.fw; c0 += 32) {
                uint32_t r[2][16];
                tmem_ld16_nowait(tb + (uint32_t)c0, r[0]);
                tmem_ld16_nowait(tb + (uint32_t)c0 + 16u, r[1]);
                tmem_wait_ld();
                if (mine) {
#pragma unroll
                    for (int g = 0; g < 4; ++g) {
                        const int col = c0 + 8 * g;
                        if (col < it.fw) {
                            const uint4 e = tvalid ? *reinterpret_cast<const uint4 *>(
                                                         eb + erow_chunk(et, col >> 3, ecpr))
                                                   : zero;
                            *reinterpret_cast<uint4 *>(yr + col) = add_scaled8(e, &r[g >> 1][(g & 1) * 8], sc);
                        }
                    }
                }
            }
        }
        tc_fence_before();
        named_bar_sync(BAR_EPI, GRP); // accumulator b and row buffer b are read
        if (et == 0) {
            mbar_arrive(&bars->acc_empty[b]);
            mbar_arrive(&bars->e_empty[b]);
        }
        ++u[b];
        ++d;
    }
}

// This CTA's own routing pass over a batch of at most EMBED_LOCAL_ROWS rows:
// a stable counting sort of the rows by bucket (0 = no valid slot, s + 1 =
// slot s) into sperm / stok, bucket starts into seg. Stable, so every CTA
// cuts a bucket into the same chunks (a chunk's feature tiles run on
// different CTAs). Rows go in rounds of 256 in input order; inside a round a
// row's place among equal keys is the count in earlier warps (per-warp counts
// tagged with the round, so they need no clearing) plus its rank in its own
// warp. CTA 0 writes the call's status word (there is no routing kernel).
// fill: [nb] scratch; wc: [8][nb] scratch.
__device__ void local_route(const EmbedParams &p, int *seg, int *fill, uint32_t *wc, int32_t *sperm,
                            int32_t *stok, int nb, int *scan_tmp)
{
    constexpr int LR = EMBED_LOCAL_ROWS / EMB_THREADS;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int b = tid; b < nb; b += EMB_THREADS)
        fill[b] = 0;
    for (int q = tid; q < (EMB_THREADS / 32) * nb; q += EMB_THREADS)
        wc[q] = 0; // tag 0: no round
    int key[LR], tok[LR];
#pragma unroll
    for (int k = 0; k < LR; ++k) { // every load issued before any is used
        const int i = tid + k * EMB_THREADS;
        key[k] = i < p.M ? p.seq_slot[i] : -1;
        tok[k] = i < p.M ? p.tokens[i] : 0;
    }
    __syncthreads();
    uint32_t fl = 0;
#pragma unroll
    for (int k = 0; k < LR; ++k) {
        const int i = tid + k * EMB_THREADS;
        if (i < p.M) {
            const int sl = key[k];
            if (sl >= p.L)
                fl |= LORA_FLAG_SLOT_RANGE;
            key[k] = (sl >= 0 && sl < p.L) ? sl + 1 : 0;
            atomicAdd(&fill[key[k]], 1);
            if (tok[k] < 0 || tok[k] >= p.vocab) {
                fl |= LORA_FLAG_TOKEN_RANGE;
                tok[k] = -1;
            }
        }
    }
    __syncthreads();
    int cnt[4], sum = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int b = tid * 4 + q;
        cnt[q] = b < nb ? fill[b] : 0;
        sum += cnt[q];
    }
    int total;
    int ex = block_scan_256(sum, scan_tmp, total);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int b = tid * 4 + q;
        if (b < nb) {
            seg[b] = ex;
            fill[b] = ex; // next free position of the bucket
            ex += cnt[q];
        }
    }
    if (tid == 0)
        seg[nb] = total;
    __syncthreads();
#pragma unroll
    for (int k = 0; k < LR; ++k) {
        if (k * EMB_THREADS >= p.M)
            break; // uniform
        const int i = tid + k * EMB_THREADS;
        const int b = i < p.M ? key[k] : -1;
        const unsigned peers = __match_any_sync(0xffffffffu, b);
        const int rk = __popc(peers & ((1u << lane) - 1u));
        const uint32_t tag = (uint32_t)(k + 1) << 16;
        if (b >= 0 && rk == 0)
            wc[warp * nb + b] = tag | (uint32_t)__popc(peers);
        __syncthreads();
        if (b >= 0) {
            int pos = fill[b] + rk;
            for (int w = 0; w < warp; ++w) {
                const uint32_t v = wc[w * nb + b];
                if ((v & 0xffff0000u) == tag)
                    pos += (int)(v & 0xffffu);
            }
            sperm[pos] = i;
            stok[pos] = tok[k];
        }
        __syncthreads();
        if (b >= 0 && rk == 0)
            atomicAdd(&fill[b], __popc(peers));
        __syncthreads();
    }
    const int any_slot = __syncthreads_or((int)(fl & LORA_FLAG_SLOT_RANGE));
    const int any_tok = __syncthreads_or((int)(fl & LORA_FLAG_TOKEN_RANGE));
    if (blockIdx.x == 0 && tid == 0)
        *p.ws.status = (any_slot ? (uint32_t)LORA_FLAG_SLOT_RANGE : 0u) |
                       (any_tok ? (uint32_t)LORA_FLAG_TOKEN_RANGE : 0u);
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
    const int warp = threadIdx.x >> 5;

    // The next call's routing kernel may launch now; it reads nothing before
    // this kernel has completed.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (threadIdx.x == 0) {
        for (int b = 0; b < 2; ++b) {
            mbar_init(&bars->op_empty[b], 1);
            mbar_init(&bars->acc_full[b], 1);
            mbar_init(&bars->acc_empty[b], 1);
            mbar_init(&bars->e_full[b], GRP); // one cp.async arrival per loader thread
            mbar_init(&bars->e_empty[b], 1);
        }
        mbar_init(&bars->fin, 1);
        bars->abort_flag = 0;
        bars->go[0] = bars->go[1] = 0;
        fence_barrier_init();
    }
    if (warp == 0)
        tmem_alloc(&bars->tmem_base, c.tmem_cols);

    // The routing sort: this CTA's own pass over the batch (small batches),
    // or the routing kernel's result. Then the active flag and chunk count of
    // each bucket (four buckets per thread, one scan).
    grid_dependency_wait();
    const int nb = p.L + 1;
    RowView rv;
    if (p.local) {
        int32_t *sperm = reinterpret_cast<int32_t *>(smem + c.sperm_off);
        int32_t *stok = reinterpret_cast<int32_t *>(smem + c.stok_off);
        // scratch: the row and operand buffers hold nothing yet (fill [nb] in
        // the first row buffer, the per-warp counts [8][nb] from the first
        // operand buffer on, at least 32 KB of buffers)
        local_route(p, seg, reinterpret_cast<int *>(smem + c.e_off[0]),
                    reinterpret_cast<uint32_t *>(smem + c.g_off[0]), sperm, stok, nb, scan_tmp);
        rv.perm = sperm;
        rv.stok = stok;
    } else {
        for (int b = threadIdx.x; b <= nb; b += EMB_THREADS)
            seg[b] = p.ws.seg_off[b];
        rv.perm = p.ws.perm;
        rv.stok = nullptr;
        __syncthreads();
    }
    int nch[4], sum = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int b = threadIdx.x * 4 + q;
        nch[q] = 0;
        if (b < nb) {
            const int cnt = seg[b + 1] - seg[b];
            bool on = false;
            if (b > 0) {
                const int s = b - 1;
                on = p.tab.a_table[s] != nullptr && p.tab.b_table[s] != nullptr &&
                     p.tab.scale_table[s] != 0.0f && p.tab.rank_table[s] > 0;
            }
            act[b] = on ? 1 : 0;
            nch[q] = cnt > 0 ? (cnt + CH - 1) / CH : 0;
            sum += nch[q];
        }
    }
    int chunks;
    int ex = block_scan_256(sum, scan_tmp, chunks);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int b = threadIdx.x * 4 + q;
        if (b < nb) {
            cpre[b] = ex;
            ex += nch[q];
        }
    }
    if (threadIdx.x == 0)
        cpre[nb] = chunks;
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;
    const int total = chunks * p.nft;

    if (threadIdx.x < GRP)
        embed_loader(p, c, bars, smem, tmem, seg, cpre, act, nb, total, rv);
    else
        embed_epilogue(p, c, bars, smem, tmem, seg, cpre, act, nb, total, rv);
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
    c.seg_off = o;  o = au(o + 4u * (nb + 1), 16);
    c.cpre_off = o; o = au(o + 4u * (nb + 1), 16);
    c.act_off = o;  o = au(o + nb, 16);
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
    return M <= EMBED_LOCAL_ROWS && make_embed_cfg(ft, R, L, M).smem_bytes <= SMEM_LIMIT;
}

cudaError_t launch_embed(const EmbedParams &p, int num_sms, cudaStream_t st)
{
    const EmbCfg c = make_embed_cfg(p.ft, p.R, p.L, p.local ? p.M : 0);
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(embed_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)SMEM_LIMIT);
        if (e != cudaSuccess)
            return e;
        attr_set = true;
    }
    // chunks at most: every non-empty bucket adds at most one partial chunk
    const long long nb = p.L + 1;
    const long long chunks = p.M / CH + (p.M < nb ? p.M : nb);
    const long long items = chunks * p.nft;
    const int grid = (int)(items < num_sms ? (items > 0 ? items : 1) : num_sms);
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(EMB_THREADS);
    cfg.dynamicSmemBytes = c.smem_bytes;
    cfg.stream = st;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, embed_kernel, p, c);
}

} // namespace rd
