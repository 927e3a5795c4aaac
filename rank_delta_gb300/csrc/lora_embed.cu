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
// of rows is cut into balanced chunks of at most tn rows; a work item is one
// chunk x one tile of 128 embedding features (f0 .. f0 + 127).
//   delta chunk (an active slot): D[e][j] = sum_r At[f0 + e][r] * B[t_j][r] on the
//     tensor cores (UMMA M = 128 features, N = the chunk's rows rounded up to 16,
//     K = the slot's rank rounded up to 16), fp32 in TMEM; y = bf16(E + s * D),
//     one rounding.
//   copy chunk (no delta): y = the E row's bytes.
// The E rows of an item come into shared memory by bulk copies (one 16-byte
// aligned run of up to 256 bytes per row); the delta is added in place and the
// same buffer goes out to y by bulk stores.
//
// Warps 0-3 (loader): per item the E rows and, for a delta chunk, the A^T tile
// and the chunk's B rows (cp.async into the 128-byte-swizzled K-major layout);
// thread 0 issues the UMMAs. Warps 4-7 (epilogue): TMEM -> scale -> add ->
// store. Two buffers of each kind: one item loads while the previous drains.
// Every wait is bounded; a wait that gives up sets LORA_FLAG_WAIT_TIMEOUT and
// the CTA unwinds (its copies and UMMAs in flight are waited for first).
#include <cstring>

#include "lora_internal.cuh"
#include "ptx.cuh"

namespace rd {

namespace {

constexpr int EMB_THREADS = 256;
constexpr int GRP = 128;             // threads of the loader and of the epilogue group
constexpr int FT = 128;              // features per item (UMMA M)
constexpr uint32_t KB_BYTES_A = FT * 128; // one 64-wide k block of the A^T tile
constexpr int BAR_LOAD = 1, BAR_EPI = 2; // named barriers of the two groups

struct EmbBars {
    uint64_t op_empty[2];  // the UMMAs that read operand buffer b are done
    uint64_t acc_full[2];  // accumulator b holds an item's D
    uint64_t acc_empty[2]; // the epilogue has read accumulator b
    uint64_t e_full[2];    // E rows of the item in row buffer b have landed
    uint64_t e_empty[2];   // the bulk stores of row buffer b have read it
    uint64_t fin;          // every UMMA of this CTA is done
    uint32_t tmem_base;
    int abort_flag;
    int go[2];             // a group leader's wait result, broadcast to its group
};

struct EmbCfg {
    int nkb;                     // 64-wide k blocks of the operands (max_rank / 64 rounded up)
    uint32_t a_bytes, b_bytes;   // one operand buffer of A^T / of B rows
    uint32_t e_bytes;            // one row buffer: tn rows of 256 bytes
    uint32_t a_off[2], b_off[2], e_off[2];
    uint32_t seg_off, cpre_off, act_off, lrow_off, erow_off, bar_off;
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
    it.f0 = f * FT;
    it.fw = min(FT, p.n_embd - it.f0);
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

} // namespace

namespace {

__device__ __forceinline__ float bf16_bits_to_f32(uint16_t h) { return __uint_as_float((uint32_t)h << 16); }

// Round to nearest even (no NaN inputs reach here: E and the pool are finite).
__device__ __forceinline__ uint16_t f32_to_bf16_bits(float f)
{
    const uint32_t u = __float_as_uint(f);
    return (uint16_t)((u + 0x7fffu + ((u >> 16) & 1u)) >> 16);
}

// Loader group (threads 0 .. 127). Per item: the leader waits until the row
// buffer (and for a delta chunk the operand buffer) is free; the group reads
// the chunk's tokens, issues the E row copies, and for a delta chunk stages
// A^T rows f0.. and the chunk's B rows; thread 0 then issues the UMMAs.
__device__ void embed_loader(const EmbedParams &p, const EmbCfg &c, EmbBars *bars, uint8_t *smem,
                             uint32_t tmem, const int *seg, const int *cpre, const uint8_t *act, int nb,
                             int total)
{
    const int t = threadIdx.x;
    int32_t *ltok = reinterpret_cast<int32_t *>(smem + c.lrow_off); // [2][tn]: token of each row, -1 = out of range
    int eu[2] = {0, 0}, ou[2] = {0, 0};
    int k = 0, d = 0;
    bool issued = false;
    for (int w = blockIdx.x; w < total; w += gridDim.x, ++k) {
        const Item it = get_item(p, seg, cpre, act, nb, w);
        const int rb = k & 1, ob = d & 1;
        if (t == 0) {
            bool ok = !aborted(bars) && mbar_wait(&bars->e_empty[rb], ((uint32_t)eu[rb] & 1u) ^ 1u);
            if (ok && it.delta)
                ok = mbar_wait(&bars->op_empty[ob], ((uint32_t)ou[ob] & 1u) ^ 1u);
            if (!ok && !aborted(bars))
                flag_abort(p, bars);
            *(volatile int *)&bars->go[0] = ok ? 1 : 0;
        }
        named_bar_sync(BAR_LOAD, GRP);
        if (*(volatile int *)&bars->go[0] == 0)
            break;
        int32_t *tok = ltok + rb * p.tn;
        uint8_t *eb = smem + c.e_off[rb];
        const uint32_t ebytes = (uint32_t)it.fw * 2u;
        for (int j = t; j < it.n; j += GRP) {
            const int i = p.ws.perm[it.lo + j];
            int tk = p.tokens[i];
            if (tk < 0 || tk >= p.vocab) {
                tk = -1;
                atomicOr(p.ws.status, (uint32_t)LORA_FLAG_TOKEN_RANGE);
            } else {
                mbar_expect_tx(&bars->e_full[rb], ebytes);
                bulk_load(eb + (size_t)j * 256, p.E + (size_t)tk * p.n_embd + it.f0, ebytes, &bars->e_full[rb]);
            }
            tok[j] = tk;
        }
        named_bar_sync(BAR_LOAD, GRP); // every expect_tx posted, tok[] complete
        if (t == 0)
            mbar_arrive(&bars->e_full[rb]);
        ++eu[rb];
        if (!it.delta)
            continue;

        const int rank = p.tab.rank_table[it.slot];
        const int pk = (rank + 15) & ~15; // UMMA K granularity; k >= rank is zero-filled
        const int cpr = pk >> 3;          // 16-byte chunks of a staged row
        const uint16_t *At = p.tab.a_table[it.slot];
        const uint16_t *Bt = p.tab.b_table[it.slot];
        uint8_t *abuf = smem + c.a_off[ob], *bbuf = smem + c.b_off[ob];
        const uint32_t b_kb = (uint32_t)p.tn * 128u; // bytes of one 64-wide k block of the B rows
        for (int f = t; f < FT * cpr; f += GRP) {
            const int e = f / cpr, q = f - e * cpr;
            const bool has = e < it.fw && q * 8 < rank;
            const uint16_t *src = At + (has ? (size_t)(it.f0 + e) * p.R + q * 8 : 0);
            cp_async_16(abuf + (q >> 3) * KB_BYTES_A + e * 128 + (((q & 7) ^ (e & 7)) << 4), src,
                        has ? 16u : 0u);
        }
        const int nmma = (it.n + 15) & ~15;
        for (int f = t; f < nmma * cpr; f += GRP) {
            const int j = f / cpr, q = f - j * cpr;
            const int tk = j < it.n ? tok[j] : -1;
            const bool has = tk >= 0 && q * 8 < rank;
            const uint16_t *src = Bt + (has ? (size_t)tk * p.R + q * 8 : 0);
            cp_async_16(bbuf + (q >> 3) * b_kb + j * 128 + (((q & 7) ^ (j & 7)) << 4), src, has ? 16u : 0u);
        }
        cp_async_wait_all();
        fence_proxy_async_smem(); // generic-proxy copies, read by the UMMAs
        named_bar_sync(BAR_LOAD, GRP);
        if (t == 0) {
            // A failed wait only skips the issue: the group learns of the abort
            // at the next item's leader wait, so no thread leaves a barrier early.
            if (!aborted(bars) && mbar_wait(&bars->acc_empty[ob], ((uint32_t)ou[ob] & 1u) ^ 1u)) {
                tc_fence_after();
                const uint32_t acc = tmem + (uint32_t)(ob * p.tn);
                const uint32_t idesc = idesc_bf16_f32(FT, (uint32_t)nmma);
                const uint32_t ab = smem_u32(abuf), bb = smem_u32(bbuf);
                for (int k16 = 0; k16 < pk / 16; ++k16) {
                    const uint32_t kb = (uint32_t)k16 >> 2, kk = ((uint32_t)k16 & 3u) * 32u;
                    umma_bf16(acc, sw128_kmajor_desc(ab + kb * KB_BYTES_A + kk),
                              sw128_kmajor_desc(bb + kb * b_kb + kk), idesc, k16 > 0 ? 1u : 0u);
                }
                umma_commit(&bars->op_empty[ob]);
                umma_commit(&bars->acc_full[ob]);
                issued = true;
            } else if (!aborted(bars)) {
                flag_abort(p, bars);
            }
        }
        ++ou[ob];
        ++d;
    }
    // Nothing of this CTA may still be in flight when it exits: the cp.async
    // copies (waited per item), the E row copies, the UMMAs.
    if (t == 0) {
        for (int b = 0; b < 2; ++b)
            if (eu[b] > 0 && !mbar_wait(&bars->e_full[b], ((uint32_t)eu[b] - 1u) & 1u))
                flag_abort(p, bars);
        if (issued) {
            umma_commit(&bars->fin);
            if (!mbar_wait(&bars->fin, 0))
                flag_abort(p, bars);
        }
    }
}

// Epilogue group (threads 128 .. 255; warp 4 + q reads TMEM lanes 32q ..
// 32q + 31, so thread et owns feature f0 + et of every row). Per item: y rows
// of the chunk, then the leader waits for the E rows (and the accumulator);
// a delta chunk gets y = bf16(E + s * D) written over its E row in place;
// then the rows go out by bulk stores.
__device__ void embed_epilogue(const EmbedParams &p, const EmbCfg &c, EmbBars *bars, uint8_t *smem,
                               uint32_t tmem, const int *seg, const int *cpre, const uint8_t *act, int nb,
                               int total)
{
    const int et = threadIdx.x - GRP;
    const int wq = (threadIdx.x >> 5) & 3;
    int32_t *erow = reinterpret_cast<int32_t *>(smem + c.erow_off); // [2][tn]: y row, ~row if the token is out of range
    int eu[2] = {0, 0}, ou[2] = {0, 0};
    int k = 0, d = 0;
    for (int w = blockIdx.x; w < total; w += gridDim.x, ++k) {
        const Item it = get_item(p, seg, cpre, act, nb, w);
        const int rb = k & 1, ob = d & 1;
        int32_t *rows = erow + rb * p.tn;
        for (int j = et; j < it.n; j += GRP) {
            const int i = p.ws.perm[it.lo + j];
            const int tk = p.tokens[i];
            rows[j] = (tk >= 0 && tk < p.vocab) ? i : ~i;
        }
        if (et == 0) {
            bool ok = !aborted(bars) && mbar_wait(&bars->e_full[rb], (uint32_t)eu[rb] & 1u);
            if (ok && it.delta)
                ok = mbar_wait(&bars->acc_full[ob], (uint32_t)ou[ob] & 1u);
            if (!ok && !aborted(bars))
                flag_abort(p, bars);
            *(volatile int *)&bars->go[1] = ok ? 1 : 0;
        }
        named_bar_sync(BAR_EPI, GRP);
        if (*(volatile int *)&bars->go[1] == 0)
            break;
        mbar_wait(&bars->e_full[rb], (uint32_t)eu[rb] & 1u); // complete: orders the copied rows for this thread
        uint8_t *eb = smem + c.e_off[rb];
        if (it.delta) {
            tc_fence_after();
            const float sc = p.tab.scale_table[it.slot];
            const uint32_t tb = tmem + ((uint32_t)(wq * 32) << 16) + (uint32_t)(ob * p.tn);
            const bool fe = et < it.fw;
            for (int c0 = 0; c0 < it.n; c0 += 16) {
                float v[16];
                tmem_ld16(tb + (uint32_t)c0, v);
#pragma unroll
                for (int q = 0; q < 16; ++q) {
                    const int j = c0 + q;
                    if (j < it.n && fe) {
                        uint16_t *dst = reinterpret_cast<uint16_t *>(eb + (size_t)j * 256) + et;
                        const float e = rows[j] >= 0 ? bf16_bits_to_f32(*dst) : 0.0f;
                        *dst = f32_to_bf16_bits(e + sc * v[q]);
                    }
                }
            }
            tc_fence_before();
            named_bar_sync(BAR_EPI, GRP); // every TMEM read of accumulator ob is done
            if (et == 0)
                mbar_arrive(&bars->acc_empty[ob]);
            ++ou[ob];
            ++d;
        } else {
            // rows of out-of-range tokens were not copied: zero them
            for (int f = et; f < it.n * 16; f += GRP) {
                const int j = f >> 4, q = f & 15;
                if (rows[j] < 0 && q * 8 < it.fw)
                    *reinterpret_cast<uint4 *>(eb + (size_t)j * 256 + q * 16) = make_uint4(0u, 0u, 0u, 0u);
            }
        }
        fence_proxy_async_smem(); // generic writes above, read by the bulk stores
        named_bar_sync(BAR_EPI, GRP);
        for (int j = et; j < it.n; j += GRP) {
            const int v = rows[j], i = v >= 0 ? v : ~v;
            bulk_store(p.y + (size_t)i * p.y_stride + it.f0, eb + (size_t)j * 256, (uint32_t)it.fw * 2u);
        }
        bulk_commit();
        bulk_wait_read_all();
        named_bar_sync(BAR_EPI, GRP); // every store of row buffer rb has read it
        if (et == 0)
            mbar_arrive(&bars->e_empty[rb]);
        ++eu[rb];
    }
    bulk_wait_all();
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
            mbar_init(&bars->e_full[b], 1);
            mbar_init(&bars->e_empty[b], 1);
        }
        mbar_init(&bars->fin, 1);
        bars->abort_flag = 0;
        bars->go[0] = bars->go[1] = 0;
        fence_barrier_init();
    }
    if (warp == 0)
        tmem_alloc(&bars->tmem_base, c.tmem_cols);

    // Buckets of the routing sort: rows, active flag and chunk count of each
    // (four buckets per thread, then one scan).
    grid_dependency_wait();
    const int nb = p.L + 1;
    int nch[4], sum = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int b = threadIdx.x * 4 + q;
        nch[q] = 0;
        if (b < nb) {
            const int s0 = p.ws.seg_off[b], cnt = p.ws.seg_off[b + 1] - s0;
            bool on = false;
            if (b > 0) {
                const int s = b - 1;
                on = p.tab.a_table[s] != nullptr && p.tab.b_table[s] != nullptr &&
                     p.tab.scale_table[s] != 0.0f && p.tab.rank_table[s] > 0;
            }
            seg[b] = s0;
            act[b] = on ? 1 : 0;
            nch[q] = cnt > 0 ? (cnt + p.tn - 1) / p.tn : 0;
            sum += nch[q];
        }
    }
    if (threadIdx.x == 0)
        seg[nb] = p.ws.seg_off[nb];
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
        embed_loader(p, c, bars, smem, tmem, seg, cpre, act, nb, total);
    else
        embed_epilogue(p, c, bars, smem, tmem, seg, cpre, act, nb, total);
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

EmbCfg make_embed_cfg(int tn, int R, int L)
{
    EmbCfg c;
    memset(&c, 0, sizeof c);
    c.nkb = (R + 63) / 64;
    c.a_bytes = (uint32_t)c.nkb * KB_BYTES_A;
    c.b_bytes = (uint32_t)c.nkb * (uint32_t)tn * 128u;
    c.e_bytes = (uint32_t)tn * 256u;
    uint32_t o = 0;
    for (int b = 0; b < 2; ++b) {
        c.a_off[b] = o;
        o += c.a_bytes;
    }
    for (int b = 0; b < 2; ++b) {
        c.b_off[b] = o;
        o += c.b_bytes;
    }
    for (int b = 0; b < 2; ++b) {
        c.e_off[b] = o;
        o += c.e_bytes;
    }
    const uint32_t nb = (uint32_t)L + 1;
    c.seg_off = o;  o = au(o + 4u * (nb + 1), 16);
    c.cpre_off = o; o = au(o + 4u * (nb + 1), 16);
    c.act_off = o;  o = au(o + nb, 16);
    c.lrow_off = o; o = au(o + 8u * (uint32_t)tn, 16);
    c.erow_off = o; o = au(o + 8u * (uint32_t)tn, 16);
    c.bar_off = o;  o = au(o + (uint32_t)sizeof(EmbBars), 16);
    c.smem_bytes = o + 1024; // slack to align the base to 1024
    c.tmem_cols = pow2_cols(2u * (uint32_t)tn);
    return c;
}

} // namespace

int embed_chunk_rows(int M, int R)
{
    int tn = (M + 15) / 16 * 16;
    tn = tn < 16 ? 16 : (tn > 256 ? 256 : tn);
    // sized for the largest slot count, so the choice depends on M and R only
    while (tn > 16 && make_embed_cfg(tn, R, MAX_BUCKETS - 1).smem_bytes > SMEM_LIMIT)
        tn -= 16;
    return tn;
}

cudaError_t launch_embed(const EmbedParams &p, int num_sms, cudaStream_t st)
{
    const EmbCfg c = make_embed_cfg(p.tn, p.R, p.L);
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
    const long long chunks = p.M / p.tn + (p.M < nb ? p.M : nb);
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
