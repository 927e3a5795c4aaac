// One-launch tensor-core projection for batches of up to 256 rows (decode,
// fused QKV): y = W x + s B (A x) per row, every step in one kernel.
//
// The base product is computed transposed, D[n, t] = sum_k W[n, k] x[t, k]
// (UMMA M = 128 output features, N = the rows of the batch), so W -- the
// bytes that bound these shapes -- streams through shared memory once. Each
// 128-feature tile is split along K into C parts (64-wide chunks, fixed by K
// and C alone), one CTA each; the parts' fp32 tiles are summed in part order,
// so every element is computed the same way for a given (rows, K) whatever N
// is: a fused q/k/v call equals its split calls byte for byte.
//
// The shrink h_t = A_{s_t} x_t (ferrox-core `weight_matrix/lora.rs`,
// `LoraDelta::project`) runs on the tensor cores inside the same K loop,
// reading the x tile already staged for the base product:
//   D_h^T[q, t] = sum_k A_rows[q, k] x[t, k]   (UMMA M = 128 rank rows, N = the batch)
// The "rank rows" of the call are the touched slots' A rows at their true
// ranks (each rounded up to 8), concatenated in slot order; cluster c owns
// rows [c Q, (c + 1) Q) and each of its CTAs covers its own K part. The
// routing reads are issued at kernel entry, ahead of the W stream; the A rows
// of the CTA's whole K part are then copied in one batch (cp.async, through
// a_table). The MMA warp issues the base UMMAs of a stage as soon as W and x
// land, and that stage's shrink UMMAs once the A rows are in, releasing the
// stage after both.
//
// Exchange of h: after the K loop every CTA writes its fp32 partial h of its
// rank rows to the workspace and arrives on one counter tagged with the
// call's epoch (a word in the workspace that each call advances by one), so
// nothing needs clearing between calls. CTAs that add a delta wait (bounded,
// one polling thread with back-off) for every CTA's arrival, then stage the
// expand operands:
//   XB[n, k]  B rows n of the slots this K part owns (slot mod C), ranks
//             rounded to 16 -- copied before the wait, they do not need h,
//   XH[t, k]  s_t * comp * h_t (the K parts' partials summed in part order)
//             in row t's slot range, zero elsewhere, bf16 hi + lo planes,
// and the MMA warp accumulates D'[n, t] = sum_k XB[n, k] XH[t, k] in TMEM
// columns of its own. The drain adds D' only to the rows whose slot this
// part owns (spark_model `layers/ops/lora_delta.rs`: the fold fused with the
// base product instead of a scaled-add pass), so rows without a delta are
// the base product byte for byte.
//
// Gated variant (frink `lora_attach.rs`, `parts_mut`: a fused ffn_up holds
// the gate rows, then the up rows, with B rows split the same way over one
// A): tile f holds gate features f*64.. and up features I + f*64..; the sum
// rounds both halves to bf16 and writes act = silu(g) * u, rounded once.
//
// Residency: every CTA waits for every other CTA's arrival, so the whole
// grid must be resident at once. When the device can hold all the clusters
// of C CTAs (the host asks the occupancy API), the K parts of a feature tile
// form a cluster and sum over distributed shared memory. Otherwise (the
// fused QKV shape: 48 clusters of 3, one GB300 holds 46) the launch is
// cooperative -- the whole grid resident, or no launch -- and each CTA writes
// its fp32 tile to the workspace and sums its share of the rows from its
// peers' tiles, in the same part order: the same bytes in both modes.
//
// Warp roles (256 threads): warp 0 TMA producer of W and x; warp 1 TMEM
// owner and UMMA issuer; warps 2-3 A-row loaders; warps 4-7 epilogue. Warps
// 2-7 resolve the routing together at the start. Every wait is bounded
// (%globaltimer); on a timeout the CTA records LORA_FLAG_WAIT_TIMEOUT in the
// status word, skips the delta, and still takes part in both cluster
// barriers, so its peers never wait on it.
#include <cstdio>
#include <mutex>

#include "lora_internal.cuh"
#include "ptx.cuh"
#include "vec.cuh"

namespace rd {

namespace {

constexpr int DC_THREADS = 256;
constexpr int DC_EPI = 128;
constexpr int DC_ROUTE = 192; // warps 2..7
constexpr int DC_MAX_TN = 256;
constexpr int DC_MAX_STAGES = 8;
constexpr int DC_MAX_Q = 128;
constexpr int DC_MAX_L = 256;
constexpr int DC_MAX_NA = 32; // A-row chunk slots
constexpr uint32_t DC_W_CHUNK = 128u * 128u; // 128 rows x 64 bf16
constexpr uint32_t DC_XB_BLOCK = 128u * 128u;
constexpr uint64_t DC_FLAG_MARK = 0xA5A5A5A5ull << 32;
constexpr int DC_HCNT_WORD = 8; // u64 index in the workspace status block: the h arrival counter

struct DecCfg {
    int tn, kc, stages, C, ncl;
    int kchunks, use3d;
    int Q;           // shrink rank rows per cluster (the UMMA M side holds 128: rows past Q are ignored)
    int gated, I;
    int yvec;        // 1: y / act rows take 8-byte stores
    int blocks;      // 64-wide k blocks of one expand round (XB + two XH planes)
    int na;          // A-row slots, one 64-wide chunk of the CTA's shrink rows each
    uint32_t x_chunk, stage_bytes, a_chunk, region;
    uint32_t a_off, aux_off, bar_off, smem_bytes;
    uint32_t tmem_cols, col_h, col_d;
    uint64_t wait_ns;
    int extra_arrivals; // test hook: arrivals that never come (the exchange wait then runs out)
    int l2sum;       // 1: the K parts' tiles are summed through the workspace (no clusters; cooperative launch)
    int gb_mask;     // bit lg: a box of 2^lg groups x nchb chunks fits the A region (the 5D A-row maps)
    int nchb;        // chunks of one such box: the most of any K part
};

// The pool's A rows as boxes of 2^lg 8-row groups of one slot over nchb
// 64-wide chunks, lg = 0..4, laid out chunk by chunk as the shrink reads them.
struct AMap5 {
    CUtensorMap m[5];
};

struct DecParams {
    const uint16_t *x;
    int64_t x_stride;
    uint16_t *y;
    int64_t y_stride;
    const int32_t *seq_slot;
    int M, K, N, L, R;
    Tables tab;
    uint32_t *ws_status; // [0] flags, [1] tag (epoch of the call that set them), [2] epoch
    int32_t *perm;       // routing export (CTA 0)
    int32_t *seg_off;
    float *hpart;        // [C][ncl][M][Q]: block [M][Q] per CTA (its rank rows q_lo.., columns past q_n unused)
    float *gpart;        // [ncl * C][M][128] fp32 tiles of the K parts (l2sum)
    unsigned long long *pflags; // [ncl * C] tile published (l2sum)
    const uint8_t *pool; // the route's pool: slot s's A at pool + s * slot_bytes (the A-row tensor map's view)
    size_t slot_bytes;
};

struct DecAux {
    // rows
    int16_t tslot[DC_MAX_TN];      // slot of row t if it takes a delta, else -1
    int16_t tkey[DC_MAX_TN];       // routing key of row t: slot + 1, 0 without a valid slot
    // slots (the route tables, read once at kernel entry)
    const uint16_t *s_a[DC_MAX_L];
    const uint16_t *s_b[DC_MAX_L];
    float s_scale[DC_MAX_L];
    int16_t s_rank[DC_MAX_L];
    int32_t s_u[DC_MAX_L];         // touched index of slot s, or -1
    uint32_t tmask[DC_MAX_L / 32]; // slots that some row names
    // touched slots, ascending
    int16_t u_slot[DC_MAX_TN];
    int16_t u_rank[DC_MAX_TN];
    int32_t u_grow[DC_MAX_TN + 1]; // first rank row of touched slot u (ranks rounded to 8)
    int32_t u_koff[DC_MAX_TN];     // k offset in this part's expand (owned slots, ranks rounded to 16)
    // rows whose delta this part adds, in row order
    int16_t own_t[DC_MAX_TN];
    int16_t own_u[DC_MAX_TN];      // touched slots this part owns (touched index), ascending
    int32_t ewsum[4], ewmax[4];
    int32_t nownu;
    const uint16_t *q_src[DC_MAX_Q]; // A row of shrink row q at k = 0, or null (not used)
    int16_t g_slot[DC_MAX_Q / 8];  // slot of 8-row group g of this CTA's shrink rows, or -1
    int16_t g_r0[DC_MAX_Q / 8];    // its first rank row
    int32_t a_tma;                 // 1: every group's A lies in the pool layout (one TMA copy per group and chunk)
    int32_t ngroups;               // groups with rows
    uint32_t onbits[DC_MAX_TN / 32];
    int32_t wsum[4];
    int32_t nu, trows, kx, nq, nown, gmax;
    int32_t q_lo, q_n;             // this cluster's shrink rows: rank rows [q_lo, q_lo + q_n)
    int32_t amode, a_lg;           // 1: one copy of 2^a_lg groups over the whole K part (g_slot[0], g_r0[0])
    int16_t u_pfx[DC_MAX_TN];      // amode 1: the run (cluster) of touched slot u's first groups
    int32_t psum[2], pool_bad;
    int32_t a_go[2];               // cp.async A loaders: 1 while thread 0 found the next slot free
    int32_t xr_nk16, xr_last;
    uint32_t epoch;
    int32_t abort_flag;
    int32_t slot_range;
};

struct DecBars {
    uint64_t full[DC_MAX_STAGES];
    uint64_t empty[DC_MAX_STAGES];
    uint64_t a_full[DC_MAX_NA];
    uint64_t a_empty[DC_MAX_NA];
    uint64_t route_done;
    uint64_t base_done;
    uint64_t acc_full;
    uint64_t x_full;
    uint64_t x_empty;
    uint64_t epi_done;
    uint32_t tmem_base;
};

// ------------------------------------------------------------ cluster PTX
__device__ __forceinline__ uint32_t cluster_ctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Every thread of every CTA of the cluster arrives (release) and waits (acquire).
__device__ __forceinline__ void cluster_sync_all()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// 16 bytes of CTA `rank`'s shared memory at the address of `p` in this CTA
// (read between two cluster barriers: no ordering of its own needed).
__device__ __forceinline__ float4 ld_dsmem_f4(const void *p, uint32_t rank)
{
    uint32_t a = smem_u32(p), ra;
    asm("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(a), "r"(rank));
    float4 v;
    asm("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(ra));
    return v;
}

__device__ __forceinline__ void st_release_u64(unsigned long long *p, unsigned long long v)
{
    asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long *p)
{
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

// Record flag bits for the call with epoch `e`: the status word keeps the
// tag of the call that set its bits, so bits of an earlier call are replaced.
__device__ __forceinline__ void dec_set_flag(uint32_t *status, uint32_t e, uint32_t f)
{
    unsigned long long *w = reinterpret_cast<unsigned long long *>(status);
    unsigned long long old = *reinterpret_cast<volatile unsigned long long *>(w);
    const uint32_t te = status_tag(e);
    for (;;) {
        const uint32_t tag = (uint32_t)(old >> 32), fl = (uint32_t)old;
        const unsigned long long nw = ((unsigned long long)te << 32) | (unsigned long long)((tag == te ? fl : 0u) | f);
        const unsigned long long prev = atomicCAS(w, old, nw);
        if (prev == old)
            return;
        old = prev;
    }
}

// Tag of the call with epoch e in the arrival counter's high half: a value
// that neither zeroed memory nor small leftover integers hold.
__device__ __forceinline__ uint32_t arrive_tag(uint32_t e) { return e ^ 0x9E3779B9u; }

// One arrival on the call's counter: (tag << 32) | arrivals. The first
// arrival of a call replaces whatever an earlier call (or anything else) left
// there (one compare-and-swap); every other arrival is one add on the low half.
__device__ __forceinline__ void dec_arrive(unsigned long long *w, uint32_t e)
{
    const uint32_t tg = arrive_tag(e);
    unsigned long long old = ld_acquire_u64(w);
    while ((uint32_t)(old >> 32) != tg) {
        const unsigned long long prev = atomicCAS(w, old, ((unsigned long long)tg << 32) | 1ull);
        if (prev == old)
            return;
        old = prev;
    }
    atomicAdd(w, 1ull);
}

// Wait (one thread, bounded, with back-off) until the counter holds `want`
// arrivals of epoch e.
__device__ __forceinline__ bool dec_wait_count(const unsigned long long *w, uint32_t e, uint32_t want, uint64_t wait_ns)
{
    const unsigned long long target = ((unsigned long long)arrive_tag(e) << 32) | want;
    if (ld_acquire_u64(w) == target)
        return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        __nanosleep(128);
        if (ld_acquire_u64(w) == target)
            return true;
        if (globaltimer_ns() - t0 > wait_ns)
            return false;
    }
}

// One arrival on a counter that already carries the call's tag: a release
// add whose result nobody waits for (it orders the CTA's earlier writes,
// gathered by a CTA barrier, before it).
__device__ __forceinline__ void red_release_add_u64(unsigned long long *w, unsigned long long v)
{
    asm volatile("red.release.gpu.global.add.u64 [%0], %1;" ::"l"(w), "l"(v) : "memory");
}

// Once the arrivals of the call with epoch e have been counted (or the wait
// gave up): advance the epoch, and, when every arrival came, tag the counter
// of the next call (the one nobody in this call polls) with that call's tag
// and no arrivals, so its arrivals can be plain adds. A call that finds its
// counter untagged (the first on a workspace, one after a timeout, or after
// other kernels moved the epoch on) takes the compare-and-swap counter instead.
__device__ __forceinline__ void dec_next_epoch(const DecParams &p, unsigned long long *hpre, uint32_t e, bool all_came)
{
    if (all_came)
        *reinterpret_cast<volatile unsigned long long *>(hpre + ((e + 1u) & 1u)) =
            (unsigned long long)arrive_tag(e + 1u) << 32;
    *reinterpret_cast<volatile uint32_t *>(p.ws_status + 2) = e + 1;
}

__device__ __forceinline__ void dec_abort(const DecParams &p, DecAux *aux)
{
    if (atomicExch(&aux->abort_flag, 1) == 0)
        dec_set_flag(p.ws_status, aux->epoch, LORA_FLAG_WAIT_TIMEOUT);
}

__device__ __forceinline__ bool dec_aborted(const DecAux *aux) { return *(volatile const int32_t *)&aux->abort_flag != 0; }

// Non-blocking test of an mbarrier phase (mbarrier.try_wait may park the
// thread for a while, which a loop polling several barriers cannot afford).
__device__ __forceinline__ bool mbar_test(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait on an mbarrier phase. With `aux`, it also gives up as soon as
// the CTA has aborted, so one timeout unwinds every role quickly.
__device__ __forceinline__ bool dec_wait(uint64_t *bar, uint32_t parity, uint64_t wait_ns,
                                         const DecAux *aux = nullptr)
{
    const uint32_t a = smem_u32(bar);
    if (mbar_try_wait(a, parity))
        return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(a, parity))
            return true;
        if ((i & 255u) == 0 && (globaltimer_ns() - t0 > wait_ns || (aux != nullptr && dec_aborted(aux))))
            return false;
    }
}

// W is read once per call: its TMA loads carry an L2 evict-first policy, so
// the weight stream does not push out what the call reads again (x, the
// route tables, the h exchange, B rows, the kernel's own instructions).
__device__ __forceinline__ uint64_t l2_evict_first_policy()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ void tma_load_3d_hint(void *dst, const CUtensorMap *map, int32_t c0, int32_t c1,
                                                 int32_t c2, uint64_t *bar, uint64_t pol)
{
    asm volatile("cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
                 " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(dst)),
                 "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar)), "l"(pol)
                 : "memory");
}

__device__ __forceinline__ void tma_load_2d_hint(void *dst, const CUtensorMap *map, int32_t c0, int32_t c1,
                                                 uint64_t *bar, uint64_t pol)
{
    asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
                 " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
                 "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar)), "l"(pol)
                 : "memory");
}

__device__ __forceinline__ void tma_load_5d(void *dst, const CUtensorMap *map, int32_t c0, int32_t c1, int32_t c2,
                                            int32_t c3, int32_t c4, uint64_t *bar)
{
    asm volatile("cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                 " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(smem_u32(dst)),
                 "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4),
                 "r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void split_hl(float v, uint32_t &hi, uint32_t &lo)
{
    const uint16_t h = f32_to_bf16_bits(v);
    hi = h;
    lo = f32_to_bf16_bits(v - __uint_as_float((uint32_t)h << 16));
}

// What an A-loader thread (lt = 0..63) reads at kernel entry: the table
// entries of slots 4 lt .. 4 lt + 3 and the slots of rows lt + 64 i
// (L <= 256, M <= 256).
struct RouteLoads {
    int32_t slot[4];
    const uint16_t *a[4], *b[4];
    float scale[4];
    int32_t rank[4];
};

__device__ __forceinline__ RouteLoads route_load(const DecParams &p, int lt)
{
    RouteLoads r;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int j = lt + i * 64, s = lt * 4 + i;
        r.slot[i] = j < p.M ? p.seq_slot[j] : -1;
        r.a[i] = s < p.L ? p.tab.a_table[s] : nullptr;
        r.b[i] = s < p.L ? p.tab.b_table[s] : nullptr;
        r.scale[i] = s < p.L ? p.tab.scale_table[s] : 0.0f;
        r.rank[i] = s < p.L ? p.tab.rank_table[s] : 0;
    }
    return r;
}

// The touched slot owning rank row gr (< trows): the last u with u_grow[u] <= gr.
__device__ __forceinline__ int dec_find_u(const DecAux *aux, int nu, int gr)
{
    int lo = 0, hi = nu;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (aux->u_grow[mid] <= gr)
            lo = mid;
        else
            hi = mid;
    }
    return lo;
}

// Routing for the shrink, by the two A-loader warps alone (lt = 0..63,
// barrier 3), from the values read at kernel entry, so the A-row copies go
// out about one table read after the kernel starts. Every CTA resolves the
// same tables:
//  - a row takes a delta when its slot is in [0, L), the slot is filled and
//    its scale is not 0 (a rank past R counts as R: the pool has R rows);
//  - the touched slots (ascending) and their ranks; rank rows: touched slot
//    u owns rows [u_grow[u], u_grow[u + 1]) of the shrink, its rank rounded
//    up to 8;
//  - the rank rows in 8-row groups, spread evenly over the clusters: cluster
//    cl shrinks groups [cl G / ncl, (cl + 1) G / ncl), and where their A rows are.
// The slot tables and the rows' keys are left in shared memory for the epilogue.
__device__ void dec_route(const DecParams &p, const DecCfg &c, DecAux *aux, const RouteLoads &ld, int cl, int lt)
{
    const int L = p.L, M = p.M;
    bool range = false;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int j = lt + i * 64;
        if (j < M) {
            const int s = ld.slot[i];
            const bool ok = s >= 0 && s < L;
            range |= s >= L;
            aux->tkey[j] = (int16_t)(ok ? s + 1 : 0);
            if (ok)
                atomicOr(&aux->tmask[s >> 5], 1u << (s & 31));
        }
        const int s = lt * 4 + i;
        if (s < L) {
            aux->s_a[s] = ld.a[i];
            aux->s_b[s] = ld.b[i];
            aux->s_scale[s] = ld.scale[i];
        }
    }
    if (range)
        aux->slot_range = 1;
    named_bar_sync(3, 64);
    // touched slots and their rank rows in slot order: one inclusive scan of
    // (slots, rows) over the 64 threads, four slots each
    int rk[4], cnt = 0, rows = 0;
    bool on[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int s = lt * 4 + i;
        rk[i] = min(max(ld.rank[i], 0), p.R);
        on[i] = s < L && ((aux->tmask[s >> 5] >> (s & 31)) & 1u) && ld.a[i] != nullptr && ld.b[i] != nullptr &&
                ld.scale[i] != 0.0f && rk[i] > 0;
        cnt += on[i] ? 1 : 0;
        rows += on[i] ? (rk[i] + 7) & ~7 : 0;
    }
    const int lane = lt & 31, w = lt >> 5;
    int ic = cnt, ir = rows;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int a = __shfl_up_sync(0xffffffffu, ic, o), d = __shfl_up_sync(0xffffffffu, ir, o);
        if (lane >= o) {
            ic += a;
            ir += d;
        }
    }
    if (lane == 31) {
        aux->wsum[2 * w] = ic;
        aux->wsum[2 * w + 1] = ir;
    }
    named_bar_sync(3, 64);
    const int nu = aux->wsum[0] + aux->wsum[2], trows = aux->wsum[1] + aux->wsum[3];
    int u = ic - cnt + (w ? aux->wsum[0] : 0), g = ir - rows + (w ? aux->wsum[1] : 0);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int s = lt * 4 + i;
        if (s < L) {
            aux->s_rank[s] = (int16_t)rk[i];
            if (on[i]) {
                aux->u_slot[u] = (int16_t)s;
                aux->u_rank[u] = (int16_t)rk[i];
                aux->u_grow[u] = g;
                aux->s_u[s] = u;
                ++u;
                g += (rk[i] + 7) & ~7;
            } else {
                aux->s_u[s] = -1;
            }
        }
    }
    const int G = trows >> 3;
    // One copy per CTA when it can: the rank rows go to the clusters in runs of
    // 2^lg 8-row groups that never cross a slot (each slot's groups cut into
    // runs from its first), run j to cluster j, when there are no more runs than
    // clusters, every touched slot's A lies in the pool, and a box of 2^lg
    // groups over the whole K part fits the A region (c.gb_mask).
    int lg = 0;
    while ((1 << lg) < max(1, (G + c.ncl - 1) / c.ncl))
        ++lg;
    const bool try5 = G > 0 && lg <= 4 && ((c.gb_mask >> lg) & 1);
    int pc[4], pcs = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        pc[i] = (try5 && on[i]) ? ((((rk[i] + 7) >> 3) + (1 << lg) - 1) >> lg) : 0;
        pcs += pc[i];
        if (on[i] && reinterpret_cast<const uint8_t *>(ld.a[i]) != p.pool + (size_t)(lt * 4 + i) * p.slot_bytes)
            aux->pool_bad = 1;
    }
    int ip = pcs;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, ip, o);
        if (lane >= o)
            ip += t;
    }
    if (lane == 31)
        aux->psum[w] = ip;
    if (lt == 0) {
        aux->u_grow[nu] = trows;
        aux->nu = nu;
        aux->trows = trows;
    }
    named_bar_sync(3, 64);
    const int ptot = aux->psum[0] + aux->psum[1];
    const bool m5 = try5 && ptot <= c.ncl && aux->pool_bad == 0;
    if (lt == 0) {
        aux->amode = m5 ? 1 : 0;
        aux->a_lg = lg;
    }
    if (m5) {
        // the run of this cluster: slot s, groups [gi, gi + 2^lg) (fewer at the slot's end)
        int pp = ip - pcs + (w ? aux->psum[0] : 0);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            if (pc[i] > 0 && cl >= pp && cl < pp + pc[i]) {
                const int sl = lt * 4 + i, gi = (cl - pp) << lg;
                const int n = min(1 << lg, ((rk[i] + 7) >> 3) - gi);
                aux->q_lo = aux->u_grow[aux->s_u[sl]] + gi * 8;
                aux->q_n = n * 8;
                aux->nq = 1;
                aux->ngroups = n;
                aux->g_slot[0] = (int16_t)sl;
                aux->g_r0[0] = (int16_t)(gi * 8);
                aux->a_tma = 1;
            }
            if (on[i])
                aux->u_pfx[aux->s_u[lt * 4 + i]] = (int16_t)pp;
            pp += pc[i];
        }
        if (lt == 0 && cl >= ptot) {
            aux->q_lo = 0;
            aux->q_n = 0;
            aux->nq = 0;
            aux->ngroups = 0;
            aux->a_tma = 1;
        }
        named_bar_sync(3, 64);
        return;
    }
    // else the rank rows' groups spread evenly over the clusters: cluster cl
    // shrinks groups [cl G / ncl, (cl + 1) G / ncl)
    const int g0 = cl * G / c.ncl, ng = min(c.Q / 8, (cl + 1) * G / c.ncl - g0);
    if (lt == 0) {
        aux->q_lo = g0 * 8;
        aux->q_n = ng * 8;
        aux->nq = ng > 0 ? 1 : 0;
        aux->ngroups = ng;
    }
    if (w == 0) {
        // one TMA copy per group and chunk when every group's A lies in the pool
        bool pool_ok = true;
        if (lane < ng) {
            const int gr = (g0 + lane) * 8;
            const int v = dec_find_u(aux, nu, gr);
            const int sl = aux->u_slot[v];
            aux->g_slot[lane] = (int16_t)sl;
            aux->g_r0[lane] = (int16_t)(gr - aux->u_grow[v]);
            pool_ok = reinterpret_cast<const uint8_t *>(aux->s_a[sl]) == p.pool + (size_t)sl * p.slot_bytes;
        }
        const bool all_ok = __all_sync(0xffffffffu, pool_ok);
        if (lane == 0)
            aux->a_tma = all_ok ? 1 : 0;
    } else {
        // else each shrink row's A row (rows past the slot's rank stay zero)
        for (int q = lane; q < ng * 8; q += 32) {
            const int gr = g0 * 8 + q;
            const int v = dec_find_u(aux, nu, gr);
            const int r = gr - aux->u_grow[v];
            aux->q_src[q] = r < aux->u_rank[v] ? aux->s_a[aux->u_slot[v]] + (size_t)r * p.K : nullptr;
        }
    }
    named_bar_sync(3, 64);
}

// What only the epilogue needs, by its 128 threads (et), once the A loaders
// have resolved the shrink: each row's delta slot, the rows whose delta this
// part adds, in row order (and as a bit set), the widest of their slots in
// 8-wide groups, and this part's slots (slot mod C) in slot order with their
// k offsets in the expand (ranks rounded to 16).
__device__ void dec_route_epi(const DecParams &p, const DecCfg &c, DecAux *aux, int part, int et)
{
    const int M = p.M;
    int mine = 0, gm = 0;
    const int j0 = et * 2;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int j = j0 + i;
        if (j < M) {
            const int key = aux->tkey[j];
            const int s = (key > 0 && aux->s_u[key - 1] >= 0) ? key - 1 : -1;
            aux->tslot[j] = (int16_t)s;
            if (s >= 0 && s % c.C == part) {
                mine |= 1 << i;
                gm = max(gm, (aux->s_rank[s] + 7) >> 3);
            }
        }
    }
    // exclusive scan of the owned-row counts over the 128 threads (barrier 2)
    const int lane = et & 31, w = et >> 5;
    const int cnt = __popc(mine);
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o)
            incl += t;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        gm = max(gm, __shfl_xor_sync(0xffffffffu, gm, off));
    if (lane == 31) {
        aux->ewsum[w] = incl;
        aux->ewmax[w] = gm;
    }
    const uint32_t bal0 = __ballot_sync(0xffffffffu, mine & 1), bal1 = __ballot_sync(0xffffffffu, (mine >> 1) & 1);
    if (w == 0) {
        // this part's touched slots, ascending, and their k offsets
        const int nu = aux->nu;
        int n = 0, kx = 0;
        for (int u0 = 0; u0 < nu; u0 += 32) {
            const int u = u0 + lane;
            const bool own = u < nu && aux->u_slot[u] % c.C == part;
            const int k16 = own ? (aux->u_rank[u] + 15) & ~15 : 0;
            int ik = k16;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int t = __shfl_up_sync(0xffffffffu, ik, o);
                if (lane >= o)
                    ik += t;
            }
            const uint32_t bal = __ballot_sync(0xffffffffu, own);
            if (own) {
                aux->u_koff[u] = kx + ik - k16;
                aux->own_u[n + __popc(bal & ((1u << lane) - 1u))] = (int16_t)u;
            }
            n += __popc(bal);
            kx += __shfl_sync(0xffffffffu, ik, 31);
        }
        if (lane == 0) {
            aux->nownu = n;
            aux->kx = kx;
        }
    }
    named_bar_sync(2, DC_EPI);
    int pre = 0, nown = 0, gmax = 0;
#pragma unroll
    for (int q = 0; q < DC_EPI / 32; ++q) {
        pre += q < w ? aux->ewsum[q] : 0;
        nown += aux->ewsum[q];
        gmax = max(gmax, aux->ewmax[q]);
    }
    int o = pre + incl - cnt;
#pragma unroll
    for (int i = 0; i < 2; ++i)
        if ((mine >> i) & 1)
            aux->own_t[o++] = (int16_t)(j0 + i);
    // rows 64 w .. 64 w + 63 of this warp as two 32-bit words, rows interleaved
    if (lane == 0) {
        uint32_t lo = 0, hi = 0;
        for (int b = 0; b < 16; ++b) {
            lo |= ((bal0 >> b) & 1u) << (2 * b) | ((bal1 >> b) & 1u) << (2 * b + 1);
            hi |= ((bal0 >> (16 + b)) & 1u) << (2 * b) | ((bal1 >> (16 + b)) & 1u) << (2 * b + 1);
        }
        aux->onbits[2 * w] = lo;
        aux->onbits[2 * w + 1] = hi;
    }
    if (et == 0) {
        aux->nown = nown;
        aux->gmax = gmax;
    }
    named_bar_sync(2, DC_EPI);
}

// Routing export of CTA 0 (the stable grouping of rows by slot: bucket 0 =
// no valid slot, then slot 0, 1, ...), by the 128 epilogue threads.
__device__ void dec_export_routing(const DecParams &p, DecAux *aux, int et)
{
    const int M = p.M, L = p.L;
    for (int j = et; j < M; j += DC_EPI) {
        const int key = aux->tkey[j];
        int before = 0, same = 0;
        for (int i = 0; i < M; ++i) {
            const int ki = aux->tkey[i];
            before += ki < key;
            same += (ki == key) & (i < j);
        }
        p.perm[before + same] = j;
    }
    for (int b = et; b <= L + 1; b += DC_EPI) {
        int before = 0;
        for (int i = 0; i < M; ++i)
            before += aux->tkey[i] < b;
        p.seg_off[b] = before;
    }
}

__global__ void __launch_bounds__(DC_THREADS, 1)
    dec_kernel(const __grid_constant__ TmapSet maps, const __grid_constant__ CUtensorMap amap,
               const __grid_constant__ AMap5 a5m, const __grid_constant__ DecParams p,
               const __grid_constant__ DecCfg c)
{
    extern __shared__ uint8_t dc_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(dc_raw) + 1023) & ~uintptr_t(1023));
    DecAux *aux = reinterpret_cast<DecAux *>(smem + c.aux_off);
    DecBars *bars = reinterpret_cast<DecBars *>(smem + c.bar_off);
    uint8_t *abuf = smem + c.a_off;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // K part: the CTA's rank in its cluster (blockIdx.x % C also without clusters)
    const int part = c.l2sum ? (int)blockIdx.x % c.C : (int)cluster_ctarank();
    const int cl = (int)blockIdx.x / c.C;
    const int nmma = (p.M + 15) & ~15;
    // 64-wide chunks [kc0, kc1), fixed by (K, C) alone -- never by the stage
    // grouping -- so every element sums the same chunks in the same order
    const int kc0 = part * c.kchunks / c.C, kc1 = (part + 1) * c.kchunks / c.C;
    const int nfill = (kc1 - kc0 + c.kc - 1) / c.kc;
    unsigned long long *hcnt = reinterpret_cast<unsigned long long *>(p.ws_status) + DC_HCNT_WORD;
    unsigned long long *hpre = hcnt + 1; // two counters, tagged ahead for the call of epoch e in [e & 1]

    // the routing reads go out first, ahead of the W stream
    RouteLoads rl;
    if (warp == 2 || warp == 3)
        rl = route_load(p, threadIdx.x - 64);
    if (threadIdx.x == 0) {
        for (int i = 0; i < c.stages; ++i) {
            mbar_init(bars->full + i, 1);
            mbar_init(bars->empty + i, 1);
        }
        for (int i = 0; i < c.na; ++i) {
            // full: one arrival (with the copies' bytes, or after the loaders' cp.async)
            mbar_init(bars->a_full + i, 1);
            mbar_init(bars->a_empty + i, 1);
        }
        mbar_init(&bars->route_done, 1);
        mbar_init(&bars->base_done, 1);
        mbar_init(&bars->acc_full, 1);
        mbar_init(&bars->x_full, 1);
        mbar_init(&bars->x_empty, 1);
        mbar_init(&bars->epi_done, DC_EPI);
        aux->abort_flag = 0;
        aux->slot_range = 0;
        for (int i = 0; i < DC_MAX_L / 32; ++i)
            aux->tmask[i] = 0;
        aux->pool_bad = 0;
        aux->epoch = *reinterpret_cast<volatile uint32_t *>(p.ws_status + 2);
        fence_barrier_init();
        prefetch_tmap(&maps.x);
        prefetch_tmap(&maps.w[0]);
        prefetch_tmap(&amap);
    }
    if (warp == 1)
        tmem_alloc(&bars->tmem_base, c.tmem_cols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;
    const uint32_t e = aux->epoch;
    const int ncta = c.ncl * c.C;

    // CTA 0 opens the call's status word: its tag becomes this call's, with no
    // bits unless a CTA has already set one (so bits an earlier call or other
    // data left there never read as this call's)
    if (blockIdx.x == 0 && threadIdx.x == 1)
        dec_set_flag(p.ws_status, e, 0u);
    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            const uint64_t pol = l2_evict_first_policy();
            int last_par[DC_MAX_STAGES];
            for (int i = 0; i < DC_MAX_STAGES; ++i)
                last_par[i] = -1;
            for (int g = 0; g < nfill; ++g) {
                const int st = g % c.stages;
                const uint32_t ph = (uint32_t)(g / c.stages) & 1u;
                if (dec_aborted(aux) || !dec_wait(bars->empty + st, ph ^ 1u, c.wait_ns, aux)) {
                    dec_abort(p, aux);
                    break;
                }
                const int ch0 = kc0 + g * c.kc; // first chunk of the fill (chunks past kc1 are not used)
                uint8_t *stage = smem + (size_t)st * c.stage_bytes;
                mbar_arrive_expect_tx(bars->full + st, (uint32_t)c.kc * (DC_W_CHUNK + c.x_chunk));
                uint8_t *xdst = stage + (size_t)c.kc * DC_W_CHUNK;
                if (c.gated) {
                    // 4D view [chunks][2 halves][I rows][64]: gate rows then up rows
                    asm volatile(
                        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
                        " [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(smem_u32(stage)),
                        "l"(reinterpret_cast<uint64_t>(&maps.w[0])), "r"(0), "r"(cl * 64), "r"(0), "r"(ch0),
                        "r"(smem_u32(bars->full + st)), "l"(pol)
                        : "memory");
                } else if (c.use3d) {
                    tma_load_3d_hint(stage, &maps.w[0], 0, cl * 128, ch0, bars->full + st, pol);
                } else {
                    tma_load_2d_hint(stage, &maps.w[0], ch0 * 64, cl * 128, bars->full + st, pol);
                }
                if (c.use3d)
                    tma_load_3d(xdst, &maps.x, 0, 0, ch0, bars->full + st);
                else
                    tma_load_2d(xdst, &maps.x, ch0 * 64, 0, bars->full + st);
                last_par[st] = (int)ph;
            }
            if (dec_aborted(aux)) // let this thread's copies land before shared memory goes away
                for (int i = 0; i < c.stages; ++i)
                    if (last_par[i] >= 0)
                        dec_wait(bars->full + i, (uint32_t)last_par[i], c.wait_ns);
        }
    } else if (warp == 1) {
        // ------------------------------------------------ UMMA issuer
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16_f32(128, (uint32_t)nmma);
            uint32_t acc_on = 0, h_on = 0;
            int gb = 0, gs = 0, nq = 0;
            int stb = 0, sts = 0, asl = 0; // stage of fill gb, of fill gs; A slot of the next chunk to shrink
            uint32_t phb = 0, aph = 0;     // their phase parities
            bool routed = false, ok = true, afence = false, a5 = false, a5_in = false;
            uint32_t a5_stride = 0;
            uint32_t idle = 0;
            uint64_t t_idle = 0;
            // The loop serves the W stages and the A slots as each lands, polling
            // with non-blocking tests; stage and slot indices advance without
            // divisions, and the wall clock is read only while nothing lands.
            while (gs < nfill) {
                bool prog = false;
                if (!routed && mbar_test(&bars->route_done, 0)) {
                    routed = true;
                    nq = aux->nq;
                    afence = aux->a_tma == 0;
                    a5 = aux->amode != 0;
                    a5_stride = 1024u << aux->a_lg;
                    prog = true;
                }
                if (gb < nfill && gb - gs < c.stages && mbar_test(bars->full + stb, phb)) {
                    tc_fence_after();
                    const uint32_t wb = smem_u32(smem + (size_t)stb * c.stage_bytes);
                    const uint32_t xb = wb + (uint32_t)c.kc * DC_W_CHUNK;
                    const int nch = min(c.kc, kc1 - (kc0 + gb * c.kc));
                    for (int q = 0; q < nch; ++q) {
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            umma_bf16(tmem, sw128_kmajor_desc(wb + q * DC_W_CHUNK + j * 32),
                                      sw128_kmajor_desc(xb + q * c.x_chunk + j * 32), idesc, acc_on);
                            acc_on = 1;
                        }
                    }
                    ++gb;
                    if (++stb == c.stages) {
                        stb = 0;
                        phb ^= 1u;
                    }
                    prog = true;
                }
                while (gs < gb && routed) {
                    const int nch = min(c.kc, kc1 - (kc0 + gs * c.kc));
                    if (nq) {
                        if (a5) {
                            // one copy brought the A rows of every chunk
                            if (!a5_in) {
                                if (!mbar_test(bars->a_full, 0))
                                    break;
                                a5_in = true;
                            }
                        } else {
                            // the A rows of every chunk of fill gs are in their slots
                            bool in = true;
                            int sl = asl;
                            uint32_t ph = aph;
                            for (int q = 0; q < nch; ++q) {
                                if (!mbar_test(bars->a_full + sl, ph)) {
                                    in = false;
                                    break;
                                }
                                if (++sl == c.na) {
                                    sl = 0;
                                    ph ^= 1u;
                                }
                            }
                            if (!in)
                                break;
                        }
                        tc_fence_after();
                        if (afence)
                            fence_proxy_async_smem(); // cp.async (generic proxy) wrote the A rows
                        const uint32_t xb = smem_u32(smem + (size_t)sts * c.stage_bytes) + (uint32_t)c.kc * DC_W_CHUNK;
                        for (int q = 0; q < nch; ++q) {
                            const uint32_t ab = a5 ? smem_u32(abuf) + (uint32_t)(gs * c.kc + q) * a5_stride
                                                   : smem_u32(abuf) + (uint32_t)asl * c.a_chunk;
                            // D_h^T[q, t] += A_rows[q, k] x[t, k]: the rank rows are the
                            // UMMA M side (128 lanes; past Q they are ignored), the rows
                            // of the batch its N side -- the same instruction shape in any
                            // call of the same batch size, one per 16-wide k step
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                umma_bf16(tmem + c.col_h, sw128_kmajor_desc(ab + j * 32),
                                          sw128_kmajor_desc(xb + q * c.x_chunk + j * 32), idesc, h_on);
                                h_on = 1; // the first k step writes, the rest add
                            }
                            if (!a5) {
                                umma_commit(bars->a_empty + asl);
                                if (++asl == c.na) {
                                    asl = 0;
                                    aph ^= 1u;
                                }
                            }
                        }
                    }
                    umma_commit(bars->empty + sts);
                    if (++sts == c.stages)
                        sts = 0;
                    ++gs;
                    prog = true;
                }
                if (prog) {
                    idle = 0;
                } else if ((++idle & 63u) == 0) {
                    const uint64_t now = globaltimer_ns();
                    if (idle == 64)
                        t_idle = now;
                    else if (dec_aborted(aux) || now - t_idle > c.wait_ns) {
                        dec_abort(p, aux);
                        ok = false;
                        break;
                    }
                }
            }
            umma_commit(&bars->base_done);
            // expand rounds staged by the epilogue
            for (int round = 0; ok; ++round) {
                if (!dec_wait(&bars->x_full, (uint32_t)round & 1u, c.wait_ns, aux)) {
                    dec_abort(p, aux);
                    break;
                }
                tc_fence_after();
                const int nk16 = *(volatile int32_t *)&aux->xr_nk16;
                const int last = *(volatile int32_t *)&aux->xr_last;
                const uint32_t xbb = smem_u32(smem);
                const uint32_t xhb = xbb + (uint32_t)c.blocks * DC_XB_BLOCK;
                const uint32_t hblk = (uint32_t)c.tn * 128u;
                const uint32_t plane = (uint32_t)c.blocks * hblk;
                for (int k = 0; k < nk16; ++k) {
                    const uint32_t ko = (uint32_t)(k >> 2) * DC_XB_BLOCK + (uint32_t)(k & 3) * 32u;
                    const uint32_t ho = (uint32_t)(k >> 2) * hblk + (uint32_t)(k & 3) * 32u;
                    for (int h = 0; h < 2; ++h)
                        umma_bf16(tmem + c.col_d, sw128_kmajor_desc(xbb + ko), sw128_kmajor_desc(xhb + h * plane + ho),
                                  idesc, round > 0 || k > 0 || h > 0);
                }
                umma_commit(&bars->x_empty);
                if (last)
                    break;
            }
            umma_commit(&bars->acc_full);
        }
        __syncwarp();
        // TMEM is freed once the epilogue has read it (the epilogue's own
        // waits are bounded and give up together once the CTA aborts)
        dec_wait(&bars->epi_done, 0, 8 * c.wait_ns);
        tc_fence_after();
        tmem_dealloc(tmem, c.tmem_cols);
    } else {
        if (warp < 4) {
            // ------------------------------------------ routing, then the A-row
            // loaders: the CTA's shrink rows, one 64-wide chunk per slot, as far
            // ahead as the slots go
            const int lt = threadIdx.x - 64; // 0..63
            dec_route(p, c, aux, rl, cl, lt);
            const bool tma = aux->a_tma != 0;
            if (lt == 0)
                mbar_arrive(&bars->route_done);
            named_bar_arrive(1, DC_ROUTE); // the epilogue may read the routing
            const int nch = kc1 - kc0;
            if (aux->nq && aux->amode) {
                // one copy: 2^lg groups of slot g_slot[0] from rank row g_r0[0], over
                // nchb chunks from the part's first, chunk by chunk; the thread then
                // waits (bounded) for it to land, so an abort never leaves it in flight
                if (lt == 0) {
                    const int lg = aux->a_lg;
                    mbar_arrive_expect_tx(bars->a_full, (1024u << lg) * (uint32_t)c.nchb);
                    tma_load_5d(abuf, &a5m.m[lg], 0, 0, aux->g_r0[0] >> 3, kc0, aux->g_slot[0], bars->a_full);
                    dec_wait(bars->a_full, 0, c.wait_ns);
                }
            } else if (aux->nq && tma) {
                // one thread: one copy per 8-row group and chunk, [64 k][8 rows] of
                // slot g_slot at rank row g_r0 (k past K zero-filled), 128-byte swizzled
                if (lt == 0) {
                    const int ng = aux->ngroups;
                    int sl = 0, i = 0;
                    uint32_t ph = 0;
                    for (; i < nch; ++i) {
                        if (!dec_wait(bars->a_empty + sl, ph ^ 1u, c.wait_ns, aux)) {
                            dec_abort(p, aux);
                            break;
                        }
                        uint8_t *dst = abuf + (size_t)sl * c.a_chunk;
                        mbar_arrive_expect_tx(bars->a_full + sl, (uint32_t)ng * 1024u);
                        for (int g = 0; g < ng; ++g)
                            tma_load_3d(dst + g * 1024, &amap, (kc0 + i) * 64, aux->g_r0[g], aux->g_slot[g],
                                        bars->a_full + sl);
                        if (++sl == c.na) {
                            sl = 0;
                            ph ^= 1u;
                        }
                    }
                    if (dec_aborted(aux)) // let the copies in flight land before shared memory goes away
                        for (int j = max(0, i - c.na); j < i; ++j)
                            dec_wait(bars->a_full + j % c.na, (uint32_t)(j / c.na) & 1u, c.wait_ns);
                }
            } else if (aux->nq) {
                // all 64 threads copy with cp.async; each makes the slot's barrier
                // wait for its copies, and after a barrier thread 0 gives the one
                // arrival. Thread 0 alone waits for a free slot and passes its verdict
                // on through shared memory (two words: one for this chunk, one for the
                // next), so every thread leaves the loop at the same chunk.
                int sl = 0;
                uint32_t ph = 0;
                for (int i = 0; i < nch; ++i, sl = sl + 1 == c.na ? 0 : sl + 1, ph ^= sl == 0 ? 1u : 0u) {
                    if (lt == 0) {
                        const bool free = dec_wait(bars->a_empty + sl, ph ^ 1u, c.wait_ns, aux);
                        if (!free)
                            dec_abort(p, aux);
                        aux->a_go[i & 1] = free ? 1 : 0;
                    }
                    named_bar_sync(3, 64);
                    if (!aux->a_go[i & 1])
                        break;
                    uint8_t *dst = abuf + (size_t)sl * c.a_chunk;
                    const int k0 = (kc0 + i) * 64;
                    for (int pc = lt; pc < aux->q_n * 8; pc += 64) {
                        const int q = pc >> 3, cq = pc & 7;
                        const uint16_t *src = aux->q_src[q];
                        const int k = k0 + cq * 8;
                        if (src != nullptr) // rows without an A row are never read from D_h
                            cp_async_16(dst + q * 128 + ((cq ^ (q & 7)) << 4), k < p.K ? src + k : src,
                                        k < p.K ? 16u : 0u);
                    }
                    cp_async_mbar_arrive(bars->a_full + sl);
                    named_bar_sync(3, 64);
                    if (lt == 0)
                        mbar_arrive(bars->a_full + sl);
                }
            }
            cp_async_wait_all();
        } else {
            // ------------------------------------------ epilogue
            const int et = threadIdx.x - (DC_THREADS - DC_EPI);
            const int ew = et >> 5;
            // the arrival counter the previous call tagged for this one, if it did
            bool fast = false;
            if (et == 0)
                fast = (uint32_t)(*reinterpret_cast<volatile unsigned long long *>(hpre + (e & 1u)) >> 32) ==
                       arrive_tag(e);
            named_bar_sync(1, DC_ROUTE);
            dec_route_epi(p, c, aux, part, et);
            if (blockIdx.x == 0) {
                dec_export_routing(p, aux, et);
                if (et == 0 && aux->slot_range)
                    dec_set_flag(p.ws_status, e, LORA_FLAG_SLOT_RANGE);
            }
            const bool exch = aux->trows > 0;
            const int kx = aux->kx;
            const bool expand = exch && kx > 0;
            if (!expand && et == 0) { // no expand: the MMA warp finishes with an empty round
                aux->xr_nk16 = 0;
                aux->xr_last = 1;
                mbar_arrive(&bars->x_full);
            }
            const int kround = c.blocks * 64;
            const uint32_t hblk = (uint32_t)c.tn * 128u;
            uint8_t *XB = smem;
            uint8_t *XH = smem + (size_t)c.blocks * DC_XB_BLOCK;
            const uint32_t plane = (uint32_t)c.blocks * hblk;
            // B row of this thread's feature
            int nrow;
            bool row_ok;
            if (c.gated) {
                const int fi = cl * 64 + (et & 63);
                row_ok = fi < c.I;
                nrow = (et < 64 ? 0 : c.I) + fi;
            } else {
                nrow = cl * 128 + et;
                row_ok = nrow < p.N;
            }
            // B rows of the owned slots in the k range [r0k, r0k + kr), into XB
            auto stage_b = [&](int r0k, int kr) {
                const int nownu = aux->nownu;
                for (int iv = 0; iv < nownu; ++iv) {
                    const int v = aux->own_u[iv];
                    const int s = aux->u_slot[v];
                    const int so = aux->u_koff[v] - r0k;
                    const int rk = aux->u_rank[v];
                    const int pk = (rk + 15) & ~15;
                    if (so + pk <= 0 || so >= kr)
                        continue;
                    const uint16_t *src = aux->s_b[s] + (size_t)(row_ok ? nrow : 0) * p.R;
                    for (int q = max(0, -so); q < pk && so + q < kr; q += 8) {
                        const int kl = so + q, cq = kl >> 3;
                        const bool has = row_ok && q < rk;
                        cp_async_16(XB + (size_t)(cq >> 3) * DC_XB_BLOCK + et * 128 + (((cq & 7) ^ (et & 7)) << 4),
                                    src + (has ? q : 0), has ? 16u : 0u);
                    }
                }
            };
            // (1) the K loop (base and shrink UMMAs) has finished
            if (!dec_wait(&bars->base_done, 0, c.wait_ns, aux))
                dec_abort(p, aux);
            tc_fence_after();
            // (2) publish this CTA's partial h of its rank rows (the other CTAs
            // wait for it), then arrive: the CTA barrier orders every thread's
            // stores before thread 0's fence and arrival
            const int q_n = aux->q_n;
            // this CTA's block of h: [t][Q] floats at hpart[part][cl], staged in the
            // A region (free once the K loop is done) and stored with one bulk copy
            const bool pub = exch && aux->nq && !dec_aborted(aux);
            float *hs = reinterpret_cast<float *>(abuf);
            if (pub && ew * 32 < q_n) {
                // lane q of D_h^T is rank row q_lo + q; its columns are the rows of the batch
                const int q = et;
                const uint32_t ta = tmem + ((uint32_t)(ew * 32) << 16) + c.col_h;
                for (int t0 = 0; t0 < nmma; t0 += 32) {
                    uint32_t v[2][16];
                    tmem_ld16_nowait(ta + (uint32_t)t0, v[0]);
                    if (t0 + 16 < nmma)
                        tmem_ld16_nowait(ta + (uint32_t)(t0 + 16), v[1]);
                    tmem_wait_ld();
                    if (q < q_n) {
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            if (t0 + i < p.M)
                                hs[(t0 + i) * c.Q + q] = __uint_as_float(v[i >> 4][i & 15]);
                    }
                }
                fence_proxy_async_smem(); // the bulk copy reads them through the async proxy
            }
            tc_fence_before();
            named_bar_sync(2, DC_EPI);
            // every CTA arrives, with or without h: a CTA that has seen every
            // arrival knows the whole grid has started (and read the epoch)
            if (et == 0) {
                if (pub) {
                    bulk_store_1d(p.hpart + ((size_t)part * c.ncl + cl) * p.M * c.Q, hs, (uint32_t)(p.M * c.Q * 4));
                    bulk_commit();
                    bulk_wait_all();
                    fence_proxy_async_global(); // the block is written before the arrival releases it
                }
                if (fast) {
                    red_release_add_u64(hpre + (e & 1u), 1ull);
                } else {
                    __threadfence();
                    dec_arrive(hcnt, e);
                }
            }
            // the first round's B rows (the stage region is free)
            if (expand)
                stage_b(0, min(kround, kx));
            // (3) the expand: every CTA's arrival, then the operands, round by round
            int mode = 0; // 0: no delta in this part, 1: D' in its own columns
            if (expand) {
                if (et == 0) {
                    if (!dec_wait_count(fast ? hpre + (e & 1u) : hcnt, e, (uint32_t)(ncta + c.extra_arrivals),
                                        c.wait_ns))
                        dec_abort(p, aux);
                    dec_next_epoch(p, hpre, e, !dec_aborted(aux));
                }
                named_bar_sync(2, DC_EPI);
                if (!dec_aborted(aux)) {
                    mode = 1;
                    // where h of touched slot v's rank rows r.. r + 7 lies: the block of
                    // the cluster that shrank them, and the column in it
                    const int hG = aux->trows >> 3, a_lg = aux->a_lg;
                    const bool hm5 = aux->amode != 0;
                    auto h_loc = [&](int v, int r, int &hcl, int &hoff) {
                        if (hm5) {
                            hcl = aux->u_pfx[v] + (r >> (3 + a_lg));
                            hoff = r & ((8 << a_lg) - 1);
                        } else {
                            const int gr = aux->u_grow[v] + r, g = gr >> 3;
                            int cc = g * c.ncl / hG;
                            while (cc + 1 < c.ncl && (cc + 1) * hG / c.ncl <= g)
                                ++cc;
                            while (cc > 0 && cc * hG / c.ncl > g)
                                --cc;
                            hcl = cc;
                            hoff = gr - 8 * (cc * hG / c.ncl);
                        }
                    };
                    const size_t hpart_stride = (size_t)c.ncl * p.M * c.Q;
                    const int nown = aux->nown, gmax = aux->gmax;
                    for (int r0k = 0, round = 0; r0k < kx; r0k += kround, ++round) {
                        const int kr = min(kround, kx - r0k);
                        if (round > 0) { // the previous round's UMMAs have read the buffers
                            if (!dec_wait(&bars->x_empty, (uint32_t)(round - 1) & 1u, c.wait_ns, aux))
                                dec_abort(p, aux);
                            named_bar_sync(2, DC_EPI);
                            stage_b(r0k, kr);
                        }
                        // XH: zeros over the round's k range (rows 0..nmma-1, both planes) ...
                        const int nblk = (kr + 63) >> 6;
                        const uint4 z = make_uint4(0, 0, 0, 0);
                        for (int idx = et; idx < nblk * nmma * 8; idx += DC_EPI) {
                            const int b = idx / (nmma * 8), rem = idx - b * nmma * 8;
                            uint8_t *dst = XH + (size_t)b * hblk + rem * 16;
                            *reinterpret_cast<uint4 *>(dst) = z;
                            *reinterpret_cast<uint4 *>(dst + plane) = z;
                        }
                        named_bar_sync(2, DC_EPI);
                        // ... then s * comp * h of each owned row's 8-wide groups in the round
                        for (int idx = et; idx < nown * gmax; idx += DC_EPI) {
                            const int t = aux->own_t[idx / gmax], gq = idx - (idx / gmax) * gmax;
                            const int s = aux->tslot[t], v = aux->s_u[s];
                            const int rk = aux->u_rank[v], r = gq * 8;
                            const int kl = aux->u_koff[v] + r - r0k;
                            if (r >= rk || kl < 0 || kl >= kr)
                                continue;
                            int hcl, hoff;
                            h_loc(v, r, hcl, hoff);
                            const float *hrow = p.hpart + ((size_t)hcl * p.M + t) * c.Q + hoff;
                            float4 x0[4], x1[4];
#pragma unroll
                            for (int q = 0; q < 4; ++q)
                                if (q < c.C) {
                                    const float *hq = hrow + (size_t)q * hpart_stride;
                                    x0[q] = __ldcg(reinterpret_cast<const float4 *>(hq));
                                    x1[q] = __ldcg(reinterpret_cast<const float4 *>(hq + 4));
                                }
                            const float *cr = p.tab.comp_table + (size_t)s * LORA_COMP_STRIDE + r;
                            const float4 c0 = __ldg(reinterpret_cast<const float4 *>(cr));
                            const float4 c1 = __ldg(reinterpret_cast<const float4 *>(cr + 4));
                            float a[8] = {x0[0].x, x0[0].y, x0[0].z, x0[0].w, x1[0].x, x1[0].y, x1[0].z, x1[0].w};
#pragma unroll
                            for (int q = 1; q < 4; ++q) // K parts summed in part order
                                if (q < c.C) {
                                    a[0] += x0[q].x; a[1] += x0[q].y; a[2] += x0[q].z; a[3] += x0[q].w;
                                    a[4] += x1[q].x; a[5] += x1[q].y; a[6] += x1[q].z; a[7] += x1[q].w;
                                }
                            const float sc = aux->s_scale[s];
                            const float cf[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
                            uint32_t h8[8], l8[8];
#pragma unroll
                            for (int i = 0; i < 8; ++i) {
                                h8[i] = 0;
                                l8[i] = 0;
                                if (r + i < rk)
                                    split_hl(a[i] * (sc * cf[i]), h8[i], l8[i]);
                            }
                            const int cq = kl >> 3;
                            uint8_t *dst = XH + (size_t)(cq >> 3) * hblk + t * 128 + (((cq & 7) ^ (t & 7)) << 4);
                            *reinterpret_cast<uint4 *>(dst) = make_uint4(h8[0] | (h8[1] << 16), h8[2] | (h8[3] << 16),
                                                                         h8[4] | (h8[5] << 16), h8[6] | (h8[7] << 16));
                            *reinterpret_cast<uint4 *>(dst + plane) =
                                make_uint4(l8[0] | (l8[1] << 16), l8[2] | (l8[3] << 16), l8[4] | (l8[5] << 16),
                                           l8[6] | (l8[7] << 16));
                        }
                        cp_async_wait_all();
                        fence_proxy_async_smem(); // generic-proxy writes, read by the UMMAs
                        named_bar_sync(2, DC_EPI);
                        if (et == 0) {
                            aux->xr_nk16 = (kr + 15) / 16;
                            aux->xr_last = r0k + kround >= kx ? 1 : 0;
                            mbar_arrive(&bars->x_full);
                        }
                    }
                }
            }
            cp_async_wait_all();
            // (4) drain base (+ D' on the rows this part owns) into an fp32 tile
            // [rows][128 features]: in the stage region (every UMMA is done), or
            // in the workspace (read by the CTAs of the same feature tile)
            const bool got = dec_wait(&bars->acc_full, 0, c.wait_ns);
            tc_fence_after();
            if (!got)
                dec_abort(p, aux);
            float *ptile = c.l2sum ? p.gpart + (size_t)blockIdx.x * p.M * 128 : reinterpret_cast<float *>(smem);
            const uint32_t lane_off = (uint32_t)(ew * 32) << 16;
            // 32 columns per wait: the base and D' loads of both halves in flight together
            for (int c0 = 0; c0 < nmma; c0 += 32) {
                uint32_t rb[2][16], rd[2][16];
                const uint32_t on32 = mode == 1 ? aux->onbits[c0 >> 5] : 0u;
#pragma unroll
                for (int hh = 0; hh < 2; ++hh)
                    if (c0 + 16 * hh < nmma) {
                        tmem_ld16_nowait(tmem + lane_off + (uint32_t)(c0 + 16 * hh), rb[hh]);
                        if ((on32 >> (16 * hh)) & 0xFFFFu)
                            tmem_ld16_nowait(tmem + lane_off + c.col_d + (uint32_t)(c0 + 16 * hh), rd[hh]);
                    }
                tmem_wait_ld();
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const uint32_t on16 = (on32 >> (16 * hh)) & 0xFFFFu;
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int t = c0 + 16 * hh + j;
                        const float v = (on16 >> j) & 1u ? __uint_as_float(rb[hh][j]) + __uint_as_float(rd[hh][j])
                                                         : __uint_as_float(rb[hh][j]);
                        if (t < p.M)
                            ptile[t * 128 + et] = v;
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(&bars->epi_done);
            if (c.l2sum) {
                // publish the tile, then wait (bounded) for the other K parts' tiles
                __threadfence();
                named_bar_sync(2, DC_EPI);
                if (et == 0)
                    st_release_u64(p.pflags + blockIdx.x, DC_FLAG_MARK | (unsigned long long)e);
                if (et < c.C) {
                    const unsigned long long *fp = p.pflags + cl * c.C + et;
                    const unsigned long long want = DC_FLAG_MARK | (unsigned long long)e;
                    const uint64_t t0 = globaltimer_ns();
                    while (ld_acquire_u64(fp) != want) {
                        __nanosleep(64);
                        if (globaltimer_ns() - t0 > c.wait_ns) {
                            dec_abort(p, aux);
                            break;
                        }
                    }
                }
                named_bar_sync(2, DC_EPI);
            }
            if (!expand && blockIdx.x == 0 && et == 0) {
                // the epoch advances once every CTA has started: CTA 0, when it has
                // no exchange wait of its own, waits for every arrival here
                if (!dec_wait_count(fast ? hpre + (e & 1u) : hcnt, e, (uint32_t)ncta, c.wait_ns))
                    dec_abort(p, aux);
                dec_next_epoch(p, hpre, e, !dec_aborted(aux));
            }
        }
    }
    __syncwarp();
    // (5) split-K sum: this CTA sums its share of the rows over the C parts'
    // tiles, in part order -- from the cluster's shared memory, or from the
    // workspace (the same values and order: the same bytes either way)
    if (!c.l2sum)
        cluster_sync_all();
    if (warp >= 4) {
        const int et = threadIdx.x - (DC_THREADS - DC_EPI);
        const float *ptile = reinterpret_cast<const float *>(smem);
        auto part_f4 = [&](int t, int col, int q) -> float4 {
            if (c.l2sum)
                return __ldcg(reinterpret_cast<const float4 *>(p.gpart + ((size_t)(cl * c.C + q) * p.M + t) * 128 + col));
            return ld_dsmem_f4(ptile + t * 128 + col, (uint32_t)q);
        };
        const int r0 = part * p.M / c.C, r1 = (part + 1) * p.M / c.C;
        if (!c.gated) {
            const int quad = et & 31, grp = et >> 5;
            const int n = cl * 128 + 4 * quad;
            // four rows per pass, every part's value of them loaded before any sum
            for (int t0 = r0 + grp; t0 < r1; t0 += 16) {
                float4 v[4][4];
#pragma unroll
                for (int rr = 0; rr < 4; ++rr)
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        if (q < c.C && t0 + 4 * rr < r1)
                            v[rr][q] = part_f4(t0 + 4 * rr, 4 * quad, q);
#pragma unroll
                for (int rr = 0; rr < 4; ++rr) {
                const int t = t0 + 4 * rr;
                if (t >= r1)
                    break;
                float4 s = v[rr][0];
#pragma unroll
                for (int q = 1; q < 4; ++q)
                    if (q < c.C) {
                        s.x += v[rr][q].x; s.y += v[rr][q].y; s.z += v[rr][q].z; s.w += v[rr][q].w;
                    }
                uint16_t *yr = p.y + (int64_t)t * p.y_stride;
                const uint16_t b0 = f32_to_bf16_bits(s.x), b1 = f32_to_bf16_bits(s.y), b2 = f32_to_bf16_bits(s.z),
                               b3 = f32_to_bf16_bits(s.w);
                if (c.yvec && n + 3 < p.N) {
                    *reinterpret_cast<uint2 *>(yr + n) = make_uint2((uint32_t)b0 | ((uint32_t)b1 << 16),
                                                                   (uint32_t)b2 | ((uint32_t)b3 << 16));
                } else {
                    if (n + 0 < p.N) yr[n + 0] = b0;
                    if (n + 1 < p.N) yr[n + 1] = b1;
                    if (n + 2 < p.N) yr[n + 2] = b2;
                    if (n + 3 < p.N) yr[n + 3] = b3;
                }
                }
            }
        } else {
            // act = silu(g) * u from the bf16-rounded halves, one rounding
            const int quad = et & 15, grp = et >> 4;
            const int fi = cl * 64 + 4 * quad;
            for (int t = r0 + grp; t < r1; t += 8) {
                float4 vg[4], vu[4];
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    if (q < c.C) {
                        vg[q] = part_f4(t, 4 * quad, q);
                        vu[q] = part_f4(t, 64 + 4 * quad, q);
                    }
                float4 g = vg[0], u = vu[0];
#pragma unroll
                for (int q = 1; q < 4; ++q)
                    if (q < c.C) {
                        g.x += vg[q].x; g.y += vg[q].y; g.z += vg[q].z; g.w += vg[q].w;
                        u.x += vu[q].x; u.y += vu[q].y; u.z += vu[q].z; u.w += vu[q].w;
                    }
                const float gv[4] = {g.x, g.y, g.z, g.w}, uv[4] = {u.x, u.y, u.z, u.w};
                uint16_t b[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float gb = bf_lo(f32_to_bf16_bits(gv[i]));
                    const float ub = bf_lo(f32_to_bf16_bits(uv[i]));
                    b[i] = f32_to_bf16_bits(gb / (1.0f + expf(-gb)) * ub);
                }
                uint16_t *yr = p.y + (int64_t)t * p.y_stride;
                if (c.yvec && fi + 3 < c.I) {
                    *reinterpret_cast<uint2 *>(yr + fi) = make_uint2((uint32_t)b[0] | ((uint32_t)b[1] << 16),
                                                                    (uint32_t)b[2] | ((uint32_t)b[3] << 16));
                } else {
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        if (fi + i < c.I)
                            yr[fi + i] = b[i];
                }
            }
        }
    }
    // peers are done reading this CTA's tile
    if (!c.l2sum)
        cluster_sync_all();
}

uint32_t pow2_cols(uint32_t v)
{
    uint32_t r = 32;
    while (r < v)
        r <<= 1;
    return r;
}

uint32_t align_up_u(uint32_t v, uint32_t a) { return (v + a - 1) / a * a; }

constexpr uint32_t DC_SMEM_LIMIT = 232448;

int dec_q(int M, int L, int R, int ncl)
{
    const int worst = (M < L ? M : L) * ((R + 7) & ~7); // every row a different slot at the pool rank
    int q = (worst + ncl - 1) / ncl;
    q = (q + 15) & ~15;
    return q < 16 ? 16 : q;
}

// Shared-memory layout: [stage region][A rows of the K part][aux][bars]. The
// stage region is reused after the K loop for the expand operands and the
// fp32 tile.
bool make_dec_cfg(DecCfg &c, int M, int K, int L, int R, int kc, int stages, int C, int ncl, int gated, int I,
                  int min_na)
{
    memset(&c, 0, sizeof c);
    c.tn = tc_token_tile(M);
    c.kc = kc;
    c.stages = stages;
    c.C = C;
    c.ncl = ncl;
    c.kchunks = (K + 63) / 64;
    c.use3d = (K % 64) == 0 ? 1 : 0;
    if (kc > 1 && !c.use3d)
        return false;
    if (c.kchunks < C || L > DC_MAX_L)
        return false;
    c.gated = gated;
    c.I = I;
    const int q = dec_q(M, L, R, ncl);
    if (q > DC_MAX_Q)
        return false;
    c.Q = q;
    c.x_chunk = (uint32_t)c.tn * 128u;
    c.stage_bytes = (uint32_t)kc * (DC_W_CHUNK + c.x_chunk);
    c.a_chunk = (uint32_t)q * 128u;
    c.region = (uint32_t)stages * c.stage_bytes;
    // the fp32 tile of the split-K sum
    if (c.region < (uint32_t)c.tn * 512u)
        return false;
    const uint32_t hblk = (uint32_t)c.tn * 128u;
    c.blocks = (int)(c.region / (DC_XB_BLOCK + 2 * hblk));
    if (c.blocks > 8)
        c.blocks = 8;
    if (c.blocks < 1)
        return false;
    // A-row slots: as many 64-wide chunks of the largest K part as fit, at
    // least `min_na`
    const int max_nch = (c.kchunks + C - 1) / C;
    c.a_off = c.region;
    const uint32_t fixed = c.a_off + align_up_u((uint32_t)sizeof(DecAux), 16) + (uint32_t)sizeof(DecBars) + 64u + 1024u;
    if (fixed >= DC_SMEM_LIMIT)
        return false;
    int na = (int)((DC_SMEM_LIMIT - fixed) / c.a_chunk);
    na = min(na, min(max_nch, DC_MAX_NA));
    if (na < min(min_na, max_nch) || na < kc)
        return false;
    c.na = na;
    // the CTA's h block [M][Q] fp32 is staged in the A region after the K loop
    if ((uint32_t)M * (uint32_t)q * 4u > (uint32_t)na * c.a_chunk)
        return false;
    uint32_t o = c.a_off + (uint32_t)na * c.a_chunk;
    // the shrink UMMA reads 128 rank rows from each A slot: rows past Q
    // (ignored lanes) run into the next slots and must still lie inside the
    // allocation past the last one
    const uint32_t a_tail = (128u - (uint32_t)q) * 128u;
    c.aux_off = align_up_u(o, 16);
    o = c.aux_off + (uint32_t)sizeof(DecAux);
    c.bar_off = align_up_u(o, 16);
    o = c.bar_off + (uint32_t)sizeof(DecBars);
    const uint32_t need_tail = c.a_off + (uint32_t)na * c.a_chunk + a_tail;
    if (o < need_tail)
        o = need_tail;
    c.smem_bytes = 1024u + o;
    if (c.smem_bytes > DC_SMEM_LIMIT)
        return false;
    // base [0, tn); D_h^T and then D' share [tn, 2 tn) (h is read out before the expand)
    c.col_h = (uint32_t)c.tn;
    c.col_d = (uint32_t)c.tn;
    c.tmem_cols = pow2_cols(2u * (uint32_t)c.tn);
    if (c.tmem_cols > 512)
        return false;
    c.wait_ns = WAIT_NS;
    return true;
}

// The plan: at least 8 A-row slots (or the whole K part) if any shape allows
// it, then the widest K chunk per stage that leaves three stages, then more
// stages.
bool plan_dec(DecCfg &c, int M, int K, int L, int R, int C, int ncl, int gated, int I)
{
    const int kcs[3] = {2, 1, 4};
    for (int pass = 0; pass < 2; ++pass)
        for (int i = 0; i < 3; ++i)
            for (int s = DC_MAX_STAGES; s >= 3; --s)
                if (make_dec_cfg(c, M, K, L, R, kcs[i], s, C, ncl, gated, I, pass == 0 ? 8 : 1))
                    return true;
    return false;
}

// Clusters of C CTAs that can be resident at once, per (device, C, smem).
int max_clusters(int C, uint32_t smem)
{
    static std::mutex mu;
    struct Ent {
        int dev, C;
        uint32_t smem;
        int n;
    };
    static Ent cache[64];
    static int ncache = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return 0;
    std::lock_guard<std::mutex> g(mu);
    for (int i = 0; i < ncache; ++i)
        if (cache[i].dev == dev && cache[i].C == C && cache[i].smem == smem)
            return cache[i].n;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = (unsigned)C;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.gridDim = dim3((unsigned)C);
    cfg.blockDim = dim3(DC_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, dec_kernel, &cfg) != cudaSuccess) {
        cudaGetLastError();
        n = 0;
    }
    if (ncache < 64)
        cache[ncache++] = Ent{dev, C, smem, n};
    return n;
}

std::atomic<uint64_t> g_test_wait_ns{0};
std::atomic<int> g_test_extra{0};

int dec_ncl(int N, int gated, int I) { return gated ? (I + 63) / 64 : (N + 127) / 128; }

} // namespace

size_t dec_hpart_floats(int M, int K, int N, int L, int R, int gated)
{
    const int C = tc_csplit(M, K, false);
    const int ncl = dec_ncl(N, gated, N / 2);
    return (size_t)C * (size_t)M * (size_t)ncl * (size_t)dec_q(M, L, R, ncl);
}

int dec_flag_count(int M, int K, int N, int gated)
{
    return tc_csplit(M, K, false) * dec_ncl(N, gated, N / 2);
}

void dec_test_hook(uint64_t wait_ns, int extra_arrivals)
{
    g_test_wait_ns.store(wait_ns);
    g_test_extra.store(extra_arrivals);
}

void test_hook_get(uint64_t &wait_ns, int &extra)
{
    wait_ns = g_test_wait_ns.load();
    extra = wait_ns ? g_test_extra.load() : 0;
}

// Plan and launch; returns cudaErrorNotSupported when the shape does not fit
// this kernel (the caller then takes the general tensor-core path).
cudaError_t launch_dec(const DecLaunch &d, int num_sms, cudaStream_t st)
{
    if (d.M < 1 || d.M > DC_MAX_TN || d.L > DC_MAX_L)
        return cudaErrorNotSupported;
    const int C = tc_csplit(d.M, d.K, false);
    const int ncl = dec_ncl(d.N, d.gated, d.I);
    if (ncl * C > num_sms)
        return cudaErrorNotSupported;
    DecCfg c;
    if (!plan_dec(c, d.M, d.K, d.L, d.R, C, ncl, d.gated, d.I))
        return cudaErrorNotSupported;
    c.yvec = d.yvec;
    const uint64_t tw = g_test_wait_ns.load();
    if (tw) {
        c.wait_ns = tw;
        c.extra_arrivals = g_test_extra.load();
    }
    static std::atomic<uint64_t> raised{0};
    cudaError_t e = raise_smem_limit(raised, dec_kernel, (int)DC_SMEM_LIMIT);
    if (e != cudaSuccess)
        return e;
    // Every CTA waits for every other CTA's arrival, so the whole grid must be
    // resident. When the device holds every cluster of C CTAs at once, the K
    // parts of a feature tile form a cluster and sum over distributed shared
    // memory; otherwise the launch is cooperative (the whole grid resident or
    // no launch) and the parts sum through the workspace.
    c.l2sum = max_clusters(C, c.smem_bytes) < ncl ? 1 : 0;
    // one-copy A rows: the box must land inside the A region, and the shrink's
    // 128-row reads from its last chunk must stay inside the allocation
    c.nchb = (c.kchunks + C - 1) / C;
    c.gb_mask = 0;
    AMap5 a5m;
    memset(&a5m, 0, sizeof a5m);
    for (int lg = 0; lg <= 4; ++lg) {
        const uint32_t gbytes = 1024u << lg;
        if (!((d.gb_mask >> lg) & 1) || gbytes * (uint32_t)c.nchb > (uint32_t)c.na * c.a_chunk ||
            c.a_off + (uint32_t)(c.nchb - 1) * gbytes + 16384u > c.smem_bytes - 1024u)
            continue;
        c.gb_mask |= 1 << lg;
        a5m.m[lg] = d.amap5[lg];
    }
    if (c.l2sum && (d.gpart == nullptr || d.pflags == nullptr))
        return cudaErrorNotSupported;
    DecParams p;
    memset(&p, 0, sizeof p);
    p.x = d.x;
    p.x_stride = d.x_stride;
    p.y = d.y;
    p.y_stride = d.y_stride;
    p.seq_slot = d.seq_slot;
    p.M = d.M;
    p.K = d.K;
    p.N = d.N;
    p.L = d.L;
    p.R = d.R;
    p.tab = d.tab;
    p.ws_status = d.status;
    p.perm = d.perm;
    p.seg_off = d.seg_off;
    p.hpart = d.hpart;
    p.gpart = d.gpart;
    p.pflags = d.pflags;
    p.pool = static_cast<const uint8_t *>(d.pool);
    p.slot_bytes = d.slot_bytes;
    cudaLaunchAttribute attr;
    if (c.l2sum) {
        attr.id = cudaLaunchAttributeCooperative;
        attr.val.cooperative = 1;
    } else {
        attr.id = cudaLaunchAttributeClusterDimension;
        attr.val.clusterDim.x = (unsigned)C;
        attr.val.clusterDim.y = 1;
        attr.val.clusterDim.z = 1;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(ncl * C));
    cfg.blockDim = dim3(DC_THREADS);
    cfg.dynamicSmemBytes = c.smem_bytes;
    cfg.stream = st;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, dec_kernel, d.maps, d.amap, a5m, p, c);
}

int dec_plan_info(int M, int K, int N, int L, int R, int gated, int I, int num_sms, int *clusters_needed,
                  int *clusters_resident, int *cluster_size, uint32_t *smem)
{
    *clusters_needed = 0;
    *clusters_resident = 0;
    *cluster_size = 0;
    *smem = 0;
    if (M < 1 || M > DC_MAX_TN || L > DC_MAX_L)
        return 0;
    const int C = tc_csplit(M, K, false);
    const int ncl = dec_ncl(N, gated, I);
    *clusters_needed = ncl;
    *cluster_size = C;
    if (ncl * C > num_sms)
        return 0;
    DecCfg c;
    if (!plan_dec(c, M, K, L, R, C, ncl, gated, I))
        return 0;
    *smem = c.smem_bytes;
    static std::atomic<uint64_t> raised{0};
    if (raise_smem_limit(raised, dec_kernel, (int)DC_SMEM_LIMIT) != cudaSuccess)
        return 0;
    *clusters_resident = max_clusters(C, c.smem_bytes);
    return 1;
}

int dec_plan_kc(int M, int K, int N, int L, int R, int gated, int I)
{
    const int C = tc_csplit(M, K, false);
    DecCfg c;
    return plan_dec(c, M, K, L, R, C, dec_ncl(N, gated, I), gated, I) ? c.kc : 0;
}

} // namespace rd
