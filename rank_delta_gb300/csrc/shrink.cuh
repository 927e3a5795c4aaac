// The LoRA shrink h_i = A_s x_i (ferrox-core `weight_matrix/lora.rs`,
// `LoraDelta::project`), as work units over the routing sort.
//
// A unit is (bucket b, rank group of 8, up to 4 rows of that bucket, one of
// kp parts of K): a group of warps splitting the K part (four in the shrink
// kernel and the epilogue, two in the projection kernel's shrink warps), lanes taking 8-element
// (16-byte) vectors, each lane accumulating 8 ranks x 4 rows. A slot's A rows
// are read once per 4 rows rather than once per row. Part q writes its
// partial sums to h[q][row][r] (fp32); readers add the kp parts in part
// order, so h is the same on every run.
// Ranks between the adapter's rank and the next multiple of 8 are written as
// zero so the expand can run in 8-wide vectors.
#pragma once
#include "lora_internal.cuh"
#include "ptx.cuh"
#include "vec.cuh"

namespace rd {

constexpr int SHRINK_WARPS = 4;

struct UnitLoc {
    int b, e, s, rank, rg, r0, nrows, kpart;
};

// Units of one bucket: rank groups x row chunks x K parts.
__host__ __device__ __forceinline__ int bucket_units(int rank, int rows, int kp)
{
    return ((rank + SHRINK_RG - 1) / SHRINK_RG) * ((rows + SHRINK_TC - 1) / SHRINK_TC) * kp;
}

// K range of part q: whole 256-element steps, so every lane stays aligned.
__device__ __forceinline__ void kpart_range(int K, int kp, int q, int &k0, int &k1)
{
    const int step = ((K + kp - 1) / kp + 255) / 256 * 256;
    k0 = q * step;
    k1 = min(K, k0 + step);
}

// Locate unit u. unit_off / seg_off may be the workspace arrays or copies of
// them in shared memory (the binary search is a chain of dependent loads).
__device__ __forceinline__ UnitLoc locate_unit(const Params &p, int u, const int32_t *unit_off,
                                               const int32_t *seg_off)
{
    const int nb = p.E * (p.L + 1);
    int lo = 0, hi = nb;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (unit_off[mid] <= u)
            lo = mid;
        else
            hi = mid;
    }
    UnitLoc l;
    l.b = lo;
    l.e = lo / (p.L + 1);
    l.s = lo % (p.L + 1) - 1;
    l.rank = p.tab[l.e].rank_table[l.s];
    const int nrg = (l.rank + SHRINK_RG - 1) / SHRINK_RG;
    int local = u - unit_off[lo];
    l.kpart = local % p.kp;
    local /= p.kp;
    l.rg = local % nrg;
    const int tc = local / nrg;
    l.r0 = seg_off[lo] + tc * SHRINK_TC;
    l.nrows = min(SHRINK_TC, seg_off[lo + 1] - l.r0);
    return l;
}

// Sum v[0..31] over the 32 lanes, leaving lane l with the total of v[l]
// (reduce-scatter butterfly: 31 shuffles instead of 32 x 5).
__device__ __forceinline__ float warp_reduce_scatter32(float (&v)[32], int lane)
{
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        const bool hi = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < o; ++i) {
            const float send = hi ? v[i] : v[i + o];
            const float keep = hi ? v[i + o] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
    }
    return v[0];
}

// What a unit needs before its loads can start: A of its slot and its x
// rows. Built once per unit (table and perm reads) so that the loads of the
// unit itself depend on nothing but these fields.
struct UnitMeta {
    const uint16_t *A;       // A of the slot, [R][K]
    int32_t row[SHRINK_TC];  // x rows of the unit (the last one repeated past nrows)
    int16_t b, rank, rg, kpart, nrows, pad;
};

__device__ __forceinline__ UnitMeta unit_meta(const Params &p, int u, const int32_t *unit_off,
                                              const int32_t *seg_off)
{
    const UnitLoc l = locate_unit(p, u, unit_off, seg_off);
    UnitMeta m;
    m.A = p.tab[l.e].a_table[l.s];
#pragma unroll
    for (int j = 0; j < SHRINK_TC; ++j)
        m.row[j] = p.ws.perm[l.r0 + min(j, l.nrows - 1)];
    m.b = (int16_t)l.b;
    m.rank = (int16_t)l.rank;
    m.rg = (int16_t)l.rg;
    m.kpart = (int16_t)l.kpart;
    m.nrows = (int16_t)l.nrows;
    m.pad = 0;
    return m;
}

// Unit m, executed by NW warps (w = 0..NW-1) of one group that shares named
// barrier `bar_id` and the float scratch `red` [NW][32]: the warps split the
// unit's K part NW ways, each lane accumulating 8 ranks x 4 rows over its
// 8-element K slices so every load of a pass is in flight at once; lane sums
// are reduce-scattered, then the warps' sums are added (warp order) and
// written to h.
template <int NW = SHRINK_WARPS>
__device__ __forceinline__ void shrink_unit(const Params &p, const UnitMeta &m, int w, int lane,
                                            float *red, int bar_id)
{
    int kb, ke;
    kpart_range(p.K, p.kp, m.kpart, kb, ke);
    // this warp's quarter of the K part, in whole 256-element steps
    const int steps = (ke - kb + 255) / 256;
    const int s0 = kb + (steps * w / NW) * 256, s1 = min(ke, kb + (steps * (w + 1) / NW) * 256);
    const uint16_t *arow[SHRINK_RG];
#pragma unroll
    for (int r = 0; r < SHRINK_RG; ++r) {
        const int rr = m.rg * SHRINK_RG + r;
        arow[r] = m.A + (size_t)(rr < m.rank ? rr : 0) * p.K;
    }
    float *hpart = p.ws.h + (size_t)m.kpart * p.rows * p.R;
    const int nr = m.nrows;
    const uint16_t *xr[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
        xr[j] = p.x + (int64_t)m.row[j] * p.x_stride;
    float acc[32]; // [rank][row]
#pragma unroll
    for (int i = 0; i < 32; ++i)
        acc[i] = 0.0f;
#pragma unroll 2
    for (int k0 = s0 + lane * 8; k0 < s1; k0 += 256) {
        uint4 xv[4], av[SHRINK_RG];
#pragma unroll
        for (int j = 0; j < 4; ++j)
            xv[j] = ld_nc_16(xr[j] + k0); // rows past nrows repeat the last row; their sums are dropped
#pragma unroll
        for (int r = 0; r < SHRINK_RG; ++r)
            av[r] = ld_nc_16(arow[r] + k0); // ranks past the rank read row 0; their sums are dropped
#pragma unroll
        for (int r = 0; r < SHRINK_RG; ++r)
#pragma unroll
            for (int j = 0; j < 4; ++j)
                acc[r * 4 + j] = dot8_acc(acc[r * 4 + j], av[r], xv[j]);
    }
    const float mine = warp_reduce_scatter32(acc, lane); // lane = rank * 4 + row
    red[w * 32 + lane] = mine;
    named_bar_sync(bar_id, NW * 32);
    if (w == 0) {
        float t = red[lane];
#pragma unroll
        for (int q = 1; q < NW; ++q)
            t += red[q * 32 + lane];
        const int r = m.rg * SHRINK_RG + lane / 4, j = lane % 4;
        if (j < nr)
            hpart[(size_t)m.row[j] * p.R + r] = r < m.rank ? t : 0.0f;
    }
    named_bar_sync(bar_id, NW * 32);
}

// h[row][r..r+8) summed over the kp parts (part order), for readers running
// after the producing units have been waited for (L2 reads: the parts are
// written during the same kernel).
__device__ __forceinline__ void h_sum8(const Params &p, int row, int r, float4 &a, float4 &b)
{
    const size_t part = (size_t)p.rows * p.R;
    const float *h = p.ws.h + (size_t)row * p.R + r;
    a = __ldcg(reinterpret_cast<const float4 *>(h));
    b = __ldcg(reinterpret_cast<const float4 *>(h + 4));
    for (int q = 1; q < p.kp; ++q) {
        const float4 c = __ldcg(reinterpret_cast<const float4 *>(h + q * part));
        const float4 d = __ldcg(reinterpret_cast<const float4 *>(h + q * part + 4));
        a.x += c.x; a.y += c.y; a.z += c.z; a.w += c.w;
        b.x += d.x; b.y += d.y; b.z += d.z; b.w += d.w;
    }
}

// Mark one more unit of bucket b finished (after the group's h writes).
__device__ __forceinline__ void shrink_unit_done(const Params &p, int b)
{
    __threadfence();
    atomicAdd(p.ws.done + b, 1);
}

__device__ __forceinline__ int ld_acquire_gpu(const int *p)
{
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Wait until every shrink unit of bucket b has finished; false after ~1 s.
__device__ __forceinline__ bool wait_bucket(const Params &p, int b, const int32_t *unit_off)
{
    const int need = unit_off[b + 1] - unit_off[b];
    if (ld_acquire_gpu(p.ws.done + b) >= need)
        return true;
    uint64_t t0;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t0));
    for (;;) {
        if (ld_acquire_gpu(p.ws.done + b) >= need)
            return true;
        uint64_t t;
        asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
        if (t - t0 > 1000000000ull)
            return false;
    }
}

} // namespace rd
