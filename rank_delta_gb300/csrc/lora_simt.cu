// CUDA-core GEMV path of the LoRA projection, for batches of a few rows.
//
// One warp per output row n (grid-stride), rows of x taken 8 at a time: the
// warp streams W[n, :] once per 8 rows with 16-byte loads, keeps 8 fp32
// partial sums per lane and reduces them with shuffles. The expand-fold is in
// the same pass: y = base + s * (B_s[n, :] . (c_s * h_i)), rounded once to bf16
// (ferrox-core `weight_matrix/lora.rs`, `LoraDelta::accumulate`), with h_i
// the rank-sized shrink of the row produced by shrink_kernel and c_s the
// slot's per-rank factors (1 for a single adapter, each member's scale for a
// stack of adapters).
#include "lora_internal.cuh"
#include "shrink.cuh"
#include "vec.cuh"

namespace rd {

constexpr int SIMT_ROWS = 8;

__global__ void __launch_bounds__(256) simt_kernel(Params p)
{
    const int lane = threadIdx.x & 31;
    const int gwarp = blockIdx.x * 8 + (threadIdx.x >> 5);
    const int nwarps = gridDim.x * 8;
    for (int e = 0; e < p.E; ++e) {
        int s0 = 0, s1 = p.rows;
        if (p.expert_offsets) {
            s0 = p.expert_offsets[e];
            s1 = p.expert_offsets[e + 1];
            s0 = max(s0, 0);
            s1 = min(s1, p.rows);
        }
        const uint16_t *W = p.W[e];
        const Tables &tab = p.tab[e];
        for (int n = gwarp; n < p.N; n += nwarps) {
            const uint16_t *wrow = W + (size_t)n * p.K;
            for (int t0 = s0; t0 < s1; t0 += SIMT_ROWS) {
                const int nr = min(SIMT_ROWS, s1 - t0);
                float acc[SIMT_ROWS];
#pragma unroll
                for (int j = 0; j < SIMT_ROWS; ++j)
                    acc[j] = 0.0f;
                for (int k0 = lane * 8; k0 < p.K; k0 += 256) {
                    const uint4 w8 = ld_nc_16(wrow + k0);
#pragma unroll
                    for (int j = 0; j < SIMT_ROWS; ++j)
                        if (j < nr)
                            acc[j] = dot8_acc(acc[j], w8,
                                              ld_16(p.x + (int64_t)(t0 + j) * p.x_stride + k0));
                }
#pragma unroll
                for (int j = 0; j < SIMT_ROWS; ++j)
                    acc[j] = warp_sum(acc[j]);
                if (lane < nr) {
                    const int t = t0 + lane;
                    float v = 0.0f;
#pragma unroll
                    for (int j = 0; j < SIMT_ROWS; ++j)
                        if (j == lane)
                            v = acc[j];
                    const SlotInfo si = slot_info(tab, p.seq_slot[t], p.L);
                    if (si.on) {
                        const uint16_t *brow = si.b + (size_t)n * p.R;
                        const float *cr = tab.comp_table + (size_t)p.seq_slot[t] * LORA_COMP_STRIDE;
                        float d = 0.0f;
                        for (int q = 0; q < si.rank; q += 8) {
                            float4 h0, h1;
                            h_sum8(p, t, q, h0, h1);
                            // the rank's factor (1 unless the slot holds a stack of adapters)
                            const float4 c0 = __ldg(reinterpret_cast<const float4 *>(cr + q));
                            const float4 c1 = __ldg(reinterpret_cast<const float4 *>(cr + q + 4));
                            h0.x *= c0.x; h0.y *= c0.y; h0.z *= c0.z; h0.w *= c0.w;
                            h1.x *= c1.x; h1.y *= c1.y; h1.z *= c1.z; h1.w *= c1.w;
                            d = dot8_bf_f32(d, ld_nc_16(brow + q), h0, h1);
                        }
                        v = v + si.scale * d;
                    }
                    p.y[(int64_t)t * p.y_stride + n] = f32_to_bf16_bits(v);
                }
            }
        }
    }
}

cudaError_t launch_simt(const Params &p, int num_sms, cudaStream_t st)
{
    const int warps_needed = p.N;
    int blocks = (warps_needed + 7) / 8;
    blocks = blocks < 4 * num_sms ? blocks : 4 * num_sms;
    if (blocks < 1)
        blocks = 1;
    simt_kernel<<<blocks, 256, 0, st>>>(p);
    return cudaGetLastError();
}

} // namespace rd
