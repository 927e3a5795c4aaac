// Gated MLP input from a fused [gate|up] projection's output:
//
//   act[i][n] = silu(g) * u,  g = y[i][n], u = y[i][I + n], silu(g) = g / (1 + e^-g)
//
// frink `lora_attach.rs`, `parts_mut`: a fused ffn_up holds the gate rows, then
// the up rows (Phi-3), and its adapter's B rows split the same way over one A,
// so one projection call produces both halves. fp32 arithmetic from the bf16
// halves, one rounding to bf16 (nearest even).
#include "lora_internal.cuh"

namespace rd {

namespace {

__device__ __forceinline__ float silu_mul1(float g, float u) { return g / (1.0f + expf(-g)) * u; }

__device__ __forceinline__ float lo_f(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float hi_f(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ uint32_t pack2(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ uint32_t act2(uint32_t g, uint32_t u)
{
    return pack2(silu_mul1(lo_f(g), lo_f(u)), silu_mul1(hi_f(g), hi_f(u)));
}

// Eight outputs per thread and step: 16-byte loads of g and u, one 16-byte
// store (I, the strides and the bases multiples of 8 elements).
__global__ void silu_mul_vec_kernel(const uint16_t *__restrict__ y, int64_t y_stride, int M, int I,
                                    uint16_t *__restrict__ act, int64_t act_stride)
{
    const int per_row = I >> 3;
    const long long total = (long long)M * per_row;
    for (long long v = (long long)blockIdx.x * blockDim.x + threadIdx.x; v < total;
         v += (long long)gridDim.x * blockDim.x) {
        const int i = (int)(v / per_row), n = (int)(v - (long long)i * per_row) * 8;
        const uint16_t *row = y + (size_t)i * y_stride;
        const uint4 g = *reinterpret_cast<const uint4 *>(row + n);
        const uint4 u = *reinterpret_cast<const uint4 *>(row + I + n);
        *reinterpret_cast<uint4 *>(act + (size_t)i * act_stride + n) =
            make_uint4(act2(g.x, u.x), act2(g.y, u.y), act2(g.z, u.z), act2(g.w, u.w));
    }
}

// Any shape: one output per thread and step.
__global__ void silu_mul_kernel(const uint16_t *__restrict__ y, int64_t y_stride, int M, int I,
                                uint16_t *__restrict__ act, int64_t act_stride)
{
    const long long total = (long long)M * I;
    for (long long v = (long long)blockIdx.x * blockDim.x + threadIdx.x; v < total;
         v += (long long)gridDim.x * blockDim.x) {
        const int i = (int)(v / I), n = (int)(v - (long long)i * I);
        const uint16_t *row = y + (size_t)i * y_stride;
        const float g = __uint_as_float((uint32_t)row[n] << 16);
        const float u = __uint_as_float((uint32_t)row[I + n] << 16);
        act[(size_t)i * act_stride + n] = (uint16_t)(pack2(silu_mul1(g, u), 0.0f) & 0xffffu);
    }
}

} // namespace

cudaError_t launch_silu_mul(const uint16_t *y, int64_t y_stride, int M, int I, uint16_t *act,
                            int64_t act_stride, int num_sms, cudaStream_t st)
{
    const bool vec = I % 8 == 0 && y_stride % 8 == 0 && act_stride % 8 == 0 &&
                     (reinterpret_cast<uintptr_t>(y) & 15u) == 0 && (reinterpret_cast<uintptr_t>(act) & 15u) == 0;
    const long long work = vec ? (long long)M * (I / 8) : (long long)M * I;
    const int threads = 256;
    long long blocks = (work + threads - 1) / threads;
    const long long cap = 8LL * num_sms; // a few waves, grid-stride beyond
    if (blocks > cap)
        blocks = cap;
    if (blocks < 1)
        blocks = 1;
    if (vec)
        silu_mul_vec_kernel<<<(unsigned)blocks, threads, 0, st>>>(y, y_stride, M, I, act, act_stride);
    else
        silu_mul_kernel<<<(unsigned)blocks, threads, 0, st>>>(y, y_stride, M, I, act, act_stride);
    return cudaGetLastError();
}

} // namespace rd
