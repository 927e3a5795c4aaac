// lora_proj_apply_static_ws: the projection for callers that cannot allocate
// device memory.
//
// lora_proj_apply needs a caller-provided workspace (routing sort, shrink work
// list, the rank-sized h of every row, the status word). Some callers have no
// way to provide one: plugins whose host framework owns all device memory and
// hands them no allocator, or services that must not grow device memory after
// start-up and so never call cudaMalloc on a request path. This entry point
// runs the same kernels with that scratch taken from a fixed array compiled
// into the library instead.
//
// The array lives for as long as the library is loaded, on every GPU that
// loads it (LORA_STATIC_WS_BYTES each). Its device address is looked up once
// per device, with that device current, on the first call made there; that
// first call should come before any stream capture. Every call on a device
// shares the one array: calls whose kernels may overlap on the GPU (different
// streams, or host threads without ordering between them) race and give
// wrong results, so issue them on one stream. The kernels rewrite every part
// of the scratch they read within the call (counters, status word, sort, h),
// so what an earlier call left there is never used and nothing needs
// clearing in advance.
#include <cstdio>
#include <mutex>

#include "lora_internal.cuh"

// Scratch of lora_proj_apply_static_ws (host code must use its device
// address from cudaGetSymbolAddress, never this name).
static __device__ __align__(256) unsigned char lora_static_scratch[LORA_STATIC_WS_BYTES];

namespace {

constexpr int MAX_DEVICES = 64;
std::mutex g_mu;
void *g_addr[MAX_DEVICES] = {};

// Device address of the scratch array on the current device.
lora_status scratch_address(void **out)
{
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return rd::api_fail(LORA_ERR_CUDA, "lora_proj_apply_static_ws: cudaGetDevice failed");
    if (dev < 0 || dev >= MAX_DEVICES)
        return rd::api_fail(LORA_ERR_UNSUPPORTED, "lora_proj_apply_static_ws: device index out of range");
    std::lock_guard<std::mutex> g(g_mu);
    if (g_addr[dev] == nullptr) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, lora_static_scratch);
        if (e != cudaSuccess || p == nullptr) {
            char msg[256];
            snprintf(msg, sizeof msg,
                     "lora_proj_apply_static_ws: cudaGetSymbolAddress of the scratch array failed "
                     "on device %d: %s",
                     dev, cudaGetErrorString(e));
            return rd::api_fail(LORA_ERR_CUDA, msg);
        }
        g_addr[dev] = p;
    }
    *out = g_addr[dev];
    return LORA_OK;
}

} // namespace

extern "C" lora_status lora_proj_apply_static_ws(const void *x, int64_t x_stride, const void *W,
                                                 int M, int K, int N, const int32_t *seq_slot,
                                                 const lora_route *rt, void *y, int64_t y_stride,
                                                 lora_stream_t stream)
{
    const size_t need = lora_proj_workspace_bytes(M, rt);
    if (need > (size_t)LORA_STATIC_WS_BYTES) {
        char msg[512];
        snprintf(msg, sizeof msg,
                 "lora_proj_apply_static_ws: %d rows at max_rank %d with %d slots need %zu bytes of "
                 "scratch, more than the built-in %zu; pass a workspace to lora_proj_apply instead",
                 M, rt->max_rank, rt->max_loras, need, (size_t)LORA_STATIC_WS_BYTES);
        return rd::api_fail(LORA_ERR_UNSUPPORTED, msg);
    }
    void *ws = nullptr;
    if (M > 0) {
        lora_status s = scratch_address(&ws);
        if (s != LORA_OK)
            return s;
    }
    return lora_proj_apply(x, x_stride, W, M, K, N, seq_slot, rt, y, y_stride, ws,
                           (size_t)LORA_STATIC_WS_BYTES, stream);
}
