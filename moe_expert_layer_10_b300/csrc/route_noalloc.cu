// moe_route_noalloc: the router for callers that cannot allocate device memory.
//
// Such callers (code running where device allocation is forbidden, processes whose device
// memory belongs to another allocator, fixed-footprint deployments) cannot create a context,
// because a context allocates its pool, arena and scratch. This entry point needs only the
// caller's inputs and outputs: the logits between the two router kernels go to a static
// device array of this file, sized MOE_NOALLOC_MAX_LOGITS floats.
#include <cstdio>
#include <mutex>

#include "../../include/moe.h"
#include "kernels.cuh"

namespace moe {
int set_error(int code, const char* msg);
}

namespace {

// The logits scratch. Every GPU that loads the library holds this array until exit.
static __device__ __align__(256) float g_noalloc_logits[MOE_NOALLOC_MAX_LOGITS];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
float* g_logits_addr[kMaxDevices] = {};  // device address of the array, per device

int err(int code, const char* fmt, long long a = 0, long long b = 0) {
    char buf[256];
    std::snprintf(buf, sizeof(buf), fmt, a, b);
    return moe::set_error(code, buf);
}

}  // namespace

extern "C" int moe_route_noalloc(const void* x, int T, int H, int E, int k, const float* Wr, const float* b,
                                 int32_t* idx, float* w, void* stream) {
    moe::set_error(MOE_OK, "");
    if (T < 0) return err(MOE_E_INVAL, "T=%lld is negative", T);
    if (H < 256 || H % 256) return err(MOE_E_INVAL, "hidden=%lld is not a positive multiple of 256", H);
    if (E < 1 || E > 1024) return err(MOE_E_INVAL, "num_experts=%lld outside [1, 1024]", E);
    if (k < 1 || k > 32 || k > E) return err(MOE_E_INVAL, "top_k=%lld outside [1, min(num_experts, 32)]", k);
    if (static_cast<long long>(T) * E > MOE_NOALLOC_MAX_LOGITS)
        return err(MOE_E_INVAL, "T * num_experts = %lld exceeds the static scratch of %lld logits",
                   static_cast<long long>(T) * E, MOE_NOALLOC_MAX_LOGITS);
    if (T == 0) return MOE_OK;
    if (!x || !Wr || !idx || !w) return err(MOE_E_INVAL, "null device pointer");
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return moe::set_error(MOE_E_CUDA, cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices) return err(MOE_E_INVAL, "device %lld beyond the %lld supported", dev, kMaxDevices);
    float* z = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        if (!g_logits_addr[dev]) {
            void* p = nullptr;
            e = cudaGetSymbolAddress(&p, g_noalloc_logits);
            if (e != cudaSuccess) return moe::set_error(MOE_E_CUDA, cudaGetErrorString(e));
            g_logits_addr[dev] = static_cast<float*>(p);
        }
        z = g_logits_addr[dev];
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    e = moe::launch_router_logits(static_cast<const uint16_t*>(x), Wr, b, T, H, E, z, st);
    if (e == cudaSuccess) e = moe::launch_router_topk(z, T, E, k, nullptr, idx, w, nullptr, st);
    if (e != cudaSuccess) return moe::set_error(MOE_E_CUDA, cudaGetErrorString(e));
    return MOE_OK;
}
