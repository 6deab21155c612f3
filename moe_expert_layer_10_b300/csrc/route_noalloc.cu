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
// Per device: the array's device address and the id of the context it was looked up in. A
// context that is destroyed and created again (cudaDeviceReset, or another context made current
// on the device) gets a new id, and the address is looked up again in the new context.
struct SymbolAddr {
    unsigned long long ctx_id = 0;
    bool valid = false;
    float* addr = nullptr;
};
SymbolAddr g_logits_addr[kMaxDevices];

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

template <typename Fn>
Fn driver_fn(const char* name) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
        return nullptr;
    return reinterpret_cast<Fn>(p);
}

// Id of the calling thread's current context (cuCtxGetId: unique for the life of the process).
cudaError_t current_ctx_id(unsigned long long* id) {
    static CtxGetCurrentFn get_cur = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent");
    static CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId");
    if (!get_cur || !get_id) return cudaErrorNotSupported;
    CUcontext ctx = nullptr;
    if (get_cur(&ctx) != CUDA_SUCCESS || !ctx) return cudaErrorContextIsDestroyed;
    if (get_id(ctx, id) != CUDA_SUCCESS) return cudaErrorContextIsDestroyed;
    return cudaSuccess;
}

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
        unsigned long long ctx_id = 0;
        if (current_ctx_id(&ctx_id) != cudaSuccess) {
            // no context is current on this thread yet: cudaSetDevice creates (or, after a
            // cudaDeviceReset, re-creates) the device's primary context and makes it current
            e = cudaSetDevice(dev);
            if (e != cudaSuccess) return moe::set_error(MOE_E_CUDA, cudaGetErrorString(e));
            if (current_ctx_id(&ctx_id) != cudaSuccess)
                return moe::set_error(MOE_E_CUDA, "no current CUDA context to look the scratch up in");
        }
        std::lock_guard<std::mutex> lock(g_mu);
        SymbolAddr& a = g_logits_addr[dev];
        if (!a.valid || a.ctx_id != ctx_id) {
            void* p = nullptr;
            e = cudaGetSymbolAddress(&p, g_noalloc_logits);
            if (e != cudaSuccess) return moe::set_error(MOE_E_CUDA, cudaGetErrorString(e));
            a.addr = static_cast<float*>(p);
            a.ctx_id = ctx_id;
            a.valid = true;
        }
        z = a.addr;
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    e = moe::launch_router_logits(static_cast<const uint16_t*>(x), Wr, b, T, H, E, z, st);
    if (e == cudaSuccess) e = moe::launch_router_topk(z, T, E, k, nullptr, idx, w, nullptr, st);
    if (e != cudaSuccess) return moe::set_error(MOE_E_CUDA, cudaGetErrorString(e));
    return MOE_OK;
}
