// Router of the routed-MoE layer: logits, top-k and renormalised softmax gates.
//
// Source: "FreeToken rtx 4090" (freetoken.wiki/hardware), "How the MoE Memory Hierarchy
// Works" -- each token activates a small subset of routed experts per layer (six of 256).
// The gate arithmetic (softmax renormalised over the chosen k) is this library's
// specification; the pages do not state it.
//
// Logits are fp32 in one fixed evaluation order so that the chosen experts are
// reproducible bit for bit: lane l of a warp accumulates fmaf(W_r[e,h], x[t,h], s_l) over
// h = 256m + 8l + r (m ascending, then r = 0..7); the 32 partials are folded by xor
// shuffles at distances 16, 8, 4, 2, 1 (fp32 addition is commutative, so both lanes of a
// pair hold the same sum); the bias is added last.
#include <cfloat>
#include <climits>

#include "kernels.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kWarpsPerBlockLargeT = 8;

// One warp per expert e, TB tokens per CTA; warps of a CTA take consecutive experts.
template <int TB>
__global__ void __launch_bounds__(256) router_logits_kernel(const uint16_t* __restrict__ x,
                                                            const float* __restrict__ Wr,
                                                            const float* __restrict__ bias, int T, int H, int E,
                                                            float* __restrict__ z) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e = blockIdx.x * (blockDim.x >> 5) + warp;
    const int t0 = blockIdx.y * TB;
    if (e >= E || t0 >= T) return;
    const int nt = min(TB, T - t0);
    float acc[TB];
#pragma unroll
    for (int i = 0; i < TB; ++i) acc[i] = 0.0f;
    const float* wrow = Wr + static_cast<size_t>(e) * H + 8 * lane;
    const uint16_t* xrow = x + static_cast<size_t>(t0) * H + 8 * lane;
    for (int m = 0; m < H / 256; ++m) {
        const float4 wa = __ldg(reinterpret_cast<const float4*>(wrow + 256 * m));
        const float4 wb = __ldg(reinterpret_cast<const float4*>(wrow + 256 * m + 4));
        const float wv[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
#pragma unroll
        for (int i = 0; i < TB; ++i) {
            if (i < nt) {
                const uint4 xv = __ldg(reinterpret_cast<const uint4*>(xrow + static_cast<size_t>(i) * H + 256 * m));
                const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
                float a = acc[i];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    a = __fmaf_rn(wv[2 * q], bf16lo(xw[q]), a);
                    a = __fmaf_rn(wv[2 * q + 1], bf16hi(xw[q]), a);
                }
                acc[i] = a;
            }
        }
    }
    const float b = bias ? bias[e] : 0.0f;
#pragma unroll
    for (int i = 0; i < TB; ++i) {
        if (i < nt) {
            float v = acc[i];
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
            if (lane == 0) z[static_cast<size_t>(t0 + i) * E + e] = __fadd_rn(v, b);
        }
    }
}

// Small batches (decode): latency-bound, so a CTA first stages its EPB experts' router
// rows and the whole batch of activations in shared memory, every load in flight at once,
// then evaluates the same fixed fp32 order from shared memory. Warp w computes expert
// e0 + w % EPB for tokens t = w / EPB + (8 / EPB) * i.
template <int EPB, int TPW>
__global__ void __launch_bounds__(256) router_logits_staged_kernel(const uint16_t* __restrict__ x,
                                                                   const float* __restrict__ Wr,
                                                                   const float* __restrict__ bias, int T, int H,
                                                                   int E, float* __restrict__ z) {
    extern __shared__ __align__(16) uint8_t smem[];
    float* wr = reinterpret_cast<float*>(smem);                   // [EPB][H]
    uint16_t* xs = reinterpret_cast<uint16_t*>(wr + EPB * H);     // [T][H]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e0 = blockIdx.x * EPB;
    const int ne = min(EPB, E - e0);
    {
        const float4* src = reinterpret_cast<const float4*>(Wr + static_cast<size_t>(e0) * H);
        float4* dst = reinterpret_cast<float4*>(wr);
        const int n4 = ne * H / 4;
        for (int i = threadIdx.x; i < n4; i += 256) dst[i] = __ldg(src + i);
        const uint4* xsrc = reinterpret_cast<const uint4*>(x);
        uint4* xdst = reinterpret_cast<uint4*>(xs);
        const int nx = T * H / 8;
        for (int i = threadIdx.x; i < nx; i += 256) xdst[i] = __ldg(xsrc + i);
    }
    __syncthreads();
    constexpr int WPE = 8 / EPB;  // warps per expert
    const int el = warp % EPB;
    if (el >= ne) return;
    const int e = e0 + el;
    const int tw = warp / EPB;
    float acc[TPW];
#pragma unroll
    for (int i = 0; i < TPW; ++i) acc[i] = 0.0f;
    const float* wrow = wr + el * H + 8 * lane;
    for (int m = 0; m < H / 256; ++m) {
        const float4 wa = *reinterpret_cast<const float4*>(wrow + 256 * m);
        const float4 wb = *reinterpret_cast<const float4*>(wrow + 256 * m + 4);
        const float wv[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
#pragma unroll
        for (int i = 0; i < TPW; ++i) {
            const int t = tw + WPE * i;
            if (t < T) {
                const uint4 xv = *reinterpret_cast<const uint4*>(xs + static_cast<size_t>(t) * H + 256 * m + 8 * lane);
                const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
                float a = acc[i];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    a = __fmaf_rn(wv[2 * q], bf16lo(xw[q]), a);
                    a = __fmaf_rn(wv[2 * q + 1], bf16hi(xw[q]), a);
                }
                acc[i] = a;
            }
        }
    }
    const float b = bias ? bias[e] : 0.0f;
#pragma unroll
    for (int i = 0; i < TPW; ++i) {
        const int t = tw + WPE * i;
        if (t < T) {
            float v = acc[i];
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
            if (lane == 0) z[static_cast<size_t>(t) * E + e] = __fadd_rn(v, b);
        }
    }
}

template <int EPB, int TPW>
cudaError_t launch_staged(const uint16_t* x, const float* Wr, const float* b, int T, int H, int E, float* z,
                          cudaStream_t st) {
    auto kern = router_logits_staged_kernel<EPB, TPW>;
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    const size_t smem = static_cast<size_t>(EPB) * H * 4 + static_cast<size_t>(T) * H * 2;
    kern<<<(E + EPB - 1) / EPB, 256, smem, st>>>(x, Wr, b, T, H, E, z);
    return cudaGetLastError();
}

__device__ __forceinline__ bool ranks_before(float za, int ea, float zb, int eb) {
    return za > zb || (za == zb && ea < eb);
}

// One warp per token. Lane l holds the logits of experts l, l+32, ... (E <= 1024).
__global__ void __launch_bounds__(256) router_topk_kernel(const float* __restrict__ z, int T, int E, int k,
                                                          const int32_t* __restrict__ forced,
                                                          int32_t* __restrict__ idx, float* __restrict__ w,
                                                          int* status) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = blockIdx.x * (blockDim.x >> 5) + warp;
    if (t >= T) return;
    const float* zt = z + static_cast<size_t>(t) * E;
    int my_e = -1;       // lane j < k: the expert it outputs at position j
    float my_z = 0.0f;   // and its logit
    if (forced == nullptr) {
        float v[32];
        uint32_t taken = 0;
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = (lane + 32 * i < E) ? zt[lane + 32 * i] : -FLT_MAX;
        for (int j = 0; j < k; ++j) {
            float bv = -INFINITY;
            int be = INT_MAX;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const int e = lane + 32 * i;
                if (e < E && !((taken >> i) & 1u) && ranks_before(v[i], e, bv, be)) {
                    bv = v[i];
                    be = e;
                }
            }
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
                const int oe = __shfl_xor_sync(0xffffffffu, be, o);
                if (ranks_before(ov, oe, bv, be)) {
                    bv = ov;
                    be = oe;
                }
            }
            if ((be & 31) == lane) taken |= 1u << (be >> 5);
            if (lane == j) {
                my_e = be;
                my_z = bv;
            }
        }
    } else {
        // Validate the forced set, then rank it by (z desc, id asc).
        int fe = lane < k ? forced[static_cast<size_t>(t) * k + lane] : -1;
        const bool in_range = fe >= 0 && fe < E;
        const uint32_t lanes_k = (k >= 32) ? 0xffffffffu : ((1u << k) - 1u);
        const uint32_t peers = __match_any_sync(0xffffffffu, fe);
        const bool bad_here = lane < k && (!in_range || (peers & lanes_k) != (1u << lane));
        if (__any_sync(0xffffffffu, bad_here)) {
            if (lane == 0) raise_status(status, kDevBadForcedSet);
            if (lane < k) {
                idx[static_cast<size_t>(t) * k + lane] = lane;
                w[static_cast<size_t>(t) * k + lane] = 0.0f;
            }
            return;
        }
        const float fz = lane < k ? zt[fe] : 0.0f;
        int rank = 0;
        for (int i = 0; i < k; ++i) {
            const float oz = __shfl_sync(0xffffffffu, fz, i);
            const int oe = __shfl_sync(0xffffffffu, fe, i);
            if (i != lane && ranks_before(oz, oe, fz, fe)) ++rank;
        }
        // lane j takes the expert whose rank is j
        for (int i = 0; i < k; ++i) {
            const int ri = __shfl_sync(0xffffffffu, rank, i);
            const float oz = __shfl_sync(0xffffffffu, fz, i);
            const int oe = __shfl_sync(0xffffffffu, fe, i);
            if (ri == lane) {
                my_e = oe;
                my_z = oz;
            }
        }
    }
    // Gates: w_j = exp(z_j - z_0) / sum_j' exp(z_j' - z_0), the sum taken in j order.
    const float z0 = __shfl_sync(0xffffffffu, my_z, 0);
    const float ex = lane < k ? expf(my_z - z0) : 0.0f;
    float s = 0.0f;
    for (int j = 0; j < k; ++j) s += __shfl_sync(0xffffffffu, ex, j);
    if (lane < k) {
        idx[static_cast<size_t>(t) * k + lane] = my_e;
        w[static_cast<size_t>(t) * k + lane] = ex / s;
    }
}

}  // namespace

cudaError_t launch_router_logits(const uint16_t* x, const float* Wr, const float* b, int T, int H, int E, float* z,
                                 cudaStream_t st) {
    if (T <= 0) return cudaSuccess;
    // staged kernel when the experts' rows and the batch fit in shared memory
    const size_t smem4 = 4ull * H * 4 + static_cast<size_t>(T) * H * 2;
    if (T <= 2 && 2ull * H * 4 + static_cast<size_t>(T) * H * 2 <= 200 * 1024)
        return launch_staged<2, 1>(x, Wr, b, T, H, E, z, st);
    if (T <= 8 && smem4 <= 200 * 1024) return launch_staged<4, 4>(x, Wr, b, T, H, E, z, st);
    if (T <= 16 && smem4 <= 200 * 1024) return launch_staged<4, 8>(x, Wr, b, T, H, E, z, st);
    if (T <= 32 && smem4 <= 200 * 1024) return launch_staged<4, 16>(x, Wr, b, T, H, E, z, st);
    {
        const int wpb = kWarpsPerBlockLargeT;
        router_logits_kernel<16>
            <<<dim3((E + wpb - 1) / wpb, (T + 15) / 16), dim3(32 * wpb), 0, st>>>(x, Wr, b, T, H, E, z);
    }
    return cudaGetLastError();
}

cudaError_t launch_router_topk(const float* z, int T, int E, int k, const int32_t* forced, int32_t* idx, float* w,
                               int* status, cudaStream_t st) {
    if (T <= 0) return cudaSuccess;
    router_topk_kernel<<<(T + 7) / 8, 256, 0, st>>>(z, T, E, k, forced, idx, w, status);
    return cudaGetLastError();
}

}  // namespace moe
