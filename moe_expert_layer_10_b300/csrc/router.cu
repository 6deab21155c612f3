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

// Large batches (prefill): a register-tiled evaluation of the same order. A CTA of 16 warps
// owns a tile of 32 tokens x 32 experts and walks H in chunks of 256 columns (a ring of 3
// chunks in shared memory). The 32 lanes of the order are split over warps, not over the lanes
// of a warp: warp w evaluates the partials s_w and s_{w+16} of every (token, expert) of the
// tile, each accumulated with fused multiply-adds over exactly the columns 256m + 8l + r
// (m, then r = 0..7) that define s_l. Within the warp, lane (g, f) = (lane / 8, lane % 8) owns
// tokens g + 4i (i < 8) and experts f + 8j (j < 4), so the lanes of a warp read the same
// columns and shared memory serves them by broadcast. The 16 sums s_w + s_{w+16} -- the first
// xor-fold step -- go through shared memory and the remaining steps (distances 8, 4, 2, 1) are
// taken in the same pairing, then the bias.
//
// x is staged as fp32 pairs: token pair P = (P % 4 + 8 (P / 4), that token + 4) keeps, per
// column, the two tokens' values side by side, so one 16-byte read gives the f32x2 operands
// of two columns and two fused multiply-adds share one instruction (fma.rn.f32x2, two
// independent round-to-nearest results). W_r is copied as is with cp.async.
constexpr int kTT = 32, kTE = 32;
constexpr int kTiledThreads = 512;
constexpr int kXRow = 256 * 8 + 16;                 // bytes per token pair row (+16: bank spread)
constexpr int kWRow = 256 * 4 + 16;                 // bytes per expert row
constexpr int kXBytes = 16 * kXRow;
constexpr int kWBytes = kTE * kWRow;
constexpr int kTiledStage = kXBytes + kWBytes;
constexpr int kTiledStages = 3;
constexpr int kTiledSmem = kTiledStages * kTiledStage;
constexpr int kFoldRow = 40;                        // floats per token row of the fold buffer
static_assert(16 * kTT * kFoldRow * 4 <= kTiledSmem, "fold buffer must fit in the stage ring");

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Two independent fp32 fused multiply-adds in one instruction (round to nearest each), on
// register pairs: d = (a.lo * b.lo + c.lo, a.hi * b.hi + c.hi) -- the same two fmaf results.
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t pack2(float lo, float hi) {
    uint64_t d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(lo), "f"(hi));
    return d;
}
__device__ __forceinline__ float lo_of(uint64_t v) { return __uint_as_float(static_cast<uint32_t>(v)); }
__device__ __forceinline__ float hi_of(uint64_t v) { return __uint_as_float(static_cast<uint32_t>(v >> 32)); }

// The x granule (8 columns) of the two tokens of pair row P that thread tid stages.
struct XGranule {
    uint4 a, b;
};
__device__ __forceinline__ XGranule load_x_granule(const uint16_t* x, int t0, int T, int H, int m) {
    const int P = threadIdx.x & 15, g = threadIdx.x >> 4;
    const int ta = (P & 3) + 8 * (P >> 2);
    const size_t col = static_cast<size_t>(256) * m + 8 * g;
    XGranule r;
    r.a = __ldg(reinterpret_cast<const uint4*>(x + static_cast<size_t>(min(t0 + ta, T - 1)) * H + col));
    r.b = __ldg(reinterpret_cast<const uint4*>(x + static_cast<size_t>(min(t0 + ta + 4, T - 1)) * H + col));
    return r;
}
__device__ __forceinline__ void store_x_granule(uint8_t* xs, const XGranule& r) {
    const int P = threadIdx.x & 15, g = threadIdx.x >> 4;
    float4* dst = reinterpret_cast<float4*>(xs + P * kXRow + g * 64);
    const uint32_t a[4] = {r.a.x, r.a.y, r.a.z, r.a.w}, b[4] = {r.b.x, r.b.y, r.b.z, r.b.w};
#pragma unroll
    for (int q = 0; q < 4; ++q)  // columns 2q, 2q+1: (a, b) of each, column-major
        dst[q] = make_float4(bf16lo(a[q]), bf16lo(b[q]), bf16hi(a[q]), bf16hi(b[q]));
}
__device__ __forceinline__ void stage_w(uint8_t* ws, const float* Wr, int e0, int E, int H, int m) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int i = threadIdx.x + kTiledThreads * k;
        const int row = i >> 6, c = i & 63;
        const int e = min(e0 + row, E - 1);
        cp_async16(ws + row * kWRow + c * 16, Wr + static_cast<size_t>(e) * H + 256 * m + 4 * c);
    }
}

__global__ void __launch_bounds__(kTiledThreads, 1) router_logits_tiled_kernel(const uint16_t* __restrict__ x,
                                                                     const float* __restrict__ Wr,
                                                                     const float* __restrict__ bias, int T, int H,
                                                                     int E, float* __restrict__ z) {
    pdl_gate();  // may start while the previous kernel of the stream finishes
    extern __shared__ __align__(16) uint8_t rsm[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t0 = blockIdx.y * kTT, e0 = blockIdx.x * kTE;
    const int g = lane >> 3, f = lane & 7;
    // acc[c][j][p]: partial s_{warp + 16c} of expert f + 8j for the token pair (g + 8p, g + 8p + 4)
    uint64_t acc[2][4][4];
#pragma unroll
    for (int c = 0; c < 2; ++c)
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int p = 0; p < 4; ++p) acc[c][j][p] = 0ull;
    const int M = H / 256;
#pragma unroll
    for (int m = 0; m < kTiledStages - 1; ++m) {
        if (m < M) {
            uint8_t* st = rsm + m * kTiledStage;
            store_x_granule(st, load_x_granule(x, t0, T, H, m));
            stage_w(st + kXBytes, Wr, e0, E, H, m);
        }
        cp_async_commit();
    }
    for (int m = 0; m < M; ++m) {
        cp_async_wait<kTiledStages - 2>();  // chunk m's W_r rows have landed (this thread's copies)
        __syncthreads();                    // ... everyone's, and chunk m-1's buffer is free
        const int mn = m + kTiledStages - 1;
        uint8_t* nst = rsm + (mn % kTiledStages) * kTiledStage;
        XGranule nx;
        if (mn < M) {
            nx = load_x_granule(x, t0, T, H, mn);  // in flight while chunk m is evaluated
            stage_w(nst + kXBytes, Wr, e0, E, H, mn);
        }
        cp_async_commit();
        const uint8_t* xs = rsm + (m % kTiledStages) * kTiledStage;
        const uint8_t* ws = xs + kXBytes;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            const int l = warp + 16 * c;  // the lane of the order evaluated: columns 8l .. 8l+7
#pragma unroll
            for (int hq = 0; hq < 2; ++hq) {  // columns 8l + 4hq .. 8l + 4hq + 3
                float4 wq[4];
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    wq[j] = *reinterpret_cast<const float4*>(ws + (f + 8 * j) * kWRow + (8 * l + 4 * hq) * 4);
#pragma unroll
                for (int cp = 0; cp < 2; ++cp) {  // columns 8l + 4hq + 2cp, + 1
                    uint4 xq[4];
#pragma unroll
                    for (int p = 0; p < 4; ++p)
                        xq[p] = *reinterpret_cast<const uint4*>(xs + (g + 4 * p) * kXRow + (8 * l + 4 * hq + 2 * cp) * 8);
#pragma unroll
                    for (int q = 0; q < 2; ++q) {
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const float wf = cp == 0 ? (q == 0 ? wq[j].x : wq[j].y) : (q == 0 ? wq[j].z : wq[j].w);
                            const uint64_t wd = pack2(wf, wf);
#pragma unroll
                            for (int p = 0; p < 4; ++p) {
                                const uint64_t xp = q == 0 ? (static_cast<uint64_t>(xq[p].y) << 32 | xq[p].x)
                                                           : (static_cast<uint64_t>(xq[p].w) << 32 | xq[p].z);
                                acc[c][j][p] = fma2(wd, xp, acc[c][j][p]);
                            }
                        }
                    }
                }
            }
        }
        if (mn < M) store_x_granule(nst, nx);  // chunk m-1's buffer: free since the barrier above
    }
    cp_async_wait<0>();
    __syncthreads();  // every thread is done with the ring: reuse it for the fold
    float* fold = reinterpret_cast<float*>(rsm);  // [16][kTT][kFoldRow]
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            const int e = f + 8 * j, ta = g + 8 * p;
            fold[(warp * kTT + ta) * kFoldRow + e] = __fadd_rn(lo_of(acc[0][j][p]), lo_of(acc[1][j][p]));
            fold[(warp * kTT + ta + 4) * kFoldRow + e] = __fadd_rn(hi_of(acc[0][j][p]), hi_of(acc[1][j][p]));
        }
    __syncthreads();
#pragma unroll
    for (int o = threadIdx.x; o < kTT * kTE; o += kTiledThreads) {
        const int t = o / kTE, e = o % kTE;
        float v[16];
#pragma unroll
        for (int l = 0; l < 16; ++l) v[l] = fold[(l * kTT + t) * kFoldRow + e];
#pragma unroll
        for (int d = 8; d >= 1; d >>= 1)
#pragma unroll
            for (int l = 0; l < d; ++l) v[l] = __fadd_rn(v[l], v[l + d]);
        const int tt = t0 + t, ee = e0 + e;
        if (tt < T && ee < E) z[static_cast<size_t>(tt) * E + ee] = __fadd_rn(v[0], bias ? __ldg(bias + ee) : 0.0f);
    }
}

// Small batches (decode): latency-bound, so a CTA first stages its EPB experts' router
// rows and the whole batch of activations in shared memory with asynchronous copies, every
// one in flight at once, then evaluates the same fixed fp32 order from shared memory. Warp w
// computes expert e0 + w % EPB for tokens t = w / EPB + (8 / EPB) * i.
template <int EPB, int TPW>
__global__ void __launch_bounds__(256) router_logits_staged_kernel(const uint16_t* __restrict__ x,
                                                                   const float* __restrict__ Wr,
                                                                   const float* __restrict__ bias, int T, int H,
                                                                   int E, float* __restrict__ z) {
    pdl_gate();  // may start while the previous kernel of the stream finishes
    extern __shared__ __align__(16) uint8_t smem[];
    float* wr = reinterpret_cast<float*>(smem);                   // [EPB][H]
    uint16_t* xs = reinterpret_cast<uint16_t*>(wr + EPB * H);     // [T][H]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e0 = blockIdx.x * EPB;
    const int ne = min(EPB, E - e0);
    {
        // asynchronous copies: every 16-byte piece of the CTA's share is in flight at once
        const uint8_t* src = reinterpret_cast<const uint8_t*>(Wr + static_cast<size_t>(e0) * H);
        const int n4 = ne * H / 4;
        for (int i = threadIdx.x; i < n4; i += 256) cp_async16(smem + 16 * i, src + 16 * i);
        const uint8_t* xsrc = reinterpret_cast<const uint8_t*>(x);
        uint8_t* xdst = reinterpret_cast<uint8_t*>(xs);
        const int nx = T * H / 8;
        for (int i = threadIdx.x; i < nx; i += 256) cp_async16(xdst + 16 * i, xsrc + 16 * i);
        cp_async_commit();
        cp_async_wait<0>();
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
    static std::atomic<uint64_t> attr{0};
    const cudaError_t e = ensure_smem_limit(kern, 227 * 1024, attr);
    if (e != cudaSuccess) return e;
    const size_t smem = static_cast<size_t>(EPB) * H * 4 + static_cast<size_t>(T) * H * 2;
    return launch_pdl(kern, dim3((E + EPB - 1) / EPB), dim3(256), smem, st, x, Wr, b, T, H, E, z);
}

__device__ __forceinline__ bool ranks_before(float za, int ea, float zb, int eb) {
    return za > zb || (za == zb && ea < eb);
}

// One warp per token. Lane l holds the logits of experts l, l+32, ..., l + 32(NS-1)
// (NS >= ceil(E / 32), E <= 1024).
template <int NS>
__global__ void __launch_bounds__(256) router_topk_kernel(const float* __restrict__ z, int T, int E, int k,
                                                          const int32_t* __restrict__ forced,
                                                          int32_t* __restrict__ idx, float* __restrict__ w,
                                                          int* status) {
    pdl_gate();  // may start while the previous kernel of the stream finishes
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = blockIdx.x * (blockDim.x >> 5) + warp;
    if (t >= T) return;
    const float* zt = z + static_cast<size_t>(t) * E;
    int my_e = -1;       // lane j < k: the expert it outputs at position j
    float my_z = 0.0f;   // and its logit
    if (forced == nullptr) {
        float v[NS];
        uint32_t taken = 0;
#pragma unroll
        for (int i = 0; i < NS; ++i) v[i] = (lane + 32 * i < E) ? zt[lane + 32 * i] : -FLT_MAX;
        for (int j = 0; j < k; ++j) {
            float bv = -INFINITY;
            int be = INT_MAX;
#pragma unroll
            for (int i = 0; i < NS; ++i) {
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
    static std::atomic<uint64_t> attr{0};
    const cudaError_t e = ensure_smem_limit(router_logits_tiled_kernel, kTiledSmem, attr);
    if (e != cudaSuccess) return e;
    return launch_pdl(router_logits_tiled_kernel, dim3((E + kTE - 1) / kTE, (T + kTT - 1) / kTT), dim3(kTiledThreads),
                      kTiledSmem, st, x, Wr, b, T, H, E, z);
}

cudaError_t launch_router_topk(const float* z, int T, int E, int k, const int32_t* forced, int32_t* idx, float* w,
                               int* status, cudaStream_t st) {
    if (T <= 0) return cudaSuccess;
    const int blocks = (T + 7) / 8;
    const int ns = (E + 31) / 32;
    auto go = [&](auto kern) {
        return launch_pdl(kern, dim3(blocks), dim3(256), 0, st, z, T, E, k, forced, idx, w, status);
    };
    if (ns <= 1) return go(router_topk_kernel<1>);
    if (ns <= 2) return go(router_topk_kernel<2>);
    if (ns <= 4) return go(router_topk_kernel<4>);
    if (ns <= 8) return go(router_topk_kernel<8>);
    if (ns <= 16) return go(router_topk_kernel<16>);
    return go(router_topk_kernel<32>);
}

}  // namespace moe
