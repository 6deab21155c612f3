// Token permutation: group the T*k (token, j) pairs by routed expert so that every
// expert's tokens are contiguous, stable in (token, j). Deterministic: positions come
// from counts and prefix sums, never from the order of atomics.
//
// Outputs: offsets[E+1] (first position of each expert), perm[pos] = pair id t*k+j,
// inv_perm[pair] = pos, w_perm[pos] = gate of that pair, active[] = experts with at
// least one pair in ascending id, n_active. x_perm rows are gathered by a second kernel.
#include "kernels.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kPermThreads = 1024;
constexpr int kPermWarps = kPermThreads / 32;

// Exclusive prefix sum over the CTA (1024 threads, one value each); returns the total in *total.
__device__ int block_exclusive_scan(int v, int* scratch /* >= 33 ints */, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == 31) scratch[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int s = scratch[lane];
        int si = s;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, si, o);
            if (lane >= o) si += n;
        }
        scratch[lane] = si - s;  // exclusive over warps
        if (lane == 31) scratch[32] = si;
    }
    __syncthreads();
    const int res = scratch[warp] + incl - v;
    *total = scratch[32];
    __syncthreads();
    return res;
}

__global__ void __launch_bounds__(kPermThreads) permute_kernel(const int32_t* __restrict__ idx,
                                                               const float* __restrict__ w, int P, int E,
                                                               int32_t* __restrict__ offsets,
                                                               int32_t* __restrict__ perm,
                                                               int32_t* __restrict__ inv_perm,
                                                               float* __restrict__ w_perm,
                                                               int32_t* __restrict__ active,
                                                               int32_t* __restrict__ n_active, int* status) {
    extern __shared__ int smem[];
    int* base = smem;             // [E] first position of each expert, advanced per chunk
    int* ctot = base + E;         // [E] pairs of each expert in the current chunk
    int* scan = ctot + E;         // [33]
    uint16_t* wc = reinterpret_cast<uint16_t*>(scan + 36);  // [kPermWarps][E]
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    for (int e = tid; e < E; e += kPermThreads) ctot[e] = 0;
    for (int i = tid; i < kPermWarps * E; i += kPermThreads) wc[i] = 0;
    __syncthreads();
    for (int p = tid; p < P; p += kPermThreads) {
        int e = idx[p];
        if (e < 0 || e >= E) {
            raise_status(status, kDevBadIndex);
            e = 0;
        }
        atomicAdd(&ctot[e], 1);  // counts only: order-independent
    }
    __syncthreads();
    // offsets and the active list (E <= 1024 -> one expert per thread)
    {
        const int c = tid < E ? ctot[tid] : 0;
        int tot;
        const int ex = block_exclusive_scan(c, scan, &tot);
        if (tid < E) {
            base[tid] = ex;
            offsets[tid] = ex;
        }
        if (tid == 0) offsets[E] = tot;
        int nact;
        const int apos = block_exclusive_scan(c > 0 ? 1 : 0, scan, &nact);
        if (tid < E && c > 0) active[apos] = tid;
        if (tid == 0) *n_active = nact;
    }
    __syncthreads();
    // stable ranks, 1024 pairs per chunk: rank = earlier warps of the chunk + earlier lanes
    for (int c0 = 0; c0 < P; c0 += kPermThreads) {
        const int p = c0 + tid;
        const bool valid = p < P;
        int e = valid ? idx[p] : -1;
        if (valid && (e < 0 || e >= E)) e = 0;
        const uint32_t peers = __match_any_sync(0xffffffffu, e);
        const int lane_rank = __popc(peers & ((1u << lane) - 1u));
        const bool leader = lane == (__ffs(peers) - 1);
        if (valid && leader) wc[warp * E + e] = static_cast<uint16_t>(__popc(peers));
        __syncthreads();
        for (int x = tid; x < E; x += kPermThreads) {
            int run = 0;
            for (int q = 0; q < kPermWarps; ++q) {
                const int cnt = wc[q * E + x];
                wc[q * E + x] = static_cast<uint16_t>(run);
                run += cnt;
            }
            ctot[x] = run;
        }
        __syncthreads();
        if (valid) {
            const int pos = base[e] + wc[warp * E + e] + lane_rank;
            perm[pos] = p;
            inv_perm[p] = pos;
            w_perm[pos] = w[p];
        }
        __syncthreads();
        for (int x = tid; x < E; x += kPermThreads) {
            base[x] += ctot[x];
            for (int q = 0; q < kPermWarps; ++q) wc[q * E + x] = 0;
        }
        __syncthreads();
    }
}

// One warp per permuted row, 16-byte copies.
__global__ void __launch_bounds__(256) gather_rows_kernel(const uint16_t* __restrict__ x,
                                                          const int32_t* __restrict__ perm, int P, int k, int H,
                                                          uint16_t* __restrict__ x_perm) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int pos = blockIdx.x * 8 + warp;
    if (pos >= P) return;
    const int t = perm[pos] / k;
    const uint4* src = reinterpret_cast<const uint4*>(x + static_cast<size_t>(t) * H);
    uint4* dst = reinterpret_cast<uint4*>(x_perm + static_cast<size_t>(pos) * H);
    for (int c = lane; c < H / 8; c += 32) dst[c] = __ldg(src + c);
}

}  // namespace

cudaError_t launch_permute(const int32_t* idx, const float* w, int P, int E, int32_t* offsets, int32_t* perm,
                           int32_t* inv_perm, float* w_perm, int32_t* active, int32_t* n_active, int* status,
                           cudaStream_t st) {
    const size_t smem = sizeof(int) * (2 * E + 36) + sizeof(uint16_t) * kPermWarps * E;
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t err = cudaFuncSetAttribute(permute_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               sizeof(int) * (2 * 1024 + 36) + sizeof(uint16_t) * kPermWarps * 1024);
        if (err != cudaSuccess) return err;
        attr_set = true;
    }
    permute_kernel<<<1, kPermThreads, smem, st>>>(idx, w, P, E, offsets, perm, inv_perm, w_perm, active, n_active,
                                                  status);
    return cudaGetLastError();
}

cudaError_t launch_gather_rows(const uint16_t* x, const int32_t* perm, int P, int k, int H, uint16_t* x_perm,
                               cudaStream_t st) {
    if (P <= 0) return cudaSuccess;
    gather_rows_kernel<<<(P + 7) / 8, 256, 0, st>>>(x, perm, P, k, H, x_perm);
    return cudaGetLastError();
}

}  // namespace moe
