// Token permutation: group the T*k (token, j) pairs by routed expert so that every
// expert's tokens are contiguous, stable in (token, j). Deterministic: positions come
// from counts and prefix sums, never from the order of atomics.
//
// Outputs: offsets[E+1] (first position of each expert), perm[pos] = pair id t*k+j,
// inv_perm[pair] = pos, w_perm[pos] = gate of that pair, active[] = experts with at
// least one pair in ascending id, n_active, and x_perm[pos] = the row of token perm[pos] / k.
// Up to kSmallPairs pairs (decode batches) one launch does all of it; larger batches run the
// counting sort, then a row-gather kernel.
#include "kernels.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kPermThreads = 1024;
constexpr int kPermWarps = kPermThreads / 32;

// Exclusive prefix sum over the CTA (NW warps, one value per thread); returns the total in *total.
template <int NW = 32>
__device__ int block_exclusive_scan(int v, int* scratch /* >= 33 ints */, int* total) {
    static_assert(NW >= 1 && NW <= 32, "one warp scans the warp totals");
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
        int s = lane < NW ? scratch[lane] : 0;
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

// The routed expert of pair p, checked (an id outside [0, E) raises the status and counts as 0).
__device__ __forceinline__ int checked_expert(const int32_t* idx, int p, int E, int* status) {
    int e = idx[p];
    if (e < 0 || e >= E) {
        raise_status(status, kDevBadIndex);
        e = 0;
    }
    return e;
}

// The lanes of the warp holding the same expert id as this lane (e >= 0), from one ballot
// per bit of the id: a lane is a peer when it agrees on every bit. Lanes with e < 0 hold no
// pair and are never peers.
__device__ __forceinline__ uint32_t warp_peers(int e, int nbits) {
    uint32_t peers = __ballot_sync(0xffffffffu, e >= 0);
    for (int b = 0; b < nbits; ++b) {
        const bool bit = (e >> b) & 1;
        const uint32_t m = __ballot_sync(0xffffffffu, bit);
        peers &= bit ? m : ~m;
    }
    return peers;
}

// One warp per permuted row, 16-byte copies.
__global__ void __launch_bounds__(256) gather_rows_kernel(const uint16_t* __restrict__ x,
                                                          const int32_t* __restrict__ perm, int P, int k, int H,
                                                          uint16_t* __restrict__ x_perm) {
    pdl_gate();  // may start while the previous kernel of the stream finishes
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int pos = blockIdx.x * 8 + warp;
    if (pos >= P) return;
    const int t = perm[pos] / k;
    const uint4* src = reinterpret_cast<const uint4*>(x + static_cast<size_t>(t) * H);
    uint4* dst = reinterpret_cast<uint4*>(x_perm + static_cast<size_t>(pos) * H);
    for (int c = lane; c < H / 8; c += 32) dst[c] = __ldg(src + c);
}

// Larger batches (more than 1024 pairs): a counting sort over many CTAs, so that the
// scattered writes of perm and w_perm leave from many SMs. CTA g owns the pairs
// [1024 g, 1024 g + 1024), one per thread; warp w of it the 32 pairs 1024 g + 32 w + lane.
// The global order (expert, g, w, lane) is the order (expert, pair id).
//  permute_count_kernel: CTA g counts its pairs per expert into cells[g][e]; the last CTA to
//    finish (arrival counter) scans the cells in (expert, g) order into starts[g][e] and writes
//    offsets, the active list and n_active, then resets the counter for the next launch.
//  permute_place_kernel: CTA g turns starts[g][e] into per-warp starts (exclusive prefix over
//    its warps' counts) and places each pair at its warp's start plus its rank among the equal
//    lanes.
constexpr int kChunkPairs = kPermThreads;

__global__ void __launch_bounds__(kPermThreads) permute_count_kernel(const int32_t* __restrict__ idx, int P, int E,
                                                                     int32_t* __restrict__ cells,
                                                                     int32_t* __restrict__ starts,
                                                                     int32_t* __restrict__ offsets,
                                                                     int32_t* __restrict__ active,
                                                                     int32_t* __restrict__ n_active,
                                                                     unsigned* done, int* status) {
    pdl_gate();  // may start while the previous kernel of the stream finishes
    extern __shared__ int smem[];
    int* cnt = smem;             // [E] this CTA's pairs per expert, later first position per expert
    int* scan = cnt + E + 1;     // [33]
    __shared__ bool s_last;
    const int tid = threadIdx.x, G = gridDim.x, g = blockIdx.x;
    for (int e = tid; e < E; e += kPermThreads) cnt[e] = 0;
    __syncthreads();
    const int p = g * kChunkPairs + tid;
    if (p < P) atomicAdd(&cnt[checked_expert(idx, p, E, status)], 1);
    __syncthreads();
    for (int e = tid; e < E; e += kPermThreads) cells[static_cast<size_t>(g) * E + e] = cnt[e];
    __threadfence();
    __syncthreads();
    if (tid == 0) s_last = atomicAdd(done, 1u) == static_cast<unsigned>(G - 1);
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    // the last CTA: exclusive scan of the cells in (expert, CTA) order
    const int n_cells = E * G;
    const int per_thread = (n_cells + kPermThreads - 1) / kPermThreads;
    const int i0 = min(n_cells, tid * per_thread), i1 = min(n_cells, i0 + per_thread);
    int run = 0;
    for (int i = i0; i < i1; ++i) run += __ldcg(cells + static_cast<size_t>(i % G) * E + i / G);
    int total;
    int pos = block_exclusive_scan(run, scan, &total);
    for (int i = i0; i < i1; ++i) {
        const size_t cell = static_cast<size_t>(i % G) * E + i / G;
        const int v = __ldcg(cells + cell);
        starts[cell] = pos;
        if (i % G == 0) cnt[i / G] = pos;
        pos += v;
    }
    if (tid == 0) cnt[E] = total;
    __syncthreads();
    const int c = tid < E ? cnt[tid + 1] - cnt[tid] : 0;
    if (tid < E) offsets[tid] = cnt[tid];
    if (tid == 0) offsets[E] = cnt[E];
    int nact;
    const int apos = block_exclusive_scan(c > 0 ? 1 : 0, scan, &nact);
    if (tid < E && c > 0) active[apos] = tid;
    if (tid == 0) {
        *n_active = nact;
        *done = 0u;  // ready for the next launch (kernels on the stream run one after the other)
    }
}

__global__ void __launch_bounds__(kPermThreads) permute_place_kernel(const int32_t* __restrict__ idx,
                                                                     const float* __restrict__ w, int P, int E,
                                                                     const int32_t* __restrict__ starts,
                                                                     int32_t* __restrict__ perm,
                                                                     int32_t* __restrict__ inv_perm,
                                                                     float* __restrict__ w_perm) {
    pdl_gate();  // may start while the previous kernel of the stream finishes
    extern __shared__ int smem[];
    const int Es = E + 1;
    int* cnt = smem;  // [kPermWarps][Es]: the warp's pairs per expert, then the warp's first position
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, g = blockIdx.x;
    for (int i = tid; i < kPermWarps * Es; i += kPermThreads) cnt[i] = 0;
    __syncthreads();
    const int p = g * kChunkPairs + tid;
    const bool valid = p < P;
    int e = valid ? idx[p] : -1;
    if (valid && (e < 0 || e >= E)) e = 0;  // raised by the counting kernel
    const float wv = valid ? w[p] : 0.0f;
    const int nbits = E > 1 ? 32 - __clz(E - 1) : 0;
    const uint32_t peers = warp_peers(e, nbits);
    if (e >= 0 && lane == __ffs(peers) - 1) cnt[warp * Es + e] = __popc(peers);
    __syncthreads();
    for (int x = tid; x < E; x += kPermThreads) {
        int run = starts[static_cast<size_t>(g) * E + x];
        for (int q = 0; q < kPermWarps; ++q) {
            const int v = cnt[q * Es + x];
            cnt[q * Es + x] = run;
            run += v;
        }
    }
    __syncthreads();
    if (e >= 0) {
        const int pos = cnt[warp * Es + e] + __popc(peers & ((1u << lane) - 1u));
        perm[pos] = p;
        inv_perm[p] = pos;
        w_perm[pos] = wv;
    }
}


// Up to kSmallPairs pairs (decode batches): the permutation and the row gather in one launch
// over ceil(P / 8) CTAs. Every CTA stages the P expert ids in shared memory; warp w of CTA g
// owns pair p = 8 g + w, whose position is its rank in (expert, pair id) order,
//   pos(p) = #{q : e_q < e_p} + #{q < p : e_q = e_p},
// counted directly over the staged ids: the stable counting sort's result by definition. The
// warp writes perm, inv_perm and w_perm and copies token p / k's row into x_perm[pos]. CTA 0
// also counts the pairs per expert into offsets, the active list and n_active.
constexpr int kSmallPairs = 1024;
constexpr int kSmallThreads = 256;
constexpr int kSmallWarps = kSmallThreads / 32;
constexpr int kSmallExpertsPerThread = 1024 / kSmallThreads;  // E <= 1024

__global__ void __launch_bounds__(kSmallThreads) permute_gather_small_kernel(
    const int32_t* __restrict__ idx, const float* __restrict__ w, const uint16_t* __restrict__ x, int P, int k,
    int E, int H, int32_t* __restrict__ offsets, int32_t* __restrict__ perm, int32_t* __restrict__ inv_perm,
    float* __restrict__ w_perm, int32_t* __restrict__ active, int32_t* __restrict__ n_active,
    uint16_t* __restrict__ x_perm, int* status) {
    pdl_gate();  // may start while the previous kernel of the stream finishes
    extern __shared__ int smem[];
    int* es = smem;          // [P] routed expert of each pair (an id outside [0, E) counts as 0)
    int* cnt = es + P;       // CTA 0: [E] pairs per expert
    int* scan = cnt + E;     // CTA 0: [33]
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const bool lead = blockIdx.x == 0;
    if (lead)
        for (int e = tid; e < E; e += kSmallThreads) cnt[e] = 0;
    for (int q = tid; q < P; q += kSmallThreads) {
        int e = idx[q];
        if (e < 0 || e >= E) {
            if (lead) raise_status(status, kDevBadIndex);
            e = 0;
        }
        es[q] = e;
    }
    __syncthreads();
    const int p = blockIdx.x * kSmallWarps + warp;
    if (p < P) {
        const int ep = es[p];
        int r = 0;
        for (int q = lane; q < P; q += 32) {
            const int eq = es[q];
            r += (eq < ep || (eq == ep && q < p)) ? 1 : 0;
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) r += __shfl_xor_sync(0xffffffffu, r, o);
        if (lane == 0) {
            perm[r] = p;
            inv_perm[p] = r;
            w_perm[r] = w[p];
        }
        const uint4* src = reinterpret_cast<const uint4*>(x + static_cast<size_t>(p / k) * H);
        uint4* dst = reinterpret_cast<uint4*>(x_perm + static_cast<size_t>(r) * H);
        constexpr int kU = 8;  // 16-byte pieces per lane in flight before the first store
        const int n = H / 8;
        for (int c0 = lane; c0 < n; c0 += 32 * kU) {
            uint4 v[kU];
#pragma unroll
            for (int u = 0; u < kU; ++u)
                if (c0 + 32 * u < n) v[u] = __ldg(src + c0 + 32 * u);
#pragma unroll
            for (int u = 0; u < kU; ++u)
                if (c0 + 32 * u < n) dst[c0 + 32 * u] = v[u];
        }
    }
    if (!lead) return;
    for (int q = tid; q < P; q += kSmallThreads) atomicAdd(&cnt[es[q]], 1);  // counts: order-free
    __syncthreads();
    const int e0 = tid * kSmallExpertsPerThread;
    int c[kSmallExpertsPerThread];
    int run = 0, nz = 0;
#pragma unroll
    for (int i = 0; i < kSmallExpertsPerThread; ++i) {
        c[i] = e0 + i < E ? cnt[e0 + i] : 0;
        run += c[i];
        nz += c[i] > 0 ? 1 : 0;
    }
    int total, nact;
    int pos = block_exclusive_scan<kSmallWarps>(run, scan, &total);
    int apos = block_exclusive_scan<kSmallWarps>(nz, scan, &nact);
#pragma unroll
    for (int i = 0; i < kSmallExpertsPerThread; ++i) {
        if (e0 + i < E) {
            offsets[e0 + i] = pos;
            pos += c[i];
            if (c[i] > 0) active[apos++] = e0 + i;
        }
    }
    if (tid == 0) {
        offsets[E] = total;
        *n_active = nact;
    }
}

}  // namespace

int permute_grid(int P) { return P > 0 ? (P + kChunkPairs - 1) / kChunkPairs : 1; }

cudaError_t launch_permute(const int32_t* idx, const float* w, int P, int E, int32_t* offsets, int32_t* perm,
                           int32_t* inv_perm, float* w_perm, int32_t* active, int32_t* n_active, int* status,
                           int32_t* cells, unsigned* done, cudaStream_t st) {
    static std::atomic<uint64_t> attr_place{0};
    const cudaError_t err0 = ensure_smem_limit(permute_place_kernel, sizeof(int) * kPermWarps * 1025, attr_place);
    if (err0 != cudaSuccess) return err0;
    if (P <= 0) return cudaSuccess;
    if (!cells || !done) return cudaErrorInvalidValue;
    const int G = permute_grid(P);
    int32_t* starts = cells + static_cast<size_t>(G) * E;
    cudaError_t err = launch_pdl(permute_count_kernel, dim3(G), dim3(kPermThreads), sizeof(int) * (E + 1 + 36), st, idx,
                                 P, E, cells, starts, offsets, active, n_active, done, status);
    if (err != cudaSuccess) return err;
    return launch_pdl(permute_place_kernel, dim3(G), dim3(kPermThreads), sizeof(int) * kPermWarps * (E + 1), st, idx,
                      w, P, E, static_cast<const int32_t*>(starts), perm, inv_perm, w_perm);
}

bool permute_gathers_rows(int P) { return P <= kSmallPairs; }

cudaError_t launch_permute_gather(const int32_t* idx, const float* w, const uint16_t* x, int P, int k, int E, int H,
                                  int32_t* offsets, int32_t* perm, int32_t* inv_perm, float* w_perm,
                                  int32_t* active, int32_t* n_active, uint16_t* x_perm, int* status,
                                  cudaStream_t st) {
    if (P <= 0 || P > kSmallPairs || E > 1024 || H % 8) return cudaErrorInvalidValue;
    const size_t smem = sizeof(int) * (static_cast<size_t>(P) + E + 33);
    return launch_pdl(permute_gather_small_kernel, dim3((P + kSmallWarps - 1) / kSmallWarps), dim3(kSmallThreads),
                      smem, st, idx, w, x, P, k, E, H, offsets, perm, inv_perm, w_perm, active, n_active, x_perm,
                      status);
}

cudaError_t launch_gather_rows(const uint16_t* x, const int32_t* perm, int P, int k, int H, uint16_t* x_perm,
                               cudaStream_t st) {
    if (P <= 0) return cudaSuccess;
    return launch_pdl(gather_rows_kernel, dim3((P + 7) / 8), dim3(256), 0, st, x, perm, P, k, H, x_perm);
}

}  // namespace moe
