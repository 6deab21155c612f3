// Weighted combine back into the residual: out[t] = resid[t] + sum_{j<k} pair_out[pos(t, j)],
// where pair_out rows already carry the gate weight w_{t,j}. The k contributions are summed
// in j order by one thread per (token, 4 columns): no atomics, so the result is
// deterministic. resid may alias out (each element is read before it is written).
#include "kernels.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ pair_out,
                                                      const int32_t* __restrict__ inv_perm, const float* resid,
                                                      float* out, int T, int k, int H) {
    pdl_gate();  // may start while the previous kernel of the stream finishes
    const int H4 = H / 4;
    const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= static_cast<long long>(T) * H4) return;
    const int t = static_cast<int>(i / H4), c = static_cast<int>(i % H4);
    float4 acc = reinterpret_cast<const float4*>(resid + static_cast<size_t>(t) * H)[c];
    for (int j = 0; j < k; ++j) {
        const int pos = inv_perm[t * k + j];
        const float4 v = __ldg(reinterpret_cast<const float4*>(pair_out + static_cast<size_t>(pos) * H) + c);
        acc.x += v.x;
        acc.y += v.y;
        acc.z += v.z;
        acc.w += v.w;
    }
    reinterpret_cast<float4*>(out + static_cast<size_t>(t) * H)[c] = acc;
}

}  // namespace

cudaError_t launch_combine(const float* pair_out, const int32_t* inv_perm, const float* resid, float* out, int T,
                           int k, int H, cudaStream_t st) {
    if (T <= 0) return cudaSuccess;
    const long long n = static_cast<long long>(T) * (H / 4);
    return launch_pdl(combine_kernel, dim3(static_cast<unsigned>((n + 255) / 256)), dim3(256), 0, st, pair_out, inv_perm,
                      resid, out, T, k, H);
}

}  // namespace moe
