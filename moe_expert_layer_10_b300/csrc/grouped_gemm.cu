// Prefill expert FFN: persistent tcgen05 grouped GEMM through the cache-slot table.
//
// Source: "FreeToken rtx 4090" (freetoken.wiki/hardware), "How the MoE Memory Hierarchy
// Works" -- prefill activates a broad part of the expert pool; each routed expert is a
// complete cached (layer, expert) entry executed through one logical mapping (here the
// device slot table). The SwiGLU form is this library's specification.
//
// In prefill each expert sees many tokens, so its FFN is a dense contraction:
//   GEMM1  [n_e x H] x [H x (I gate | I up)] -> h = silu(gate) * up  (bf16, [n_e x I])
//   GEMM2  [n_e x I] x [I x H] -> w_p * y                          (fp32, [n_e x H])
// Design (one CTA of 6 warps per SM, persistent over a static tile schedule):
//  * tiles are (active expert, n-tile, m-tile of 128 tokens), m innermost, so CTAs that run
//    at the same time read the same weight tile from L2;
//  * warp 0 / one lane: TMA producer -- A tile [128 tokens x 64] and B tile [256 rows x 64]
//    (GEMM1: 128 gate rows + the 128 up rows of the same columns; GEMM2: 256 W_down rows),
//    128-byte swizzled, into a 4-stage ring (48 KB per stage);
//  * warp 1 / one lane: tcgen05.mma.cta_group::1.kind::f16, M=128 N=256 K=16, fp32
//    accumulators in TMEM, two accumulator buffers of 256 columns (512 columns);
//  * warps 2-5: epilogue -- tcgen05.ld of the thread's accumulator row (warp w reads TMEM
//    lanes 32*(w%4)...), SwiGLU or gate-weight scaling, direct 16-byte global stores of
//    the rows that belong to the expert.
// Every mbarrier wait is bounded (2 s); on a timeout the kernel raises the device status,
// drains its copies and MMAs (bounded) and frees its TMEM before returning.
#include <algorithm>

#include "kernels.cuh"
#include "ptx.cuh"
#include "umma.cuh"

namespace moe {
namespace {

constexpr int BM = 128, BN = 256, BK = 64;
constexpr int kStages = 4;
constexpr int A_BYTES = BM * BK * 2;  // 16 KB
constexpr int B_BYTES = BN * BK * 2;  // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 512;
constexpr int kMaxActive = 1024;
constexpr uint32_t kIdesc = idesc_bf16_f32(BM, BN);

struct __align__(8) Shared {
    uint64_t full[kStages], empty[kStages], acc_full[2], acc_empty[2];
    uint32_t tmem_base;
    int ex[kMaxActive], off[kMaxActive], cnt[kMaxActive], mtp[kMaxActive + 1];
};
constexpr int SMEM_BYTES = kStages * STAGE_BYTES + static_cast<int>(sizeof(Shared)) + 1024;

__device__ __forceinline__ void decode_tile(const Shared& sh, int na, int NT, int t, int& a, int& nt, int& mt) {
    int lo = 0, hi = na - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (sh.mtp[mid] * NT <= t) lo = mid;
        else hi = mid - 1;
    }
    a = lo;
    const int local = t - sh.mtp[a] * NT;
    const int mta = sh.mtp[a + 1] - sh.mtp[a];
    nt = local / mta;
    mt = local % mta;
}

template <bool GATEUP>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                const int32_t* __restrict__ offsets, const int32_t* __restrict__ active, int a_begin, int a_end,
                const int32_t* __restrict__ slot_row, int H, int I, uint16_t* __restrict__ h_out,
                const float* __restrict__ w_perm, float* __restrict__ pair_out, int* status) {
    pdl_wait();  // may start while the previous kernel of the stream finishes
    extern __shared__ uint8_t smem_raw[];
    uint8_t* tiles = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Shared& sh = *reinterpret_cast<Shared*>(tiles + kStages * STAGE_BYTES);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int K = GATEUP ? H : I;
    const int kblocks = K / BK;
    const int NT = GATEUP ? I / 128 : H / BN;
    const int na = a_end - a_begin;

    // per-CTA tile table from the device permutation (offsets, active list)
    for (int i = threadIdx.x; i < na; i += kThreads) {
        const int e = active[a_begin + i];
        sh.ex[i] = e;
        sh.off[i] = offsets[e];
        sh.cnt[i] = offsets[e + 1] - offsets[e];
    }
    __syncthreads();
    if (warp == 0) {
        int run = 0;
        for (int c0 = 0; c0 < na; c0 += 32) {
            const int i = c0 + lane;
            const int m = i < na ? (sh.cnt[i] + BM - 1) / BM : 0;
            int incl = m;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int n = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += n;
            }
            if (i < na) sh.mtp[i] = run + incl - m;
            run += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0) sh.mtp[na] = run;
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&sh.full[s], 1);
            mbar_init(&sh.empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&sh.acc_full[b], 1);
            mbar_init(&sh.acc_empty[b], 4);
        }
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(&sh.tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sh.tmem_base;
    const int total = sh.mtp[na] * NT;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            prefetch_tmap(&tm_a);
            prefetch_tmap(&tm_b);
            int stage = 0;
            uint32_t phase = 0, used = 0, last_phase = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                int a, nt, mt;
                decode_tile(sh, na, NT, t, a, nt, mt);
                int slot = slot_row[sh.ex[a]];
                if (slot < 0) {
                    raise_status(status, kDevBadSlot);
                    slot = 0;
                }
                const int row_a = sh.off[a] + mt * BM;
                const int row_b = GATEUP ? slot * 3 * I + nt * 128 : slot * 3 * H + 2 * H + nt * BN;
                const int row_b2 = GATEUP ? row_b + I : row_b + 128;
                for (int kb = 0; kb < kblocks; ++kb) {
                    if (!mbar_wait(&sh.empty[stage], phase ^ 1u)) {
                        raise_status(status, kDevWaitTimeout);
                        ok = false;
                        break;
                    }
                    uint8_t* sa = tiles + stage * STAGE_BYTES;
                    mbar_arrive_expect_tx(&sh.full[stage], STAGE_BYTES);
                    tma_load_2d(sa, &tm_a, &sh.full[stage], kb * BK, row_a);
                    tma_load_2d(sa + A_BYTES, &tm_b, &sh.full[stage], kb * BK, row_b);
                    tma_load_2d(sa + A_BYTES + B_BYTES / 2, &tm_b, &sh.full[stage], kb * BK, row_b2);
                    used |= 1u << stage;
                    last_phase = (last_phase & ~(1u << stage)) | (phase << stage);
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            for (int s = 0; s < kStages; ++s)
                if ((used >> s) & 1u)
                    if (!mbar_wait(&sh.full[s], (last_phase >> s) & 1u)) raise_status(status, kDevWaitTimeout);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            int last_acc = -1;
            uint32_t last_acc_phase = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                if (!mbar_wait(&sh.acc_empty[acc], acc_phase ^ 1u)) {
                    raise_status(status, kDevWaitTimeout);
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem + static_cast<uint32_t>(acc * BN);
                for (int kb = 0; kb < kblocks; ++kb) {
                    if (!mbar_wait(&sh.full[stage], phase)) {
                        raise_status(status, kDevWaitTimeout);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint8_t* sa = tiles + stage * STAGE_BYTES;
                    const uint64_t da = sw128_kmajor_desc(smem_u32(sa));
                    const uint64_t db = sw128_kmajor_desc(smem_u32(sa + A_BYTES));
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k)  // +32 bytes per K=16 step inside the swizzle atom
                        umma_bf16(d, da + 2 * k, db + 2 * k, kIdesc, (kb | k) != 0);
                    umma_commit(&sh.empty[stage]);
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                umma_commit(&sh.acc_full[acc]);
                last_acc = acc;
                last_acc_phase = acc_phase;
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1u;
            }
            // every issued MMA has finished once the last commit has arrived
            if (last_acc >= 0 && !mbar_wait(&sh.acc_full[last_acc], last_acc_phase))
                raise_status(status, kDevWaitTimeout);
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;  // TMEM lanes 32q .. 32q+31
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int t = blockIdx.x; t < total; t += gridDim.x) {
            int a, nt, mt;
            decode_tile(sh, na, NT, t, a, nt, mt);
            if (!mbar_wait(&sh.acc_full[acc], acc_phase)) {
                raise_status(status, kDevWaitTimeout);
                break;
            }
            tc_fence_after();
            const int row = q * 32 + lane;
            const int m = mt * BM + row;
            const bool valid = m < sh.cnt[a];
            const size_t pos = static_cast<size_t>(sh.off[a] + m);
            const uint32_t tbase = tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * BN);
            if (GATEUP) {
#pragma unroll 1
                for (int j = 0; j < 128; j += 32) {
                    uint32_t g[32], u[32];
                    tmem_ld32(tbase + j, g);
                    tmem_ld32(tbase + 128 + j, u);
                    tmem_ld_wait();
                    if (valid) {
                        uint32_t hp[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const float g0 = __uint_as_float(g[2 * i]), g1 = __uint_as_float(g[2 * i + 1]);
                            const float u0 = __uint_as_float(u[2 * i]), u1 = __uint_as_float(u[2 * i + 1]);
                            hp[i] = pack_bf16x2(g0 / (1.0f + expf(-g0)) * u0, g1 / (1.0f + expf(-g1)) * u1);
                        }
                        uint4* dst = reinterpret_cast<uint4*>(h_out + pos * I + nt * 128 + j);
#pragma unroll
                        for (int i = 0; i < 4; ++i) dst[i] = make_uint4(hp[4 * i], hp[4 * i + 1], hp[4 * i + 2], hp[4 * i + 3]);
                    }
                }
            } else {
                const float wg = valid ? w_perm[pos] : 0.0f;
#pragma unroll 1
                for (int j = 0; j < BN; j += 32) {
                    uint32_t v[32];
                    tmem_ld32(tbase + j, v);
                    tmem_ld_wait();
                    if (valid) {
                        float4* dst = reinterpret_cast<float4*>(pair_out + pos * H + nt * BN + j);
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            dst[i] = make_float4(wg * __uint_as_float(v[4 * i]), wg * __uint_as_float(v[4 * i + 1]),
                                                 wg * __uint_as_float(v[4 * i + 2]), wg * __uint_as_float(v[4 * i + 3]));
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sh.acc_empty[acc]);
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1u;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <bool GATEUP>
cudaError_t launch(const CUtensorMap& ta, const CUtensorMap& tb, const int32_t* offsets, const int32_t* active,
                   int a_begin, int a_end, int total_tiles, const int32_t* slot_row, int H, int I, uint16_t* h_out,
                   const float* w_perm, float* pair_out, int* status, int num_sms, cudaStream_t st) {
    if (a_end <= a_begin || total_tiles <= 0) return cudaSuccess;
    if (a_end - a_begin > kMaxActive) return cudaErrorInvalidValue;
    auto kern = gemm_kernel<GATEUP>;
    static std::atomic<uint64_t> attr{0};
    const cudaError_t e = ensure_smem_limit(kern, SMEM_BYTES, attr);
    if (e != cudaSuccess) return e;
    const int grid = std::min(total_tiles, num_sms);
    return launch_pdl(kern, dim3(grid), dim3(kThreads), SMEM_BYTES, st, ta, tb, offsets, active, a_begin, a_end,
                      slot_row, H, I, h_out, w_perm, pair_out, status);
}

}  // namespace

int gemm_tiles(bool gateup, const int* counts, int n, int H, int I) {
    int mt = 0;
    for (int i = 0; i < n; ++i) mt += (counts[i] + BM - 1) / BM;
    return mt * (gateup ? I / 128 : H / BN);
}

cudaError_t launch_gemm_gateup(const GemmMaps& m, const int32_t* offsets, const int32_t* active, int a_begin,
                               int a_end, int total_tiles, const int32_t* slot_row, int H, int I, uint16_t* h_perm,
                               int* status, int num_sms, cudaStream_t st) {
    return launch<true>(m.a_x, m.b_gu, offsets, active, a_begin, a_end, total_tiles, slot_row, H, I, h_perm,
                        nullptr, nullptr, status, num_sms, st);
}

cudaError_t launch_gemm_down(const GemmMaps& m, const int32_t* offsets, const int32_t* active, int a_begin,
                             int a_end, int total_tiles, const int32_t* slot_row, int H, int I, const float* w_perm,
                             float* pair_out, int* status, int num_sms, cudaStream_t st) {
    return launch<false>(m.a_h, m.b_d, offsets, active, a_begin, a_end, total_tiles, slot_row, H, I, nullptr,
                         w_perm, pair_out, status, num_sms, st);
}

}  // namespace moe
