// Decode expert FFN: HBM-streaming GEMV through the cache-slot indirection table.
//
// Source: "FreeToken rtx 4090" (freetoken.wiki/hardware), "How the MoE Memory Hierarchy
// Works" -- an expert is a complete cached (layer, expert) entry executed through one
// logical mapping; here the mapping is slot_of[layer][expert] -> arena slot. The SwiGLU
// expert form y = W_down (silu(W_gate x) * (W_up x)) is this library's specification.
//
// In decode an expert sees few tokens, so the work is bound by streaming its weights from
// HBM once. Design (one persistent CTA per SM):
//  * warp 8, one elected lane: producer. Per stage it TMA-loads a slab of KS columns of
//    ROWS weight rows (gate and up rows of the same intermediate index for GATEUP) plus
//    the matching KS columns of up to NTMAX token rows, into a ring of shared-memory
//    stages guarded by full/empty mbarriers.
//  * warps 0..7: consumers. Lane l multiplies the 16-byte (VE-element) chunk l of each of
//    its RPW rows with the same chunk of every token, accumulating in fp32 registers across
//    slabs; at the end of a row block the lanes are folded with xor shuffles.
//  * work units = (expert, token chunk, row block), contiguous ranges per CTA so the CTA
//    walks one expert's rows in order; every unit streams its weights exactly once.
//  * every mbarrier wait is bounded (2 s of %globaltimer); on a timeout the kernel raises
//    the device status, drains its in-flight copies (bounded) and returns.
#include <algorithm>

#include "kernels.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kConsumerWarps = 8;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kMaxStages = 8;
constexpr int kSmemBudget = 200 * 1024;
constexpr int kTokBox = 8;  // rows of one activation TMA box

template <bool GATEUP, int KS, int RPW, int NTMAX>
struct Cfg {
    static constexpr int VE = KS / 32;                          // elements of a lane's chunk (8 or 4)
    static constexpr int ROWS = kConsumerWarps * RPW;           // weight rows per stage
    static constexpr int W_BYTES = ROWS * KS * 2;
    static constexpr int X_BYTES = NTMAX * KS * 2;
    static constexpr int STAGE_BYTES = W_BYTES + X_BYTES;
    static constexpr int UNIT_ROWS = GATEUP ? ROWS / 2 : ROWS;  // output rows per unit
    static constexpr int STAGES = std::min(kMaxStages, kSmemBudget / STAGE_BYTES);
    static constexpr int SMEM = STAGES * STAGE_BYTES + 2 * STAGES * 8 + 1024;
    static_assert(VE == 8 || VE == 4, "slab width must be 256 or 128");
    static_assert(NTMAX % kTokBox == 0, "token chunk must be whole boxes");
    static_assert(!GATEUP || RPW % 2 == 0, "gate/up rows come in pairs");
};

// One lane's VE-element bf16 chunk (16 or 8 bytes) from shared memory.
template <int VE>
__device__ __forceinline__ void load_chunk(const uint8_t* src, uint32_t (&out)[VE / 2]) {
    if constexpr (VE == 8) {
        const uint4 v = *reinterpret_cast<const uint4*>(src);
        out[0] = v.x;
        out[1] = v.y;
        out[2] = v.z;
        out[3] = v.w;
    } else {
        const uint2 v = *reinterpret_cast<const uint2*>(src);
        out[0] = v.x;
        out[1] = v.y;
    }
}

struct UnitPos {
    int a;      // index into the wave's work list
    int chunk;  // token chunk
    int rb;     // row block
};

// Unit u -> (work entry, token chunk, row block): the last entry whose first unit is <= u.
__device__ __forceinline__ UnitPos locate(const GemvWork* work, int n_work, int u, int rbs) {
    int lo = 0, hi = n_work - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(&work[mid].unit_begin) <= u) lo = mid;
        else hi = mid - 1;
    }
    const int local = u - __ldg(&work[lo].unit_begin);
    return UnitPos{lo, local / rbs, local % rbs};
}

template <bool GATEUP, int KS, int RPW, int NTMAX>
__global__ void __launch_bounds__(kThreads, 1)
    gemv_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_v,
                const GemvWork* __restrict__ work, int n_work, int n_units, const int32_t* __restrict__ slot_row,
                int H, int I, uint16_t* __restrict__ h_out, const float* __restrict__ w_perm,
                float* __restrict__ pair_out, int* status) {
    using C = Cfg<GATEUP, KS, RPW, NTMAX>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE_BYTES);
    uint64_t* empty = full + C::STAGES;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumerWarps);
        }
        fence_mbar_init();
    }
    __syncthreads();

    const int K = GATEUP ? H : I;                 // reduction length
    const int out_rows = GATEUP ? I : H;          // output rows of one expert
    const int slabs = K / KS;
    const int rbs = out_rows / C::UNIT_ROWS;      // row blocks per token chunk
    // Round-robin units over the CTAs: units of one expert land on different SMs, so the
    // compute of experts with many tokens is spread evenly.
    const int G = gridDim.x;
    if (static_cast<int>(blockIdx.x) >= n_units) return;

    if (warp == kConsumerWarps) {
        // ------------------------------------------------------------ producer
        if (lane != 0) return;
        prefetch_tmap(&tm_w);
        prefetch_tmap(&tm_v);
        const uint64_t pol_w = policy_evict_first();
        int stage = 0;
        uint32_t phase = 0;
        uint32_t used = 0, last_phase = 0;  // per-stage bits for the drain
        bool ok = true;
        for (int u = blockIdx.x; u < n_units && ok; u += G) {
            const UnitPos up = locate(work, n_work, u, rbs);
            const GemvWork wk = work[up.a];
            int slot = slot_row[wk.expert];
            if (slot < 0) {
                raise_status(status, kDevBadSlot);
                slot = 0;  // keep every copy inside the arena; results are discarded
            }
            const int tok0 = wk.tok_off + up.chunk * NTMAX;
            const int nt = min(NTMAX, wk.n_tok - up.chunk * NTMAX);
            const int nbox = (nt + kTokBox - 1) / kTokBox;
            const int row0 = up.rb * C::UNIT_ROWS;
            const uint32_t tx = C::W_BYTES + nbox * kTokBox * KS * 2;
            for (int sl = 0; sl < slabs; ++sl) {
                if (!mbar_wait(&empty[stage], phase ^ 1u)) {
                    raise_status(status, kDevWaitTimeout);
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(&full[stage], tx);
                uint8_t* dst = smem + stage * C::STAGE_BYTES;
                if (GATEUP) {
                    const int base = slot * 3 * I;  // gate rows, then I up rows
                    tma_load_2d_hint(dst, &tm_w, &full[stage], sl * KS, base + row0, pol_w);
                    tma_load_2d_hint(dst + C::W_BYTES / 2, &tm_w, &full[stage], sl * KS, base + I + row0, pol_w);
                } else {
                    const int base = slot * 3 * H + 2 * H;  // W_down rows of the entry
                    tma_load_2d_hint(dst, &tm_w, &full[stage], sl * KS, base + row0, pol_w);
                }
                for (int b = 0; b < nbox; ++b)
                    tma_load_2d(dst + C::W_BYTES + b * kTokBox * KS * 2, &tm_v, &full[stage], sl * KS,
                                tok0 + b * kTokBox);
                used |= 1u << stage;
                last_phase = (last_phase & ~(1u << stage)) | (phase << stage);
                if (++stage == C::STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        // Drain: every issued copy must land before the CTA exits (immediate when the
        // consumers have already waited for them).
        for (int s = 0; s < C::STAGES; ++s)
            if ((used >> s) & 1u)
                if (!mbar_wait(&full[s], (last_phase >> s) & 1u)) raise_status(status, kDevWaitTimeout);
        return;
    }

    // ---------------------------------------------------------------- consumers
    int stage = 0;
    uint32_t phase = 0;
    for (int u = blockIdx.x; u < n_units; u += G) {
        const UnitPos up = locate(work, n_work, u, rbs);
        const GemvWork wk = work[up.a];
        const int tok0 = wk.tok_off + up.chunk * NTMAX;
        const int nt = min(NTMAX, wk.n_tok - up.chunk * NTMAX);
        float acc[RPW][NTMAX];
#pragma unroll
        for (int r = 0; r < RPW; ++r)
#pragma unroll
            for (int t = 0; t < NTMAX; ++t) acc[r][t] = 0.0f;

        for (int sl = 0; sl < slabs; ++sl) {
            if (!mbar_wait(&full[stage], phase)) {
                raise_status(status, kDevWaitTimeout);
                return;
            }
            const uint8_t* st = smem + stage * C::STAGE_BYTES;
            uint32_t wv[RPW][C::VE / 2];
#pragma unroll
            for (int r = 0; r < RPW; ++r) {
                // GATEUP: rows [0, ROWS/2) are gate, [ROWS/2, ROWS) up; warp w owns gate rows
                // (RPW/2)w .. +RPW/2 and the up rows of the same intermediate indices.
                const int row = GATEUP ? ((r < RPW / 2) ? (RPW / 2) * warp + r : C::ROWS / 2 + (RPW / 2) * warp + r - RPW / 2)
                                       : RPW * warp + r;
                load_chunk<C::VE>(st + row * KS * 2 + lane * C::VE * 2, wv[r]);
            }
            const uint8_t* xs = st + C::W_BYTES + lane * C::VE * 2;
            // tokens in pairs: rows up to the next even count are loaded in this stage (whole
            // 8-row boxes), and results of the padding token are never stored
#pragma unroll
            for (int tp = 0; tp < NTMAX; tp += 2) {
                if (tp < nt) {
#pragma unroll
                    for (int t = tp; t < tp + 2; ++t) {
                        uint32_t xv[C::VE / 2];
                        load_chunk<C::VE>(xs + t * KS * 2, xv);
                        float xf[C::VE];
#pragma unroll
                        for (int q = 0; q < C::VE / 2; ++q) {
                            xf[2 * q] = bf16lo(xv[q]);
                            xf[2 * q + 1] = bf16hi(xv[q]);
                        }
#pragma unroll
                        for (int r = 0; r < RPW; ++r) {
                            float sacc = acc[r][t];
#pragma unroll
                            for (int q = 0; q < C::VE / 2; ++q) {
                                sacc = __fmaf_rn(bf16lo(wv[r][q]), xf[2 * q], sacc);
                                sacc = __fmaf_rn(bf16hi(wv[r][q]), xf[2 * q + 1], sacc);
                            }
                            acc[r][t] = sacc;
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[stage]);
            if (++stage == C::STAGES) {
                stage = 0;
                phase ^= 1u;
            }
        }

        // fold the lanes, then lane t writes token t
#pragma unroll
        for (int t = 0; t < NTMAX; ++t) {
            if (t < nt) {
#pragma unroll
                for (int r = 0; r < RPW; ++r) acc[r][t] = warp_sum(acc[r][t]);
            }
        }
        const int row0 = up.rb * C::UNIT_ROWS;
#pragma unroll
        for (int t = 0; t < NTMAX; ++t) {
            if (t < nt && lane == t) {
                const int pos = tok0 + t;
                if (GATEUP) {
                    constexpr int P2 = RPW / 2;
                    const int i0 = row0 + P2 * warp;
                    float hv[P2];
#pragma unroll
                    for (int q = 0; q < P2; ++q) {
                        const float g = acc[q][t], uval = acc[P2 + q][t];
                        hv[q] = g / (1.0f + expf(-g)) * uval;
                    }
                    uint16_t* dst = h_out + static_cast<size_t>(pos) * I + i0;
                    if (P2 == 2) {
                        *reinterpret_cast<uint32_t*>(dst) = pack_bf16x2(hv[0], hv[P2 - 1]);
                    } else {
                        __nv_bfloat16 b = __float2bfloat16_rn(hv[0]);
                        *reinterpret_cast<__nv_bfloat16*>(dst) = b;
                    }
                } else {
                    const float g = w_perm[pos];
                    const int n0 = row0 + RPW * warp;
                    float* dst = pair_out + static_cast<size_t>(pos) * H + n0;
#pragma unroll
                    for (int r = 0; r < RPW; ++r) dst[r] = g * acc[r][t];
                }
            }
        }
    }
}

template <bool GATEUP, int KS, int RPW, int NTMAX>
cudaError_t launch_one(const CUtensorMap& tm_w, const CUtensorMap& tm_v, const GemvWork* work, int n_work,
                       int n_units, const int32_t* slot_row, int H, int I, uint16_t* h_out, const float* w_perm,
                       float* pair_out, int* status, int num_sms, cudaStream_t st) {
    using C = Cfg<GATEUP, KS, RPW, NTMAX>;
    auto kern = gemv_kernel<GATEUP, KS, RPW, NTMAX>;
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    const int grid = std::min(n_units, num_sms);
    if (grid <= 0) return cudaSuccess;
    kern<<<grid, kThreads, C::SMEM, st>>>(tm_w, tm_v, work, n_work, n_units, slot_row, H, I, h_out, w_perm,
                                         pair_out, status);
    return cudaGetLastError();
}

}  // namespace

int gemv_nt_bucket(int max_tokens_per_expert) {
    if (max_tokens_per_expert <= 8) return 8;
    if (max_tokens_per_expert <= 16) return 16;
    return 32;
}

static int rpw_of(int nt) { return nt <= 16 ? 4 : 2; }

int gemv_units_per_chunk(bool gateup, int nt_bucket, int H, int I) {
    const int rows = kConsumerWarps * rpw_of(nt_bucket);
    return gateup ? I / (rows / 2) : H / rows;
}

cudaError_t launch_gemv_gateup(const GemvMaps& m, int nt, const GemvWork* work, int n_work, int n_units,
                               const int32_t* slot_row, int H, int I, uint16_t* h_perm, int* status, int num_sms,
                               cudaStream_t st) {
    if (nt == 8)
        return launch_one<true, 256, 4, 8>(m.w_gu[0], m.xperm, work, n_work, n_units, slot_row, H, I, h_perm,
                                           nullptr, nullptr, status, num_sms, st);
    if (nt == 16)
        return launch_one<true, 256, 4, 16>(m.w_gu[0], m.xperm, work, n_work, n_units, slot_row, H, I, h_perm,
                                            nullptr, nullptr, status, num_sms, st);
    return launch_one<true, 256, 2, 32>(m.w_gu[1], m.xperm, work, n_work, n_units, slot_row, H, I, h_perm, nullptr,
                                        nullptr, status, num_sms, st);
}

cudaError_t launch_gemv_down(const GemvMaps& m, int nt, const GemvWork* work, int n_work, int n_units,
                             const int32_t* slot_row, int H, int I, const float* w_perm, float* pair_out,
                             int* status, int num_sms, cudaStream_t st) {
    if (m.ks_down == 256) {
        if (nt == 8)
            return launch_one<false, 256, 4, 8>(m.w_d[0], m.hperm, work, n_work, n_units, slot_row, H, I, nullptr,
                                                w_perm, pair_out, status, num_sms, st);
        if (nt == 16)
            return launch_one<false, 256, 4, 16>(m.w_d[0], m.hperm, work, n_work, n_units, slot_row, H, I, nullptr,
                                                 w_perm, pair_out, status, num_sms, st);
        return launch_one<false, 256, 2, 32>(m.w_d[1], m.hperm, work, n_work, n_units, slot_row, H, I, nullptr,
                                             w_perm, pair_out, status, num_sms, st);
    }
    if (nt == 8)
        return launch_one<false, 128, 4, 8>(m.w_d[0], m.hperm, work, n_work, n_units, slot_row, H, I, nullptr,
                                            w_perm, pair_out, status, num_sms, st);
    if (nt == 16)
        return launch_one<false, 128, 4, 16>(m.w_d[0], m.hperm, work, n_work, n_units, slot_row, H, I, nullptr,
                                             w_perm, pair_out, status, num_sms, st);
    return launch_one<false, 128, 2, 32>(m.w_d[1], m.hperm, work, n_work, n_units, slot_row, H, I, nullptr, w_perm,
                                         pair_out, status, num_sms, st);
}

}  // namespace moe
