// Decode expert FFN on the tensor cores: every weight byte streams from HBM once, the few
// tokens of each expert ride along as the narrow side of the product.
//
// Source: "FreeToken rtx 4090" (freetoken.wiki/hardware), "How the MoE Memory Hierarchy
// Works" -- an expert is a complete cached (layer, expert) entry executed through one
// logical mapping; here the mapping is slot_of[layer][expert] -> arena slot. The SwiGLU
// expert form y = W_down (silu(W_gate x) * (W_up x)) is this library's specification.
//
// In decode an expert sees a handful of tokens, so the work is a skinny product whose cost
// is reading the expert's weights. Doing the products on the SM's fp32 pipes makes a kernel
// issue-bound once an expert has more than a few tokens; here the weight rows are the M side
// of tcgen05.mma (M = 128) and the expert's tokens the N side (N = 16, 32, 48 or 64), so the
// tensor cores take the arithmetic and the SMs only move bytes:
//   gate/up: A tile = gate rows i0..i0+63 and the up rows of the same i (two 64-row TMA
//            boxes), B tile = the chunk's x_perm rows; accumulator lanes 0-63 hold gate,
//            lanes 64-127 up. The epilogue pairs them through shared memory and writes
//            h = bf16(silu(g) * u).
//   down:    A tile = W_down rows n0..n0+127, B tile = the chunk's h_perm rows; the epilogue
//            writes pair_out = w_p * y in fp32.
// Work units (work entry, token chunk of <= 64, row tile, K split) are dealt round-robin to
// one persistent CTA per SM. Entries whose cache fill was enqueued by the same forward come
// last in the list and carry the slot and fill generation to wait for: the producer polls the
// slot's fill flag (bumped by the copy stream after the copy) before streaming that expert, so
// resident experts compute while the fills cross the link and each filled expert starts as
// soon as its own bytes have landed -- one launch per wave, no host round trip. A launch with too few tiles to fill the SMs evenly splits K
// S ways (S <= 4): each split writes its fp32 partial tile to a workspace, and the split that
// finishes last (a per-tile arrival counter) adds the S partials in split order -- a fixed
// order, so results do not depend on timing -- and runs the epilogue.
// Roles (6 warps): warp 0 TMA producer, warp 1 MMA issuer (and TMEM owner), warps 2-5
// epilogue (warp w reads TMEM lanes 32*(w%4)..). Two accumulator buffers of 64 columns
// let the epilogue of one unit overlap the MMAs of the next.
// Every mbarrier wait is bounded (2 s); the epilogue's wait is taken by one thread and its
// outcome shared through a named barrier, so the four warps always leave together. On a
// timeout the kernel raises the device status, drains its copies and MMAs (bounded) and frees
// its TMEM before returning.
#include <algorithm>

#include "decode_common.cuh"

namespace moe {
namespace {

using dec::BK;
using dec::kNMax;
using dec::kXchgFloats;
using dec::Unit;
using dec::locate_unit;
using dec::decode_epilogue;

constexpr int A_BYTES = 128 * BK * 2;        // 16 KB of weights per stage
constexpr int B_BYTES = kNMax * BK * 2;      // up to 8 KB of tokens per stage
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int kMaxStages = 9;
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 128;          // 2 accumulators x 64 columns

struct __align__(8) Shared {
    uint64_t full[kMaxStages], empty[kMaxStages], acc_full[2], acc_empty[2];
    uint32_t tmem_base;
    int ok[2];
    int last[2];
};

// gate/up keeps a 16 KB exchange buffer for the up values, so it has one stage fewer
template <bool GATEUP>
struct Layout {
    static constexpr int STAGES = GATEUP ? 8 : 9;
    static constexpr int XCHG_BYTES = GATEUP ? kXchgFloats * 4 : 0;
    static constexpr int SMEM = STAGES * STAGE_BYTES + XCHG_BYTES + static_cast<int>(sizeof(Shared)) + 1024;
    static_assert(STAGES <= kMaxStages, "stage count");
    static_assert(SMEM <= 227 * 1024, "shared memory per CTA");
};



template <bool GATEUP>
__global__ void __launch_bounds__(kThreads, 1)
    decode_mma_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                      const GemvWork* __restrict__ work, int n_work, int n_units, int S,
                      const int32_t* __restrict__ slot_row, const uint32_t* __restrict__ fill_flag, int H, int I,
                      uint16_t* __restrict__ h_out,
                      const float* __restrict__ w_perm, float* __restrict__ pair_out, float* __restrict__ ws,
                      int* __restrict__ cnt, int* status, uint64_t fill_wait_ns, const int* __restrict__ dyn) {
    pdl_gate();  // may start while the previous kernel of the stream finishes
    using Lay = Layout<GATEUP>;
    if (dyn) {  // work size written on the device (device-resident policy)
        n_work = dyn[0];
        n_units = dyn[1];
        S = dyn[2];
    }
    // the MMA and epilogue roles may legitimately wait as long as the producer waits for a fill
    const uint64_t consumer_wait_ns = fill_wait_ns + kWaitDeadlineNs;
    constexpr int kStages = Lay::STAGES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* tiles = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float* xchg = reinterpret_cast<float*>(tiles + kStages * STAGE_BYTES);
    Shared& sh = *reinterpret_cast<Shared*>(tiles + kStages * STAGE_BYTES + Lay::XCHG_BYTES);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int K = GATEUP ? H : I;
    const int KB = K / BK;
    const int R = GATEUP ? I / 64 : H / 128;  // row tiles per token chunk

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

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            prefetch_tmap(&tm_a);
            prefetch_tmap(&tm_b);
            const uint64_t pol_w = policy_evict_first();
            int stage = 0;
            uint32_t phase = 0, used = 0, last_phase = 0;
            bool ok = true;
            int ready_a = -1;  // last work entry whose fill was seen (a CTA visits entries in order)
            for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
                const Unit un = locate_unit(work, n_work, u, R, S);
                const GemvWork wk = work[un.a];
                if (wk.wait_slot >= 0 && un.a != ready_a) {
                    // an entry filled by this wave: stream it once its copy has landed
                    if (!wait_fill_flag(fill_flag + wk.wait_slot, wk.gen, fill_wait_ns)) {
                        raise_status(status, kDevFillTimeout);
                        break;
                    }
                    ready_a = un.a;
                }
                int slot = slot_row[wk.expert];
                if (slot < 0) {
                    raise_status(status, kDevBadSlot);
                    slot = 0;  // keep every copy inside the arena; results are discarded
                }
                const int tok0 = wk.tok_off + un.chunk * kNMax;
                const int nt = min(kNMax, wk.n_tok - un.chunk * kNMax);
                const int nb = (nt + 15) >> 4;  // 16-row token boxes
                const int kb0 = un.split * KB / S, kb1 = (un.split + 1) * KB / S;
                const uint32_t tx = A_BYTES + nb * 16 * BK * 2;
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!mbar_wait(&sh.empty[stage], phase ^ 1u)) {
                        raise_status(status, kDevWaitTimeout);
                        ok = false;
                        break;
                    }
                    uint8_t* sa = tiles + stage * STAGE_BYTES;
                    mbar_arrive_expect_tx(&sh.full[stage], tx);
                    if (GATEUP) {
                        const int row = slot * 3 * I + un.tile * 64;
                        tma_load_2d_hint(sa, &tm_a, &sh.full[stage], kb * BK, row, pol_w);
                        tma_load_2d_hint(sa + A_BYTES / 2, &tm_a, &sh.full[stage], kb * BK, row + I, pol_w);
                    } else {
                        const int row = slot * 3 * H + 2 * H + un.tile * 128;
                        tma_load_2d_hint(sa, &tm_a, &sh.full[stage], kb * BK, row, pol_w);
                    }
                    for (int b = 0; b < nb; ++b)
                        tma_load_2d(sa + A_BYTES + b * 16 * BK * 2, &tm_b, &sh.full[stage], kb * BK, tok0 + 16 * b);
                    used |= 1u << stage;
                    last_phase = (last_phase & ~(1u << stage)) | (phase << stage);
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // every issued copy must land before the CTA exits
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
            for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
                const Unit un = locate_unit(work, n_work, u, R, S);
                const GemvWork wk = work[un.a];
                const int nt = min(kNMax, wk.n_tok - un.chunk * kNMax);
                const uint32_t idesc = idesc_bf16_f32(128, ((nt + 15) >> 4) * 16);
                const int kb0 = un.split * KB / S, kb1 = (un.split + 1) * KB / S;
                if (!mbar_wait(&sh.acc_empty[acc], acc_phase ^ 1u, consumer_wait_ns)) {
                    raise_status(status, kDevWaitTimeout);
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem + static_cast<uint32_t>(acc * kNMax);
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!mbar_wait(&sh.full[stage], phase, consumer_wait_ns)) {
                        raise_status(status, kDevWaitTimeout);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint8_t* sa = tiles + stage * STAGE_BYTES;
                    const uint64_t da = sw128_kmajor_desc(smem_u32(sa));
                    const uint64_t db = sw128_kmajor_desc(smem_u32(sa + A_BYTES));
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k)  // +32 bytes per K=16 step inside the swizzle row
                        umma_bf16(d, da + 2 * k, db + 2 * k, idesc, (kb != kb0 || k != 0) ? 1u : 0u);
                    umma_commit(&sh.empty[stage]);
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
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
        decode_epilogue<GATEUP>(sh.acc_full, sh.acc_empty, sh.ok, sh.last, tmem, xchg, work, n_work, n_units, S, R, H,
                                I, h_out, w_perm, pair_out, ws, cnt, status, consumer_wait_ns, 64);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <bool GATEUP>
cudaError_t launch(const CUtensorMap& ta, const CUtensorMap& tb, const GemvWork* work, int n_work, int n_units,
                   int S, const int32_t* slot_row, const uint32_t* fill_flag, int H, int I, uint16_t* h_out,
                   const float* w_perm, float* pair_out, float* ws, int* cnt, int* status, uint64_t fill_wait_ns,
                   int num_sms, cudaStream_t st, const int* dyn = nullptr) {
    if (!dyn) {
        if (n_units <= 0 || n_work <= 0) return cudaSuccess;
        if (S < 1 || S > kDecodeMaxSplit) return cudaErrorInvalidValue;
        if (S > 1 && n_units > kDecodeSplitUnits) return cudaErrorInvalidValue;
    }
    auto kern = decode_mma_kernel<GATEUP>;
    constexpr int smem = Layout<GATEUP>::SMEM;
    static std::atomic<uint64_t> attr{0};
    const cudaError_t e = ensure_smem_limit(kern, smem, attr);
    if (e != cudaSuccess) return e;
    const int grid = dyn ? num_sms : std::min(n_units, num_sms);
    return launch_pdl(kern, dim3(grid), dim3(kThreads), smem, st, ta, tb, work, n_work, n_units, S, slot_row, fill_flag,
                      H, I, h_out, w_perm, pair_out, ws, cnt, status, fill_wait_ns, dyn);
}

}  // namespace

int decode_row_tiles(bool gateup, int H, int I) { return gateup ? I / 64 : H / 128; }

int decode_token_chunks(int n_tok) { return (n_tok + kNMax - 1) / kNMax; }

int decode_choose_split(int n_tiles, bool gateup, int H, int I, int num_sms) {
    const int KB = (gateup ? H : I) / BK;
    auto eff = [&](int s) {
        const long long n = static_cast<long long>(n_tiles) * s;
        const long long waves = (n + num_sms - 1) / num_sms;
        return static_cast<double>(n) / static_cast<double>(waves * num_sms);
    };
    if (n_tiles <= 0 || eff(1) >= 0.85) return 1;
    int best = 1;
    double best_eff = eff(1);
    for (int s = 2; s <= kDecodeMaxSplit; ++s) {
        if (static_cast<long long>(n_tiles) * s > kDecodeSplitUnits || KB / s < 4) break;
        const double e = eff(s) - 0.02 * (s - 1);  // each split adds a partial write and read
        if (e > best_eff + 1e-9) {
            best = s;
            best_eff = e;
        }
    }
    return best;
}

cudaError_t launch_decode_gateup(const DecodeMaps& m, const GemvWork* work, int n_work, int n_units, int S,
                                 const int32_t* slot_row, const uint32_t* fill_flag, int H, int I, uint16_t* h_perm,
                                 float* ws, int* cnt, int* status, uint64_t fill_wait_ns, int num_sms,
                                 cudaStream_t st) {
    return launch<true>(m.a_gu, m.b_x, work, n_work, n_units, S, slot_row, fill_flag, H, I, h_perm, nullptr, nullptr,
                        ws, cnt, status, fill_wait_ns, num_sms, st);
}

cudaError_t launch_decode_gateup_dyn(const DecodeMaps& m, const GemvWork* work, const int* dyn,
                                     const int32_t* slot_row, int H, int I, uint16_t* h_perm, float* ws, int* cnt,
                                     int* status, int num_sms, cudaStream_t st) {
    return launch<true>(m.a_gu, m.b_x, work, 0, 0, 1, slot_row, nullptr, H, I, h_perm, nullptr, nullptr, ws, cnt, status,
                        0, num_sms, st, dyn);
}

cudaError_t launch_decode_down_dyn(const DecodeMaps& m, const GemvWork* work, const int* dyn,
                                   const int32_t* slot_row, int H, int I, const float* w_perm, float* pair_out,
                                   float* ws, int* cnt, int* status, int num_sms, cudaStream_t st) {
    return launch<false>(m.a_d, m.b_h, work, 0, 0, 1, slot_row, nullptr, H, I, nullptr, w_perm, pair_out, ws, cnt,
                         status, 0, num_sms, st, dyn);
}

cudaError_t launch_decode_down(const DecodeMaps& m, const GemvWork* work, int n_work, int n_units, int S,
                               const int32_t* slot_row, const uint32_t* fill_flag, int H, int I, const float* w_perm,
                               float* pair_out, float* ws, int* cnt, int* status, uint64_t fill_wait_ns, int num_sms,
                               cudaStream_t st) {
    return launch<false>(m.a_d, m.b_h, work, n_work, n_units, S, slot_row, fill_flag, H, I, nullptr, w_perm, pair_out,
                         ws, cnt, status, fill_wait_ns, num_sms, st);
}

}  // namespace moe
