// Decode expert FFN in one persistent launch per wave: the gate/up units and the down units of
// the wave's experts, bf16 weights, the same tcgen05 products and epilogues as decode_mma.cu.
//
// Source: "FreeToken rtx 4090" (freetoken.wiki/hardware), "How the MoE Memory Hierarchy Works"
// -- decode through the shared LRU cache, each cached (layer, expert) entry executed through one
// logical mapping (the slot table). The SwiGLU expert form is this library's specification.
//
// Why one launch: a small decode wave (batch 1: six experts) is short enough that each kernel's
// ramp (the first weight tiles in flight) and drain (the last tiles' epilogues while the SMs
// idle) are a large part of it, and the down kernel cannot start before the last gate/up tile
// has finished. Here each CTA walks one list of units -- every gate/up unit first, then every
// down unit -- so the down weights start streaming on an SM as soon as that SM is done with its
// gate/up share. A down unit of (expert, token chunk) reads h rows that gate/up units of other
// CTAs write, so it waits for them:
//  * each gate/up unit, once its h tile is written, adds 1 (release, gpu scope) to the chunk's
//    h_ready counter, after a proxy fence that orders its h stores before tensor-memory-access
//    (TMA) reads;
//  * the producer of a down unit first issues the unit's weight loads for as many stages as the
//    ring holds, then polls the counter (acquire) until all I/64 gate/up tiles of the chunk have
//    arrived, fences the async proxy, and only then loads the h tiles;
//  * the producer then adds 1 to the chunk's h_done counter; the last down unit of the chunk
//    resets both counters to zero for the next launch.
// The wait cannot deadlock: every CTA takes its gate/up units before its down units, gate/up
// units wait on nothing but fills, and the grid is at most one CTA per SM. It is bounded all the
// same (the fill deadline plus 2 s), like every wait here, and a timeout raises the device status.
// Split-K partials of the two phases use disjoint parts of the workspace and counter arrays.
// Waves whose chunks all have at most 16 tokens (nearly every decode wave) use 18 KB stages, 12
// in flight. Tried and dropped: prefetching each CTA's down-unit weights into L2 during its
// gate/up units (batch 1: 63.9 us against 55.2 us without).
#include <algorithm>

#include "decode_common.cuh"

namespace moe {
namespace {

using dec::BK;
using dec::EpiState;
using dec::epilogue_unit;
using dec::kNMax;
using dec::kXchgFloats;
using dec::locate_unit;
using dec::TensorScales;
using dec::Unit;

constexpr int A_BYTES = 128 * BK * 2;  // 16 KB of weights per stage
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 128;
constexpr int kMaxStages = 12;

// NB: the most 16-token boxes of a unit (1: every chunk of the wave has at most 16 tokens, as in
// almost every decode wave; 4: up to 64). The token tile and the up-value exchange buffer are
// sized for it, and the stages it leaves room for keep more weight bytes in flight.
template <int NB>
struct Cfg {
    static constexpr int B_BYTES = NB * 16 * BK * 2;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int XCHG_BYTES = NB * 16 * 64 * 4;
    static constexpr int STAGES = NB == 1 ? 12 : 8;
    static constexpr int SMEM = STAGES * STAGE_BYTES + XCHG_BYTES + 1024 + 1024;  // + barriers, alignment
    static_assert(STAGES <= kMaxStages, "stage count");
    static_assert(STAGE_BYTES % 1024 == 0, "stages keep the 1024-byte alignment of the swizzled tiles");
    static_assert(SMEM <= 227 * 1024, "shared memory per CTA");
};

struct __align__(8) Shared {
    uint64_t full[kMaxStages], empty[kMaxStages], acc_full[2], acc_empty[2];
    uint32_t tmem_base;
    int ok[2];
    int last[2];
};
static_assert(sizeof(Shared) <= 1024, "barrier block");

// One phase of the launch: its work list (closed by the unit total) and K split.
struct Phase {
    const GemvWork* work;
    int n_work, n_units, S;
};

__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
    int v;
    asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Wait (bounded) until *p >= target; then order later TMA reads after what the releasing
// threads wrote.
__device__ __forceinline__ bool wait_counter(const int* p, int target, uint64_t deadline_ns) {
    if (ld_acquire_gpu(p) < target) {
        const uint64_t t0 = globaltimer_ns();
        for (;;) {
            __nanosleep(64);
            if (ld_acquire_gpu(p) >= target) break;
            if (globaltimer_ns() - t0 > deadline_ns) return false;
        }
    }
    asm volatile("fence.proxy.async.global;" ::: "memory");
    return true;
}

// The i-th unit of this CTA, or -1 past its last: the joint list's round robin b, b + grid, ...
// (every gate/up unit comes before every down unit), cut to the first `keep` of them, then the
// down units pool[p0 .. p1) that the host moved here from the last round of more loaded CTAs.
// Without a schedule (sched == null), the whole round robin.
__device__ __forceinline__ int cta_unit(int i, int n_total, int keep, const int* pool, int p0, int p1) {
    const int b = blockIdx.x, G = gridDim.x;
    if (i < keep) return b + i * G;
    const int p = p0 + (i - keep);
    return p < p1 ? pool[p] : -1;
}

template <int NB>
__global__ void __launch_bounds__(kThreads, 1)
    decode_fused_kernel(const __grid_constant__ CUtensorMap tm_wgu, const __grid_constant__ CUtensorMap tm_wd,
                        const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_h, Phase gu,
                        Phase dn, const int32_t* __restrict__ slot_row, const uint32_t* __restrict__ fill_flag, int H,
                        int I, uint16_t* __restrict__ h_perm, const float* __restrict__ w_perm,
                        float* __restrict__ pair_out, float* __restrict__ ws, int* __restrict__ cnt,
                        int* __restrict__ h_ready, int* __restrict__ h_done, const int* __restrict__ sched,
                        int* status, uint64_t fill_wait_ns) {
    pdl_gate();
    using C = Cfg<NB>;
    constexpr int kStages = C::STAGES, STAGE_BYTES = C::STAGE_BYTES;
    const uint64_t consumer_wait_ns = fill_wait_ns + kWaitDeadlineNs;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* tiles = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float* xchg = reinterpret_cast<float*>(tiles + kStages * STAGE_BYTES);
    Shared& sh = *reinterpret_cast<Shared*>(tiles + kStages * STAGE_BYTES + C::XCHG_BYTES);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int R_gu = I / 64, R_d = H / 128;
    const int n_total = gu.n_units + dn.n_units;
    // the schedule: keep[G], then pool_off[G + 1], then the moved units
    const int G = static_cast<int>(gridDim.x), b_cta = static_cast<int>(blockIdx.x);
    const int rr_count = b_cta < n_total ? (n_total - b_cta + G - 1) / G : 0;
    const int keep = sched ? sched[b_cta] : rr_count;
    const int* pool = sched ? sched + 2 * G + 1 : nullptr;
    const int p0 = sched ? sched[G + b_cta] : 0, p1 = sched ? sched[G + b_cta + 1] : 0;
    // the down phase's split-K tiles follow the gate/up phase's in the workspace and counters
    float* ws_d = ws + static_cast<size_t>(gu.n_units) * kNMax * 128;
    int* cnt_d = cnt + gu.n_units;

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
            prefetch_tmap(&tm_wgu);
            prefetch_tmap(&tm_wd);
            prefetch_tmap(&tm_x);
            prefetch_tmap(&tm_h);
            const uint64_t pol_w = policy_evict_first();
            int stage = 0;
            uint32_t phase = 0, used = 0, last_phase = 0;
            bool ok = true;
            int ready_key = -1;  // (phase, entry) whose fill this CTA last saw land
            for (int iu = 0; ok; ++iu) {
                const int g = cta_unit(iu, n_total, keep, pool, p0, p1);
                if (g < 0) break;
                const bool is_gu = g < gu.n_units;
                const Phase ph = is_gu ? gu : dn;
                const int u = is_gu ? g : g - gu.n_units;
                const int R = is_gu ? R_gu : R_d;
                const Unit un = locate_unit(ph.work, ph.n_work, u, R, ph.S);
                const GemvWork wk = ph.work[un.a];
                const int key = is_gu ? un.a : (1 << 20) + un.a;
                if (wk.wait_slot >= 0 && key != ready_key) {
                    // an entry filled by this wave: stream its weights once its copy has landed
                    // (a CTA visits each phase's entries in order)
                    if (!wait_fill_flag(fill_flag + wk.wait_slot, wk.gen, fill_wait_ns)) {
                        raise_status(status, kDevFillTimeout);
                        break;
                    }
                    ready_key = key;
                }
                int slot = slot_row[wk.expert];
                if (slot < 0) {
                    raise_status(status, kDevBadSlot);
                    slot = 0;  // keep every copy inside the arena; results are discarded
                }
                const int tok0 = wk.tok_off + un.chunk * kNMax;
                const int nt = min(kNMax, wk.n_tok - un.chunk * kNMax);
                const int nb = (nt + 15) >> 4;  // 16-row token boxes
                const int KB = (is_gu ? H : I) / BK;
                const int kb0 = un.split * KB / ph.S, kb1 = (un.split + 1) * KB / ph.S;
                const uint32_t tx = A_BYTES + nb * 16 * BK * 2;  // nb <= NB (the host checked)
                auto load_a = [&](int st, int kb) {
                    uint8_t* sa = tiles + st * STAGE_BYTES;
                    if (is_gu) {
                        const int row = slot * 3 * I + un.tile * 64;
                        tma_load_2d_hint(sa, &tm_wgu, &sh.full[st], kb * BK, row, pol_w);
                        tma_load_2d_hint(sa + A_BYTES / 2, &tm_wgu, &sh.full[st], kb * BK, row + I, pol_w);
                    } else {
                        tma_load_2d_hint(sa, &tm_wd, &sh.full[st], kb * BK, slot * 3 * H + 2 * H + un.tile * 128,
                                         pol_w);
                    }
                };
                auto load_b = [&](int st, int kb) {
                    uint8_t* sb = tiles + st * STAGE_BYTES + A_BYTES;
                    for (int b = 0; b < nb; ++b)
                        tma_load_2d(sb + b * 16 * BK * 2, is_gu ? &tm_x : &tm_h, &sh.full[st], kb * BK, tok0 + 16 * b);
                };
                auto take_stage = [&](int& st_out) {
                    if (!mbar_wait(&sh.empty[stage], phase ^ 1u)) {
                        raise_status(status, kDevWaitTimeout);
                        return false;
                    }
                    mbar_arrive_expect_tx(&sh.full[stage], tx);
                    used |= 1u << stage;
                    last_phase = (last_phase & ~(1u << stage)) | (phase << stage);
                    st_out = stage;
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                    return true;
                };
                int kb = kb0;
                if (!is_gu) {
                    // weights first for as many stages as the ring holds, then the h rows once
                    // every gate/up tile of this (expert, chunk) has written them
                    const int pre = min(kb1 - kb0, kStages);
                    const int st0 = stage;  // the pre stages are consecutive in the ring
                    for (int i = 0; i < pre && ok; ++i) {
                        int st;
                        ok = take_stage(st);
                        if (ok) load_a(st, kb0 + i);
                    }
                    if (!ok) break;
                    auto pre_stage = [&](int i) { return (st0 + i) % kStages; };
                    const int chunk_id = wk.pad0 + un.chunk;
                    if (!wait_counter(h_ready + chunk_id, R_gu, consumer_wait_ns)) {
                        raise_status(status, kDevWaitTimeout);
                        // the issued stages still expect their token bytes: complete them with
                        // the (unused) rows so that every transaction count is met before exit
                        for (int i = 0; i < pre; ++i) load_b(pre_stage(i), kb0 + i);
                        break;
                    }
                    for (int i = 0; i < pre; ++i) load_b(pre_stage(i), kb0 + i);
                    // this unit no longer reads the counters; the last reader of the chunk resets
                    // them for the next launch
                    const int readers = R_d * dn.S;
                    if (atomicAdd(h_done + chunk_id, 1) == readers - 1) {
                        h_done[chunk_id] = 0;
                        h_ready[chunk_id] = 0;
                    }
                    kb = kb0 + pre;
                }
                for (; kb < kb1; ++kb) {
                    int st;
                    if (!take_stage(st)) {
                        ok = false;
                        break;
                    }
                    load_a(st, kb);
                    load_b(st, kb);
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
            for (int iu = 0; ok; ++iu) {
                const int g = cta_unit(iu, n_total, keep, pool, p0, p1);
                if (g < 0) break;
                const bool is_gu = g < gu.n_units;
                const Phase ph = is_gu ? gu : dn;
                const int u = is_gu ? g : g - gu.n_units;
                const Unit un = locate_unit(ph.work, ph.n_work, u, is_gu ? R_gu : R_d, ph.S);
                const GemvWork wk = ph.work[un.a];
                const int nt = min(kNMax, wk.n_tok - un.chunk * kNMax);
                const uint32_t idesc = idesc_bf16_f32(128, ((nt + 15) >> 4) * 16);
                const int KB = (is_gu ? H : I) / BK;
                const int kb0 = un.split * KB / ph.S, kb1 = (un.split + 1) * KB / ph.S;
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
                    for (int k = 0; k < BK / 16; ++k)
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
            if (last_acc >= 0 && !mbar_wait(&sh.acc_full[last_acc], last_acc_phase))
                raise_status(status, kDevWaitTimeout);
        }
    } else {
        // ------------------------------------------------------------ epilogue (warps 2-5)
        EpiState st;
        for (int iu = 0;; ++iu) {
            const int g = cta_unit(iu, n_total, keep, pool, p0, p1);
            if (g < 0) break;
            const bool ok = g < gu.n_units
                                ? epilogue_unit<true>(st, sh.acc_full, sh.acc_empty, sh.ok, sh.last, tmem, xchg,
                                                      gu.work, gu.n_work, g, gu.S, R_gu, H, I, h_perm, w_perm,
                                                      pair_out, ws, cnt, status, consumer_wait_ns, 64, TensorScales{},
                                                      h_ready)
                                : epilogue_unit<false>(st, sh.acc_full, sh.acc_empty, sh.ok, sh.last, tmem, xchg,
                                                       dn.work, dn.n_work, g - gu.n_units, dn.S, R_d, H, I, h_perm,
                                                       w_perm, pair_out, ws_d, cnt_d, status, consumer_wait_ns, 64,
                                                       TensorScales{}, nullptr);
            if (!ok) break;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

int decode_fused_chunk_slots(int E, int P) { return E + P / kNMax + 1; }

namespace {

template <int NB>
cudaError_t launch_nb(const DecodeMaps& m, Phase gu, Phase dn, const int32_t* slot_row, const uint32_t* fill_flag,
                      int H, int I, uint16_t* h_perm, const float* w_perm, float* pair_out, float* ws, int* cnt,
                      int* h_ready, int* h_done, const int* sched, int* status, uint64_t fill_wait_ns, int grid,
                      cudaStream_t st) {
    auto kern = decode_fused_kernel<NB>;
    constexpr int smem = Cfg<NB>::SMEM;
    static std::atomic<uint64_t> attr{0};
    const cudaError_t e = ensure_smem_limit(kern, smem, attr);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3(grid), dim3(kThreads), smem, st, m.a_gu, m.a_d, m.b_x, m.b_h, gu, dn, slot_row,
                      fill_flag, H, I, h_perm, w_perm, pair_out, ws, cnt, h_ready, h_done, sched, status,
                      fill_wait_ns);
}

}  // namespace

cudaError_t launch_decode_fused(const DecodeMaps& m, const GemvWork* work_gu, int n_work, int units_gu, int S_gu,
                                const GemvWork* work_d, int units_d, int S_d, int max_chunk_tok,
                                const int32_t* slot_row, const uint32_t* fill_flag, int H, int I, uint16_t* h_perm,
                                const float* w_perm, float* pair_out, float* ws, int* cnt, int* h_ready, int* h_done,
                                const int* sched, int* status, uint64_t fill_wait_ns, int num_sms, cudaStream_t st) {
    if (units_gu <= 0 || units_d <= 0 || n_work <= 0) return cudaSuccess;
    if (S_gu < 1 || S_gu > kDecodeMaxSplit || S_d < 1 || S_d > kDecodeMaxSplit) return cudaErrorInvalidValue;
    if ((S_gu > 1 || S_d > 1) && units_gu + units_d > kDecodeSplitUnits) return cudaErrorInvalidValue;
    if (max_chunk_tok < 1 || max_chunk_tok > kNMax) return cudaErrorInvalidValue;
    const int grid = std::min(units_gu + units_d, num_sms);
    const Phase gu{work_gu, n_work, units_gu, S_gu}, dn{work_d, n_work, units_d, S_d};
    if (max_chunk_tok <= 16)
        return launch_nb<1>(m, gu, dn, slot_row, fill_flag, H, I, h_perm, w_perm, pair_out, ws, cnt, h_ready, h_done,
                            sched, status, fill_wait_ns, grid, st);
    return launch_nb<4>(m, gu, dn, slot_row, fill_flag, H, I, h_perm, w_perm, pair_out, ws, cnt, h_ready, h_done,
                        sched, status, fill_wait_ns, grid, st);
}

}  // namespace moe
