// Decode expert FFN with MXFP4 expert weights: the 4-bit entries stream from HBM (and cross
// PCIe on a fill) at a quarter of the bf16 bytes, and are expanded to bf16 on chip.
//
// Source: "FreeToken benchmark" (freetoken.wiki/performance) -- the routed experts are
// evaluated in MXFP4 and NVFP4 as well as BF16 ("Results" tables); "FreeToken rtx 4090"
// (freetoken.wiki/hardware), "How the MoE Memory Hierarchy Works" -- an expert is a complete
// cached (layer, expert) entry executed through the slot table.
//
// An MXFP4 value is an E2M1 code (magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6) times its block's
// power-of-two scale, so it is exact in bf16: the kernel expands the weights to bf16 in shared
// memory and runs the same tcgen05 kind::f16 products as the bf16 kernel (decode_mma.cu),
// with the tokens as the N side; the epilogue is the shared one (decode_common.cuh).
// Entry layout: the blocks are stored in the order this kernel streams them, in stages of
// 4352 bytes (4096 bytes of E2M1 codes of a 128-row tile x 64-column slab, then its 256 scale
// bytes): W_gate/W_up per 64-row tile and slab (gate rows, up rows, gate scales, up scales),
// then W_down per 128-row tile and slab. A unit's weights are one contiguous run of stages.
// Roles (22 warps):
//  * warp 0, one lane: producer -- one 4352-byte bulk copy per stage into an 8-deep raw ring
//    (about 34 KB of weights in flight per SM);
//  * warps 6-21 (512 threads): converters, in groups that take successive MMA stages side by
//    side -- a thread expands 16 codes per group of one row
//    into bf16 inside the 128-byte-swizzled A tile of an MMA stage, with byte-permute
//    lookups (two 4-byte tables per scale for the high and the low byte of the bf16 pattern,
//    read from a 4 KB table of all 256 scales that the CTA builds once), 15 integer operations
//    per 8 weights; converter 0 also loads the stage's token tile (TMA);
//  * warp 1, one lane: MMA issuer, as in the bf16 kernel; warps 2-5: epilogue.
// Waits are bounded; the fill-flag wait and the split-K scheme are those of the bf16 kernel.
#include <algorithm>

#include "decode_common.cuh"

namespace moe {
namespace {

using dec::BK;
using dec::decode_epilogue;
using dec::kNMax;
using dec::kXchgFloats;
using dec::locate_unit;
using dec::Unit;

constexpr int kRawA = 128 * 32;                // E2M1 bytes of a 128-row tile slab
constexpr int kRawScales = 256;                // its E8M0 scales: 128 rows x 2
constexpr int kRawStage = kRawA + kRawScales;  // 4352 bytes (34 x 128)
constexpr int kRawStages = 8;
constexpr int kA16 = 128 * BK * 2;             // bf16 A tile: 16 KB
constexpr int kB16 = kNMax * BK * 2;           // token tile: up to 8 KB
constexpr int kMmaStage = kA16 + kB16;         // 24 KB
constexpr int kMaxMmaStages = 7;
constexpr int kConvWarps = 16;
// The converter warps form kConvGroups groups that expand successive MMA stages side by side
// (group g takes the stages n with n % kConvGroups == g), so several stages are in conversion at
// once; a thread of a group expands 16 * kConvGroups codes of one row.
constexpr int kConvGroups = 4;
constexpr int kGroupWarps = kConvWarps / kConvGroups;
constexpr int kThreadsPerRow = 4 / kConvGroups;
constexpr int kConvBase = 192;                 // first converter thread
constexpr int kThreads = kConvBase + 32 * kConvWarps;
constexpr uint32_t kTmemCols = 128;
constexpr int kScaleLutBytes = 256 * 16;      // scale_tables of every E8M0 scale, built once per CTA

struct __align__(8) Shared {
    uint64_t raw_full[kRawStages], raw_empty[kRawStages];
    uint64_t mma_full[kMaxMmaStages], mma_empty[kMaxMmaStages];
    uint64_t acc_full[2], acc_empty[2];
    uint32_t tmem_base;
    int ok[2], last[2];
};

template <bool GATEUP>
struct Layout {
    static constexpr int MMA_STAGES = kConvGroups == 4 ? 4 : 6;  // a multiple of kConvGroups
    static constexpr int XCHG_BYTES = GATEUP ? kXchgFloats * 4 : 0;
    static constexpr int SMEM = MMA_STAGES * kMmaStage + kRawStages * kRawStage + XCHG_BYTES + kScaleLutBytes +
                                static_cast<int>(sizeof(Shared)) + 1024;
    static_assert(MMA_STAGES <= kMaxMmaStages, "stages");
    // every raw and MMA slot then belongs to one converter group, so a group's waits and its
    // final drain only ever see its own phases
    static_assert(MMA_STAGES % kConvGroups == 0 && kRawStages % kConvGroups == 0, "slots per group");
    static_assert(SMEM <= 227 * 1024, "shared memory per CTA");
};

// bf16 patterns of the 8 E2M1 magnitudes times 2^(s-127): 0, then exponent field
// s + {-1, 0, 0, 1, 1, 2, 2} with the top mantissa bit set for 1.5, 3, 6. Returned as four
// byte tables for prmt: high bytes of codes 0-3 / 4-7, low bytes of codes 0-3 / 4-7.
__device__ __forceinline__ void scale_tables(uint32_t s, uint32_t& h_lo, uint32_t& h_hi, uint32_t& l_lo,
                                             uint32_t& l_hi) {
    const uint32_t b = s << 7;
    const uint32_t p1 = b - 128, p2 = b, p3 = b + 64, p4 = b + 128, p5 = b + 192, p6 = b + 256, p7 = b + 320;
    const uint32_t q01 = prmt(0u, p1, 0x5410);  // [p0 (= 0), p1] as two 16-bit halves
    const uint32_t q23 = prmt(p2, p3, 0x5410);
    const uint32_t q45 = prmt(p4, p5, 0x5410);
    const uint32_t q67 = prmt(p6, p7, 0x5410);
    h_lo = prmt(q01, q23, 0x7531);
    h_hi = prmt(q45, q67, 0x7531);
    l_lo = prmt(q01, q23, 0x6420);
    l_hi = prmt(q45, q67, 0x6420);
}

// 8 E2M1 codes (one word, element k in nibble k) -> 4 words of bf16 pairs (element 2j low).
// The magnitude (low 3 bits of a nibble) selects the pattern's high and low byte from the
// scale's tables; the sign (bit 3 of nibble k, bit 4k+3 of v) goes to bit 7 of the high byte
// before the bytes are interleaved: byte k of prmt(v << 4, v, 0x5140) holds bit 4k+3 of v in
// its bit 7 for k = 0..3, and prmt(v << 4, v, 0x7362) does the same for k = 4..7.
__device__ __forceinline__ void expand8(uint32_t v, uint32_t h_lo, uint32_t h_hi, uint32_t l_lo, uint32_t l_hi,
                                        uint32_t (&w)[4]) {
    const uint32_t mags = v & 0x77777777u, mh = mags >> 16, v4 = v << 4;
    const uint32_t ha = or_and(prmt(h_lo, h_hi, mags), prmt(v4, v, 0x5140), 0x80808080u);
    const uint32_t hb = or_and(prmt(h_lo, h_hi, mh), prmt(v4, v, 0x7362), 0x80808080u);
    const uint32_t la = prmt(l_lo, l_hi, mags), lb = prmt(l_lo, l_hi, mh);
    w[0] = prmt(la, ha, 0x5140);
    w[1] = prmt(la, ha, 0x7362);
    w[2] = prmt(lb, hb, 0x5140);
    w[3] = prmt(lb, hb, 0x7362);
}

template <bool GATEUP>
__global__ void __launch_bounds__(kThreads, 1)
    decode_fp4_kernel(const __grid_constant__ CUtensorMap tm_b, const uint8_t* __restrict__ arena,
                      uint64_t entry_bytes, const GemvWork* __restrict__ work, int n_work, int n_units, int S, const int32_t* __restrict__ slot_row,
                      const uint32_t* __restrict__ fill_flag, int H, int I, uint16_t* __restrict__ h_out,
                      const float* __restrict__ w_perm, float* __restrict__ pair_out, float* __restrict__ ws,
                      int* __restrict__ cnt, int* status, uint64_t fill_wait_ns, const int* __restrict__ dyn) {
    pdl_gate();  // may start while the previous kernel of the stream finishes
    using Lay = Layout<GATEUP>;
    constexpr int kMma = Lay::MMA_STAGES;
    if (dyn) {
        n_work = dyn[0];
        n_units = dyn[1];
        S = dyn[2];
    }
    const uint64_t consumer_wait_ns = fill_wait_ns + kWaitDeadlineNs;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* mma_tiles = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* raw_tiles = mma_tiles + kMma * kMmaStage;
    float* xchg = reinterpret_cast<float*>(raw_tiles + kRawStages * kRawStage);
    uint4* scale_lut = reinterpret_cast<uint4*>(raw_tiles + kRawStages * kRawStage + Lay::XCHG_BYTES);
    Shared& sh = *reinterpret_cast<Shared*>(raw_tiles + kRawStages * kRawStage + Lay::XCHG_BYTES + kScaleLutBytes);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int K = GATEUP ? H : I;
    const int KB = K / BK;
    const int R = GATEUP ? I / 64 : H / 128;
    // stages of the gate/up part of an entry (the down part follows)
    const uint64_t gu_bytes = static_cast<uint64_t>(I / 64) * (H / 64) * kRawStage;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kRawStages; ++s) {
            mbar_init(&sh.raw_full[s], 1);
            mbar_init(&sh.raw_empty[s], kGroupWarps);
        }
        for (int s = 0; s < kMma; ++s) {
            mbar_init(&sh.mma_full[s], kGroupWarps + 1);  // a group's warps + the token-tile arrival
            mbar_init(&sh.mma_empty[s], 1);
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
    for (int sc = threadIdx.x; sc < 256; sc += kThreads) {
        uint4 t;
        scale_tables(static_cast<uint32_t>(sc), t.x, t.y, t.z, t.w);
        scale_lut[sc] = t;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sh.tmem_base;

    if (warp == 0) {
        // ------------------------------------------------------------ producer (weights)
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0, used = 0, last_phase = 0;
            bool ok = true;
            int ready_a = -1;
            for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
                const Unit un = locate_unit(work, n_work, u, R, S);
                const GemvWork wk = work[un.a];
                if (wk.wait_slot >= 0 && un.a != ready_a) {
                    if (!wait_fill_flag(fill_flag + wk.wait_slot, wk.gen, fill_wait_ns)) {
                        raise_status(status, kDevFillTimeout);
                        break;
                    }
                    ready_a = un.a;
                }
                int slot = slot_row[wk.expert];
                if (slot < 0) {
                    raise_status(status, kDevBadSlot);
                    slot = 0;
                }
                // the unit's stages: one contiguous run in the slot's entry
                const uint8_t* src = arena + static_cast<uint64_t>(slot) * entry_bytes +
                                     (GATEUP ? static_cast<uint64_t>(un.tile) * (H / 64) * kRawStage
                                             : gu_bytes + static_cast<uint64_t>(un.tile) * (I / 64) * kRawStage);
                const int kb0 = un.split * KB / S, kb1 = (un.split + 1) * KB / S;
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!mbar_wait(&sh.raw_empty[stage], phase ^ 1u, consumer_wait_ns)) {
                        raise_status(status, kDevWaitTimeout);
                        ok = false;
                        break;
                    }
                    uint8_t* dst = raw_tiles + stage * kRawStage;
                    mbar_arrive_expect_tx(&sh.raw_full[stage], kRawStage);
                    bulk_load(dst, src + static_cast<uint64_t>(kb) * kRawStage, kRawStage, &sh.raw_full[stage]);
                    used |= 1u << stage;
                    last_phase = (last_phase & ~(1u << stage)) | (phase << stage);
                    if (++stage == kRawStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            for (int s = 0; s < kRawStages; ++s)
                if ((used >> s) & 1u)
                    if (!mbar_wait(&sh.raw_full[s], (last_phase >> s) & 1u)) raise_status(status, kDevWaitTimeout);
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
                    if (!mbar_wait(&sh.mma_full[stage], phase, consumer_wait_ns)) {
                        raise_status(status, kDevWaitTimeout);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint8_t* sa = mma_tiles + stage * kMmaStage;
                    const uint64_t da = sw128_kmajor_desc(smem_u32(sa));
                    const uint64_t db = sw128_kmajor_desc(smem_u32(sa + kA16));
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k)
                        umma_bf16(d, da + 2 * k, db + 2 * k, idesc, (kb != kb0 || k != 0) ? 1u : 0u);
                    umma_commit(&sh.mma_empty[stage]);
                    if (++stage == kMma) {
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
    } else if (warp < 6) {
        // ------------------------------------------------------------ epilogue (warps 2-5)
        decode_epilogue<GATEUP>(sh.acc_full, sh.acc_empty, sh.ok, sh.last, tmem, xchg, work, n_work, n_units, S, R, H,
                                I, h_out, w_perm, pair_out, ws, cnt, status, consumer_wait_ns, 64);
    } else {
        // ------------------------------------------------------------ converters (warps 6-21)
        const int c = threadIdx.x - kConvBase;
        const int grp = c / (32 * kGroupWarps), cl = c % (32 * kGroupWarps);
        const int row = cl / kThreadsPerRow, part = cl % kThreadsPerRow;  // codes 16G*part .. +16G-1
        const bool token_loader = cl == 0;
        if (token_loader) prefetch_tmap(&tm_b);
        uint32_t used = 0, last_phase = 0;
        bool ok = true;
        int n = 0;  // stage index over the whole run, as the producer and the MMA issuer count it
        for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
            const Unit un = locate_unit(work, n_work, u, R, S);
            const GemvWork wk = work[un.a];
            const int tok0 = wk.tok_off + un.chunk * kNMax;
            const int nt = min(kNMax, wk.n_tok - un.chunk * kNMax);
            const int nb = (nt + 15) >> 4;
            const int kb0 = un.split * KB / S, kb1 = (un.split + 1) * KB / S;
            for (int kb = kb0; kb < kb1; ++kb, ++n) {
                if (n % kConvGroups != grp) continue;
                const int rs = n % kRawStages, ms = n % kMma;
                const uint32_t rphase = (n / kRawStages) & 1, mphase = (n / kMma) & 1;
                if (!mbar_wait(&sh.raw_full[rs], rphase, consumer_wait_ns) ||
                    !mbar_wait(&sh.mma_empty[ms], mphase ^ 1u, consumer_wait_ns)) {
                    raise_status(status, kDevWaitTimeout);
                    ok = false;
                    break;
                }
                uint8_t* sm = mma_tiles + ms * kMmaStage;
                if (token_loader) {
                    mbar_arrive_expect_tx(&sh.mma_full[ms], nb * 16 * BK * 2);
                    for (int b = 0; b < nb; ++b)
                        tma_load_2d(sm + kA16 + b * 16 * BK * 2, &tm_b, &sh.mma_full[ms], kb * BK, tok0 + 16 * b);
                    used |= 1u << ms;
                    last_phase = (last_phase & ~(1u << ms)) | (mphase << ms);
                }
                const uint8_t* raw = raw_tiles + rs * kRawStage;
                uint32_t words[2 * kConvGroups];
#pragma unroll
                for (int h = 0; h < kConvGroups; ++h) {
                    const uint2 cw = *reinterpret_cast<const uint2*>(raw + row * 32 + part * 8 * kConvGroups + 8 * h);
                    words[2 * h] = cw.x;
                    words[2 * h + 1] = cw.y;
                }
#pragma unroll
                for (int q = 0; q < 2 * kConvGroups; ++q) {
                    const int chunk = part * 2 * kConvGroups + q;  // 16-byte chunk of the 128-byte row = 8 codes
                    const uint4 tab = scale_lut[raw[kRawA + row * 2 + (chunk >> 2)]];  // its 32-block's scale
                    uint32_t w[4];
                    expand8(words[q], tab.x, tab.y, tab.z, tab.w, w);
                    *reinterpret_cast<uint4*>(sm + row * 128 + ((chunk ^ (row & 7)) << 4)) =
                        make_uint4(w[0], w[1], w[2], w[3]);
                }
                fence_proxy_async_shared();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&sh.mma_full[ms]);
                    mbar_arrive(&sh.raw_empty[rs]);
                }
            }
        }
        // the token tiles this thread issued must land before the CTA exits
        if (token_loader)
            for (int s = 0; s < kMma; ++s)
                if ((used >> s) & 1u)
                    if (!mbar_wait(&sh.mma_full[s], (last_phase >> s) & 1u)) raise_status(status, kDevWaitTimeout);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <bool GATEUP>
cudaError_t launch(const CUtensorMap& tb, const uint8_t* arena, uint64_t entry_bytes,
                   const GemvWork* work, int n_work, int n_units, int S, const int32_t* slot_row,
                   const uint32_t* fill_flag, int H, int I, uint16_t* h_out, const float* w_perm, float* pair_out,
                   float* ws, int* cnt, int* status, uint64_t fill_wait_ns, int num_sms, cudaStream_t st,
                   const int* dyn) {
    if (!dyn) {
        if (n_units <= 0 || n_work <= 0) return cudaSuccess;
        if (S < 1 || S > kDecodeMaxSplit) return cudaErrorInvalidValue;
        if (S > 1 && n_units > kDecodeSplitUnits) return cudaErrorInvalidValue;
    }
    auto kern = decode_fp4_kernel<GATEUP>;
    constexpr int smem = Layout<GATEUP>::SMEM;
    static std::atomic<uint64_t> attr{0};
    const cudaError_t e = ensure_smem_limit(kern, smem, attr);
    if (e != cudaSuccess) return e;
    const int grid = dyn ? num_sms : std::min(n_units, num_sms);
    return launch_pdl(kern, dim3(grid), dim3(kThreads), smem, st, tb, arena, entry_bytes, work, n_work, n_units, S,
                      slot_row, fill_flag, H, I, h_out, w_perm, pair_out, ws, cnt, status, fill_wait_ns, dyn);
}

}  // namespace

cudaError_t launch_decode_fp4(bool gateup, const DecodeMaps& m, const uint8_t* arena, uint64_t entry_bytes,
                              const GemvWork* work, int n_work, int n_units, int S, const int* dyn,
                              const int32_t* slot_row, const uint32_t* fill_flag, int H, int I, uint16_t* h_perm,
                              const float* w_perm, float* pair_out, float* ws, int* cnt, int* status,
                              uint64_t fill_wait_ns, int num_sms, cudaStream_t st) {
    if (gateup)
        return launch<true>(m.b_x, arena, entry_bytes, work, n_work, n_units, S, slot_row, fill_flag, H, I,
                            h_perm, nullptr, nullptr, ws, cnt, status, fill_wait_ns, num_sms, st, dyn);
    return launch<false>(m.b_h, arena, entry_bytes, work, n_work, n_units, S, slot_row, fill_flag, H, I,
                         nullptr, w_perm, pair_out, ws, cnt, status, fill_wait_ns, num_sms, st, dyn);
}

}  // namespace moe
