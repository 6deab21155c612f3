// Decode expert FFN with 4-bit expert weights (MXFP4 or NVFP4 entries): the entries stream from
// HBM (and cross PCIe on a fill) at about a quarter of the bf16 bytes, and are expanded to bf16
// on chip, straight into tensor memory.
//
// Source: "FreeToken benchmark" (freetoken.wiki/performance) -- the routed experts are
// evaluated in MXFP4 and NVFP4 as well as BF16 ("Results" tables: the MXFP4 deployment of the
// 284B model, the NVFP4 laptop build); "FreeToken rtx 4090" (freetoken.wiki/hardware), "How
// the MoE Memory Hierarchy Works" -- an expert is a complete cached (layer, expert) entry
// executed through the slot table.
//
// A 4-bit weight is an E2M1 code (magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6) times its block's
// scale: a power of two (MXFP4, E8M0, blocks of 32) or an E4M3 value (NVFP4, blocks of 16,
// times one fp32 tensor scale per matrix). The code times the block scale has at most six
// significant bits, so it is exact in bf16; the kernel expands the weights to those bf16
// values and runs the tcgen05 kind::f16 products of the bf16 kernel (decode_mma.cu), tokens as
// the N side. NVFP4's tensor scale multiplies the fp32 accumulator in the epilogue (shared with
// the bf16 kernel, decode_common.cuh).
//
// Entry layout: the blocks are stored in the order this kernel streams them, in stages of
// 4096 bytes of E2M1 codes of a 128-row tile x 64-column slab (row r at bytes 32r .. 32r+31),
// then its scales (2 bytes per row for MXFP4: 4352-byte stages; 4 per row for NVFP4: 4608):
// W_gate/W_up per 64-row tile and slab (gate rows, then up rows), then W_down per 128-row tile
// and slab; an NVFP4 entry ends with the three fp32 tensor scales and 4 zero bytes. A unit's
// weights are one contiguous run of stages.
//
// Where the bytes go, per stage and SM: the raw stage lands in shared memory by one bulk copy;
// each converter thread reads its row's 32 code bytes (two 16-byte reads) and its scale bytes,
// looks up
// one 16-byte table per block scale, expands 64 codes with byte permutes (15 integer
// operations per 8 codes) and writes the 64 bf16 values into its row's TMEM lane with two
// tcgen05.st (the first overlaps the second half's expansion); the MMA then takes A from tensor
// memory (tcgen05.mma with an A address in TMEM) and only the token tile from shared memory. Keeping the expanded tile out of shared memory
// leaves the shared-memory pipe to the raw stages and the token tiles.
//
// Roles (22 warps):
//  * warp 0, one lane: producer -- one bulk copy per raw stage into a 12-deep ring;
//  * warp 1, one lane: MMA issuer and TMEM owner (512 columns: two 64-column accumulators,
//    then 8 A stages of 32 columns);
//  * warps 2-5: epilogue;
//  * warps 6-21: converters, 4 groups of 4 warps; group g takes the stages n with n % 4 == g,
//    so four stages are in conversion at once. The 4 warps of a group cover the 4 TMEM lane
//    quadrants (warp w writes lanes 32 * (w % 4) ..); each thread owns one A row. The group's
//    first thread also loads the stage's token tile (TMA).
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
using dec::TensorScales;
using dec::Unit;

template <int FMT>
struct Fp4Fmt {
    static constexpr int kScalesPerRow = FMT == kFp4Mx ? 2 : 4;   // per 64-column slab
    static constexpr int kRawStage = 4096 + 128 * kScalesPerRow;  // 4352 or 4608 bytes
    static_assert(kRawStage % 16 == 0, "bulk copies move multiples of 16 bytes");
};

constexpr int kConvGroups = 4;                 // converter groups of 4 warps (one per TMEM lane quadrant)
constexpr int kRawStages = 12;
constexpr int kMma = 2 * kConvGroups;          // MMA stages: A in TMEM, token tile in smem
constexpr int kB16 = kNMax * BK * 2;           // token tile: up to 8 KB
constexpr int kGroupWarps = 4;
constexpr int kConvWarps = kGroupWarps * kConvGroups;
constexpr int kConvBase = 192;                 // first converter thread
constexpr int kThreads = kConvBase + 32 * kConvWarps;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemA = 2 * kNMax;         // first A column: the accumulators take 0 .. 127
constexpr uint32_t kACols = BK / 2;            // 64 bf16 of K per row = 32 columns
constexpr int kLutBytes = 256 * 16;            // byte tables of every scale byte, built once per CTA
constexpr int kWorkSmem = 256;                 // work entries kept in shared memory (a wave of <= 255 experts)
constexpr int kWorkBytes = kWorkSmem * static_cast<int>(sizeof(GemvWork));

static_assert(kGroupWarps == 4, "a converter group covers the four TMEM lane quadrants");
static_assert(kTmemA + kMma * kACols <= kTmemCols, "TMEM columns");
// every raw and MMA slot belongs to one converter group, so a group's waits and its final
// drain only ever see its own phases
static_assert(kMma % kConvGroups == 0 && kRawStages % kConvGroups == 0, "slots per group");

struct __align__(8) Shared {
    uint64_t raw_full[kRawStages], raw_empty[kRawStages];
    uint64_t mma_full[kMma], mma_empty[kMma];
    uint64_t acc_full[2], acc_empty[2];
    uint32_t tmem_base;
    int ok[2], last[2];
};

template <int FMT, bool GATEUP>
struct Layout {
    static constexpr int RAW = Fp4Fmt<FMT>::kRawStage;
    static constexpr int XCHG_BYTES = GATEUP ? kXchgFloats * 4 : 0;
    static constexpr int SMEM = kMma * kB16 + kRawStages * RAW + XCHG_BYTES + kLutBytes + kWorkBytes +
                                static_cast<int>(sizeof(Shared)) + 1024;
    static_assert(SMEM <= 227 * 1024, "shared memory per CTA");
};

// Value of a block-scale byte: E8M0 2^(s-127) for MXFP4; E4M3 for NVFP4 (exponent field f with
// bias 7, mantissa m: m * 2^-9 when f = 0, else (8 + m) * 2^(f-10); the quantizer stores no sign
// and no NaN). Exact in fp32.
template <int FMT>
__device__ __forceinline__ float fp4_scale_value(uint32_t s) {
    if (FMT == kFp4Mx) return s == 0 ? __uint_as_float(0x00400000u) : __uint_as_float(s << 23);
    const uint32_t f = (s >> 3) & 15u, m = s & 7u;
    return f == 0 ? static_cast<float>(m) * __uint_as_float(118u << 23)
                  : static_cast<float>(8u + m) * __uint_as_float((f + 117u) << 23);
}

// The bf16 patterns of the 8 E2M1 magnitudes times the scale (every product exact), as four
// byte tables for prmt: high bytes of codes 0-3 / 4-7, low bytes of codes 0-3 / 4-7.
template <int FMT>
__device__ __forceinline__ uint4 scale_tables(uint32_t s) {
    const float sc = fp4_scale_value<FMT>(s);
    const float mag[8] = {0.0f, 0.5f, 1.0f, 1.5f, 2.0f, 3.0f, 4.0f, 6.0f};
    uint32_t hi[2] = {0, 0}, lo[2] = {0, 0};
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        const uint32_t p = __float_as_uint(mag[c] * sc) >> 16;
        hi[c >> 2] |= ((p >> 8) & 0xffu) << (8 * (c & 3));
        lo[c >> 2] |= (p & 0xffu) << (8 * (c & 3));
    }
    return make_uint4(hi[0], hi[1], lo[0], lo[1]);
}

// 8 E2M1 codes (one word, element k in nibble k) -> 4 words of bf16 pairs (element 2j low).
// The magnitude (low 3 bits of a nibble) selects the pattern's high and low byte from the
// scale's tables; the sign (bit 3 of nibble k, bit 4k+3 of v) goes to bit 7 of the high byte
// before the bytes are interleaved: byte k of prmt(v << 4, v, 0x5140) holds bit 4k+3 of v in
// its bit 7 for k = 0..3, and prmt(v << 4, v, 0x7362) does the same for k = 4..7.
__device__ __forceinline__ void expand8(uint32_t v, const uint4& t, uint32_t* w) {
    const uint32_t mags = v & 0x77777777u, mh = mags >> 16, v4 = v << 4;
    const uint32_t ha = or_and(prmt(t.x, t.y, mags), prmt(v4, v, 0x5140), 0x80808080u);
    const uint32_t hb = or_and(prmt(t.x, t.y, mh), prmt(v4, v, 0x7362), 0x80808080u);
    const uint32_t la = prmt(t.z, t.w, mags), lb = prmt(t.z, t.w, mh);
    w[0] = prmt(la, ha, 0x5140);
    w[1] = prmt(la, ha, 0x7362);
    w[2] = prmt(lb, hb, 0x5140);
    w[3] = prmt(lb, hb, 0x7362);
}

// locate_unit over a work list in shared or global memory (generic loads).
__device__ __forceinline__ Unit locate_unit_any(const GemvWork* work, int n_work, int u, int R, int S) {
    int lo = 0, hi = n_work - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (work[mid].unit_begin <= u) lo = mid;
        else hi = mid - 1;
    }
    const int local = u - work[lo].unit_begin;
    const int rest = local / S;
    return Unit{lo, rest / R, rest % R, local % S};
}

// Every lane waits; the warp goes on only if all lanes saw the phase complete (a warp-uniform
// outcome, so the warp-collective tcgen05 operations that follow stay convergent).
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, uint64_t deadline_ns) {
    return __all_sync(0xffffffffu, mbar_wait(bar, parity, deadline_ns)) != 0;
}

template <int FMT, bool GATEUP>
__global__ void __launch_bounds__(kThreads, 1)
    decode_fp4_kernel(const __grid_constant__ CUtensorMap tm_b, const uint8_t* __restrict__ arena,
                      uint64_t entry_bytes, const GemvWork* __restrict__ work, int n_work, int n_units, int S,
                      const int32_t* __restrict__ slot_row, const uint32_t* __restrict__ fill_flag, int H, int I,
                      uint16_t* __restrict__ h_out, const float* __restrict__ w_perm, float* __restrict__ pair_out,
                      float* __restrict__ ws, int* __restrict__ cnt, int* status, uint64_t fill_wait_ns,
                      const int* __restrict__ dyn) {
    pdl_gate();  // may start while the previous kernel of the stream finishes
    using Lay = Layout<FMT, GATEUP>;
    constexpr int RAW = Lay::RAW;
    if (dyn) {
        n_work = dyn[0];
        n_units = dyn[1];
        S = dyn[2];
    }
    const uint64_t consumer_wait_ns = fill_wait_ns + kWaitDeadlineNs;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* b_tiles = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* raw_tiles = b_tiles + kMma * kB16;
    float* xchg = reinterpret_cast<float*>(raw_tiles + kRawStages * RAW);
    uint4* scale_lut = reinterpret_cast<uint4*>(raw_tiles + kRawStages * RAW + Lay::XCHG_BYTES);
    GemvWork* work_sm = reinterpret_cast<GemvWork*>(raw_tiles + kRawStages * RAW + Lay::XCHG_BYTES + kLutBytes);
    Shared& sh =
        *reinterpret_cast<Shared*>(raw_tiles + kRawStages * RAW + Lay::XCHG_BYTES + kLutBytes + kWorkBytes);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int K = GATEUP ? H : I;
    const int KB = K / BK;
    const int R = GATEUP ? I / 64 : H / 128;
    // stages of the gate/up part of an entry (the down part follows)
    const uint64_t gu_bytes = static_cast<uint64_t>(I / 64) * (H / 64) * RAW;

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
    for (int sc = threadIdx.x; sc < 256; sc += kThreads) scale_lut[sc] = scale_tables<FMT>(static_cast<uint32_t>(sc));
    // the wave's work list (with its closing total entry) in shared memory, when it fits: the
    // producer, MMA and converter roles look their units up there
    const bool work_in_smem = n_work + 1 <= kWorkSmem;
    if (work_in_smem)
        for (int i = threadIdx.x; i <= n_work; i += kThreads) work_sm[i] = work[i];
    const GemvWork* wl = work_in_smem ? work_sm : work;
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sh.tmem_base;

    if (warp == 0) {
        // ------------------------------------------------------------ producer (raw stages)
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0, used = 0, last_phase = 0;
            bool ok = true;
            int ready_a = -1;
            for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
                const Unit un = locate_unit_any(wl, n_work, u, R, S);
                const GemvWork wk = wl[un.a];
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
                                     (GATEUP ? static_cast<uint64_t>(un.tile) * (H / 64) * RAW
                                             : gu_bytes + static_cast<uint64_t>(un.tile) * (I / 64) * RAW);
                const int kb0 = un.split * KB / S, kb1 = (un.split + 1) * KB / S;
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!mbar_wait(&sh.raw_empty[stage], phase ^ 1u, consumer_wait_ns)) {
                        raise_status(status, kDevWaitTimeout);
                        ok = false;
                        break;
                    }
                    uint8_t* dst = raw_tiles + stage * RAW;
                    mbar_arrive_expect_tx(&sh.raw_full[stage], RAW);
                    bulk_load(dst, src + static_cast<uint64_t>(kb) * RAW, RAW, &sh.raw_full[stage]);
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
                const Unit un = locate_unit_any(wl, n_work, u, R, S);
                const GemvWork wk = wl[un.a];
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
                    const uint64_t db = sw128_kmajor_desc(smem_u32(b_tiles + stage * kB16));
                    const uint32_t at = tmem + kTmemA + static_cast<uint32_t>(stage) * kACols;
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k)  // A: +8 columns, B: +32 bytes per K = 16 step
                        umma_bf16_tmem_a(d, at + 8 * k, db + 2 * k, idesc, (kb != kb0 || k != 0) ? 1u : 0u);
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
        TensorScales tsc{};
        if (FMT == kFp4Nv) tsc = TensorScales{arena, entry_bytes, slot_row};
        decode_epilogue<GATEUP, FMT == kFp4Nv>(sh.acc_full, sh.acc_empty, sh.ok, sh.last, tmem, xchg, work, n_work,
                                               n_units, S, R, H, I, h_out, w_perm, pair_out, ws, cnt, status,
                                               consumer_wait_ns, 64, tsc);
    } else {
        // ------------------------------------------------------------ converters (warps 6-21)
        const int c = threadIdx.x - kConvBase;
        const int grp = c / (32 * kGroupWarps);
        const int q = warp & 3;                 // TMEM lane quadrant of this warp
        const int row = q * 32 + lane;          // the A row (= TMEM lane) this thread expands
        const bool token_loader = (c % (32 * kGroupWarps)) == 0;
        const uint32_t t_row = tmem + (static_cast<uint32_t>(q * 32) << 16) + kTmemA;
        if (token_loader) prefetch_tmap(&tm_b);
        uint32_t used = 0, last_phase = 0;
        bool ok = true;
        int n0 = 0;  // stage index of the unit's first stage over the whole run (as the producer
                     // and the MMA issuer count stages)
        for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
            const Unit un = locate_unit_any(wl, n_work, u, R, S);
            const GemvWork wk = wl[un.a];
            const int tok0 = wk.tok_off + un.chunk * kNMax;
            const int nt = min(kNMax, wk.n_tok - un.chunk * kNMax);
            const int nb = (nt + 15) >> 4;
            const int kb0 = un.split * KB / S, kb1 = (un.split + 1) * KB / S;
            // this group's stages of the unit: n = n0 + (kb - kb0) with n % kConvGroups == grp
            const int first = kb0 + ((grp - n0 % kConvGroups) + kConvGroups) % kConvGroups;
            for (int kb = first; kb < kb1; kb += kConvGroups) {
                const int n = n0 + (kb - kb0);
                const int rs = n % kRawStages, ms = n % kMma;
                const uint32_t rphase = (n / kRawStages) & 1, mphase = (n / kMma) & 1;
                if (!warp_wait(&sh.raw_full[rs], rphase, consumer_wait_ns)) {
                    if (lane == 0) raise_status(status, kDevWaitTimeout);
                    ok = false;
                    break;
                }
                const uint8_t* raw = raw_tiles + rs * RAW;
                // this row's 32 code bytes (codes 0 .. 31 and 32 .. 63 of its slab) and its
                // scale bytes
                const uint4 a = *reinterpret_cast<const uint4*>(raw + row * 32);
                const uint4 b = *reinterpret_cast<const uint4*>(raw + row * 32 + 16);
                uint32_t sb;
                if (FMT == kFp4Mx) sb = *reinterpret_cast<const uint16_t*>(raw + 4096 + row * 2);
                else sb = *reinterpret_cast<const uint32_t*>(raw + 4096 + row * 4);
                __syncwarp();
                if (lane == 0) mbar_arrive(&sh.raw_empty[rs]);  // the raw slot may be refilled
                // the MMA stage is free once the products that read its A columns and token tile
                // have completed (usually long before: the converters set the pace)
                if (!warp_wait(&sh.mma_empty[ms], mphase ^ 1u, consumer_wait_ns)) {
                    if (lane == 0) raise_status(status, kDevWaitTimeout);
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (token_loader) {
                    uint8_t* sb_tile = b_tiles + ms * kB16;
                    mbar_arrive_expect_tx(&sh.mma_full[ms], nb * 16 * BK * 2);
                    for (int bx = 0; bx < nb; ++bx)
                        tma_load_2d(sb_tile + bx * 16 * BK * 2, &tm_b, &sh.mma_full[ms], kb * BK, tok0 + 16 * bx);
                    used |= 1u << ms;
                    last_phase = (last_phase & ~(1u << ms)) | (mphase << ms);
                }
                __syncwarp();  // converged again for the warp-collective TMEM stores
                // two halves of 32 codes: the first half's TMEM store runs while the second half
                // is expanded
                const uint32_t ta = t_row + static_cast<uint32_t>(ms) * kACols;
                uint32_t w[16];
                if (FMT == kFp4Mx) {  // one E8M0 scale per 32 codes
                    const uint4 t0 = scale_lut[sb & 0xffu];
                    expand8(a.x, t0, w + 0);
                    expand8(a.y, t0, w + 4);
                    expand8(a.z, t0, w + 8);
                    expand8(a.w, t0, w + 12);
                } else {  // one E4M3 scale per 16 codes
                    const uint4 t0 = scale_lut[sb & 0xffu], t1 = scale_lut[(sb >> 8) & 0xffu];
                    expand8(a.x, t0, w + 0);
                    expand8(a.y, t0, w + 4);
                    expand8(a.z, t1, w + 8);
                    expand8(a.w, t1, w + 12);
                }
                tmem_st16(ta, w);
                uint32_t w2[16];
                if (FMT == kFp4Mx) {
                    const uint4 t1 = scale_lut[(sb >> 8) & 0xffu];
                    expand8(b.x, t1, w2 + 0);
                    expand8(b.y, t1, w2 + 4);
                    expand8(b.z, t1, w2 + 8);
                    expand8(b.w, t1, w2 + 12);
                } else {
                    const uint4 t2 = scale_lut[(sb >> 16) & 0xffu], t3 = scale_lut[sb >> 24];
                    expand8(b.x, t2, w2 + 0);
                    expand8(b.y, t2, w2 + 4);
                    expand8(b.z, t3, w2 + 8);
                    expand8(b.w, t3, w2 + 12);
                }
                tmem_st16(ta + 16, w2);
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&sh.mma_full[ms]);
            }
            n0 += kb1 - kb0;
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

template <int FMT, bool GATEUP>
cudaError_t launch(const CUtensorMap& tb, const uint8_t* arena, uint64_t entry_bytes, const GemvWork* work,
                   int n_work, int n_units, int S, const int32_t* slot_row, const uint32_t* fill_flag, int H, int I,
                   uint16_t* h_out, const float* w_perm, float* pair_out, float* ws, int* cnt, int* status,
                   uint64_t fill_wait_ns, int num_sms, cudaStream_t st, const int* dyn) {
    if (!dyn) {
        if (n_units <= 0 || n_work <= 0) return cudaSuccess;
        if (S < 1 || S > kDecodeMaxSplit) return cudaErrorInvalidValue;
        if (S > 1 && n_units > kDecodeSplitUnits) return cudaErrorInvalidValue;
    }
    auto kern = decode_fp4_kernel<FMT, GATEUP>;
    constexpr int smem = Layout<FMT, GATEUP>::SMEM;
    static std::atomic<uint64_t> attr{0};
    const cudaError_t e = ensure_smem_limit(kern, smem, attr);
    if (e != cudaSuccess) return e;
    const int grid = dyn ? num_sms : std::min(n_units, num_sms);
    return launch_pdl(kern, dim3(grid), dim3(kThreads), smem, st, tb, arena, entry_bytes, work, n_work, n_units, S,
                      slot_row, fill_flag, H, I, h_out, w_perm, pair_out, ws, cnt, status, fill_wait_ns, dyn);
}

template <int FMT>
cudaError_t launch_fmt(bool gateup, const DecodeMaps& m, const uint8_t* arena, uint64_t entry_bytes,
                       const GemvWork* work, int n_work, int n_units, int S, const int* dyn, const int32_t* slot_row,
                       const uint32_t* fill_flag, int H, int I, uint16_t* h_perm, const float* w_perm,
                       float* pair_out, float* ws, int* cnt, int* status, uint64_t fill_wait_ns, int num_sms,
                       cudaStream_t st) {
    if (gateup)
        return launch<FMT, true>(m.b_x, arena, entry_bytes, work, n_work, n_units, S, slot_row, fill_flag, H, I,
                                 h_perm, nullptr, nullptr, ws, cnt, status, fill_wait_ns, num_sms, st, dyn);
    return launch<FMT, false>(m.b_h, arena, entry_bytes, work, n_work, n_units, S, slot_row, fill_flag, H, I,
                              nullptr, w_perm, pair_out, ws, cnt, status, fill_wait_ns, num_sms, st, dyn);
}

}  // namespace

cudaError_t launch_decode_fp4(int fmt, bool gateup, const DecodeMaps& m, const uint8_t* arena, uint64_t entry_bytes,
                              const GemvWork* work, int n_work, int n_units, int S, const int* dyn,
                              const int32_t* slot_row, const uint32_t* fill_flag, int H, int I, uint16_t* h_perm,
                              const float* w_perm, float* pair_out, float* ws, int* cnt, int* status,
                              uint64_t fill_wait_ns, int num_sms, cudaStream_t st) {
    if (fmt == kFp4Mx)
        return launch_fmt<kFp4Mx>(gateup, m, arena, entry_bytes, work, n_work, n_units, S, dyn, slot_row, fill_flag,
                                  H, I, h_perm, w_perm, pair_out, ws, cnt, status, fill_wait_ns, num_sms, st);
    if (fmt == kFp4Nv)
        return launch_fmt<kFp4Nv>(gateup, m, arena, entry_bytes, work, n_work, n_units, S, dyn, slot_row, fill_flag,
                                  H, I, h_perm, w_perm, pair_out, ws, cnt, status, fill_wait_ns, num_sms, st);
    return cudaErrorInvalidValue;
}

}  // namespace moe
