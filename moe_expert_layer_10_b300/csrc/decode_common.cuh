// Parts shared by the decode expert kernels (bf16 weights, decode_mma.cu; MXFP4 weights,
// decode_fp4.cu): the unit schedule and the epilogue. See decode_mma.cu for the design.
#pragma once

#include "kernels.cuh"
#include "ptx.cuh"
#include "umma.cuh"

namespace moe {
namespace dec {

constexpr int BK = 64;                   // K per stage (one 128-byte swizzle row of bf16)
constexpr int kNMax = 64;                // tokens per chunk (MMA N <= 64)
constexpr int kXchgFloats = kNMax * 64;  // up values of one unit: [token][64 rows]

struct Unit {
    int a;      // work entry
    int chunk;  // token chunk
    int tile;   // row tile
    int split;  // K split
};

__device__ __forceinline__ Unit locate_unit(const GemvWork* work, int n_work, int u, int R, int S) {
    int lo = 0, hi = n_work - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(&work[mid].unit_begin) <= u) lo = mid;
        else hi = mid - 1;
    }
    const int local = u - __ldg(&work[lo].unit_begin);
    const int rest = local / S;
    return Unit{lo, rest / R, rest % R, local % S};
}

__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.0f + expf(-g)) * u; }

// Arrival on a split tile's counter: a gpu-scope acquire-release add. The barrier before it
// orders the other epilogue threads' partial stores ahead of this release (cumulativity), and
// the barrier after it orders their partial loads behind this acquire.
__device__ __forceinline__ int atomic_add_acq_rel_gpu(int* p, int v) {
    int old;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

// Per-matrix fp32 scales that multiply the accumulator before the epilogue's arithmetic (the
// tensor scales of NVFP4 entries): the last 16 bytes of each entry hold the scales of W_gate,
// W_up and W_down. None for bf16 and MXFP4 entries.
struct TensorScales {
    const uint8_t* arena = nullptr;  // slot s's entry starts at arena + s * entry_bytes
    uint64_t entry_bytes = 0;
    const int32_t* slot_row = nullptr;
};

// State of the epilogue role across units: which of the two accumulators comes next, and its
// barrier phase.
struct EpiState {
    int acc = 0;
    uint32_t acc_phase = 0;
};

// gpu-scope release add, for a counter that other CTAs read with an acquire load
__device__ __forceinline__ void red_add_release_gpu(int* p, int v) {
    asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// The epilogue role on one unit: four consecutive warps (TMEM lane quadrant = warp % 4), named
// barrier 1 over their 128 threads, leader_tid = the first of them. Wait for the accumulator
// (one thread waits, the outcome is shared), then either write the split's partial and arrive
// on the tile counter, or (single split / last split) produce h = silu(g)*u (gate/up) or
// pair_out = w_p * y (down) for the chunk's tokens. With TSCALE the (summed) accumulator of a
// row is first multiplied by its matrix's tensor scale. ws / cnt: this launch's split-K
// workspace and tile counters for the unit's phase (u is the unit's index within the phase).
// h_ready (gate/up, or null): once the unit's h tile is written, the leader adds 1 to
// h_ready[wk.pad0 + chunk] with release semantics, after a proxy fence that orders the h
// stores before later tensor-memory-access (TMA) reads of them. Returns false on a timeout
// (status raised; the role must stop).
template <bool GATEUP, bool TSCALE = false>
__device__ __forceinline__ bool epilogue_unit(EpiState& st, uint64_t* acc_full, uint64_t* acc_empty, int* sh_ok,
                                              int* sh_last, uint32_t tmem, float* xchg,
                                              const GemvWork* __restrict__ work, int n_work, int u, int S, int R,
                                              int H, int I, uint16_t* __restrict__ h_out,
                                              const float* __restrict__ w_perm, float* __restrict__ pair_out,
                                              float* __restrict__ ws, int* __restrict__ cnt, int* status,
                                              uint64_t consumer_wait_ns, int leader_tid, TensorScales tsc,
                                              int* h_ready) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int q = warp & 3;         // TMEM lanes 32q .. 32q+31
    const int row = q * 32 + lane;  // accumulator row of this thread
    const bool leader = static_cast<int>(threadIdx.x) == leader_tid;
    const int acc = st.acc;
    auto advance = [&]() {
        st.acc ^= 1;
        if (st.acc == 0) st.acc_phase ^= 1u;
    };
    const Unit un = locate_unit(work, n_work, u, R, S);
    const GemvWork wk = work[un.a];
    const int tok0 = wk.tok_off + un.chunk * kNMax;
    const int nt = min(kNMax, wk.n_tok - un.chunk * kNMax);
    const int nc = (nt + 15) >> 4;  // 16-column chunks of the accumulator
    if (leader) sh_ok[acc] = mbar_wait(&acc_full[acc], st.acc_phase, consumer_wait_ns) ? 1 : 0;
    named_bar(1, 128);
    if (!sh_ok[acc]) {
        if (leader) raise_status(status, kDevWaitTimeout);
        return false;
    }
    tc_fence_after();
    const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * kNMax);
    const size_t tile_floats = static_cast<size_t>(kNMax) * 128;
    bool from_ws = false;
    if (S > 1) {
        // partial of this split -> workspace [unit][token][row], coalesced over rows
        float* wsu = ws + static_cast<size_t>(u) * tile_floats;
        for (int c = 0; c < nc; ++c) {
            uint32_t v[16];
            tmem_ld16(taddr + 16 * c, v);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 16; ++j) __stcg(wsu + (16 * c + j) * 128 + row, __uint_as_float(v[j]));
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[acc]);
        named_bar(1, 128);
        if (leader) {
            const int tile_id = u / S;
            const int old = atomic_add_acq_rel_gpu(cnt + tile_id, 1);
            const int is_last = (old == S - 1) ? 1 : 0;
            if (is_last) cnt[tile_id] = 0;  // every split has arrived; ready for the next launch
            sh_last[acc] = is_last;
        }
        named_bar(1, 128);
        const bool is_last = sh_last[acc] != 0;
        if (!is_last) {
            advance();
            return true;
        }
        from_ws = true;
    }
    float tscale = 1.0f;  // this row's tensor scale (gate rows, up rows, or W_down rows)
    if (TSCALE) {
        int slot = tsc.slot_row[wk.expert];
        if (slot < 0) slot = 0;  // the producer raised the status; results are discarded
        const float* ts = reinterpret_cast<const float*>(tsc.arena + static_cast<uint64_t>(slot) * tsc.entry_bytes +
                                                         tsc.entry_bytes - 16);
        tscale = __ldg(ts + (GATEUP ? (q >= 2 ? 1 : 0) : 2));
    }
    const float* ws0 = ws + static_cast<size_t>(u - un.split) * tile_floats;
    // 16 accumulator columns of this thread's row: TMEM, or the sum of the S partials
    auto fetch = [&](int c, float (&v)[16]) {
        if (from_ws) {
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] = __ldcg(ws0 + (16 * c + j) * 128 + row);
            for (int s = 1; s < S; ++s) {
                const float* p = ws0 + static_cast<size_t>(s) * tile_floats;
#pragma unroll
                for (int j = 0; j < 16; ++j) v[j] += __ldcg(p + (16 * c + j) * 128 + row);
            }
        } else {
            uint32_t r[16];
            tmem_ld16(taddr + 16 * c, r);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
        }
        if (TSCALE) {
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] *= tscale;
        }
    };
    auto release = [&]() {
        if (!from_ws) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[acc]);
        }
    };
    if (GATEUP) {
        float* xc = xchg;
        const int i0 = un.tile * 64;
        if (q >= 2) {  // up rows: hand them to the gate warps
            for (int c = 0; c < nc; ++c) {
                float v[16];
                fetch(c, v);
#pragma unroll
                for (int j = 0; j < 16; ++j) xc[(16 * c + j) * 64 + row - 64] = v[j];
            }
            release();
        }
        named_bar(1, 128);
        if (q < 2) {  // gate rows: h = silu(g) * u for the chunk's tokens
            for (int c = 0; c < nc; ++c) {
                float v[16];
                fetch(c, v);
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int n = 16 * c + j;
                    if (n < nt) {
                        const float h = silu_mul(v[j], xc[n * 64 + row]);
                        reinterpret_cast<__nv_bfloat16*>(h_out)[static_cast<size_t>(tok0 + n) * I + i0 + row] =
                            __float2bfloat16_rn(h);
                    }
                }
            }
            release();
            if (h_ready) asm volatile("fence.proxy.async.global;" ::: "memory");
        }
        named_bar(1, 128);  // the exchange buffer is free for the next unit; every h store is done
        if (h_ready && leader) red_add_release_gpu(h_ready + wk.pad0 + un.chunk, 1);
    } else {
        const int n0 = un.tile * 128;
        for (int c = 0; c < nc; ++c) {
            float v[16];
            fetch(c, v);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int n = 16 * c + j;
                if (n < nt) {
                    const size_t pos = static_cast<size_t>(tok0 + n);
                    pair_out[pos * H + n0 + row] = __ldg(w_perm + pos) * v[j];
                }
            }
        }
        release();
    }
    advance();
    return true;
}

// The epilogue role over a launch's units u = blockIdx.x, blockIdx.x + gridDim.x, ...
template <bool GATEUP, bool TSCALE = false>
__device__ __forceinline__ void decode_epilogue(uint64_t* acc_full, uint64_t* acc_empty, int* sh_ok, int* sh_last,
                                                uint32_t tmem, float* xchg, const GemvWork* __restrict__ work,
                                                int n_work, int n_units, int S, int R, int H, int I,
                                                uint16_t* __restrict__ h_out, const float* __restrict__ w_perm,
                                                float* __restrict__ pair_out, float* __restrict__ ws,
                                                int* __restrict__ cnt, int* status, uint64_t consumer_wait_ns,
                                                int leader_tid, TensorScales tsc = TensorScales{}) {
    EpiState st;
    for (int u = blockIdx.x; u < n_units; u += gridDim.x)
        if (!epilogue_unit<GATEUP, TSCALE>(st, acc_full, acc_empty, sh_ok, sh_last, tmem, xchg, work, n_work, u, S, R,
                                           H, I, h_out, w_perm, pair_out, ws, cnt, status, consumer_wait_ns,
                                           leader_tid, tsc, nullptr))
            break;
}

}  // namespace dec
}  // namespace moe
