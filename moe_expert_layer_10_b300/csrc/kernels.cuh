// Kernel launchers of the routed-MoE hot path (sm_103a). Each launcher enqueues on the
// given stream and returns the launch's cudaError_t. Pointers are device pointers.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <utility>

namespace moe {

// Raise a kernel's dynamic shared-memory limit to `bytes` once per device: `done` keeps one bit
// per device id (ids >= 64 share bit 63 and simply set the attribute again).
template <typename... KArgs>
inline cudaError_t ensure_smem_limit(void (*kern)(KArgs...), size_t bytes, std::atomic<uint64_t>& done) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = dev < 63 ? (1ull << dev) : 0ull;
    if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
    if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_acq_rel);
    return e;
}

// Launch a kernel of the layer's chain with programmatic stream serialization: it may be
// scheduled while the previous kernel of the stream is still running, and waits for it in
// pdl_gate (ptx.cuh) before touching memory.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args&&... args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// --- router: logits in the fixed fp32 order, then top-k + softmax gates ---
cudaError_t launch_router_logits(const uint16_t* x, const float* Wr, const float* b, int T, int H, int E, float* z,
                                 cudaStream_t st);
// forced == nullptr: top-k by (z desc, id asc); else order the forced sets the same way.
cudaError_t launch_router_topk(const float* z, int T, int E, int k, const int32_t* forced, int32_t* idx, float* w,
                               int* status, cudaStream_t st);

// --- permutation: stable grouping of the T*k pairs by expert ---
// permute_grid(P) CTAs of 1024 pairs, with `cells` holding 2 * permute_grid(P) * E ints of
// scratch and `done` an arrival counter that is 0 before the first launch (the kernels leave it
// 0). Decode batches (up to 1024 pairs) take launch_permute_gather below instead.
int permute_grid(int P);
cudaError_t launch_permute(const int32_t* idx, const float* w, int P, int E, int32_t* offsets, int32_t* perm,
                           int32_t* inv_perm, float* w_perm, int32_t* active, int32_t* n_active, int* status,
                           int32_t* cells, unsigned* done, cudaStream_t st);
// Up to 1024 pairs: the permutation and x_perm[pos] = x[perm[pos] / k] in one launch, the
// same outputs as launch_permute followed by launch_gather_rows.
bool permute_gathers_rows(int P);
cudaError_t launch_permute_gather(const int32_t* idx, const float* w, const uint16_t* x, int P, int k, int E, int H,
                                  int32_t* offsets, int32_t* perm, int32_t* inv_perm, float* w_perm,
                                  int32_t* active, int32_t* n_active, uint16_t* x_perm, int* status,
                                  cudaStream_t st);
// x_perm[pos] = x[perm[pos] / k]  (bf16 rows of H)
cudaError_t launch_gather_rows(const uint16_t* x, const int32_t* perm, int P, int k, int H, uint16_t* x_perm,
                               cudaStream_t st);

// --- decode expert FFN: work list of one wave (one entry per routed expert) ---
struct GemvWork {
    int expert;      // expert id
    int tok_off;     // first permuted position of its tokens
    int n_tok;       // tokens routed to it
    int unit_begin;  // first work unit of this expert (entry n_work holds the total)
    int wait_slot;   // slot whose fill flag must reach `gen` before its weights are read, or -1
    uint32_t gen;    // fill generation of that slot (written by the copy stream after the copy)
    int pad0, pad1;
};

// --- decode expert FFN on the tensor cores (weights as M = 128, tokens as N <= 64) ---
constexpr int kDecodeMaxSplit = 4;       // largest K split of one launch
constexpr int kDecodeSplitUnits = 1024;  // most units of a split launch (workspace tiles)
constexpr int kDecodeTileFloats = 64 * 128;  // fp32 partial tile: [64 tokens][128 rows]

struct DecodeMaps {
    CUtensorMap a_gu;  // arena [C*3I rows x H], box 64 x 64 rows, 128B swizzle
    CUtensorMap a_d;   // arena [C*3H rows x I], box 64 x 128 rows
    CUtensorMap b_x;   // x_perm [P_max x H], box 64 x 16 rows
    CUtensorMap b_h;   // h_perm [P_max x I], box 64 x 16 rows
};

int decode_row_tiles(bool gateup, int H, int I);   // row tiles per token chunk
int decode_token_chunks(int n_tok);                // chunks of <= 64 tokens
int decode_choose_split(int n_tiles, bool gateup, int H, int I, int num_sms);  // K split S of a launch
// h_perm[pos, i] = bf16( silu(W_gate[i] . x) * (W_up[i] . x) ) for the wave's experts.
// work[a].unit_begin counts units = chunks * row tiles * S per entry (entry n_work: total).
// fill_flag[slot] is the device word the copy stream bumps after each fill of the slot.
cudaError_t launch_decode_gateup(const DecodeMaps& maps, const GemvWork* work, int n_work, int n_units, int S,
                                 const int32_t* slot_row, const uint32_t* fill_flag, int H, int I, uint16_t* h_perm,
                                 float* ws, int* cnt, int* status, uint64_t fill_wait_ns, int num_sms,
                                 cudaStream_t st);
// Same kernels with the work size read on the device: dyn = {n_work, n_units, S} (written by
// the policy kernel); the grid is one CTA per SM.
cudaError_t launch_decode_gateup_dyn(const DecodeMaps& maps, const GemvWork* work, const int* dyn,
                                     const int32_t* slot_row, int H, int I, uint16_t* h_perm, float* ws, int* cnt,
                                     int* status, int num_sms, cudaStream_t st);
cudaError_t launch_decode_down_dyn(const DecodeMaps& maps, const GemvWork* work, const int* dyn,
                                   const int32_t* slot_row, int H, int I, const float* w_perm, float* pair_out,
                                   float* ws, int* cnt, int* status, int num_sms, cudaStream_t st);
// pair_out[pos, n] = w_perm[pos] * (W_down[n] . h[pos])
cudaError_t launch_decode_down(const DecodeMaps& maps, const GemvWork* work, int n_work, int n_units, int S,
                               const int32_t* slot_row, const uint32_t* fill_flag, int H, int I, const float* w_perm,
                               float* pair_out, float* ws, int* cnt, int* status, uint64_t fill_wait_ns, int num_sms,
                               cudaStream_t st);

// --- decode expert FFN, gate/up and down in one persistent launch (bf16; decode_fused.cu) ---
// work_gu / work_d: the wave's two work lists in the same entry order, each closed by its unit
// total, with GemvWork::pad0 = the entry's first token-chunk index (chunks of all entries
// numbered consecutively). h_ready / h_done: decode_fused_chunk_slots(E, P) ints each, zero
// before the first launch (every launch leaves them zero). The down phase's split-K tiles follow
// the gate/up phase's in ws and cnt.
int decode_fused_chunk_slots(int E, int P);
// max_chunk_tok: the most tokens of any chunk of the wave (<= 16 selects the small-token kernel).
cudaError_t launch_decode_fused(const DecodeMaps& maps, const GemvWork* work_gu, int n_work, int units_gu, int S_gu,
                                const GemvWork* work_d, int units_d, int S_d, int max_chunk_tok, const int32_t* slot_row,
                                const uint32_t* fill_flag, int H, int I, uint16_t* h_perm, const float* w_perm,
                                float* pair_out, float* ws, int* cnt, int* h_ready, int* h_done, const int* sched,
                                int* status, uint64_t fill_wait_ns, int num_sms, cudaStream_t st);
// A unit schedule for a fused launch of `grid` CTAs that keeps the joint list's round robin but
// moves the last down unit of each most-loaded CTA to a least-loaded one, when that lowers the
// largest per-CTA K-block total (kb_gu / kb_d: K blocks of one unit of each phase). Writes
// keep[grid] (round-robin units a CTA runs), pool_off[grid + 1] and the moved units into sched
// (at most cap ints) and returns the ints written, or 0 if the plain round robin is as level
// (the launch then takes sched = null).
int decode_fused_schedule(int units_gu, int units_d, int kb_gu, int kb_d, int grid, int* sched, int cap);
// K splits (S_gu, S_d) of a fused launch: the pair that minimises the largest per-CTA load
// under the round-robin assignment of the concatenated unit list. chunk_tok: token count of each
// chunk of the wave's entries, in work-list order.
void decode_fused_choose_split(const int* chunk_tok, int n_chunks, int H, int I, int num_sms, int* S_gu, int* S_d);

// --- decode expert FFN with 4-bit entries (expanded to bf16 on chip; decode_fp4.cu) ---
// fmt: kFp4Mx (MXFP4: E8M0 scale per 32 weights) or kFp4Nv (NVFP4: E4M3 scale per 16 weights
// and an fp32 tensor scale per matrix, in the entry's last 16 bytes). Same work lists, splits
// and epilogues as the bf16 kernels; dyn as for the _dyn launchers.
enum : int { kFp4Mx = 1, kFp4Nv = 2 };
cudaError_t launch_decode_fp4(int fmt, bool gateup, const DecodeMaps& maps, const uint8_t* arena, uint64_t entry_bytes,
                              const GemvWork* work, int n_work, int n_units, int S, const int* dyn,
                              const int32_t* slot_row, const uint32_t* fill_flag, int H, int I, uint16_t* h_perm,
                              const float* w_perm, float* pair_out, float* ws, int* cnt, int* status,
                              uint64_t fill_wait_ns, int num_sms, cudaStream_t st);

// --- device-resident cache policy (decode forward with no host round trip) ---
enum : int { kEvHit = 0, kEvFill = 1, kEvPrefetchFill = 2, kEvPrefetchHit = 3 };

struct DevLruState {
    int head, tail, n_used, pad;  // most / least recently used slot, slots handed out so far
};
struct DevStats {  // the fields of moe_stats_t that the device policy counts
    unsigned long long expert_reads, hits, misses, prefetch_fills, prefetch_hits, evictions, fill_bytes, trace_len,
        forwards, waves, resize_evictions;
};
struct DevEvent {
    int kind, layer, expert, slot, ev_layer, ev_expert;
};
struct WaveHdr {  // written by the policy kernel, read by the fill and decode kernels
    int n_fill;
    int hit_gu[3], hit_d[3], miss_gu[3], miss_d[3];  // {n_work, n_units, S} per decode launch
};
struct DevPolicyArgs {
    DevLruState* state;
    int *lru_prev, *lru_next, *lru_key;  // [C]
    int32_t* slot_of;                    // [L*E] device slot table
    int C, E, H, I, layer, num_sms;
    int prefetch;                        // accesses are prefetches (no compute)
    // keys: the routed wave (active list of the permutation) or an explicit expert list
    const int32_t* active;
    const int32_t* n_active;
    int wave;
    const int32_t* keys;
    int n_keys;
    const int32_t* offsets;              // expert offsets of the permutation (for work lists)
    int2* fill_list;                     // [C] (key, slot)
    GemvWork* work_hit;                  // [2*(E+1)]: gate/up list, then down list (or null)
    GemvWork* work_miss;                 // [2*(E+1)]
    int* order;                          // [2*C] scratch: hit experts, then filled experts
    WaveHdr* hdr;
    DevStats* stats;
    DevEvent* trace;                     // ring of trace_cap events (or null)
    unsigned long long trace_cap;
    unsigned long long entry_bytes;
};
cudaError_t launch_policy(const DevPolicyArgs& a, cudaStream_t st);
// copy the fill list's entries from the host pool (device-mapped) into their slots
cudaError_t launch_fill(const void* pool_dev, void* arena, const int2* fill_list, const int* n_fill,
                        size_t entry_bytes, int num_sms, cudaStream_t st);

// --- combine: out[t] = resid[t] + sum_j pair_out[inv_perm[t*k+j]] (j order) ---
cudaError_t launch_combine(const float* pair_out, const int32_t* inv_perm, const float* resid, float* out, int T,
                           int k, int H, cudaStream_t st);

// --- prefill expert FFN: tcgen05 grouped GEMM ---
struct GemmMaps {
    CUtensorMap a_x;    // x_perm [P_max x H], box 64 x 128, 128B swizzle
    CUtensorMap b_gu;   // arena [C*3I rows x H], box 64 x 128, 128B swizzle
    CUtensorMap a_h;    // h_perm [P_max x I], box 64 x 128
    CUtensorMap b_d;    // arena [C*3H rows x I], box 64 x 128
};
int gemm_tiles(bool gateup, const int* counts, int n, int H, int I);  // grid bound for a wave
cudaError_t launch_gemm_gateup(const GemmMaps& maps, const int32_t* offsets, const int32_t* active, int a_begin,
                               int a_end, int total_tiles, const int32_t* slot_row, int H, int I, uint16_t* h_perm,
                               int* status, int num_sms, cudaStream_t st);
cudaError_t launch_gemm_down(const GemmMaps& maps, const int32_t* offsets, const int32_t* active, int a_begin,
                             int a_end, int total_tiles, const int32_t* slot_row, int H, int I, const float* w_perm,
                             float* pair_out, int* status, int num_sms, cudaStream_t st);

}  // namespace moe
