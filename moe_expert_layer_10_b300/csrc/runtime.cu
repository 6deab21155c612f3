// Host runtime and C ABI of the routed-MoE layer (see include/moe.h for the contract).
//
// Sources (page title, section):
//  * "FreeToken rtx 4090" (freetoken.wiki/hardware), "How the MoE Memory Hierarchy Works":
//    the complete expert pool stays in host memory as the source of truth; VRAM holds a
//    cache of complete (layer, expert) entries; decode follows routing with a shared LRU;
//    prefill loads the next layer's experts while the current layer computes; startup
//    writes weights straight into the final host layout (moe_host_entry).
//  * "FreeToken benchmark" (freetoken.wiki/performance), "How FreeToken Serves Large MoE
//    Models": full-layer double buffering; the PCIe link moves selected experts into the
//    GPU cache; the runtime console reports cache activity (moe_stats).
//
// B300 design: one context owns a pinned pool (cudaHostAlloc), a device arena of C whole
// entries, a device slot table slot_of[L][E], a compute stream and a copy stream.
//  * Host policy (default): the LRU runs here. A fill is one cudaMemcpyAsync of a contiguous
//    entry on the copy stream, followed by a write of the slot's fill generation to a device
//    flag. A fill into a slot waits (event) for the last compute wave that read the slot. The
//    decode kernels of a wave wait on the device for the flags of the entries the wave filled,
//    so resident experts compute while the copies cross the link; the prefill GEMM waits
//    (event) for its wave's fills.
//  * Device policy (MOE_DEVICE_POLICY): the LRU, the trace and the fills run in kernels
//    (device_policy.cu); a forward enqueues work only, so a decode step can be graph-captured.
//  * Elastic capacity (moe_cache_resize) and MXFP4 entries (MOE_MXFP4) apply to both.
// Every host wait polls with a deadline.
#include <algorithm>
#include <chrono>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <string>
#include <thread>
#include <vector>

#include "../../include/moe.h"
#include "kernels.cuh"
#include "lru.h"

using moe::ExpertLru;
using moe::GemvWork;

namespace {

thread_local std::string g_last_error;

int fail(int code, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return code;
}

#define CUDA_TRY(call)                                                                                 \
    do {                                                                                               \
        cudaError_t e_ = (call);                                                                       \
        if (e_ != cudaSuccess) return fail(MOE_E_CUDA, "%s: %s (%s:%d)", #call, cudaGetErrorString(e_), \
                                           __FILE__, __LINE__);                                        \
    } while (0)

constexpr int kEvRing = 256;     // compute-wave and per-fill completion events
constexpr int kFillStreams = 2;  // copy streams the fills of a batch take in turn
constexpr int kStageRing = 16;   // pinned staging buffers for small H2D copies
constexpr uint64_t kFillWaitNs = 20000000000ull;  // 20 s: a wave's own fills must land by then
constexpr uint64_t kInjectedFillWaitNs = 200000000ull;  // 0.2 s under injection kind 3
constexpr int kDecodeMaxTokens = 64;  // AUTO path: tensor-core decode kernels up to this many tokens per expert
// work-list entries of one wave: a gate/up and a down list, each closed by a total entry
// A wave's uploaded work: the gate/up and down lists (E + 1 entries each), then the fused
// launch's unit schedule (up to kSchedInts ints).
constexpr int kSchedInts = 1024;
static_assert(kSchedInts * sizeof(int) % sizeof(GemvWork) == 0, "the schedule fills whole work entries");
constexpr size_t kWorkEntries(int E) {
    return 2 * (static_cast<size_t>(E) + 1) + kSchedInts * sizeof(int) / sizeof(GemvWork);
}

enum KernelId { kRouterLogits, kRouterTopk, kPermute, kGather, kDecodeGateUp, kDecodeDown, kGemmGateUp, kGemmDown,
                kCombine, kPolicy, kFill, kDecodeFused, kNumKernels };
const char* kKernelNames[kNumKernels] = {"router_logits", "router_topk",  "permute",     "gather_rows",
                                         "decode_gateup", "decode_down",  "gemm_gateup", "gemm_down",
                                         "combine",       "device_policy", "device_fill", "decode_fused"};

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

typedef CUresult (*WriteValue32Fn)(CUstream, CUdeviceptr, cuuint32_t, unsigned int);

// cuStreamWriteValue32: a stream memory operation that writes a 32-bit word in stream order
// (with a memory barrier before the write, so the stream's earlier copies are visible first).
WriteValue32Fn write_value_fn() {
    static WriteValue32Fn fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuStreamWriteValue32", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<WriteValue32Fn>(p);
    }
    return fn;
}

// bf16 2-D view [rows x cols] (cols contiguous) with a box of [box_rows x box_cols].
bool make_map(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint32_t box_cols, uint32_t box_rows,
              CUtensorMapSwizzle sw) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t es[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

double wait_deadline_s() {
    static double v = [] {
        const char* s = getenv("MOE_WAIT_TIMEOUT_S");
        double d = s ? atof(s) : 120.0;
        return d > 0 ? d : 120.0;
    }();
    return v;
}

struct ProfRec {
    int kernel;
    cudaEvent_t start, stop;
    double bytes, flops;
};

struct FillRec {
    cudaEvent_t start, stop;
};

}  // namespace

struct moe_ctx {
    moe_config_t cfg{};
    int dev = 0, num_sms = 148;
    int L = 0, E = 0, H = 0, I = 0, k = 0, C = 0, Tmax = 0, Pmax = 0;
    size_t entry_elems = 0, entry_bytes = 0;
    int path = MOE_PATH_AUTO;
    bool fp4 = false;  // 4-bit entries (MOE_MXFP4 or MOE_NVFP4)
    int fp4_fmt = 0;   // moe::kFp4Mx or moe::kFp4Nv when fp4

    uint16_t* pool = nullptr;   // pinned host, L*E entries
    uint16_t* arena = nullptr;  // device, C entries
    std::vector<int32_t> slot_host;   // [L*E]
    int32_t* slot_dev = nullptr;      // [L*E]
    bool table_dirty = true;
    ExpertLru lru;

    cudaStream_t s_comp = nullptr, s_copy = nullptr;
    // fills take s_copy and kFillStreams - 1 internal streams in turn, so that one entry's copy
    // crosses the link while another stream finishes its previous copy (flag write, completion
    // event); every fill batch ends with s_copy waiting for the others
    cudaStream_t s_fill[kFillStreams] = {};
    cudaEvent_t ev_fill_join[kFillStreams] = {};
    bool own_comp = false, own_copy = false;

    // scratch (device)
    float* logits = nullptr;
    int32_t *offsets = nullptr, *perm = nullptr, *inv_perm = nullptr, *active = nullptr, *n_active = nullptr;
    int32_t* perm_cells = nullptr;         // multi-CTA permutation: per-CTA counts and starts
    unsigned* perm_done = nullptr;         // its arrival counter (0 between launches)
    float *w_perm = nullptr, *pair_out = nullptr;
    uint16_t *x_perm = nullptr, *h_perm = nullptr;
    int* status = nullptr;
    GemvWork* work_dev = nullptr;

    // pinned host staging
    int32_t* idx_host = nullptr;   // [Pmax]
    int* status_host = nullptr;    // [1]
    int32_t* table_stage = nullptr;        // [kStageRing][L*E]
    GemvWork* work_stage = nullptr;        // [kStageRing][kWorkEntries(E)]
    cudaEvent_t stage_ev[kStageRing] = {};
    int stage_next = 0;
    cudaEvent_t ev_d2h = nullptr;

    // ordering between fills and compute
    cudaEvent_t comp_ev[kEvRing] = {}, fill_ev[kEvRing] = {};
    int64_t comp_seq = -1, fill_seq = -1;
    std::vector<int64_t> slot_last_use, slot_fill;
    // per-slot fill generation: the copy stream writes fill_gen[slot] to fill_flag[slot] after
    // each fill, and the decode kernels poll it before streaming a freshly filled slot
    uint32_t* fill_flag = nullptr;     // device [C]
    std::vector<uint32_t> fill_gen;    // host [C], the generation of the last enqueued fill

    moe::DecodeMaps dec_maps{};
    float* dec_ws = nullptr;  // split-K partial tiles of the decode kernels
    int* dec_cnt = nullptr;   // per-tile arrival counters (zero between launches)
    int *dec_ready = nullptr, *dec_done = nullptr;  // fused decode: per-chunk h counters (zero between launches)
    int dec_chunk_slots = 0;
    moe::GemmMaps gemm_maps{};

    // stats and trace
    moe_stats_t stats{};
    std::vector<moe_event_t> trace;
    std::vector<FillRec> fill_pending;
    std::vector<cudaEvent_t> ev_pool;
    std::vector<ProfRec> prof_pending;
    moe_kernel_stat_t kstats[kNumKernels] = {};

    int inject_kind = 0, inject_count = 0;
    uint64_t fill_wait_ns = kFillWaitNs;  // device-side deadline of a wait for a fill

    // device-resident policy (MOE_DEVICE_POLICY): LRU, stats, trace and fills on the GPU
    bool dev_policy = false;
    void* pool_dev = nullptr;              // the pinned pool's device-mapped address
    moe::DevLruState* d_lru = nullptr;
    int *d_prev = nullptr, *d_next = nullptr, *d_key = nullptr;  // [C]
    moe::DevStats* d_stats = nullptr;
    moe::DevEvent* d_trace = nullptr;
    uint64_t d_trace_cap = 0;
    int2* d_fill_list = nullptr;           // [C]
    GemvWork* d_work = nullptr;            // [4*(E+1)]: hit lists, then miss lists
    int* d_order = nullptr;                // [2*C]
    moe::WaveHdr* d_hdr = nullptr;
    int32_t* d_keys = nullptr;             // [E]: explicit key lists of moe_cache_fill
    int32_t* d_iota = nullptr;             // [E]: 0..E-1
    cudaEvent_t ev_fork = nullptr, ev_join = nullptr;
};

namespace {

cudaEvent_t pool_event(moe_ctx* c) {
    if (!c->ev_pool.empty()) {
        cudaEvent_t e = c->ev_pool.back();
        c->ev_pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    return e;
}

// Fold completed timing records into the counters (no waiting).
void harvest(moe_ctx* c) {
    size_t keep = 0;
    for (size_t i = 0; i < c->prof_pending.size(); ++i) {
        ProfRec& r = c->prof_pending[i];
        if (cudaEventQuery(r.stop) == cudaSuccess) {
            float ms = 0.f;
            cudaEventElapsedTime(&ms, r.start, r.stop);
            moe_kernel_stat_t& s = c->kstats[r.kernel];
            s.launches++;
            s.total_ms += ms;
            s.bytes += r.bytes;
            s.flops += r.flops;
            c->ev_pool.push_back(r.start);
            c->ev_pool.push_back(r.stop);
        } else {
            c->prof_pending[keep++] = r;
        }
    }
    c->prof_pending.resize(keep);
    keep = 0;
    for (size_t i = 0; i < c->fill_pending.size(); ++i) {
        FillRec& r = c->fill_pending[i];
        if (cudaEventQuery(r.stop) == cudaSuccess) {
            float ms = 0.f;
            cudaEventElapsedTime(&ms, r.start, r.stop);
            c->stats.fill_ms += ms;
            c->ev_pool.push_back(r.start);
            c->ev_pool.push_back(r.stop);
        } else {
            c->fill_pending[keep++] = r;
        }
    }
    c->fill_pending.resize(keep);
    cudaGetLastError();  // cudaEventQuery's cudaErrorNotReady is not an error here
}

struct ProfScope {
    moe_ctx* c;
    int kernel;
    double bytes, flops;
    cudaEvent_t start = nullptr;
    ProfScope(moe_ctx* c_, int kid, double b, double f) : c(c_), kernel(kid), bytes(b), flops(f) {
        cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
        cudaStreamIsCapturing(c->s_comp, &cap);
        if ((c->cfg.flags & MOE_PROFILE) && cap == cudaStreamCaptureStatusNone) {
            start = pool_event(c);
            if (start) cudaEventRecord(start, c->s_comp);
        }
    }
    ~ProfScope() {
        if (start) {
            cudaEvent_t stop = pool_event(c);
            if (stop) {
                cudaEventRecord(stop, c->s_comp);
                c->prof_pending.push_back(ProfRec{kernel, start, stop, bytes, flops});
            }
        }
    }
};

int wait_event(moe_ctx* c, cudaEvent_t ev, const char* what) {
    if (c->inject_kind == 2 && c->inject_count > 0) {
        c->inject_count--;
        return fail(MOE_E_TIMEOUT, "%s: injected host wait timeout", what);
    }
    const auto t0 = std::chrono::steady_clock::now();
    for (long it = 0;; ++it) {
        cudaError_t e = cudaEventQuery(ev);
        if (e == cudaSuccess) return MOE_OK;
        if (e != cudaErrorNotReady) return fail(MOE_E_CUDA, "%s: %s", what, cudaGetErrorString(e));
        if ((it & 255) == 255) {
            const double dt = std::chrono::duration<double>(std::chrono::steady_clock::now() - t0).count();
            if (dt > wait_deadline_s()) return fail(MOE_E_TIMEOUT, "%s: no completion after %.0f s", what, dt);
            std::this_thread::yield();
        }
    }
}

int check_status(moe_ctx* c) {
    if (*c->status_host != 0) {
        const int code = *c->status_host;
        *c->status_host = 0;
        // clear the device word too, in stream order, so the context stays usable
        cudaMemsetAsync(c->status, 0, sizeof(int), c->s_comp);
        // a kernel that stopped early may have left split-K arrival or h counters behind
        cudaMemsetAsync(c->dec_cnt, 0, moe::kDecodeSplitUnits * sizeof(int), c->s_comp);
        cudaMemsetAsync(c->dec_ready, 0, c->dec_chunk_slots * sizeof(int), c->s_comp);
        cudaMemsetAsync(c->dec_done, 0, c->dec_chunk_slots * sizeof(int), c->s_comp);
        return fail(MOE_E_DEVICE, "a kernel raised device status %d (1 wait timeout, 2 bad forced set, 3 bad slot, "
                                  "4 bad expert index, 5 fill wait timeout)", code);
    }
    return MOE_OK;
}

// Pinned staging slot for a small H2D copy; waits (bounded) until its previous copy is done.
int next_stage(moe_ctx* c, int* slot_out) {
    const int s = c->stage_next;
    c->stage_next = (s + 1) % kStageRing;
    int rc = wait_event(c, c->stage_ev[s], "staging buffer reuse");
    if (rc) return rc;
    *slot_out = s;
    return MOE_OK;
}

int upload_table(moe_ctx* c) {
    if (!c->table_dirty) return MOE_OK;
    int s;
    int rc = next_stage(c, &s);
    if (rc) return rc;
    const size_t n = static_cast<size_t>(c->L) * c->E;
    int32_t* host = c->table_stage + static_cast<size_t>(s) * n;
    std::memcpy(host, c->slot_host.data(), n * sizeof(int32_t));
    CUDA_TRY(cudaMemcpyAsync(c->slot_dev, host, n * sizeof(int32_t), cudaMemcpyHostToDevice, c->s_comp));
    CUDA_TRY(cudaEventRecord(c->stage_ev[s], c->s_comp));
    c->table_dirty = false;
    return MOE_OK;
}

// A fill copy into p.slot was enqueued but the fill failed before it was committed: the slot's
// previous entry (p.victim, if any) is overwritten, so it leaves the cache and the slot returns
// to the free set. A later copy into the slot runs after this one on the copy stream.
void abandon_slot(moe_ctx* c, const ExpertLru::Plan& p) {
    if (p.victim < 0) return;  // the slot was free and stays free
    c->lru.release_slot(p.slot);
    c->slot_host[p.victim] = -1;
    c->stats.evictions++;
    c->table_dirty = true;
}

void record_event(moe_ctx* c, int kind, int key, int slot, int victim) {
    c->stats.trace_len++;
    if (!(c->cfg.flags & MOE_TRACE) || c->trace.empty()) return;
    moe_event_t ev;
    ev.kind = kind;
    ev.layer = key / c->E;
    ev.expert = key % c->E;
    ev.slot = slot;
    ev.ev_layer = victim >= 0 ? victim / c->E : -1;
    ev.ev_expert = victim >= 0 ? victim % c->E : -1;
    c->trace[(c->stats.trace_len - 1) % c->trace.size()] = ev;
}

// Make `st` wait until every fill numbered <= seq has landed. Within a batch the fills take the
// kFillStreams copy streams in turn, and a batch starts after the previous one has ended, so the
// completion events of fill seq and of the kFillStreams - 1 fills before it (one per other
// stream) cover all of them.
cudaError_t wait_fills_through(moe_ctx* c, cudaStream_t st, int64_t seq) {
    cudaError_t e = cudaSuccess;
    for (int64_t q = seq; e == cudaSuccess && q >= 0 && q > seq - kFillStreams; --q)
        e = cudaStreamWaitEvent(st, c->fill_ev[q % kEvRing], 0);
    return e;
}

// Access the given keys in order (routed or prefetch), enqueue the fills as one batch on
// the copy streams. Each filled slot remembers the batch, whose event compute waits for.
// On any failure the batch opened so far is still closed with its event, and the access
// that failed is not committed, so the policy and the slot table stay consistent. If the
// failure comes after the copy into the slot was enqueued, the slot's previous entry is
// evicted as well (its bytes are being overwritten) and the slot returns to the free set.
int access_keys(moe_ctx* c, const std::vector<int>& keys, bool prefetch) {
    bool batch_open = false;
    bool used[kFillStreams] = {};
    FillRec fr{nullptr, nullptr};
    int rc = MOE_OK;
    int n_fill = 0;                           // fills of this batch: fill i takes copy stream i % kFillStreams
    const uint64_t batch_seq0 = c->fill_seq;  // fills numbered above this one belong to this batch
    for (int key : keys) {
        ExpertLru::Plan p = c->lru.plan(key, prefetch);
        const bool fill = p.kind == ExpertLru::kFill || p.kind == ExpertLru::kPrefetchFill;
        if (fill) {
            if (c->inject_kind == 1 && c->inject_count > 0) {
                c->inject_count--;
                rc = fail(MOE_E_CUDA, "injected fill failure (layer %d expert %d)", key / c->E, key % c->E);
                break;
            }
            if (!batch_open) {
                fr.start = pool_event(c);
                if (fr.start) cudaEventRecord(fr.start, c->s_copy);
                batch_open = true;
            }
            const int si = n_fill % kFillStreams;
            const cudaStream_t cs = c->s_fill[si];
            cudaError_t e = cudaSuccess;
            if (si > 0 && !used[si]) {
                // an internal stream starts after everything enqueued on s_copy so far
                if (fr.start) e = cudaStreamWaitEvent(cs, fr.start, 0);
                used[si] = true;
            }
            // the slot's previous entry may still be read by an enqueued wave
            const int64_t last = c->slot_last_use[p.slot];
            if (e == cudaSuccess && last >= 0) e = cudaStreamWaitEvent(cs, c->comp_ev[last % kEvRing], 0);
            // a slot filled earlier in this batch (maybe on another stream): after that copy
            const uint64_t prev_fill = static_cast<uint64_t>(c->slot_fill[p.slot]);
            if (e == cudaSuccess && c->slot_fill[p.slot] >= 0 && prev_fill > batch_seq0)
                e = cudaStreamWaitEvent(cs, c->fill_ev[prev_fill % kEvRing], 0);
            if (e == cudaSuccess)
                e = cudaMemcpyAsync(c->arena + static_cast<size_t>(p.slot) * c->entry_elems,
                                    c->pool + static_cast<size_t>(key) * c->entry_elems, c->entry_bytes,
                                    cudaMemcpyHostToDevice, cs);
            if (e != cudaSuccess) {
                rc = fail(MOE_E_CUDA, "fill of layer %d expert %d: %s", key / c->E, key % c->E,
                          cudaGetErrorString(e));
                break;
            }
            // from here on the slot's old bytes are being overwritten
            const uint32_t gen = c->fill_gen[p.slot] + 1;
            CUresult r = write_value_fn()(reinterpret_cast<CUstream>(cs),
                                          reinterpret_cast<CUdeviceptr>(c->fill_flag + p.slot), gen, 0);
            if (c->inject_kind == 4 && c->inject_count > 0) {
                c->inject_count--;
                r = CUDA_ERROR_UNKNOWN;  // injected: report the flag write as failed
            }
            // the generation is used up even if the write failed (it may have landed), so the
            // next fill of the slot waits for a strictly newer one
            c->fill_gen[p.slot] = gen;
            if (r != CUDA_SUCCESS) {
                rc = fail(MOE_E_CUDA, "fill flag write for layer %d expert %d: driver error %d", key / c->E,
                          key % c->E, static_cast<int>(r));
                abandon_slot(c, p);
                break;
            }
        }
        c->lru.commit(p);
        record_event(c, p.kind, key, p.slot, p.victim);
        switch (p.kind) {
            case ExpertLru::kHit: c->stats.expert_reads++; c->stats.hits++; break;
            case ExpertLru::kFill: c->stats.expert_reads++; c->stats.misses++; break;
            case ExpertLru::kPrefetchFill: c->stats.prefetch_fills++; break;
            case ExpertLru::kPrefetchHit: c->stats.prefetch_hits++; break;
        }
        if (fill) {
            c->stats.fill_bytes += c->entry_bytes;
            if (p.victim >= 0) {
                c->stats.evictions++;
                c->slot_host[p.victim] = -1;
            }
            c->slot_host[key] = p.slot;
            // each fill gets its own completion event, so compute can start on the entries
            // that have landed while later copies are still crossing the link
            c->fill_seq++;
            c->slot_fill[p.slot] = c->fill_seq;
            c->table_dirty = true;
            cudaError_t e = cudaEventRecord(c->fill_ev[c->fill_seq % kEvRing], c->s_fill[n_fill % kFillStreams]);
            n_fill++;
            if (e != cudaSuccess) {
                // compute could not be ordered after this copy: the new entry is not usable
                rc = fail(MOE_E_CUDA, "fill event: %s", cudaGetErrorString(e));
                c->lru.release_slot(p.slot);
                c->slot_host[key] = -1;
                break;
            }
        }
    }
    if (batch_open) {
        // s_copy joins the internal streams, so that waiting on s_copy waits for every fill
        for (int si = 1; si < kFillStreams; ++si) {
            if (!used[si]) continue;
            cudaError_t e = cudaEventRecord(c->ev_fill_join[si], c->s_fill[si]);
            if (e == cudaSuccess) e = cudaStreamWaitEvent(c->s_copy, c->ev_fill_join[si], 0);
            if (e != cudaSuccess && rc == MOE_OK) rc = fail(MOE_E_CUDA, "joining the fill streams: %s", cudaGetErrorString(e));
        }
        fr.stop = pool_event(c);
        if (fr.start && fr.stop) {
            cudaEventRecord(fr.stop, c->s_copy);
            c->fill_pending.push_back(fr);
        }
    }
    return rc;
}

// TMA views of the slot arena (they change when the arena is reallocated).
bool make_arena_maps(moe_ctx* c) {
    const uint64_t H = c->H, I = c->I, C = c->C;
    if (c->fp4) return true;  // 4-bit stages are fetched with plain bulk copies
    return make_map(&c->dec_maps.a_gu, c->arena, H, C * 3 * I, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B) &&
           make_map(&c->dec_maps.a_d, c->arena, I, C * 3 * H, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B) &&
           make_map(&c->gemm_maps.b_gu, c->arena, H, C * 3 * I, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B) &&
           make_map(&c->gemm_maps.b_d, c->arena, I, C * 3 * H, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B);
}

int validate_layer(moe_ctx* c, int layer) {
    if (!c) return fail(MOE_E_INVAL, "null context");
    if (layer < 0 || layer >= c->L) return fail(MOE_E_INVAL, "layer %d outside [0, %d)", layer, c->L);
    return MOE_OK;
}

void free_all(moe_ctx* c) {
    if (c->s_comp) cudaStreamSynchronize(c->s_comp);
    if (c->s_copy) cudaStreamSynchronize(c->s_copy);
    for (int si = 1; si < kFillStreams; ++si)
        if (c->s_fill[si]) cudaStreamSynchronize(c->s_fill[si]);
    harvest(c);
    for (auto& r : c->prof_pending) {
        cudaEventDestroy(r.start);
        cudaEventDestroy(r.stop);
    }
    for (auto& r : c->fill_pending) {
        cudaEventDestroy(r.start);
        cudaEventDestroy(r.stop);
    }
    for (cudaEvent_t e : c->ev_pool) cudaEventDestroy(e);
    for (int i = 0; i < kEvRing; ++i) {
        if (c->comp_ev[i]) cudaEventDestroy(c->comp_ev[i]);
        if (c->fill_ev[i]) cudaEventDestroy(c->fill_ev[i]);
    }
    for (int i = 0; i < kStageRing; ++i)
        if (c->stage_ev[i]) cudaEventDestroy(c->stage_ev[i]);
    if (c->ev_d2h) cudaEventDestroy(c->ev_d2h);
    if (c->ev_fork) cudaEventDestroy(c->ev_fork);
    if (c->ev_join) cudaEventDestroy(c->ev_join);
    for (int si = 1; si < kFillStreams; ++si)
        if (c->ev_fill_join[si]) cudaEventDestroy(c->ev_fill_join[si]);
    void* dev_ptrs[] = {c->arena, c->slot_dev, c->logits, c->offsets, c->perm, c->inv_perm, c->active,
                        c->perm_cells, c->perm_done, c->n_active, c->w_perm, c->pair_out, c->x_perm, c->h_perm, c->status, c->work_dev,
                        c->dec_ws,   c->dec_cnt, c->dec_ready, c->dec_done, c->fill_flag, c->d_lru,   c->d_prev, c->d_next,  c->d_key,
                        c->d_stats,  c->d_trace, c->d_fill_list, c->d_work, c->d_order, c->d_hdr, c->d_keys,
                        c->d_iota};
    for (void* p : dev_ptrs)
        if (p) cudaFree(p);
    void* host_ptrs[] = {c->pool, c->idx_host, c->status_host, c->table_stage, c->work_stage};
    for (void* p : host_ptrs)
        if (p) cudaFreeHost(p);
    if (c->own_comp && c->s_comp) cudaStreamDestroy(c->s_comp);
    if (c->own_copy && c->s_copy) cudaStreamDestroy(c->s_copy);
    for (int si = 1; si < kFillStreams; ++si)
        if (c->s_fill[si]) cudaStreamDestroy(c->s_fill[si]);
    delete c;
}

}  // namespace

namespace {

// The decode expert kernels for the context's weight format: a work list with its size given
// here (n_work, n_units, S) or read on the device from dyn = {n_work, n_units, S}.
cudaError_t run_gateup(moe_ctx* c, const GemvWork* work, int n_work, int n_units, int S, const int* dyn,
                       const int32_t* slot_row, uint64_t fill_wait_ns) {
    if (c->fp4)
        return moe::launch_decode_fp4(c->fp4_fmt, true, c->dec_maps, reinterpret_cast<const uint8_t*>(c->arena), c->entry_bytes,
                                      work, n_work, n_units, S, dyn, slot_row, c->fill_flag, c->H, c->I, c->h_perm,
                                      nullptr, nullptr, c->dec_ws, c->dec_cnt, c->status, fill_wait_ns, c->num_sms,
                                      c->s_comp);
    if (dyn)
        return moe::launch_decode_gateup_dyn(c->dec_maps, work, dyn, slot_row, c->H, c->I, c->h_perm, c->dec_ws,
                                             c->dec_cnt, c->status, c->num_sms, c->s_comp);
    return moe::launch_decode_gateup(c->dec_maps, work, n_work, n_units, S, slot_row, c->fill_flag, c->H, c->I,
                                     c->h_perm, c->dec_ws, c->dec_cnt, c->status, fill_wait_ns, c->num_sms, c->s_comp);
}

cudaError_t run_down(moe_ctx* c, const GemvWork* work, int n_work, int n_units, int S, const int* dyn,
                     const int32_t* slot_row, uint64_t fill_wait_ns) {
    if (c->fp4)
        return moe::launch_decode_fp4(c->fp4_fmt, false, c->dec_maps, reinterpret_cast<const uint8_t*>(c->arena), c->entry_bytes,
                                      work, n_work, n_units, S, dyn, slot_row, c->fill_flag, c->H, c->I, nullptr,
                                      c->w_perm, c->pair_out, c->dec_ws, c->dec_cnt, c->status, fill_wait_ns,
                                      c->num_sms, c->s_comp);
    if (dyn)
        return moe::launch_decode_down_dyn(c->dec_maps, work, dyn, slot_row, c->H, c->I, c->w_perm, c->pair_out,
                                           c->dec_ws, c->dec_cnt, c->status, c->num_sms, c->s_comp);
    return moe::launch_decode_down(c->dec_maps, work, n_work, n_units, S, slot_row, c->fill_flag, c->H, c->I,
                                   c->w_perm, c->pair_out, c->dec_ws, c->dec_cnt, c->status, fill_wait_ns, c->num_sms,
                                   c->s_comp);
}

// Bytes of one weight as stored: 2 (bf16), 17/32 (MXFP4: E2M1 half byte plus a scale per 32) or
// 9/16 (NVFP4: a scale per 16; the 16-byte tensor-scale trailer is not counted).
double weight_bytes(const moe_ctx* c) {
    if (!c->fp4) return 2.0;
    return c->fp4_fmt == moe::kFp4Nv ? 9.0 / 16.0 : 17.0 / 32.0;
}

// The device policy on one key set, then the fills it chose on the copy stream (forked from
// and, when `join`, joined back into the compute stream). No host wait: capturable.
int dev_policy_run(moe_ctx* c, moe::DevPolicyArgs a, bool join) {
    a.state = c->d_lru;
    a.lru_prev = c->d_prev;
    a.lru_next = c->d_next;
    a.lru_key = c->d_key;
    a.slot_of = c->slot_dev;
    a.C = c->C;
    a.E = c->E;
    a.H = c->H;
    a.I = c->I;
    a.num_sms = c->num_sms;
    a.fill_list = c->d_fill_list;
    a.order = c->d_order;
    a.hdr = c->d_hdr;
    a.stats = c->d_stats;
    a.trace = c->d_trace;
    a.trace_cap = c->d_trace_cap;
    a.entry_bytes = c->entry_bytes;
    {
        ProfScope ps(c, kPolicy, 0.0, 0.0);
        CUDA_TRY(moe::launch_policy(a, c->s_comp));
    }
    CUDA_TRY(cudaEventRecord(c->ev_fork, c->s_comp));
    CUDA_TRY(cudaStreamWaitEvent(c->s_copy, c->ev_fork, 0));
    CUDA_TRY(moe::launch_fill(c->pool_dev, c->arena, c->d_fill_list, &c->d_hdr->n_fill, c->entry_bytes, c->num_sms,
                              c->s_copy));
    CUDA_TRY(cudaEventRecord(c->ev_join, c->s_copy));
    if (join) CUDA_TRY(cudaStreamWaitEvent(c->s_comp, c->ev_join, 0));
    return MOE_OK;
}

// The permutation of the T * k pairs and the gather of their token rows into x_perm: one
// launch for decode batches, the counting sort and a row-gather kernel for larger ones.
int permute_and_gather(moe_ctx* c, const void* x, int T, const int32_t* idx, const float* w) {
    const int P = T * c->k, E = c->E, H = c->H;
    const double perm_bytes = 8.0 * P + 12.0 * P + 8.0 * E;
    // the gather's bytes: each of the T rows read once (L2 serves its k - 1 repeats), each of
    // the P permuted rows written once
    const double gather_bytes = 2.0 * T * H + 2.0 * P * H;
    if (moe::permute_gathers_rows(P)) {
        ProfScope ps(c, kPermute, perm_bytes + gather_bytes, 0.0);
        CUDA_TRY(moe::launch_permute_gather(idx, w, static_cast<const uint16_t*>(x), P, c->k, E, H, c->offsets,
                                            c->perm, c->inv_perm, c->w_perm, c->active, c->n_active, c->x_perm,
                                            c->status, c->s_comp));
        return MOE_OK;
    }
    {
        ProfScope ps(c, kPermute, perm_bytes, 0.0);
        CUDA_TRY(moe::launch_permute(idx, w, P, E, c->offsets, c->perm, c->inv_perm, c->w_perm, c->active,
                                     c->n_active, c->status, c->perm_cells, c->perm_done, c->s_comp));
    }
    ProfScope ps(c, kGather, gather_bytes, 0.0);
    CUDA_TRY(moe::launch_gather_rows(static_cast<const uint16_t*>(x), c->perm, P, c->k, H, c->x_perm, c->s_comp));
    return MOE_OK;
}

// Decode forward with the device-resident policy: permutation, then per wave the policy,
// the fills (copy stream) alongside the resident experts' kernels, the filled experts'
// kernels after the fills, then the combine. Enqueues only; never waits on the host.
int forward_device(moe_ctx* c, int layer, const void* x, const float* resid, float* out, int T, const int32_t* idx,
                   const float* w) {
    const int P = T * c->k, E = c->E, H = c->H;
    if (c->path == MOE_PATH_GEMM)
        return fail(MOE_E_INVAL, "the device-resident policy runs the decode kernels only (MOE_PATH_GEMM unsupported)");
    int rc = permute_and_gather(c, x, T, idx, w);
    if (rc) return rc;
    const int32_t* slot_row = c->slot_dev + static_cast<size_t>(layer) * E;
    GemvWork* wh = c->d_work;
    GemvWork* wm = c->d_work + 2 * (E + 1);
    const int waves = (std::min(P, E) + c->C - 1) / c->C;  // the most the routed set can need
    for (int wv = 0; wv < waves; ++wv) {
        moe::DevPolicyArgs a{};
        a.layer = layer;
        a.active = c->active;
        a.n_active = c->n_active;
        a.wave = wv;
        a.offsets = c->offsets;
        a.work_hit = wh;
        a.work_miss = wm;
        int rc = dev_policy_run(c, a, false);
        if (rc) return rc;
        {
            ProfScope ps(c, kDecodeGateUp, 0.0, 0.0);
            CUDA_TRY(run_gateup(c, wh, 0, 0, 1, c->d_hdr->hit_gu, slot_row, 0));
        }
        {
            ProfScope ps(c, kDecodeDown, 0.0, 0.0);
            CUDA_TRY(run_down(c, wh + (E + 1), 0, 0, 1, c->d_hdr->hit_d, slot_row, 0));
        }
        CUDA_TRY(cudaStreamWaitEvent(c->s_comp, c->ev_join, 0));
        {
            ProfScope ps(c, kDecodeGateUp, 0.0, 0.0);
            CUDA_TRY(run_gateup(c, wm, 0, 0, 1, c->d_hdr->miss_gu, slot_row, 0));
        }
        {
            ProfScope ps(c, kDecodeDown, 0.0, 0.0);
            CUDA_TRY(run_down(c, wm + (E + 1), 0, 0, 1, c->d_hdr->miss_d, slot_row, 0));
        }
    }
    {
        ProfScope ps(c, kCombine, 4.0 * P * H + 8.0 * T * H + 4.0 * P, 1.0 * P * H);
        CUDA_TRY(moe::launch_combine(c->pair_out, c->inv_perm, resid, out, T, c->k, H, c->s_comp));
    }
    return MOE_OK;
}

// Wait for both streams (bounded) without touching the device status.
int drain(moe_ctx* c) {
    cudaEvent_t e1 = pool_event(c), e2 = pool_event(c);
    if (!e1 || !e2) return fail(MOE_E_CUDA, "event creation failed");
    CUDA_TRY(cudaEventRecord(e1, c->s_comp));
    CUDA_TRY(cudaEventRecord(e2, c->s_copy));
    int rc = wait_event(c, e1, "compute stream");
    if (!rc) rc = wait_event(c, e2, "copy stream");
    c->ev_pool.push_back(e1);
    c->ev_pool.push_back(e2);
    return rc;
}

// The device policy's recency list into the host LRU (the device owns it between calls).
int dev_state_pull(moe_ctx* c) {
    std::vector<int> prev(c->C), next(c->C), key(c->C);
    moe::DevLruState st{};
    CUDA_TRY(cudaMemcpy(prev.data(), c->d_prev, c->C * sizeof(int), cudaMemcpyDeviceToHost));
    CUDA_TRY(cudaMemcpy(next.data(), c->d_next, c->C * sizeof(int), cudaMemcpyDeviceToHost));
    CUDA_TRY(cudaMemcpy(key.data(), c->d_key, c->C * sizeof(int), cudaMemcpyDeviceToHost));
    CUDA_TRY(cudaMemcpy(&st, c->d_lru, sizeof(st), cudaMemcpyDeviceToHost));
    c->lru.import_state(prev, next, key, st.head, st.tail, st.n_used);
    return MOE_OK;
}

int dev_state_push(moe_ctx* c) {
    std::vector<int> prev, next, key;
    moe::DevLruState st{};
    c->lru.export_state(&prev, &next, &key, &st.head, &st.tail, &st.n_used);
    CUDA_TRY(cudaMemcpy(c->d_prev, prev.data(), c->C * sizeof(int), cudaMemcpyHostToDevice));
    CUDA_TRY(cudaMemcpy(c->d_next, next.data(), c->C * sizeof(int), cudaMemcpyHostToDevice));
    CUDA_TRY(cudaMemcpy(c->d_key, key.data(), c->C * sizeof(int), cudaMemcpyHostToDevice));
    CUDA_TRY(cudaMemcpy(c->d_lru, &st, sizeof(st), cudaMemcpyHostToDevice));
    return MOE_OK;
}

}  // namespace

namespace moe {
// Record a thread-local error message for moe_last_error() and return `code`.
int set_error(int code, const char* msg) { return fail(code, "%s", msg); }
}  // namespace moe

extern "C" {

const char* moe_last_error(void) { return g_last_error.c_str(); }

uint64_t moe_entry_bytes(const moe_ctx* c) { return c ? c->entry_bytes : 0; }

int moe_cache_init(const moe_config_t* cfg, void* stream_compute, void* stream_copy, moe_ctx** out) {
    g_last_error.clear();
    if (!cfg || !out) return fail(MOE_E_INVAL, "null argument");
    *out = nullptr;
    const moe_config_t& f = *cfg;
    if (f.num_layers < 1 || f.num_experts < 1 || f.num_experts > 1024 || f.top_k < 1 || f.top_k > 32 ||
        f.top_k > f.num_experts || f.hidden < 256 || f.hidden % 256 || f.inter < 128 || f.inter % 128 ||
        f.max_tokens < 1)
        return fail(MOE_E_INVAL, "shape outside the limits (hidden %% 256, inter %% 128, 1 <= k <= min(E, 32), "
                                 "E <= 1024, max_tokens >= 1)");
    if ((f.flags & MOE_MXFP4) && (f.flags & MOE_NVFP4))
        return fail(MOE_E_INVAL, "MOE_MXFP4 and MOE_NVFP4 are exclusive");
    if (f.capacity < 1) return fail(MOE_E_CAPACITY, "capacity must be >= 1");
    if ((f.flags & MOE_PREFILL_DB) && f.capacity < 2 * f.num_experts)
        return fail(MOE_E_CAPACITY, "double buffering needs capacity >= 2 * num_experts (%d < %d)", f.capacity,
                    2 * f.num_experts);
    const uint64_t keys = static_cast<uint64_t>(f.num_layers) * f.num_experts;
    const uint64_t entry_elems = 3ull * f.hidden * f.inter;
    if (static_cast<uint64_t>(f.capacity) * 3ull * f.inter >= (1ull << 31) ||
        static_cast<uint64_t>(f.capacity) * 3ull * f.hidden >= (1ull << 31) || keys >= (1ull << 31))
        return fail(MOE_E_INVAL, "arena too large for 32-bit row coordinates");
    if (!encode_fn()) return fail(MOE_E_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    if (!write_value_fn()) return fail(MOE_E_CUDA, "cuStreamWriteValue32 is not available from the driver");

    moe_ctx* c = new moe_ctx();
    c->cfg = f;
    c->L = f.num_layers;
    c->E = f.num_experts;
    c->H = f.hidden;
    c->I = f.inter;
    c->k = f.top_k;
    c->C = f.capacity;
    c->Tmax = f.max_tokens;
    c->Pmax = f.max_tokens * f.top_k;
    c->fp4 = (f.flags & (MOE_MXFP4 | MOE_NVFP4)) != 0;
    c->fp4_fmt = (f.flags & MOE_NVFP4) ? moe::kFp4Nv : ((f.flags & MOE_MXFP4) ? moe::kFp4Mx : 0);
    // bf16: 2 bytes per weight; MXFP4: E2M1 halves plus one scale byte per 32 weights; NVFP4:
    // E2M1 halves, one scale byte per 16 weights and a 16-byte trailer of tensor scales
    if (!c->fp4) c->entry_bytes = entry_elems * 2;
    else if (c->fp4_fmt == moe::kFp4Mx) c->entry_bytes = entry_elems / 2 + entry_elems / 32;
    else c->entry_bytes = entry_elems / 2 + entry_elems / 16 + 16;
    c->entry_elems = c->entry_bytes / 2;  // 16-bit units (pool and arena pointers are uint16_t)
    c->lru.reset(c->C, static_cast<int>(keys));
    c->slot_host.assign(keys, -1);
    c->slot_last_use.assign(c->C, -1);
    c->slot_fill.assign(c->C, -1);
    c->fill_gen.assign(c->C, 0);
    if (f.flags & MOE_TRACE) c->trace.resize(f.trace_capacity ? f.trace_capacity : (1u << 20));

#define INIT_TRY(call)                                                                          \
    do {                                                                                        \
        cudaError_t e_ = (call);                                                                \
        if (e_ != cudaSuccess) {                                                                \
            int code_ = (e_ == cudaErrorMemoryAllocation) ? MOE_E_NOMEM : MOE_E_CUDA;           \
            fail(code_, "%s: %s", #call, cudaGetErrorString(e_));                               \
            std::string msg_ = g_last_error;                                                    \
            free_all(c);                                                                        \
            g_last_error = msg_;                                                                \
            return code_;                                                                       \
        }                                                                                       \
    } while (0)

    INIT_TRY(cudaGetDevice(&c->dev));
    INIT_TRY(cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, c->dev));
    if (stream_compute) {
        c->s_comp = static_cast<cudaStream_t>(stream_compute);
    } else {
        INIT_TRY(cudaStreamCreateWithFlags(&c->s_comp, cudaStreamNonBlocking));
        c->own_comp = true;
    }
    if (stream_copy) {
        c->s_copy = static_cast<cudaStream_t>(stream_copy);
    } else {
        INIT_TRY(cudaStreamCreateWithFlags(&c->s_copy, cudaStreamNonBlocking));
        c->own_copy = true;
    }
    c->s_fill[0] = c->s_copy;
    for (int si = 1; si < kFillStreams; ++si) {
        INIT_TRY(cudaStreamCreateWithFlags(&c->s_fill[si], cudaStreamNonBlocking));
        INIT_TRY(cudaEventCreateWithFlags(&c->ev_fill_join[si], cudaEventDisableTiming));
    }
    const size_t pool_bytes = keys * c->entry_bytes;
    c->dev_policy = (f.flags & MOE_DEVICE_POLICY) != 0;
    INIT_TRY(cudaHostAlloc(reinterpret_cast<void**>(&c->pool), pool_bytes,
                           cudaHostAllocPortable | (c->dev_policy ? cudaHostAllocMapped : 0)));
    if (c->dev_policy) INIT_TRY(cudaHostGetDevicePointer(&c->pool_dev, c->pool, 0));
    std::memset(c->pool, 0, pool_bytes);
    INIT_TRY(cudaMalloc(&c->arena, static_cast<size_t>(c->C) * c->entry_bytes));
    INIT_TRY(cudaMalloc(&c->slot_dev, keys * sizeof(int32_t)));
    INIT_TRY(cudaMalloc(&c->logits, static_cast<size_t>(c->Tmax) * c->E * sizeof(float)));
    INIT_TRY(cudaMalloc(&c->offsets, (c->E + 1) * sizeof(int32_t)));
    INIT_TRY(cudaMalloc(&c->active, c->E * sizeof(int32_t)));
    INIT_TRY(cudaMalloc(&c->n_active, sizeof(int32_t)));
    INIT_TRY(cudaMalloc(&c->perm, c->Pmax * sizeof(int32_t)));
    INIT_TRY(cudaMalloc(&c->inv_perm, c->Pmax * sizeof(int32_t)));
    INIT_TRY(cudaMalloc(&c->perm_cells, 2ull * moe::permute_grid(c->Pmax) * c->E * sizeof(int32_t)));
    INIT_TRY(cudaMalloc(&c->perm_done, sizeof(unsigned)));
    INIT_TRY(cudaMemset(c->perm_done, 0, sizeof(unsigned)));
    INIT_TRY(cudaMalloc(&c->w_perm, c->Pmax * sizeof(float)));
    INIT_TRY(cudaMalloc(&c->x_perm, static_cast<size_t>(c->Pmax) * c->H * 2));
    INIT_TRY(cudaMalloc(&c->h_perm, static_cast<size_t>(c->Pmax) * c->I * 2));
    INIT_TRY(cudaMalloc(&c->pair_out, static_cast<size_t>(c->Pmax) * c->H * sizeof(float)));
    INIT_TRY(cudaMalloc(&c->status, sizeof(int)));
    INIT_TRY(cudaMalloc(&c->work_dev, kWorkEntries(c->E) * sizeof(GemvWork)));
    INIT_TRY(cudaMalloc(&c->dec_ws, static_cast<size_t>(moe::kDecodeSplitUnits) * moe::kDecodeTileFloats * sizeof(float)));
    INIT_TRY(cudaMalloc(&c->dec_cnt, moe::kDecodeSplitUnits * sizeof(int)));
    c->dec_chunk_slots = moe::decode_fused_chunk_slots(c->E, c->Pmax);
    INIT_TRY(cudaMalloc(&c->dec_ready, c->dec_chunk_slots * sizeof(int)));
    INIT_TRY(cudaMalloc(&c->dec_done, c->dec_chunk_slots * sizeof(int)));
    INIT_TRY(cudaMemset(c->dec_ready, 0, c->dec_chunk_slots * sizeof(int)));
    INIT_TRY(cudaMemset(c->dec_done, 0, c->dec_chunk_slots * sizeof(int)));
    INIT_TRY(cudaMalloc(&c->fill_flag, static_cast<size_t>(c->C) * sizeof(uint32_t)));
    INIT_TRY(cudaMemset(c->fill_flag, 0, static_cast<size_t>(c->C) * sizeof(uint32_t)));
    INIT_TRY(cudaMemset(c->dec_cnt, 0, moe::kDecodeSplitUnits * sizeof(int)));
    INIT_TRY(cudaMemset(c->status, 0, sizeof(int)));
    INIT_TRY(cudaMemset(c->x_perm, 0, static_cast<size_t>(c->Pmax) * c->H * 2));
    INIT_TRY(cudaMemset(c->h_perm, 0, static_cast<size_t>(c->Pmax) * c->I * 2));
    INIT_TRY(cudaHostAlloc(reinterpret_cast<void**>(&c->idx_host), c->Pmax * sizeof(int32_t), 0));
    INIT_TRY(cudaHostAlloc(reinterpret_cast<void**>(&c->status_host), sizeof(int), 0));
    *c->status_host = 0;
    INIT_TRY(cudaHostAlloc(reinterpret_cast<void**>(&c->table_stage), kStageRing * keys * sizeof(int32_t), 0));
    INIT_TRY(cudaHostAlloc(reinterpret_cast<void**>(&c->work_stage),
                           static_cast<size_t>(kStageRing) * kWorkEntries(c->E) * sizeof(GemvWork), 0));
    for (int i = 0; i < kStageRing; ++i) {
        INIT_TRY(cudaEventCreateWithFlags(&c->stage_ev[i], cudaEventDisableTiming));
        INIT_TRY(cudaEventRecord(c->stage_ev[i], c->s_comp));
    }
    for (int i = 0; i < kEvRing; ++i) {
        INIT_TRY(cudaEventCreateWithFlags(&c->comp_ev[i], cudaEventDisableTiming));
        INIT_TRY(cudaEventCreateWithFlags(&c->fill_ev[i], cudaEventDisableTiming));
    }
    INIT_TRY(cudaEventCreateWithFlags(&c->ev_d2h, cudaEventDisableTiming));
    if (c->dev_policy) {
        const size_t Cn = static_cast<size_t>(c->C);
        INIT_TRY(cudaMalloc(&c->d_lru, sizeof(moe::DevLruState)));
        INIT_TRY(cudaMalloc(&c->d_prev, Cn * sizeof(int)));
        INIT_TRY(cudaMalloc(&c->d_next, Cn * sizeof(int)));
        INIT_TRY(cudaMalloc(&c->d_key, Cn * sizeof(int)));
        INIT_TRY(cudaMalloc(&c->d_stats, sizeof(moe::DevStats)));
        c->d_trace_cap = (f.flags & MOE_TRACE) ? (f.trace_capacity ? f.trace_capacity : (1u << 20)) : 0;
        if (c->d_trace_cap) INIT_TRY(cudaMalloc(&c->d_trace, c->d_trace_cap * sizeof(moe::DevEvent)));
        INIT_TRY(cudaMalloc(&c->d_fill_list, Cn * sizeof(int2)));
        INIT_TRY(cudaMalloc(&c->d_work, 4 * (static_cast<size_t>(c->E) + 1) * sizeof(GemvWork)));
        INIT_TRY(cudaMalloc(&c->d_order, 2 * Cn * sizeof(int)));
        INIT_TRY(cudaMalloc(&c->d_hdr, sizeof(moe::WaveHdr)));
        INIT_TRY(cudaMalloc(&c->d_keys, c->E * sizeof(int32_t)));
        INIT_TRY(cudaMalloc(&c->d_iota, c->E * sizeof(int32_t)));
        std::vector<int32_t> iota(c->E);
        for (int e = 0; e < c->E; ++e) iota[e] = e;
        INIT_TRY(cudaMemcpy(c->d_iota, iota.data(), c->E * sizeof(int32_t), cudaMemcpyHostToDevice));
        const moe::DevLruState st0{-1, -1, 0, 0};
        INIT_TRY(cudaMemcpy(c->d_lru, &st0, sizeof(st0), cudaMemcpyHostToDevice));
        INIT_TRY(cudaMemset(c->d_prev, 0xff, Cn * sizeof(int)));
        INIT_TRY(cudaMemset(c->d_next, 0xff, Cn * sizeof(int)));
        INIT_TRY(cudaMemset(c->d_key, 0xff, Cn * sizeof(int)));
        INIT_TRY(cudaMemset(c->d_stats, 0, sizeof(moe::DevStats)));
        INIT_TRY(cudaMemset(c->d_hdr, 0, sizeof(moe::WaveHdr)));
        INIT_TRY(cudaEventCreateWithFlags(&c->ev_fork, cudaEventDisableTiming));
        INIT_TRY(cudaEventCreateWithFlags(&c->ev_join, cudaEventDisableTiming));
    }

    // TMA views. Arena rows: [C*3I x H] for gate/up, [C*3H x I] for down.
    const uint64_t H = c->H, I = c->I, P = c->Pmax;
    bool ok = make_arena_maps(c) &&
              make_map(&c->dec_maps.b_x, c->x_perm, H, P, 64, 16, CU_TENSOR_MAP_SWIZZLE_128B) &&
              make_map(&c->dec_maps.b_h, c->h_perm, I, P, 64, 16, CU_TENSOR_MAP_SWIZZLE_128B) &&
              make_map(&c->gemm_maps.a_x, c->x_perm, H, P, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B) &&
              make_map(&c->gemm_maps.a_h, c->h_perm, I, P, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B);
    if (!ok) {
        free_all(c);
        return fail(MOE_E_CUDA, "cuTensorMapEncodeTiled rejected a tensor view");
    }
    if (upload_table(c) != MOE_OK) {
        std::string msg = g_last_error;
        free_all(c);
        g_last_error = msg;
        return MOE_E_CUDA;
    }
    INIT_TRY(cudaStreamSynchronize(c->s_comp));
#undef INIT_TRY
    *out = c;
    return MOE_OK;
}

void moe_cache_destroy(moe_ctx* c) {
    if (!c) return;
    cudaSetDevice(c->dev);
    free_all(c);
}

void* moe_host_entry(moe_ctx* c, int layer, int expert) {
    if (!c || layer < 0 || layer >= c->L || expert < 0 || expert >= c->E) return nullptr;
    return c->pool + (static_cast<size_t>(layer) * c->E + expert) * c->entry_elems;
}

int moe_set_path(moe_ctx* c, int path) {
    if (!c) return fail(MOE_E_INVAL, "null context");
    if (path != MOE_PATH_AUTO && path != MOE_PATH_GEMV && path != MOE_PATH_GEMM && path != MOE_PATH_GEMV_UNFUSED)
        return fail(MOE_E_INVAL, "unknown path %d", path);
    c->path = path;
    return MOE_OK;
}

int moe_cache_resize(moe_ctx* c, int new_C) {
    g_last_error.clear();
    if (!c) return fail(MOE_E_INVAL, "null context");
    if (new_C < 1) return fail(MOE_E_INVAL, "capacity %d < 1", new_C);
    if ((c->cfg.flags & MOE_PREFILL_DB) && new_C < 2 * c->E)
        return fail(MOE_E_CAPACITY, "double buffering needs capacity >= 2 * num_experts (%d < %d)", new_C, 2 * c->E);
    if (static_cast<uint64_t>(new_C) * 3ull * c->I >= (1ull << 31) ||
        static_cast<uint64_t>(new_C) * 3ull * c->H >= (1ull << 31))
        return fail(MOE_E_INVAL, "arena too large for 32-bit row coordinates");
    CUDA_TRY(cudaSetDevice(c->dev));
    int rc = drain(c);  // the safe point: nothing enqueued reads or writes the arena any more
    if (rc) return rc;
    harvest(c);
    if (c->dev_policy && (rc = dev_state_pull(c))) return rc;

    ExpertLru next = c->lru;
    std::vector<std::pair<int, int>> evicted, moved;
    next.resize(new_C, &evicted, &moved);

    // every new buffer first, so a failed allocation leaves the cache as it was
    uint16_t* arena2 = nullptr;
    uint32_t* flag2 = nullptr;
    int *prev2 = nullptr, *next2 = nullptr, *key2 = nullptr, *order2 = nullptr;
    int2* fl2 = nullptr;
    auto release = [&]() {
        void* ps[] = {arena2, flag2, prev2, next2, key2, order2, fl2};
        for (void* p : ps)
            if (p) cudaFree(p);
    };
    const size_t Cn = static_cast<size_t>(new_C);
    bool ok = cudaMalloc(&arena2, Cn * c->entry_bytes) == cudaSuccess &&
              cudaMalloc(&flag2, Cn * sizeof(uint32_t)) == cudaSuccess;
    if (ok && c->dev_policy)
        ok = cudaMalloc(&prev2, Cn * sizeof(int)) == cudaSuccess && cudaMalloc(&next2, Cn * sizeof(int)) == cudaSuccess &&
             cudaMalloc(&key2, Cn * sizeof(int)) == cudaSuccess &&
             cudaMalloc(&order2, 2 * Cn * sizeof(int)) == cudaSuccess &&
             cudaMalloc(&fl2, Cn * sizeof(int2)) == cudaSuccess;
    if (!ok) {
        cudaGetLastError();
        release();
        return fail(MOE_E_NOMEM, "could not allocate a %d-entry arena", new_C);
    }
    // survivors into their new slots (slot r of the new arena holds next.key_in(r))
    for (int r = 0; r < next.used(); ++r) {
        const int old = c->lru.slot_of(next.key_in(r));
        cudaError_t e = cudaMemcpyAsync(arena2 + static_cast<size_t>(r) * c->entry_elems,
                                        c->arena + static_cast<size_t>(old) * c->entry_elems, c->entry_bytes,
                                        cudaMemcpyDeviceToDevice, c->s_comp);
        if (e != cudaSuccess) {
            release();
            return fail(MOE_E_CUDA, "moving a cache entry: %s", cudaGetErrorString(e));
        }
    }
    cudaError_t e = cudaMemsetAsync(flag2, 0, Cn * sizeof(uint32_t), c->s_comp);
    if (e == cudaSuccess) e = cudaStreamSynchronize(c->s_comp);
    if (e != cudaSuccess) {
        release();
        return fail(MOE_E_CUDA, "resize copies: %s", cudaGetErrorString(e));
    }
    // commit
    cudaFree(c->arena);
    cudaFree(c->fill_flag);
    c->arena = arena2;
    c->fill_flag = flag2;
    c->lru = next;
    c->C = new_C;
    c->cfg.capacity = new_C;
    c->fill_gen.assign(new_C, 0);
    c->slot_last_use.assign(new_C, -1);
    c->slot_fill.assign(new_C, -1);
    for (size_t k = 0; k < c->slot_host.size(); ++k) c->slot_host[k] = c->lru.slot_of(static_cast<int>(k));
    c->table_dirty = true;
    if (c->dev_policy) {
        cudaFree(c->d_prev);
        cudaFree(c->d_next);
        cudaFree(c->d_key);
        cudaFree(c->d_order);
        cudaFree(c->d_fill_list);
        c->d_prev = prev2;
        c->d_next = next2;
        c->d_key = key2;
        c->d_order = order2;
        c->d_fill_list = fl2;
        if ((rc = dev_state_push(c))) return rc;
    }
    if (!make_arena_maps(c)) return fail(MOE_E_CUDA, "cuTensorMapEncodeTiled rejected the resized arena");
    if ((rc = upload_table(c))) return rc;
    // trace and counters
    if (c->dev_policy) {
        moe::DevStats d{};
        CUDA_TRY(cudaMemcpy(&d, c->d_stats, sizeof(d), cudaMemcpyDeviceToHost));
        for (const auto& kv : evicted) {
            if (c->d_trace_cap) {
                const moe::DevEvent ev{MOE_EV_RESIZE_EVICT, kv.first / c->E, kv.first % c->E, kv.second, -1, -1};
                CUDA_TRY(cudaMemcpy(c->d_trace + d.trace_len % c->d_trace_cap, &ev, sizeof(ev),
                                    cudaMemcpyHostToDevice));
            }
            d.trace_len++;
            d.resize_evictions++;
        }
        CUDA_TRY(cudaMemcpy(c->d_stats, &d, sizeof(d), cudaMemcpyHostToDevice));
    } else {
        for (const auto& kv : evicted) {
            record_event(c, MOE_EV_RESIZE_EVICT, kv.first, kv.second, -1);
            c->stats.resize_evictions++;
        }
    }
    CUDA_TRY(cudaStreamSynchronize(c->s_comp));
    return MOE_OK;
}

int moe_set_profile(moe_ctx* c, int on) {
    if (!c) return fail(MOE_E_INVAL, "null context");
    if (on) c->cfg.flags |= MOE_PROFILE;
    else c->cfg.flags &= ~MOE_PROFILE;
    return MOE_OK;
}

int moe_resident_slot(moe_ctx* c, int layer, int expert) {
    if (!c || layer < 0 || layer >= c->L || expert < 0 || expert >= c->E) return -1;
    if (c->dev_policy) {
        int32_t s = -1;
        if (cudaSetDevice(c->dev) != cudaSuccess || drain(c) != MOE_OK ||
            cudaMemcpy(&s, c->slot_dev + static_cast<size_t>(layer) * c->E + expert, sizeof(s),
                       cudaMemcpyDeviceToHost) != cudaSuccess)
            return -1;
        return s;
    }
    return c->lru.slot_of(layer * c->E + expert);
}

int moe_debug_inject(moe_ctx* c, int kind, int count) {
    if (!c) return fail(MOE_E_INVAL, "null context");
    if (kind < 0 || kind > 4 || count < 0) return fail(MOE_E_INVAL, "bad injection");
    c->inject_kind = kind;
    c->inject_count = kind ? count : 0;
    return MOE_OK;
}

static int route_impl(moe_ctx* c, int layer, const void* x, int T, const float* Wr, const float* b,
                      const int32_t* forced, int32_t* idx, float* w, float* logits) {
    g_last_error.clear();
    int rc = validate_layer(c, layer);
    if (rc) return rc;
    if (T < 0 || T > c->Tmax) return fail(MOE_E_INVAL, "T=%d outside [0, %d]", T, c->Tmax);
    if (T == 0) return MOE_OK;
    if (!x || !Wr || !idx || !w) return fail(MOE_E_INVAL, "null device pointer");
    CUDA_TRY(cudaSetDevice(c->dev));
    float* z = logits ? logits : c->logits;
    {
        ProfScope ps(c, kRouterLogits, 4.0 * c->E * c->H + 2.0 * T * c->H + 4.0 * T * c->E,
                     2.0 * T * c->E * c->H);
        CUDA_TRY(moe::launch_router_logits(static_cast<const uint16_t*>(x), Wr, b, T, c->H, c->E, z, c->s_comp));
    }
    {
        ProfScope ps(c, kRouterTopk, 4.0 * T * c->E + 8.0 * T * c->k, 0.0);
        CUDA_TRY(moe::launch_router_topk(z, T, c->E, c->k, forced, idx, w, c->status, c->s_comp));
    }
    return MOE_OK;
}

int moe_route(moe_ctx* c, int layer, const void* x, int T, const float* Wr, const float* b, int32_t* idx, float* w,
              float* logits) {
    return route_impl(c, layer, x, T, Wr, b, nullptr, idx, w, logits);
}

int moe_route_forced(moe_ctx* c, int layer, const void* x, int T, const float* Wr, const float* b,
                     const int32_t* forced, int32_t* idx, float* w, float* logits) {
    if (!forced && T > 0) return fail(MOE_E_INVAL, "null forced sets");
    return route_impl(c, layer, x, T, Wr, b, forced, idx, w, logits);
}

int moe_cache_fill(moe_ctx* c, int layer, const int32_t* idx_host, int n, int mode) {
    g_last_error.clear();
    int rc = validate_layer(c, layer);
    if (rc) return rc;
    CUDA_TRY(cudaSetDevice(c->dev));
    if (c->dev_policy) {
        moe::DevPolicyArgs a{};
        a.layer = layer;
        if (mode == MOE_FILL_FULL_LAYER) {
            if (c->C < c->E) return fail(MOE_E_CAPACITY, "a whole layer (%d) does not fit in %d slots", c->E, c->C);
            a.keys = c->d_iota;
            a.n_keys = c->E;
            a.prefetch = 1;
        } else if (mode == MOE_FILL_DEMAND) {
            if (n < 0 || (n > 0 && !idx_host)) return fail(MOE_E_INVAL, "bad index list");
            std::vector<char> used(c->E, 0);
            for (int i = 0; i < n; ++i) {
                if (idx_host[i] < 0 || idx_host[i] >= c->E)
                    return fail(MOE_E_INVAL, "expert id %d out of range", idx_host[i]);
                used[idx_host[i]] = 1;
            }
            std::vector<int32_t> ids;
            for (int e = 0; e < c->E; ++e)
                if (used[e]) ids.push_back(e);
            if (static_cast<int>(ids.size()) > c->C)
                return fail(MOE_E_CAPACITY, "%zu distinct experts exceed %d slots", ids.size(), c->C);
            if (ids.empty()) return MOE_OK;
            CUDA_TRY(cudaMemcpyAsync(c->d_keys, ids.data(), ids.size() * sizeof(int32_t), cudaMemcpyHostToDevice,
                                     c->s_comp));
            CUDA_TRY(cudaStreamSynchronize(c->s_comp));  // the host list goes out of scope
            a.keys = c->d_keys;
            a.n_keys = static_cast<int>(ids.size());
        } else {
            return fail(MOE_E_INVAL, "unknown fill mode %d", mode);
        }
        return dev_policy_run(c, a, true);
    }
    std::vector<int> keys;
    if (mode == MOE_FILL_FULL_LAYER) {
        if (c->C < c->E) return fail(MOE_E_CAPACITY, "a whole layer (%d) does not fit in %d slots", c->E, c->C);
        for (int e = 0; e < c->E; ++e) keys.push_back(layer * c->E + e);
        rc = access_keys(c, keys, true);
        return rc ? rc : upload_table(c);
    }
    if (mode != MOE_FILL_DEMAND) return fail(MOE_E_INVAL, "unknown fill mode %d", mode);
    if (n < 0 || (n > 0 && !idx_host)) return fail(MOE_E_INVAL, "bad index list");
    std::vector<char> used(c->E, 0);
    for (int i = 0; i < n; ++i) {
        if (idx_host[i] < 0 || idx_host[i] >= c->E) return fail(MOE_E_INVAL, "expert id %d out of range", idx_host[i]);
        used[idx_host[i]] = 1;
    }
    for (int e = 0; e < c->E; ++e)
        if (used[e]) keys.push_back(layer * c->E + e);
    if (static_cast<int>(keys.size()) > c->C)
        return fail(MOE_E_CAPACITY, "%zu distinct experts exceed %d slots", keys.size(), c->C);
    rc = access_keys(c, keys, false);
    return rc ? rc : upload_table(c);
}

int moe_layer_forward(moe_ctx* c, int layer, const void* x, const float* resid, float* out, int T,
                      const int32_t* idx, const float* w) {
    g_last_error.clear();
    int rc = validate_layer(c, layer);
    if (rc) return rc;
    if (T < 0 || T > c->Tmax) return fail(MOE_E_INVAL, "T=%d outside [0, %d]", T, c->Tmax);
    if (T == 0) return MOE_OK;
    if (!x || !resid || !out || !idx || !w) return fail(MOE_E_INVAL, "null device pointer");
    CUDA_TRY(cudaSetDevice(c->dev));
    if (c->dev_policy) return forward_device(c, layer, x, resid, out, T, idx, w);
    const int P = T * c->k;
    const int E = c->E, H = c->H, I = c->I;
    c->stats.forwards++;

    // 1. routed indices to the host (the LRU needs them), plus the device status word
    CUDA_TRY(cudaMemcpyAsync(c->idx_host, idx, P * sizeof(int32_t), cudaMemcpyDeviceToHost, c->s_comp));
    CUDA_TRY(cudaMemcpyAsync(c->status_host, c->status, sizeof(int), cudaMemcpyDeviceToHost, c->s_comp));
    CUDA_TRY(cudaEventRecord(c->ev_d2h, c->s_comp));
    // 2. permutation and row gather run while the host waits and plans
    rc = permute_and_gather(c, x, T, idx, w);
    if (rc) return rc;
    rc = wait_event(c, c->ev_d2h, "routed indices copy");
    if (rc) return rc;
    harvest(c);
    rc = check_status(c);
    if (rc) return rc;

    // 3. counts, offsets and the distinct experts in ascending id
    std::vector<int> count(E, 0);
    for (int p = 0; p < P; ++p) {
        const int e = c->idx_host[p];
        if (e < 0 || e >= E) return fail(MOE_E_INVAL, "routed expert id %d out of range", e);
        count[e]++;
    }
    std::vector<int> offs(E + 1, 0), distinct;
    int max_n = 0;
    for (int e = 0; e < E; ++e) {
        offs[e + 1] = offs[e] + count[e];
        if (count[e]) {
            distinct.push_back(e);
            max_n = std::max(max_n, count[e]);
        }
    }
    const int U = static_cast<int>(distinct.size());
    int path = c->path;
    if (c->fp4 && path == MOE_PATH_GEMM)
        return fail(MOE_E_INVAL, "4-bit entries run on the decode kernels only (MOE_PATH_GEMM unsupported)");
    if (path == MOE_PATH_AUTO) path = (c->fp4 || max_n <= kDecodeMaxTokens) ? MOE_PATH_GEMV : MOE_PATH_GEMM;

    // 4. waves of at most C experts
    for (int a0 = 0; a0 < U; a0 += c->C) {
        const int a1 = std::min(U, a0 + c->C);
        std::vector<int> keys;
        for (int a = a0; a < a1; ++a) keys.push_back(layer * E + distinct[a]);
        const int64_t seq_before = c->fill_seq;
        rc = access_keys(c, keys, false);
        if (rc) return rc;
        rc = upload_table(c);
        if (rc) return rc;

        const int32_t* slot_row = c->slot_dev + static_cast<size_t>(layer) * E;
        if (path == MOE_PATH_GEMM) {
            int64_t need_fill = -1;
            for (int key : keys) need_fill = std::max(need_fill, c->slot_fill[c->lru.slot_of(key)]);
            CUDA_TRY(wait_fills_through(c, c->s_comp, need_fill));
            std::vector<int> wc;
            int pw = 0;
            for (int a = a0; a < a1; ++a) {
                wc.push_back(count[distinct[a]]);
                pw += count[distinct[a]];
            }
            const int nw = a1 - a0;
            const int tiles_gu = moe::gemm_tiles(true, wc.data(), nw, H, I);
            const int tiles_d = moe::gemm_tiles(false, wc.data(), nw, H, I);
            {
                ProfScope ps(c, kGemmGateUp, 4.0 * nw * I * H + 2.0 * pw * H + 2.0 * pw * I, 4.0 * pw * I * H);
                CUDA_TRY(moe::launch_gemm_gateup(c->gemm_maps, c->offsets, c->active, a0, a1, tiles_gu, slot_row, H,
                                                 I, c->h_perm, c->status, c->num_sms, c->s_comp));
            }
            {
                ProfScope ps(c, kGemmDown, 2.0 * nw * H * I + 2.0 * pw * I + 4.0 * pw * H + 4.0 * pw,
                             2.0 * pw * I * H);
                CUDA_TRY(moe::launch_gemm_down(c->gemm_maps, c->offsets, c->active, a0, a1, tiles_d, slot_row, H, I,
                                               c->w_perm, c->pair_out, c->status, c->num_sms, c->s_comp));
            }
            c->comp_seq++;
            CUDA_TRY(cudaEventRecord(c->comp_ev[c->comp_seq % kEvRing], c->s_comp));
            for (int key : keys) c->slot_last_use[c->lru.slot_of(key)] = c->comp_seq;
            c->stats.waves++;
            continue;
        }

        // One launch per kernel for the whole wave. The work list holds the resident experts
        // first and then the ones this wave filled, in fill order; those carry their slot and
        // fill generation, and the kernel waits on the slot's fill flag before streaming them.
        // So resident experts compute while the copies cross the link, and each filled expert
        // starts as soon as its own copy has landed. Fills enqueued before this wave (a
        // prefetch still in flight) are waited for here, on the stream. Each expert writes only
        // its own pair_out rows, and every unit is computed the same way whatever the order, so
        // results do not depend on which entries had to be filled.
        bool inject_wave = false;
        std::vector<int> order;          // indices a into distinct[]: hits, then misses
        std::vector<char> filled_now(a1 - a0, 0);
        int64_t older_fill = -1;
        for (int a = a0; a < a1; ++a) {
            const int64_t f = c->slot_fill[c->lru.slot_of(keys[a - a0])];
            if (f > seq_before) filled_now[a - a0] = 1;
            else older_fill = std::max(older_fill, f);
        }
        for (int a = a0; a < a1; ++a)
            if (!filled_now[a - a0]) order.push_back(a);
        for (int a = a0; a < a1; ++a)
            if (filled_now[a - a0]) order.push_back(a);
        CUDA_TRY(wait_fills_through(c, c->s_comp, older_fill));

        // Work lists (gate/up, then down), each closed by an entry holding the unit total.
        // Units are token chunks x row tiles x K splits; the split of each kernel fills the SMs
        // evenly and depends only on the wave's routed set. bf16 entries run both phases in one
        // fused launch (unless MOE_PATH_GEMV_UNFUSED), whose splits balance the joint unit list.
        int pw = 0, chunks = 0;
        for (int a = a0; a < a1; ++a) {
            pw += count[distinct[a]];
            chunks += moe::decode_token_chunks(count[distinct[a]]);
        }
        const int nw = a1 - a0;
        const bool fused = !c->fp4 && path != MOE_PATH_GEMV_UNFUSED;
        const int Rg = moe::decode_row_tiles(true, H, I), Rd = moe::decode_row_tiles(false, H, I);
        int Sg = 1, Sd = 1, max_chunk_tok = 1;
        if (fused) {
            std::vector<int> chunk_tok;
            for (int i = 0; i < nw; ++i) {
                const int e = distinct[order[i]];
                for (int ch = 0; ch < moe::decode_token_chunks(count[e]); ++ch) {
                    chunk_tok.push_back(std::min(64, count[e] - 64 * ch));
                    max_chunk_tok = std::max(max_chunk_tok, chunk_tok.back());
                }
            }
            moe::decode_fused_choose_split(chunk_tok.data(), static_cast<int>(chunk_tok.size()), H, I, c->num_sms,
                                           &Sg, &Sd);
        } else {
            Sg = moe::decode_choose_split(chunks * Rg, true, H, I, c->num_sms);
            Sd = moe::decode_choose_split(chunks * Rd, false, H, I, c->num_sms);
        }
        int s;
        rc = next_stage(c, &s);
        if (rc) return rc;
        GemvWork* wk = c->work_stage + static_cast<size_t>(s) * kWorkEntries(E);
        GemvWork* wk2 = wk + (E + 1);
        int units_gu = 0, units_d = 0, chunk_base = 0;
        for (int i = 0; i < nw; ++i) {
            const int a = order[i];
            const int e = distinct[a];
            const int ch = moe::decode_token_chunks(count[e]);
            const int slot = c->lru.slot_of(keys[a - a0]);
            const int wait_slot = filled_now[a - a0] ? slot : -1;
            uint32_t gen = c->fill_gen[slot];
            if (wait_slot >= 0 && c->inject_kind == 3 && c->inject_count > 0) {
                gen += 1000;  // injected: a generation the copy stream will not write for a long time
                inject_wave = true;
            }
            wk[i] = GemvWork{e, offs[e], count[e], units_gu, wait_slot, gen, chunk_base, 0};
            wk2[i] = GemvWork{e, offs[e], count[e], units_d, wait_slot, gen, chunk_base, 0};
            units_gu += ch * Rg * Sg;
            units_d += ch * Rd * Sd;
            chunk_base += ch;
        }
        const uint64_t fill_wait_ns = inject_wave ? kInjectedFillWaitNs : c->fill_wait_ns;
        if (inject_wave) c->inject_count--;
        wk[nw] = GemvWork{-1, 0, 0, units_gu, -1, 0, 0, 0};
        wk2[nw] = GemvWork{-1, 0, 0, units_d, -1, 0, 0, 0};
        // the fused launch's unit schedule, after the two lists (null: the plain round robin)
        const int* sched_dev = nullptr;
        if (fused) {
            int* sched = reinterpret_cast<int*>(wk + 2 * (E + 1));
            const int grid = std::min(units_gu + units_d, c->num_sms);
            if (moe::decode_fused_schedule(units_gu, units_d, std::max(1, (H / 64) / Sg), std::max(1, (I / 64) / Sd),
                                           grid, sched, kSchedInts) > 0)
                sched_dev = reinterpret_cast<const int*>(c->work_dev + 2 * (E + 1));
        }
        // both lists (and the schedule) in one copy: gate/up at work_dev, down at work_dev + E + 1
        CUDA_TRY(cudaMemcpyAsync(c->work_dev, wk, kWorkEntries(E) * sizeof(GemvWork), cudaMemcpyHostToDevice,
                                 c->s_comp));
        CUDA_TRY(cudaEventRecord(c->stage_ev[s], c->s_comp));
        const double gu_bytes = 2.0 * nw * I * H * weight_bytes(c) + 2.0 * pw * H + 2.0 * pw * I;
        const double d_bytes = 1.0 * nw * H * I * weight_bytes(c) + 2.0 * pw * I + 4.0 * pw * H + 4.0 * pw;
        if (fused) {
            ProfScope ps(c, kDecodeFused, gu_bytes + d_bytes, 6.0 * pw * I * H);
            CUDA_TRY(moe::launch_decode_fused(c->dec_maps, c->work_dev, nw, units_gu, Sg, c->work_dev + (E + 1),
                                              units_d, Sd, max_chunk_tok, slot_row, c->fill_flag, H, I, c->h_perm,
                                              c->w_perm,
                                              c->pair_out, c->dec_ws, c->dec_cnt, c->dec_ready, c->dec_done,
                                              sched_dev, c->status, fill_wait_ns, c->num_sms, c->s_comp));
        } else {
            {
                ProfScope ps(c, kDecodeGateUp, gu_bytes, 4.0 * pw * I * H);
                CUDA_TRY(run_gateup(c, c->work_dev, nw, units_gu, Sg, nullptr, slot_row, fill_wait_ns));
            }
            {
                ProfScope ps(c, kDecodeDown, d_bytes, 2.0 * pw * I * H);
                CUDA_TRY(run_down(c, c->work_dev + (E + 1), nw, units_d, Sd, nullptr, slot_row, fill_wait_ns));
            }
        }
        c->comp_seq++;
        CUDA_TRY(cudaEventRecord(c->comp_ev[c->comp_seq % kEvRing], c->s_comp));
        for (int key : keys) c->slot_last_use[c->lru.slot_of(key)] = c->comp_seq;
        c->stats.waves++;
    }

    // 5. combine in j order
    {
        ProfScope ps(c, kCombine, 4.0 * P * H + 8.0 * T * H + 4.0 * P, 1.0 * P * H);
        CUDA_TRY(moe::launch_combine(c->pair_out, c->inv_perm, resid, out, T, c->k, H, c->s_comp));
    }
    return MOE_OK;
}

int moe_sync(moe_ctx* c) {
    g_last_error.clear();
    if (!c) return fail(MOE_E_INVAL, "null context");
    CUDA_TRY(cudaSetDevice(c->dev));
    CUDA_TRY(cudaMemcpyAsync(c->status_host, c->status, sizeof(int), cudaMemcpyDeviceToHost, c->s_comp));
    cudaEvent_t e1 = pool_event(c), e2 = pool_event(c);
    if (!e1 || !e2) return fail(MOE_E_CUDA, "event creation failed");
    CUDA_TRY(cudaEventRecord(e1, c->s_comp));
    CUDA_TRY(cudaEventRecord(e2, c->s_copy));
    int rc = wait_event(c, e1, "compute stream");
    if (!rc) rc = wait_event(c, e2, "copy stream");
    c->ev_pool.push_back(e1);
    c->ev_pool.push_back(e2);
    if (rc) return rc;
    harvest(c);
    return check_status(c);
}

int moe_stats(moe_ctx* c, moe_stats_t* out, moe_event_t* trace, uint64_t cap, int reset) {
    g_last_error.clear();
    if (!c) return fail(MOE_E_INVAL, "null context");
    if (c->dev_policy) {
        CUDA_TRY(cudaSetDevice(c->dev));
        int rc = drain(c);
        if (rc) return rc;
        moe::DevStats d{};
        CUDA_TRY(cudaMemcpy(&d, c->d_stats, sizeof(d), cudaMemcpyDeviceToHost));
        if (out) {
            *out = moe_stats_t{};
            out->expert_reads = d.expert_reads;
            out->hits = d.hits;
            out->misses = d.misses;
            out->prefetch_fills = d.prefetch_fills;
            out->prefetch_hits = d.prefetch_hits;
            out->evictions = d.evictions;
            out->fill_bytes = d.fill_bytes;
            out->fill_ms = 0.0;  // fills run inside kernels here; no per-batch copy timing
            out->trace_len = d.trace_len;
            out->forwards = d.forwards;
            out->waves = d.waves;
            out->resize_evictions = d.resize_evictions;
        }
        int written = 0;
        if (trace && cap > 0 && c->d_trace_cap) {
            const uint64_t have = std::min<uint64_t>(d.trace_len, c->d_trace_cap);
            const uint64_t n = std::min<uint64_t>(have, cap);
            for (uint64_t i = 0; i < n;) {
                const uint64_t pos = (d.trace_len - n + i) % c->d_trace_cap;
                const uint64_t run = std::min<uint64_t>(n - i, c->d_trace_cap - pos);
                static_assert(sizeof(moe::DevEvent) == sizeof(moe_event_t), "event layout");
                CUDA_TRY(cudaMemcpy(trace + i, c->d_trace + pos, run * sizeof(moe_event_t), cudaMemcpyDeviceToHost));
                i += run;
            }
            written = static_cast<int>(n);
        }
        if (reset) CUDA_TRY(cudaMemset(c->d_stats, 0, sizeof(moe::DevStats)));
        harvest(c);
        return written;
    }
    harvest(c);
    if (out) *out = c->stats;
    int written = 0;
    if (trace && cap > 0 && !c->trace.empty()) {
        const uint64_t have = std::min<uint64_t>(c->stats.trace_len, c->trace.size());
        const uint64_t n = std::min<uint64_t>(have, cap);
        const uint64_t first = c->stats.trace_len - n;
        for (uint64_t i = 0; i < n; ++i) trace[i] = c->trace[(first + i) % c->trace.size()];
        written = static_cast<int>(n);
    }
    if (reset) {
        c->stats = moe_stats_t{};
    }
    return written;
}

int moe_kernel_stats(moe_ctx* c, moe_kernel_stat_t* out, int cap, int reset) {
    if (!c) return fail(MOE_E_INVAL, "null context");
    harvest(c);
    for (int i = 0; i < kNumKernels && i < cap; ++i) {
        if (!out) break;
        out[i] = c->kstats[i];
        std::snprintf(out[i].name, sizeof(out[i].name), "%s", kKernelNames[i]);
    }
    if (reset)
        for (auto& s : c->kstats) s = moe_kernel_stat_t{};
    return kNumKernels;
}

int moe_debug_read(moe_ctx* c, int what, void* dst, uint64_t bytes) {
    g_last_error.clear();
    if (!c || !dst) return fail(MOE_E_INVAL, "null argument");
    const void* src = nullptr;
    uint64_t cap = 0;
    switch (what) {
        case MOE_DBG_OFFSETS: src = c->offsets; cap = (c->E + 1) * 4ull; break;
        case MOE_DBG_PERM: src = c->perm; cap = c->Pmax * 4ull; break;
        case MOE_DBG_INV_PERM: src = c->inv_perm; cap = c->Pmax * 4ull; break;
        case MOE_DBG_ACTIVE: src = c->active; cap = c->E * 4ull; break;
        case MOE_DBG_N_ACTIVE: src = c->n_active; cap = 4; break;
        case MOE_DBG_SLOT_TABLE: src = c->slot_dev; cap = static_cast<uint64_t>(c->L) * c->E * 4; break;
        case MOE_DBG_H_PERM: src = c->h_perm; cap = static_cast<uint64_t>(c->Pmax) * c->I * 2; break;
        case MOE_DBG_X_PERM: src = c->x_perm; cap = static_cast<uint64_t>(c->Pmax) * c->H * 2; break;
        case MOE_DBG_W_PERM: src = c->w_perm; cap = c->Pmax * 4ull; break;
        default: return fail(MOE_E_INVAL, "unknown buffer %d", what);
    }
    if (bytes > cap) return fail(MOE_E_INVAL, "%llu bytes requested, buffer holds %llu",
                                 static_cast<unsigned long long>(bytes), static_cast<unsigned long long>(cap));
    int rc = moe_sync(c);
    if (rc) return rc;
    CUDA_TRY(cudaMemcpy(dst, src, bytes, cudaMemcpyDeviceToHost));
    return MOE_OK;
}

int moe_measure_bandwidth(moe_ctx* c, int host_threads, int reps, moe_bandwidth_t* out) {
    g_last_error.clear();
    if (!c || !out || host_threads < 1 || reps < 1) return fail(MOE_E_INVAL, "bad arguments");
    CUDA_TRY(cudaSetDevice(c->dev));
    *out = moe_bandwidth_t{};
    out->entry_bytes = static_cast<double>(c->entry_bytes);
    out->host_threads = host_threads;
    // pinned host -> device: whole-entry copies on the copy stream, into a scratch buffer
    void* scratch = nullptr;
    cudaError_t e = cudaMalloc(&scratch, c->entry_bytes);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(MOE_E_NOMEM, "bandwidth probe buffer: %s", cudaGetErrorString(e));
    }
    cudaEvent_t e0 = pool_event(c), e1 = pool_event(c);
    int rc = MOE_OK;
    if (!e0 || !e1) rc = fail(MOE_E_CUDA, "event creation failed");
    for (int i = 0; i <= reps && rc == MOE_OK; ++i) {  // copy 0 warms up, the next reps are timed
        if (i == 1 && cudaEventRecord(e0, c->s_copy) != cudaSuccess) rc = fail(MOE_E_CUDA, "event record");
        if (rc == MOE_OK && cudaMemcpyAsync(scratch, c->pool, c->entry_bytes, cudaMemcpyHostToDevice, c->s_copy) !=
                                cudaSuccess)
            rc = fail(MOE_E_CUDA, "probe copy failed");
    }
    if (rc == MOE_OK && cudaEventRecord(e1, c->s_copy) != cudaSuccess) rc = fail(MOE_E_CUDA, "event record");
    if (rc == MOE_OK) rc = wait_event(c, e1, "bandwidth probe");
    if (rc == MOE_OK) {
        float ms = 0.f;
        cudaEventElapsedTime(&ms, e0, e1);
        out->pcie_h2d_gbps = ms > 0.f ? reps * static_cast<double>(c->entry_bytes) / (ms * 1e-3) / 1e9 : 0.0;
    }
    if (e0) c->ev_pool.push_back(e0);
    if (e1) c->ev_pool.push_back(e1);
    cudaFree(scratch);
    if (rc) return rc;
    // host expert FFN on entry (0, 0) with one token (bf16 entries only)
    if (!c->fp4) {
        std::vector<uint16_t> x(c->H, 0x3f80);  // 1.0
        std::vector<float> y(c->H);
        std::vector<double> t;
        for (int i = 0; i <= reps; ++i) {
            const auto t0 = std::chrono::steady_clock::now();
            rc = moe_host_expert_ffn(c->pool, c->H, c->I, x.data(), 1, y.data(), host_threads);
            if (rc) return rc;
            if (i > 0) t.push_back(std::chrono::duration<double>(std::chrono::steady_clock::now() - t0).count());
        }
        std::sort(t.begin(), t.end());
        const double med = t[t.size() / 2];
        out->host_expert_gbps = med > 0 ? static_cast<double>(c->entry_bytes) / med / 1e9 : 0.0;
    }
    return MOE_OK;
}

int moe_lru_simulate(int capacity, int n, const int32_t* layer, const int32_t* expert, const int32_t* kind,
                     moe_event_t* events, uint64_t events_cap) {
    if (capacity < 1 || n < 0 || (n > 0 && (!layer || !expert || !kind || !events)))
        return fail(MOE_E_INVAL, "bad arguments");
    int L = 1, E = 1;
    for (int i = 0; i < n; ++i) {
        if (kind[i] == 2) {
            if (expert[i] < 1) return fail(MOE_E_INVAL, "capacity change to %d", expert[i]);
            continue;
        }
        if (layer[i] < 0 || expert[i] < 0) return fail(MOE_E_INVAL, "negative key");
        L = std::max(L, layer[i] + 1);
        E = std::max(E, expert[i] + 1);
    }
    ExpertLru lru(capacity, L * E);
    uint64_t m = 0;
    for (int i = 0; i < n; ++i) {
        if (kind[i] == 2) {
            std::vector<std::pair<int, int>> evicted, moved;
            lru.resize(expert[i], &evicted, &moved);
            for (const auto& kv : evicted) {
                if (m >= events_cap) return fail(MOE_E_INVAL, "more events than events_cap");
                events[m++] = moe_event_t{MOE_EV_RESIZE_EVICT, kv.first / E, kv.first % E, kv.second, -1, -1};
            }
            continue;
        }
        if (m >= events_cap) return fail(MOE_E_INVAL, "more events than events_cap");
        const int key = layer[i] * E + expert[i];
        ExpertLru::Plan p = lru.plan(key, kind[i] == 1);
        lru.commit(p);
        events[m++] = moe_event_t{p.kind, layer[i], expert[i], p.slot, p.victim >= 0 ? p.victim / E : -1,
                                  p.victim >= 0 ? p.victim % E : -1};
    }
    return static_cast<int>(m);
}

}  // extern "C"
