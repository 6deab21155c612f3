/*
 * moe.h -- C ABI of the B300 (sm_103a) routed Mixture-of-Experts layer served from a
 * shared VRAM LRU cache of whole (layer, expert) entries, with the complete expert pool
 * in pinned host memory as the source of truth.
 *
 * What the calls implement, by page (title, section):
 *  - "FreeToken rtx 4090" (freetoken.wiki/hardware), "How the MoE Memory Hierarchy Works":
 *    the host keeps the complete expert pool; VRAM keeps a cache of complete
 *    layer-and-expert entries executed through one logical mapping; a router selects a
 *    few routed experts per token per layer ("six of 256"); decode keeps a shared LRU
 *    cache across layers and tokens; prefill streams the next layer's experts while the
 *    current layer computes; startup loads weights directly into the final host layout.
 *  - "FreeToken benchmark" (freetoken.wiki/performance), "How FreeToken Serves Large MoE
 *    Models": full-layer double buffering in prefill; shared least-recently-used expert
 *    cache in decode; misses move experts over the PCIe link into the GPU cache.
 *  - The per-layer arithmetic, which the pages do not state, is this library's
 *    specification: logits z = W_r x + b (fp32), top-k by (z desc, id asc), gates
 *    w_j = softmax of the k chosen logits, SwiGLU experts
 *    y_e(x) = W_down (silu(W_gate x) * (W_up x)), out = resid + sum_j w_j y_{e_j}(x).
 *
 * Conventions for every call:
 *  - Return 0 on success or a negative MOE_E_* code; moe_last_error() then holds a
 *    thread-local message. No call aborts or throws across the ABI. A failed call leaves
 *    the LRU bookkeeping consistent (an entry is only marked resident once its fill is
 *    enqueued successfully).
 *  - "device" pointers are CUDA device memory owned by the caller. All device work runs
 *    in order on the context's compute stream; fills run on its copy stream.
 *  - A context is used by one host thread at a time.
 *  - Device buffers passed to a call must stay valid until that call's work has finished on
 *    the compute stream (moe_sync, or any later synchronising call).
 *  - Activations are bf16 (raw 16-bit patterns), row-major [T x hidden].
 *  - Entry layout (host pool and device slot alike), bf16 row-major, contiguous:
 *      W_gate [inter x hidden] | W_up [inter x hidden] | W_down [hidden x inter]
 *    i.e. 3 * hidden * inter * 2 bytes per (layer, expert).
 *  - Shape limits: hidden % 256 == 0, inter % 128 == 0, 1 <= top_k <= num_experts <= 1024,
 *    top_k <= 32.
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- error codes ---- */
#define MOE_OK 0
#define MOE_E_INVAL (-1)    /* bad argument or shape */
#define MOE_E_NOMEM (-2)    /* host pinned or device allocation failed */
#define MOE_E_CUDA (-3)     /* a CUDA runtime call failed (message has the CUDA error) */
#define MOE_E_TIMEOUT (-4)  /* a host wait on the GPU passed its deadline */
#define MOE_E_CAPACITY (-5) /* the request needs more cache entries than configured */
#define MOE_E_DEVICE (-6)   /* a kernel reported an error through the device status word */

/* ---- config flags ---- */
#define MOE_TRACE 1u      /* keep a ring of LRU events, readable through moe_stats */
#define MOE_PROFILE 2u    /* time every kernel launch with CUDA events (moe_kernel_stats) */
#define MOE_PREFILL_DB 4u /* full-layer double buffering is intended: requires capacity >= 2*num_experts */
/* Keep the LRU policy, the slot table, the counters and the trace on the GPU, and issue the
 * fills from a kernel that reads the pinned pool through its device mapping: moe_layer_forward
 * then never waits on the host, and a decode step (moe_route + moe_layer_forward per layer) can
 * be captured into a CUDA graph on the compute stream. Same policy and traces as the host
 * policy. Decode kernels only (MOE_PATH_GEMM is refused); moe_cache_fill joins its fills
 * back into the compute stream (no prefill overlap); moe_stats reports fill_ms = 0. Run one
 * call of each shape before capturing, and keep MOE_PROFILE timing off while capturing. */
#define MOE_DEVICE_POLICY 8u
/* Expert entries in MXFP4 (OCP Microscaling: E2M1 weights, the even element in the low nibble,
 * one E8M0 scale per 32 consecutive weights of a row), stored in the order the kernels stream
 * them: stages of 4352 bytes, each the 4096 code bytes of a 128-row tile x 64-column slab
 * followed by its 256 scale bytes. W_gate/W_up come first, per 64-row tile (tile-major) and
 * slab: gate rows (64 x 32 bytes), up rows (64 x 32), gate scales (64 x 2), up scales (64 x 2);
 * then W_down per 128-row tile and slab: rows (128 x 32), scales (128 x 2). Within a row, its
 * two 32-blocks of the slab take bytes 0-15 and 16-31 and scale bytes 2r and 2r+1. An entry is
 * 3*hidden*inter*17/32 bytes, 17/64 of bf16, so fills move 3.8x fewer bytes. The kernels expand
 * the weights to bf16 on chip -- every MXFP4 value is exact in bf16 -- and run the decode
 * kernels (MOE_PATH_GEMM is refused); activations stay bf16. Needs inter % 128 == 0 and
 * hidden % 256 == 0 (as for every context). */
#define MOE_MXFP4 16u
/* Expert entries in NVFP4: E2M1 weights as in MOE_MXFP4, one FP8 E4M3 scale per 16 consecutive
 * weights of a row, and one fp32 tensor scale per matrix; a weight's value is
 * e2m1 * e4m3(block scale) * tensor scale. Same streaming order as MOE_MXFP4, in stages of 4608
 * bytes (4096 code bytes, then 4 scale bytes per row: block j of a row's 64-column slab takes
 * code bytes 8j .. 8j+7 and scale byte 4r + j; gate/up stages hold gate scales (64 x 4) then up
 * scales (64 x 4)), then a 16-byte trailer: the tensor scales of W_gate, W_up, W_down (fp32) and
 * 4 zero bytes. An entry is 3*hidden*inter*9/16 + 16 bytes. The kernels expand code times block
 * scale to bf16 on chip (exact: at most six significant bits) and multiply the fp32 accumulator
 * by the tensor scale; decode kernels only (MOE_PATH_GEMM is refused). Exclusive with MOE_MXFP4. */
#define MOE_NVFP4 32u

/* ---- fill modes (moe_cache_fill) ---- */
#define MOE_FILL_DEMAND 0     /* access the distinct experts of the given top-k indices */
#define MOE_FILL_FULL_LAYER 1 /* prefetch every expert of the layer (prefill double buffering) */

/* ---- expert-FFN path selection (moe_set_path) ---- */
#define MOE_PATH_AUTO 0 /* decode kernels when every routed expert has <= 64 tokens, else grouped GEMM */
#define MOE_PATH_GEMV 1 /* decode kernels: weight-streaming tcgen05 products, tokens as the narrow side */
#define MOE_PATH_GEMM 2 /* tcgen05 grouped GEMM kernels (prefill) */
/* decode kernels as two launches per wave (gate/up, then down); MOE_PATH_AUTO and MOE_PATH_GEMV
 * run bf16 entries' gate/up and down units in one persistent launch per wave */
#define MOE_PATH_GEMV_UNFUSED 3

/* ---- LRU event kinds ---- */
#define MOE_EV_HIT 0           /* routed access, entry resident */
#define MOE_EV_FILL 1          /* routed access, entry copied in (a miss) */
#define MOE_EV_PREFETCH_FILL 2 /* whole-layer prefetch copied the entry in */
#define MOE_EV_PREFETCH_HIT 3  /* whole-layer prefetch found the entry resident */
#define MOE_EV_RESIZE_EVICT 4  /* moe_cache_resize evicted the entry (slot = the slot it held) */
#define MOE_EV_HOST_EXEC 5     /* q-star simulation: a miss executed on the host (not filled; slot -1) */

typedef struct moe_ctx moe_ctx; /* opaque: pinned pool, slot arena, LRU, streams, scratch */

typedef struct {
    int32_t num_layers;  /* L: layers sharing the cache */
    int32_t num_experts; /* E: routed experts per layer */
    int32_t hidden;      /* H */
    int32_t inter;       /* I: expert SwiGLU intermediate size */
    int32_t top_k;       /* k */
    int32_t capacity;    /* C: cache slots, in whole entries */
    int32_t max_tokens;  /* largest T passed to moe_route / moe_layer_forward */
    uint32_t flags;      /* MOE_TRACE | MOE_PROFILE | MOE_PREFILL_DB | MOE_DEVICE_POLICY | MOE_MXFP4 | MOE_NVFP4 */
    uint64_t trace_capacity; /* events kept by MOE_TRACE (0: 1<<20) */
} moe_config_t;

typedef struct {
    uint64_t expert_reads;   /* routed accesses: one per distinct (layer, expert) per forward */
    uint64_t hits;           /* routed accesses that found the entry resident */
    uint64_t misses;         /* routed accesses that filled the entry */
    uint64_t prefetch_fills; /* whole-layer prefetches that filled an entry */
    uint64_t prefetch_hits;  /* whole-layer prefetches that found the entry resident */
    uint64_t evictions;      /* fills that replaced a resident entry */
    uint64_t fill_bytes;     /* bytes copied host -> device by fills */
    double fill_ms;          /* copy-stream time of completed fills, per call that filled (CUDA events;
                                0 under MOE_DEVICE_POLICY) */
    uint64_t trace_len;      /* events recorded since the last reset (the ring keeps the newest) */
    uint64_t forwards;       /* moe_layer_forward calls */
    uint64_t waves;          /* expert waves run (a layer routing to more than C experts runs several) */
    uint64_t resize_evictions; /* entries evicted by moe_cache_resize */
} moe_stats_t;

typedef struct {
    int32_t kind;      /* MOE_EV_* */
    int32_t layer;     /* accessed entry */
    int32_t expert;
    int32_t slot;      /* cache slot that holds it afterwards */
    int32_t ev_layer;  /* entry evicted to make room, or -1 */
    int32_t ev_expert; /* or -1 */
} moe_event_t;

typedef struct {
    char name[32];     /* kernel name */
    uint64_t launches; /* launches timed */
    double total_ms;   /* summed CUDA-event durations */
    double bytes;      /* algorithmic HBM bytes of those launches (weights + activations + outputs) */
    double flops;      /* algorithmic flops of those launches */
} moe_kernel_stat_t;

/*
 * Source: "FreeToken rtx 4090", "How the MoE Memory Hierarchy Works" -- the host keeps the
 * complete expert pool as the source of truth, the GPU keeps a cache of complete layer-expert
 * entries; "FreeToken benchmark", "How FreeToken Serves Large MoE Models" -- remaining VRAM is
 * an elastic expert cache. This call sets up both tiers.
 * Create a context: pinned host pool of L*E entries (zeroed), device arena of C entries,
 * slot-indirection table slot_of[L][E] (all -1), host LRU, scratch for max_tokens.
 * stream_compute / stream_copy: cudaStream_t handles to use, or NULL to create private
 * streams. Fills also take one private copy stream in turn with stream_copy; every batch of
 * fills ends with stream_copy waiting for it, so work ordered after stream_copy is ordered
 * after every fill. The caller then writes each entry straight into moe_host_entry(). Ownership:
 * the context owns everything it allocates; moe_cache_destroy frees it.
 * Errors: MOE_E_INVAL (shape limits above), MOE_E_CAPACITY (MOE_PREFILL_DB with C < 2E, or
 * C < 1), MOE_E_NOMEM, MOE_E_CUDA.
 */
int moe_cache_init(const moe_config_t* cfg, void* stream_compute, void* stream_copy, moe_ctx** out);

/* Free every resource of the context (waits for its streams first). NULL is a no-op. */
void moe_cache_destroy(moe_ctx* ctx);

/*
 * Host pointer (pinned, writable) to entry (layer, expert) of the pool, in the final
 * layout given above, so loaders write weights in place. NULL if out of range.
 * Entries must not change while a fill of that entry may be in flight.
 */
void* moe_host_entry(moe_ctx* ctx, int layer, int expert);

/*
 * Elastic cache: change the capacity to new_capacity entries at a safe point. The call waits
 * (with the deadline) until the context's enqueued work has finished, then:
 *  - keeps the min(n_resident, new_capacity) most recently used entries and evicts the
 *    others, least recent first (trace events MOE_EV_RESIZE_EVICT, counter resize_evictions);
 *  - moves the survivors into a new device arena of new_capacity slots, renumbered 0, 1, ...
 *    in the order of their old slots (growing moves nothing); the slots above are free;
 *  - keeps the recency order, the host pool and every counter.
 * Later misses take the lowest free slot, then the least recently used entry, as before. The
 * old arena is freed after the copy, so the device holds both for the duration of the call.
 * Kernel launches captured into a CUDA graph before the call hold the old arena's and state's
 * addresses: a graph of this context's calls must be captured again after a resize, not
 * replayed.
 * Errors: MOE_E_INVAL (new_capacity < 1, or arena too large), MOE_E_CAPACITY (MOE_PREFILL_DB
 * with new_capacity < 2*num_experts), MOE_E_NOMEM (the new arena could not be allocated; the
 * cache is unchanged), MOE_E_TIMEOUT, MOE_E_CUDA.
 */
int moe_cache_resize(moe_ctx* ctx, int new_capacity);

/* Bytes of one entry: 3 * hidden * inter * 2 (bf16), 3 * hidden * inter * 17/32 (MOE_MXFP4), or
 * 3 * hidden * inter * 9/16 + 16 (MOE_NVFP4). */
uint64_t moe_entry_bytes(const moe_ctx* ctx);

/*
 * Source: "FreeToken rtx 4090", "How the MoE Memory Hierarchy Works" -- each token activates a
 * small subset of the routed experts per layer ("six of 256"). The gating arithmetic below is
 * this library's specification (the pages state none).
 * Router for one layer: logits z[t,e] = fp32(sum_h W_r[e,h] x[t,h]) + b[e] in a fixed
 * order (32 lane partials over h = 256m + 8l + r, m then r ascending, fmaf; pairwise folds
 * at distances 16,8,4,2,1; bias last), top-k by (z desc, id asc), gates = softmax over the
 * k chosen logits (fp32).
 * x_bf16 [T x H], router_w fp32 [E x H], router_b fp32 [E] (NULL: zero), outputs
 * topk_idx int32 [T x k], topk_w fp32 [T x k], logits_or_null fp32 [T x E] -- all device.
 * Asynchronous on the compute stream. Errors: MOE_E_INVAL (T < 0 or T > max_tokens, layer
 * out of range, NULL pointer), MOE_E_CUDA. T == 0 is a no-op.
 */
int moe_route(moe_ctx* ctx, int layer, const void* x_bf16, int T, const float* router_w, const float* router_b,
              int32_t* topk_idx, float* topk_w, float* logits_or_null);

/*
 * Forced routing: token t uses the k distinct experts forced_sets[t*k .. t*k+k-1] (device
 * int32). The router logits are computed as in moe_route; the forced experts are ordered
 * by (z desc, id asc) and gated by the softmax over their k logits. A set with a repeated
 * or out-of-range id makes the kernel raise the device status (MOE_E_DEVICE at the next
 * synchronising call) and write expert 0 / gate 0 for that token.
 */
int moe_route_forced(moe_ctx* ctx, int layer, const void* x_bf16, int T, const float* router_w,
                     const float* router_b, const int32_t* forced_sets, int32_t* topk_idx, float* topk_w,
                     float* logits_or_null);

/*
 * Source: "FreeToken rtx 4090", "How the MoE Memory Hierarchy Works" -- during prefill the
 * runtime loads the next layer's experts while the GPU computes the current layer (full-layer
 * streaming, MOE_FILL_FULL_LAYER); "FreeToken benchmark", "How FreeToken Serves Large MoE
 * Models" -- the PCIe link moves selected experts into the GPU cache (MOE_FILL_DEMAND).
 * Cache fill without compute.
 *  MOE_FILL_DEMAND: topk_idx_host holds n host int32 expert ids (e.g. a T*k top-k block);
 *    their distinct values are accessed in ascending id. Errors: MOE_E_CAPACITY if more than
 *    C distinct experts are given (moe_layer_forward runs such layers in waves instead).
 *  MOE_FILL_FULL_LAYER: every expert 0..E-1 of the layer is accessed as a prefetch; the
 *    copies are enqueued on the copy stream and the call returns without waiting, so they
 *    overlap compute already enqueued (prefill double buffering). topk_idx_host/n ignored.
 *    Errors: MOE_E_CAPACITY if C < E.
 * Copies into a slot wait (on the GPU) for every enqueued compute that read the slot's
 * previous entry; compute that reads a filled slot waits (on the GPU) for its copy.
 */
int moe_cache_fill(moe_ctx* ctx, int layer, const int32_t* topk_idx_host, int n, int mode);

/*
 * Source: "FreeToken rtx 4090", "How the MoE Memory Hierarchy Works" -- decode keeps a shared
 * LRU expert cache across layers and tokens, and a cached entry is executed through one logical
 * mapping (here the slot table); "FreeToken benchmark", "How FreeToken Serves Large MoE Models"
 * -- recently routed experts stay in VRAM and misses are filled over PCIe. The SwiGLU expert
 * form and the weighted combine are this library's specification (the pages state neither).
 * One MoE layer on T tokens (device pointers): out = resid + sum_j w_j y_{e_j}(x).
 * x_bf16 [T x H], resid fp32 [T x H] (may equal out), out fp32 [T x H],
 * topk_idx int32 [T x k], topk_w fp32 [T x k] (as written by moe_route).
 * Steps: a D2H copy of topk_idx and a host wait (the host LRU needs the routed experts);
 * the distinct experts D (ascending) are accessed in the LRU in waves of at most C;
 * missing entries are copied in on the copy streams; per wave the expert FFN runs through
 * the device slot table; a deterministic combine sums the k contributions in j order.
 * On the decode path each fill is followed, on its copy stream, by a write of the slot's
 * fill generation to a device flag, and the expert kernels stream a filled entry only once
 * its flag shows the copy has landed: resident experts compute while the fills cross the
 * link. Results do not depend on which entries had to be filled.
 * Returns after enqueuing the last kernel (no wait at the end).
 * Errors: MOE_E_INVAL, MOE_E_CUDA, MOE_E_TIMEOUT (host wait deadline), MOE_E_DEVICE (a kernel
 * of an earlier call reported an error).
 */
int moe_layer_forward(moe_ctx* ctx, int layer, const void* x_bf16, const float* resid, float* out, int T,
                      const int32_t* topk_idx, const float* topk_w);

/*
 * Source: "FreeToken benchmark", overview -- the runtime reports token speed, processed tokens,
 * requests and cache activity; "FreeToken rtx 4090", "Benchmarks, Comparisons, and Tradeoffs"
 * -- the miss rate over expert reads is the measure of the cache (hits / expert_reads here).
 * Counters and trace. out may be NULL. trace_or_null receives up to trace_cap of the
 * newest events, oldest first; the return value is the number written (>= 0), or a
 * negative error. reset != 0 clears counters and trace after reading.
 */
int moe_stats(moe_ctx* ctx, moe_stats_t* out, moe_event_t* trace_or_null, uint64_t trace_cap, int reset);

/* ---- helpers ---- */

/* Thread-local message of the last failing call on this thread ("" if none). */
const char* moe_last_error(void);

/* Choose the expert-FFN path for later moe_layer_forward calls (MOE_PATH_*). */
int moe_set_path(moe_ctx* ctx, int path);

/* Turn the per-launch CUDA-event timing of MOE_PROFILE on (on != 0) or off for later calls,
 * e.g. to time a region without the events and then profile a separate pass. */
int moe_set_profile(moe_ctx* ctx, int on);

/* Wait (with a deadline) until all enqueued work of the context has finished; reports any
 * device status raised by its kernels (MOE_E_DEVICE). */
int moe_sync(moe_ctx* ctx);

/* Slot of entry (layer, expert) if resident, else -1 (host bookkeeping, no GPU access). */
int moe_resident_slot(moe_ctx* ctx, int layer, int expert);

/*
 * Per-kernel timing gathered under MOE_PROFILE (complete launches only; call moe_sync
 * first). Writes up to cap records, returns how many kernels there are. reset != 0 clears.
 */
int moe_kernel_stats(moe_ctx* ctx, moe_kernel_stat_t* out, int cap, int reset);

/*
 * Host-only run of this library's LRU policy (no GPU, no context): capacity slots, n
 * operations (layer[i], expert[i], kind[i]: 0 routed access, 1 prefetch, 2 capacity change to
 * expert[i] slots as moe_cache_resize does it). Writes one event per access and one
 * MOE_EV_RESIZE_EVICT event per entry a capacity change evicts, at most events_cap. Lets the
 * host policy be checked against a reference without a GPU. Returns the number of events
 * written, or MOE_E_INVAL (bad arguments, or more events than events_cap).
 */
int moe_lru_simulate(int capacity, int n, const int32_t* layer, const int32_t* expert, const int32_t* kind,
                     moe_event_t* events, uint64_t events_cap);

/*
 * Host-side fault injection for tests: the next `count` fill copies of this context report
 * failure before any copy is enqueued (kind 1), or the next `count` host waits report a
 * timeout (kind 2), or the next `count` decode waves that fill entries tell their kernels to
 * wait for a fill generation that the copy stream does not write, with a 0.2 s device-side
 * deadline (kind 3): the kernels give up, raise device status 5 (MOE_E_DEVICE at the next
 * synchronising call) and the context stays usable; or the next `count` fills report a failed
 * fill-flag write after their copy was enqueued (kind 4): the call fails with MOE_E_CUDA, the
 * entry is not made resident, and the entry the copy overwrites is evicted. kind 0 clears. No
 * GPU fault is ever produced.
 */
int moe_debug_inject(moe_ctx* ctx, int kind, int count);

/*
 * Copy an internal device buffer of the last moe_layer_forward to host memory, for tests.
 * Waits (with the deadline) for the compute stream first. bytes must not exceed the
 * buffer's size for the last call; returns MOE_E_INVAL otherwise.
 */
#define MOE_DBG_OFFSETS 0    /* int32 [E+1]: first permuted position of each expert */
#define MOE_DBG_PERM 1       /* int32 [T*k]: pair id t*k+j at each permuted position */
#define MOE_DBG_INV_PERM 2   /* int32 [T*k]: permuted position of each pair id */
#define MOE_DBG_ACTIVE 3     /* int32 [E]: experts with >= 1 pair, ascending (first n_active valid) */
#define MOE_DBG_N_ACTIVE 4   /* int32 [1] */
#define MOE_DBG_SLOT_TABLE 5 /* int32 [L*E]: device slot table */
#define MOE_DBG_H_PERM 6     /* bf16 [T*k x inter]: SwiGLU activations per permuted position */
#define MOE_DBG_X_PERM 7     /* bf16 [T*k x hidden]: token row of each permuted position */
#define MOE_DBG_W_PERM 8     /* fp32 [T*k]: gate of each permuted position */
int moe_debug_read(moe_ctx* ctx, int what, void* host_dst, uint64_t bytes);

/*
 * Router that allocates nothing: moe_route without a context, for callers that cannot call
 * cudaMalloc -- for example a process whose device memory belongs entirely to another
 * allocator (a serving engine's memory pool, where a stray cudaMalloc would break its
 * accounting), or a caller that must stay within a fixed, preallocated footprint and may not
 * grow the device heap at run time.
 * The paper has no counterpart of this call; it is a deployment convenience of this library.
 *
 * It computes what moe_route computes, with the same kernels: fp32 logits in the fixed
 * order, top-k by (z desc, id asc), softmax gates over the k chosen logits.
 * Arguments: x_bf16 [T x hidden], router_w fp32 [num_experts x hidden], router_b fp32
 * [num_experts] or NULL, outputs topk_idx int32 [T x top_k] and topk_w fp32 [T x top_k] --
 * all device pointers owned by the caller; cuda_stream is a cudaStream_t or NULL.
 * Scratch: the T x num_experts fp32 logits live in one static device array of
 * MOE_NOALLOC_MAX_LOGITS floats (256 KiB) inside the library; every GPU that loads the
 * library holds it until the process exits. T * num_experts above that limit returns
 * MOE_E_INVAL; so do hidden % 256 != 0, num_experts outside [1, 1024], top_k outside
 * [1, min(num_experts, 32)], T < 0 and NULL pointers. T == 0 is a no-op.
 * The array is shared by every call and keeps the last call's logits: calls that overlap on
 * the GPU (other streams, other host threads on the same device) race on it, so issue them
 * in order on one stream. The first call in each CUDA context looks up the array's device
 * address with that context current (cudaGetSymbolAddress) and keeps it with the context's id;
 * a later call in another context -- a different context made current on the device, or the
 * primary context created again after cudaDeviceReset -- looks it up again, so a stale address
 * is never used. Make the first call in each context before any stream capture begins.
 * Errors: MOE_E_INVAL, MOE_E_CUDA.
 */
#define MOE_NOALLOC_MAX_LOGITS 65536
int moe_route_noalloc(const void* x_bf16, int T, int hidden, int num_experts, int top_k, const float* router_w,
                      const float* router_b, int32_t* topk_idx, float* topk_w, void* cuda_stream);

/* ---- q-star: bandwidth-adaptive split of cache misses between fills and host execution ----
 *
 * Source: "FreeToken benchmark" (freetoken.wiki/performance), "How FreeToken Serves Large MoE
 * Models" -- misses are divided between GPU cache fills and direct CPU execution by the q-star
 * policy, which profiles host-side expert bandwidth and PCIe transfer bandwidth ("Adaptive
 * Misses"); "FreeToken rtx 4090" (freetoken.wiki/hardware), "Measure the Machine" and its tuning
 * table. The pages give no formula; this library's reading: a layer's miss time is
 * max(n_fill / B_pcie, n_host / B_host) * entry bytes (the link and the host cores work side by
 * side), smallest at the fill fraction q* = B_pcie / (B_pcie + B_host); ties go to more fills (a
 * fill also serves later hits). The misses with the most routed tokens fill first (ties: lower
 * expert id). These calls measure, decide and simulate; moe_layer_forward never executes an
 * expert on the host.
 */

typedef struct {
    double pcie_h2d_gbps;    /* pinned host -> device copies of whole entries (copy stream) */
    double host_expert_gbps; /* entry bytes / time of moe_host_expert_ffn on one token (0: not measured,
                                e.g. 4-bit entries) */
    int32_t host_threads;    /* threads the host expert FFN used */
    int32_t pad;
    double entry_bytes;
} moe_bandwidth_t;

/* Measure both bandwidths on this context's pool and device: `reps` timed copies of entry (0, 0)
 * into a temporary device buffer (cudaMalloc'd for the call), and `reps` host expert FFNs on it
 * with one token and host_threads threads (bf16 contexts only). Waits for its own work.
 * Errors: MOE_E_INVAL, MOE_E_NOMEM, MOE_E_CUDA. */
int moe_measure_bandwidth(moe_ctx* ctx, int host_threads, int reps, moe_bandwidth_t* out);

/* Expert FFN on the host cores, fp32 arithmetic: y[t] = W_down (silu(W_gate x_t) * (W_up x_t)) for
 * n_tok tokens, weights read from a bf16 entry in host memory (the entry layout above),
 * x_bf16 [n_tok x hidden] host bf16, y [n_tok x hidden] host fp32, `threads` worker threads.
 * Needs hidden % 16 == 0 and inter % 16 == 0. Errors: MOE_E_INVAL. */
int moe_host_expert_ffn(const void* entry_bf16, int hidden, int inter, const void* x_bf16, int n_tok, float* y,
                        int threads);

/* Host-only: the unit schedule of the fused decode launch (gate/up and down units of a wave in one
 * launch of `grid` CTAs). Units are numbered gate/up first (units_gu of kb_gu K blocks each), then
 * down (units_d of kb_d each); the launch deals them round robin (CTA b: b, b + grid, ...), and
 * this schedule moves the last down unit of each most-loaded CTA to a less-loaded one when that
 * lowers the largest per-CTA K-block total. Writes keep[grid] (round-robin units CTA b runs),
 * pool_off[grid + 1] and the moved units (CTA b runs pool[pool_off[b] .. pool_off[b+1]) after its
 * own) into sched, at most cap ints. Every CTA runs all its gate/up units before any down unit.
 * Returns the ints written, 0 when the plain round robin is as level, or MOE_E_INVAL. */
int moe_fused_schedule(int units_gu, int units_d, int kb_gu, int kb_d, int grid, int32_t* sched, int cap);

/* Number of a layer's n_miss misses to fill under the q-star rule for the given bandwidths
 * (host_gbps == 0: all; pcie_gbps == 0: none). Returns the count (>= 0) or MOE_E_INVAL. */
int moe_qstar_fills(double pcie_gbps, double host_gbps, int n_miss);

typedef struct {
    uint64_t expert_reads; /* routed accesses (distinct experts per invocation) */
    uint64_t hits;         /* resident when accessed */
    uint64_t fills;        /* misses filled (they enter the LRU) */
    uint64_t host_execs;   /* misses executed on the host (the LRU does not see them) */
    uint64_t evictions;
    uint64_t events;       /* events written */
    double modeled_ms;     /* sum over invocations of max(link, host) + GPU streaming time */
    double link_ms, host_ms;
} moe_qstar_sim_t;

/* Host-only run of the LRU under the q-star split (no GPU, no context). Invocation v (one layer
 * forward) holds accesses inv_offsets[v] .. inv_offsets[v+1]-1: (layer, expert, routed token
 * count), the distinct experts of that forward in ascending id. Per invocation: the misses at
 * its start are split -- q in [0, 1]: round(q * n_miss) fill; q < 0: moe_qstar_fills(pcie, host)
 * -- the fills in the order above; then the accesses run in order through the LRU, except the
 * host-executed ones (event MOE_EV_HOST_EXEC). Modeled time per invocation: max(n_fill * entry /
 * B_pcie, n_host * entry / B_host) + (n_hit + n_fill) * entry / B_hbm. events may be NULL.
 * Returns the number of events written, or MOE_E_INVAL. */
int moe_qstar_simulate(int capacity, int n_inv, const int32_t* inv_offsets, const int32_t* layer,
                       const int32_t* expert, const int32_t* n_tok, double q, double pcie_gbps, double host_gbps,
                       double hbm_gbps, double entry_bytes, moe_qstar_sim_t* out, moe_event_t* events,
                       uint64_t events_cap);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H */
