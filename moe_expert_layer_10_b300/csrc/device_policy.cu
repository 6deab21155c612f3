// Device-resident cache policy and fills: a decode forward that never waits on the host, so
// that a whole decode step can be captured in a CUDA graph.
//
// Sources (page title, section):
//  * "FreeToken rtx 4090" (freetoken.wiki/hardware), "How the MoE Memory Hierarchy Works":
//    one shared LRU cache of complete (layer, expert) entries across layers and tokens,
//    following routing; the host pool stays the source of truth.
//  * "FreeToken benchmark" (freetoken.wiki/performance), "Graph Compatibility": the decode
//    path is kept compatible with CUDA graphs by holding its control data on the device.
//
// The policy is the same as the host policy (lru.h), so the traces are identical: the wave's
// distinct routed experts are accessed in ascending id; a resident entry is a HIT and moves
// to most-recently-used; a missing one takes the lowest free slot, else the slot of the
// least recently used entry (evicting it). Free slots are taken in increasing order and a
// used slot is never freed, so "lowest free" is the count of slots used so far.
//
// policy_kernel (one CTA): stages the recency list in shared memory, walks the wave in one
// thread (the accesses depend on each other), writes the slot table, the trace ring and the
// counters, and emits (a) the fill list (key, slot) and (b) the decode work lists: the wave's
// resident experts, and the experts it filled, with units and K split as the host path
// computes them (the split is chosen from the whole wave, so results do not depend on which
// experts were resident).
// fill_kernel: copies the listed entries from the pinned host pool (mapped into the device
// address space) into their slots with 16-byte loads over PCIe, the entries in list order.
#include <algorithm>

#include "kernels.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kPolicyThreads = 256;

__device__ __forceinline__ void lru_unlink(int* prev, int* next, int& head, int& tail, int s) {
    if (prev[s] >= 0) next[prev[s]] = next[s];
    else head = next[s];
    if (next[s] >= 0) prev[next[s]] = prev[s];
    else tail = prev[s];
    prev[s] = next[s] = -1;
}

__device__ __forceinline__ void lru_push_front(int* prev, int* next, int& head, int& tail, int s) {
    prev[s] = -1;
    next[s] = head;
    if (head >= 0) prev[head] = s;
    head = s;
    if (tail < 0) tail = s;
}

// Units of one expert for the decode kernels: token chunks of <= 64 x row tiles x split.
__device__ __forceinline__ int dev_chunks(int n) { return (n + 63) / 64; }

// The host's split rule (decode_choose_split), evaluated the same way on the device.
__device__ int dev_choose_split(int n_tiles, int KB, int num_sms) {
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
        const double e = eff(s) - 0.02 * (s - 1);
        if (e > best_eff + 1e-9) {
            best = s;
            best_eff = e;
        }
    }
    return best;
}

__global__ void __launch_bounds__(kPolicyThreads) policy_kernel(DevPolicyArgs a) {
    extern __shared__ int psm[];
    int* prev = psm;              // [C]
    int* next = prev + a.C;       // [C]
    int* key_in = next + a.C;     // [C]
    __shared__ int s_head, s_tail, s_used;
    DevLruState* st = a.state;
    for (int i = threadIdx.x; i < a.C; i += blockDim.x) {
        prev[i] = a.lru_prev[i];
        next[i] = a.lru_next[i];
        key_in[i] = a.lru_key[i];
    }
    if (threadIdx.x == 0) {
        s_head = st->head;
        s_tail = st->tail;
        s_used = st->n_used;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        // the keys of this call: a wave of the routed experts, or an explicit list
        int n_keys, k0;
        const int* keys_src;
        if (a.active) {
            const int n_act = *a.n_active;
            k0 = a.wave * a.C;
            n_keys = max(0, min(n_act, k0 + a.C) - k0);
            keys_src = a.active + k0;
        } else {
            k0 = 0;
            n_keys = a.n_keys;
            keys_src = a.keys;
        }
        int head = s_head, tail = s_tail, used = s_used;
        int n_fill = 0, n_hit = 0, n_miss = 0;
        DevStats& stats = *a.stats;
        for (int i = 0; i < n_keys; ++i) {
            const int e = keys_src[i];
            const int key = a.layer * a.E + e;
            int s = a.slot_of[key];
            int kind, victim = -1;
            if (s >= 0) {
                kind = a.prefetch ? kEvPrefetchHit : kEvHit;
                lru_unlink(prev, next, head, tail, s);
                lru_push_front(prev, next, head, tail, s);
                if (a.work_hit) a.order[n_hit++] = e;
            } else {
                kind = a.prefetch ? kEvPrefetchFill : kEvFill;
                if (used < a.C) {
                    s = used++;
                } else {
                    s = tail;
                    victim = key_in[s];
                    lru_unlink(prev, next, head, tail, s);
                    a.slot_of[victim] = -1;
                    stats.evictions++;
                }
                key_in[s] = key;
                a.slot_of[key] = s;
                lru_push_front(prev, next, head, tail, s);
                a.fill_list[n_fill++] = make_int2(key, s);
                stats.fill_bytes += a.entry_bytes;
                if (a.work_hit) a.order[a.C + n_miss++] = e;
            }
            switch (kind) {
                case kEvHit: stats.expert_reads++; stats.hits++; break;
                case kEvFill: stats.expert_reads++; stats.misses++; break;
                case kEvPrefetchFill: stats.prefetch_fills++; break;
                default: stats.prefetch_hits++; break;
            }
            if (a.trace_cap > 0) {
                DevEvent ev;
                ev.kind = kind;
                ev.layer = a.layer;
                ev.expert = e;
                ev.slot = s;
                ev.ev_layer = victim >= 0 ? victim / a.E : -1;
                ev.ev_expert = victim >= 0 ? victim % a.E : -1;
                a.trace[stats.trace_len % a.trace_cap] = ev;
            }
            stats.trace_len++;
        }
        if (a.active && a.wave == 0) stats.forwards++;
        if (n_keys > 0 && a.active) stats.waves++;
        s_head = head;
        s_tail = tail;
        s_used = used;
        a.hdr->n_fill = n_fill;
        if (a.work_hit) {
            // work lists: units = chunks x row tiles x split, the split chosen from the whole wave
            int chunks = 0;
            for (int i = 0; i < n_hit; ++i) {
                const int e = a.order[i];
                chunks += dev_chunks(a.offsets[e + 1] - a.offsets[e]);
            }
            for (int i = 0; i < n_miss; ++i) {
                const int e = a.order[a.C + i];
                chunks += dev_chunks(a.offsets[e + 1] - a.offsets[e]);
            }
            const int Rg = a.I / 64, Rd = a.H / 128;
            const int Sg = dev_choose_split(chunks * Rg, a.H / 64, a.num_sms);
            const int Sd = dev_choose_split(chunks * Rd, a.I / 64, a.num_sms);
            for (int g = 0; g < 2; ++g) {
                const int n = g == 0 ? n_hit : n_miss;
                const int* ord = a.order + (g == 0 ? 0 : a.C);
                GemvWork* wg = g == 0 ? a.work_hit : a.work_miss;
                GemvWork* wd = wg + (a.E + 1);
                int ug = 0, ud = 0;
                for (int i = 0; i < n; ++i) {
                    const int e = ord[i];
                    const int off = a.offsets[e], cnt = a.offsets[e + 1] - off;
                    const int ch = dev_chunks(cnt);
                    wg[i] = GemvWork{e, off, cnt, ug, -1, 0u, 0, 0};
                    wd[i] = GemvWork{e, off, cnt, ud, -1, 0u, 0, 0};
                    ug += ch * Rg * Sg;
                    ud += ch * Rd * Sd;
                }
                wg[n] = GemvWork{-1, 0, 0, ug, -1, 0u, 0, 0};
                wd[n] = GemvWork{-1, 0, 0, ud, -1, 0u, 0, 0};
                // dynamic launch headers: {n_work, n_units, S}
                int* hg = g == 0 ? a.hdr->hit_gu : a.hdr->miss_gu;
                int* hd = g == 0 ? a.hdr->hit_d : a.hdr->miss_d;
                hg[0] = n;
                hg[1] = n ? ug : 0;
                hg[2] = Sg;
                hd[0] = n;
                hd[1] = n ? ud : 0;
                hd[2] = Sd;
            }
        }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < a.C; i += blockDim.x) {
        a.lru_prev[i] = prev[i];
        a.lru_next[i] = next[i];
        a.lru_key[i] = key_in[i];
    }
    if (threadIdx.x == 0) {
        st->head = s_head;
        st->tail = s_tail;
        st->n_used = s_used;
    }
}

// Copy the listed entries host pool -> slots, one entry after the other (every CTA works on
// the same entry, so the first listed entries land first), 16-byte loads unrolled so many
// PCIe reads are in flight.
__global__ void __launch_bounds__(512) fill_kernel(const uint4* __restrict__ pool, uint4* __restrict__ arena,
                                                   const int2* __restrict__ fill_list, const int* __restrict__ n_fill,
                                                   size_t entry16) {
    const int nf = *n_fill;
    const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
    const size_t t0 = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x;
    constexpr int U = 8;
    for (int f = 0; f < nf; ++f) {
        const int2 kv = fill_list[f];
        const uint4* src = pool + static_cast<size_t>(kv.x) * entry16;
        uint4* dst = arena + static_cast<size_t>(kv.y) * entry16;
        size_t i = t0;
        for (; i + (U - 1) * stride < entry16; i += U * stride) {
            uint4 v[U];
#pragma unroll
            for (int u = 0; u < U; ++u) v[u] = src[i + u * stride];
#pragma unroll
            for (int u = 0; u < U; ++u) dst[i + u * stride] = v[u];
        }
        for (; i < entry16; i += stride) dst[i] = src[i];
    }
}

}  // namespace

cudaError_t launch_policy(const DevPolicyArgs& a, cudaStream_t st) {
    const size_t smem = 3ull * a.C * sizeof(int);
    if (smem > 200 * 1024) return cudaErrorInvalidValue;
    if (smem > 48 * 1024) {  // above the default limit: raise it to 200 KB once per device
        static std::atomic<uint64_t> attr{0};
        const cudaError_t e = ensure_smem_limit(policy_kernel, 200 * 1024, attr);
        if (e != cudaSuccess) return e;
    }
    policy_kernel<<<1, kPolicyThreads, smem, st>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_fill(const void* pool_dev, void* arena, const int2* fill_list, const int* n_fill,
                        size_t entry_bytes, int num_sms, cudaStream_t st) {
    fill_kernel<<<num_sms * 2, 512, 0, st>>>(static_cast<const uint4*>(pool_dev), static_cast<uint4*>(arena),
                                              fill_list, n_fill, entry_bytes / 16);
    return cudaGetLastError();
}

}  // namespace moe
