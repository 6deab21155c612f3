// Host-side pieces of the bandwidth-adaptive miss split ("q-star"): an expert FFN that runs on
// the host cores straight from a bf16 entry in host memory, and the split rule that divides a
// layer's cache misses between cache fills (PCIe, then the GPU) and host execution.
//
// Source: "FreeToken benchmark" (freetoken.wiki/performance), "How FreeToken Serves Large MoE
// Models" -- the runtime profiles host-side expert bandwidth and PCIe transfer bandwidth and
// uses them to decide how many missing experts move to the GPU and how many execute on the
// CPU ("Adaptive Misses"); "FreeToken rtx 4090" (freetoken.wiki/hardware), "Measure the
// Machine" -- the split should be measured with the deployed tensor shapes and the actual CPU
// expert kernel, and the tuning table: use fills where future reuse justifies the movement.
//
// The pages give no formula. The reading taken here: a miss filled over PCIe costs entry/B_pcie
// on the link, a miss run on the host costs entry/B_host on the host cores (both measured), the
// two paths run side by side, so the layer's miss time max(n_fill / B_pcie, n_host / B_host) *
// entry is smallest at n_fill / n_miss = q* = B_pcie / (B_pcie + B_host); ties go to the larger
// fill count (a fill also serves later hits). Which misses fill: the ones with the most routed
// tokens (the host's cost grows with tokens, the link's does not), ties to the lower expert id.
//
// None of this runs inside moe_layer_forward: the GPU path never executes an expert on the host.
#include <algorithm>
#include <chrono>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

#include "../../include/moe.h"
#include "lru.h"

namespace moe {
int set_error(int code, const char* msg);
}

namespace {

inline float bf16f(uint16_t b) {
    uint32_t u = static_cast<uint32_t>(b) << 16;
    float f;
    std::memcpy(&f, &u, 4);
    return f;
}

// acc[t] = sum_c W[c] * x[t][c] for a block of 4 tokens (or 1) over one weight row of K bf16
// values (x as fp32, row-major [tokens x K]): one pass over the row, 16 partial sums per token.
// Built for three instruction-set levels; the loader picks the best one the CPU has.
__attribute__((target_clones("arch=x86-64-v4", "arch=x86-64-v3", "default"))) void row_dot4(
    const uint16_t* __restrict__ w, const float* __restrict__ x, int K, float* __restrict__ acc) {
    float s[4][16] = {};
    for (int c = 0; c < K; c += 16) {
        float wf[16];
        for (int l = 0; l < 16; ++l) wf[l] = bf16f(w[c + l]);
        for (int t = 0; t < 4; ++t)
            for (int l = 0; l < 16; ++l) s[t][l] += wf[l] * x[static_cast<size_t>(t) * K + c + l];
    }
    for (int t = 0; t < 4; ++t) {
        float r = 0.0f;
        for (int l = 0; l < 16; ++l) r += s[t][l];
        acc[t] = r;
    }
}

__attribute__((target_clones("arch=x86-64-v4", "arch=x86-64-v3", "default"))) float row_dot1(
    const uint16_t* __restrict__ w, const float* __restrict__ x, int K) {
    float s[16] = {};
    for (int c = 0; c < K; c += 16)
        for (int l = 0; l < 16; ++l) s[l] += bf16f(w[c + l]) * x[c + l];
    float r = 0.0f;
    for (int l = 0; l < 16; ++l) r += s[l];
    return r;
}

// The dot products of rows [r0, r1) of W ([rows x K] bf16) with n_tok tokens: out[t * ld + r].
void rows_dot(const uint16_t* W, int K, int r0, int r1, const float* x, int n_tok, float* out, int ld) {
    for (int r = r0; r < r1; ++r) {
        const uint16_t* w = W + static_cast<size_t>(r) * K;
        int t = 0;
        float acc[4];
        for (; t + 4 <= n_tok; t += 4) {
            row_dot4(w, x + static_cast<size_t>(t) * K, K, acc);
            for (int j = 0; j < 4; ++j) out[static_cast<size_t>(t + j) * ld + r] = acc[j];
        }
        for (; t < n_tok; ++t) out[static_cast<size_t>(t) * ld + r] = row_dot1(w, x + static_cast<size_t>(t) * K, K);
    }
}

template <typename F>
void parallel_rows(int rows, int threads, F&& f) {
    threads = std::max(1, std::min(threads, rows));
    if (threads == 1) {
        f(0, rows);
        return;
    }
    std::vector<std::thread> pool;
    pool.reserve(threads);
    for (int i = 0; i < threads; ++i) {
        const int r0 = static_cast<int>(static_cast<int64_t>(rows) * i / threads);
        const int r1 = static_cast<int>(static_cast<int64_t>(rows) * (i + 1) / threads);
        pool.emplace_back([&f, r0, r1] { f(r0, r1); });
    }
    for (auto& t : pool) t.join();
}

int fills_for(double q, int n_miss) {
    if (n_miss <= 0) return 0;
    const int n = static_cast<int>(std::floor(q * n_miss + 0.5));
    return std::min(n_miss, std::max(0, n));
}

}  // namespace

extern "C" {

int moe_host_expert_ffn(const void* entry_bf16, int H, int I, const void* x_bf16, int n_tok, float* y, int threads) {
    if (!entry_bf16 || !x_bf16 || !y || H < 16 || H % 16 || I < 16 || I % 16 || n_tok < 0 || threads < 1)
        return moe::set_error(MOE_E_INVAL, "host expert FFN: bad arguments (hidden, inter multiples of 16)");
    if (n_tok == 0) return MOE_OK;
    const uint16_t* Wg = static_cast<const uint16_t*>(entry_bf16);
    const uint16_t* Wu = Wg + static_cast<size_t>(I) * H;
    const uint16_t* Wd = Wu + static_cast<size_t>(I) * H;
    const uint16_t* xb = static_cast<const uint16_t*>(x_bf16);
    std::vector<float> x(static_cast<size_t>(n_tok) * H), g(static_cast<size_t>(n_tok) * I),
        u(static_cast<size_t>(n_tok) * I), h(static_cast<size_t>(n_tok) * I);
    for (size_t i = 0; i < x.size(); ++i) x[i] = bf16f(xb[i]);
    // gate and up rows: one pass over each row for all tokens
    parallel_rows(I, threads, [&](int r0, int r1) {
        rows_dot(Wg, H, r0, r1, x.data(), n_tok, g.data(), I);
        rows_dot(Wu, H, r0, r1, x.data(), n_tok, u.data(), I);
        for (int t = 0; t < n_tok; ++t)
            for (int i = r0; i < r1; ++i) {
                const size_t p = static_cast<size_t>(t) * I + i;
                h[p] = g[p] / (1.0f + std::exp(-g[p])) * u[p];
            }
    });
    // down rows
    parallel_rows(H, threads, [&](int r0, int r1) { rows_dot(Wd, I, r0, r1, h.data(), n_tok, y, H); });
    return MOE_OK;
}

int moe_qstar_fills(double pcie_gbps, double host_gbps, int n_miss) {
    if (n_miss < 0 || !(pcie_gbps >= 0.0) || !(host_gbps >= 0.0) || pcie_gbps + host_gbps <= 0.0)
        return moe::set_error(MOE_E_INVAL, "q-star split: bandwidths must be >= 0, not both 0, and n_miss >= 0");
    if (host_gbps == 0.0) return n_miss;
    if (pcie_gbps == 0.0) return 0;
    // n minimising max(n / B_pcie, (m - n) / B_host): floor or ceil of m * q*, ties to the larger
    const double q = pcie_gbps / (pcie_gbps + host_gbps);
    const int lo = static_cast<int>(std::floor(q * n_miss)), hi = std::min(n_miss, lo + 1);
    auto cost = [&](int n) { return std::max(n / pcie_gbps, (n_miss - n) / host_gbps); };
    return cost(hi) <= cost(lo) ? hi : lo;
}

int moe_qstar_simulate(int capacity, int n_inv, const int32_t* inv_offsets, const int32_t* layer,
                       const int32_t* expert, const int32_t* n_tok, double q, double pcie_gbps, double host_gbps,
                       double hbm_gbps, double entry_bytes, moe_qstar_sim_t* out, moe_event_t* events,
                       uint64_t events_cap) {
    if (capacity < 1 || n_inv < 0 || (n_inv > 0 && (!inv_offsets || !layer || !expert || !n_tok)) || !out ||
        !(pcie_gbps > 0.0) || !(host_gbps > 0.0) || !(hbm_gbps > 0.0) || !(entry_bytes > 0.0) || q > 1.0)
        return moe::set_error(MOE_E_INVAL, "q-star simulation: bad arguments");
    int L = 1, E = 1;
    const int n = n_inv > 0 ? inv_offsets[n_inv] : 0;
    for (int i = 0; i < n; ++i) {
        if (layer[i] < 0 || expert[i] < 0 || n_tok[i] < 1)
            return moe::set_error(MOE_E_INVAL, "q-star simulation: negative key or a key without tokens");
        L = std::max(L, layer[i] + 1);
        E = std::max(E, expert[i] + 1);
    }
    moe::ExpertLru lru(capacity, L * E);
    *out = moe_qstar_sim_t{};
    uint64_t m = 0;
    auto emit = [&](const moe_event_t& ev) {
        if (!events) return true;
        if (m >= events_cap) return false;
        events[m++] = ev;
        return true;
    };
    for (int v = 0; v < n_inv; ++v) {
        const int a = inv_offsets[v], b = inv_offsets[v + 1];
        if (b < a) return moe::set_error(MOE_E_INVAL, "q-star simulation: offsets must not decrease");
        // the invocation's misses at its start, the ones to fill first by (tokens desc, id asc)
        std::vector<int> miss;
        for (int i = a; i < b; ++i)
            if (lru.slot_of(layer[i] * E + expert[i]) < 0) miss.push_back(i);
        const int m_miss = static_cast<int>(miss.size());
        const int n_fill = q < 0.0 ? moe_qstar_fills(pcie_gbps, host_gbps, m_miss) : fills_for(q, m_miss);
        std::stable_sort(miss.begin(), miss.end(), [&](int x, int y) {
            if (n_tok[x] != n_tok[y]) return n_tok[x] > n_tok[y];
            return expert[x] < expert[y];
        });
        std::vector<char> host(b - a, 0);
        for (int j = n_fill; j < m_miss; ++j) host[miss[j] - a] = 1;
        uint64_t fills = 0, hits = 0, hosts = 0;
        for (int i = a; i < b; ++i) {
            const int key = layer[i] * E + expert[i];
            out->expert_reads++;
            if (host[i - a]) {
                hosts++;
                if (!emit(moe_event_t{MOE_EV_HOST_EXEC, layer[i], expert[i], -1, -1, -1}))
                    return moe::set_error(MOE_E_INVAL, "q-star simulation: more events than events_cap");
                continue;
            }
            moe::ExpertLru::Plan p = lru.plan(key, false);
            lru.commit(p);
            if (p.kind == moe::ExpertLru::kHit) hits++;
            else fills++;
            if (p.victim >= 0) out->evictions++;
            if (!emit(moe_event_t{p.kind, layer[i], expert[i], p.slot, p.victim >= 0 ? p.victim / E : -1,
                                  p.victim >= 0 ? p.victim % E : -1}))
                return moe::set_error(MOE_E_INVAL, "q-star simulation: more events than events_cap");
        }
        out->hits += hits;
        out->fills += fills;
        out->host_execs += hosts;
        // fills and host execution run side by side; the GPU then streams every entry it computes
        const double t_link = fills * entry_bytes / (pcie_gbps * 1e9), t_host = hosts * entry_bytes / (host_gbps * 1e9);
        const double t_gpu = (hits + fills) * entry_bytes / (hbm_gbps * 1e9);
        out->modeled_ms += 1e3 * (std::max(t_link, t_host) + t_gpu);
        out->link_ms += 1e3 * t_link;
        out->host_ms += 1e3 * t_host;
    }
    out->events = m;
    return static_cast<int>(std::min<uint64_t>(m, 0x7fffffff));
}

}  // extern "C"
