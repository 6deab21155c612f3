// CPU oracle for the routed Mixture-of-Experts layer served from a VRAM LRU cache of
// whole (layer, expert) entries.
//
// TEST INFRASTRUCTURE ONLY. The tests, the smoke check and the benchmark's CPU-baseline
// leg may call this file; the library never does. It shares no code with the CUDA
// path. It is plain and slow on purpose: every function computes its definition
// directly, in double precision except where a stated fp32 order is the definition.
//
// Sources (page title, section):
//  * "FreeToken rtx 4090" (freetoken.wiki/hardware), section "How the MoE Memory
//    Hierarchy Works": a token activates a few of many routed experts per layer
//    ("six of 256 routed experts"); a cache entry is one whole (layer, expert) pair,
//    executed through the same logical mapping on CPU and GPU; decode keeps a shared
//    LRU expert cache across layers and tokens; prefill streams whole layers.
//  * "FreeToken benchmark" (freetoken.wiki/performance), section "How FreeToken Serves
//    Large MoE Models": full-layer double buffering in prefill, shared least-recently-
//    used cache in decode.
//  * The layer's arithmetic, which the pages leave unstated, is the library's stated
//    specification: softmax gating renormalised over the top-k, SwiGLU experts
//    y = W_down (silu(W_gate x) * (W_up x)), combine out = resid + sum_j w_j y_j.
//
// Readings where the pages are silent (each repeated at its function):
//  R1 router logits are fp32 in one fixed order (below), so top-k is reproducible bit
//     for bit; a double copy is kept to flag near-ties;
//  R2 top-k orders by (logit desc, expert id asc): ties go to the lower id;
//  R3 gates are the softmax restricted to the k chosen logits;
//  R4 pairs are grouped by a stable counting sort on (expert, token, j);
//  R5 the LRU sees, per layer invocation, the distinct routed experts in ascending id;
//     a miss takes the lowest free slot, else the least recently used entry's slot.
//
// Parity pins for each function live in tests/test_oracle_*.py.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <map>
#include <set>
#include <vector>
#ifdef _OPENMP
#include <omp.h>
#endif

namespace {

double bf16_to_double(uint16_t b) {
    uint32_t u = static_cast<uint32_t>(b) << 16;
    float f;
    std::memcpy(&f, &u, 4);
    return static_cast<double>(f);
}

float bf16_to_float(uint16_t b) {
    uint32_t u = static_cast<uint32_t>(b) << 16;
    float f;
    std::memcpy(&f, &u, 4);
    return f;
}

// Order of two (logit, expert) candidates under R2: larger logit first, lower id on ties.
bool ranks_before(float za, int ea, float zb, int eb) {
    if (za != zb) return za > zb;
    return ea < eb;
}

}  // namespace

extern "C" {

int orc_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Threads of later parallel regions (the host's cores by default); returns the previous count.
   Used to time the oracle single-threaded beside the all-cores figure. */
int orc_set_num_threads(int n) {
#ifdef _OPENMP
    const int prev = omp_get_max_threads();
    if (n >= 1) omp_set_num_threads(n);
    return prev;
#else
    (void)n;
    return 1;
#endif
}

// Router logits z[t,e] = sum_h W_r[e,h] x[t,h] + b[e].
// R1: z32 is evaluated in fp32 in this order. 32 partial sums s_l (l = 0..31); s_l
// accumulates fmaf(W_r[e,h], x[t,h], s_l) over h = 256*m + 8*l + r, m ascending, then
// r = 0..7. The partials are folded pairwise at distances 16, 8, 4, 2, 1
// (s_l <- s_l + s_{l+d} for the l whose bit d is clear), and b[e] is added last.
// Requires H % 256 == 0. z64 is the same sum in double (for near-tie reports).
void orc_router_logits(const uint16_t* x, const float* Wr, const float* b, int T, int H, int E,
                       float* z32, double* z64) {
#pragma omp parallel for schedule(static)
    for (int t = 0; t < T; ++t) {
        for (int e = 0; e < E; ++e) {
            const float* w = Wr + static_cast<size_t>(e) * H;
            const uint16_t* xt = x + static_cast<size_t>(t) * H;
            float s[32];
            for (int l = 0; l < 32; ++l) {
                float acc = 0.0f;
                for (int m = 0; m < H / 256; ++m)
                    for (int r = 0; r < 8; ++r) {
                        int h = 256 * m + 8 * l + r;
                        acc = std::fmaf(w[h], bf16_to_float(xt[h]), acc);
                    }
                s[l] = acc;
            }
            for (int d = 16; d >= 1; d /= 2)
                for (int l = 0; l < 32; ++l)
                    if ((l & d) == 0) s[l] = s[l] + s[l + d];
            if (z32) z32[static_cast<size_t>(t) * E + e] = s[0] + b[e];
            if (z64) {
                double acc = 0.0;
                for (int h = 0; h < H; ++h) acc += static_cast<double>(w[h]) * bf16_to_double(xt[h]);
                z64[static_cast<size_t>(t) * E + e] = acc + static_cast<double>(b[e]);
            }
        }
    }
}

// Gates over k chosen logits, R3: w_j = exp(z_j - z_0) / sum_j' exp(z_j' - z_0), where
// z_0 is the largest chosen logit. Computed in double.
static void gates_of(const float* zsel, int k, double* w) {
    double zmax = static_cast<double>(zsel[0]);
    for (int j = 1; j < k; ++j) zmax = std::max(zmax, static_cast<double>(zsel[j]));
    double den = 0.0;
    for (int j = 0; j < k; ++j) den += std::exp(static_cast<double>(zsel[j]) - zmax);
    for (int j = 0; j < k; ++j) w[j] = std::exp(static_cast<double>(zsel[j]) - zmax) / den;
}

// Top-k routing of each token by R2 (full sort of all E candidates), then R3 gates.
// idx[t*k + j] is the j-th best expert; w[t*k + j] its gate.
void orc_topk(const float* z, int T, int E, int k, int32_t* idx, double* w) {
    for (int t = 0; t < T; ++t) {
        const float* zt = z + static_cast<size_t>(t) * E;
        std::vector<int> order(E);
        for (int e = 0; e < E; ++e) order[e] = e;
        std::sort(order.begin(), order.end(), [&](int a, int c) { return ranks_before(zt[a], a, zt[c], c); });
        std::vector<float> zsel(k);
        for (int j = 0; j < k; ++j) {
            idx[static_cast<size_t>(t) * k + j] = order[j];
            zsel[j] = zt[order[j]];
        }
        gates_of(zsel.data(), k, w + static_cast<size_t>(t) * k);
    }
}

// Forced routing: token t must use the experts sets[t*k .. t*k+k-1] (distinct). They are
// ordered by R2 on the router logits z, and gated by R3 over those k logits.
// Returns 0, or -1 if a set repeats an expert or holds an id outside [0, E).
int orc_forced_gates(const float* z, const int32_t* sets, int T, int E, int k, int32_t* idx, double* w) {
    for (int t = 0; t < T; ++t) {
        const float* zt = z + static_cast<size_t>(t) * E;
        std::vector<int> s(sets + static_cast<size_t>(t) * k, sets + static_cast<size_t>(t) * k + k);
        for (int j = 0; j < k; ++j) {
            if (s[j] < 0 || s[j] >= E) return -1;
            for (int q = 0; q < j; ++q)
                if (s[q] == s[j]) return -1;
        }
        std::sort(s.begin(), s.end(), [&](int a, int c) { return ranks_before(zt[a], a, zt[c], c); });
        std::vector<float> zsel(k);
        for (int j = 0; j < k; ++j) {
            idx[static_cast<size_t>(t) * k + j] = s[j];
            zsel[j] = zt[s[j]];
        }
        gates_of(zsel.data(), k, w + static_cast<size_t>(t) * k);
    }
    return 0;
}

// Tokens whose k-th and (k+1)-th best double logits differ by less than eps: there the
// fp32 order of R1 decides the routing. Writes the flags, returns their count.
int orc_near_ties(const double* z64, int T, int E, int k, double eps, int32_t* flag) {
    int n = 0;
    for (int t = 0; t < T; ++t) {
        std::vector<double> v(z64 + static_cast<size_t>(t) * E, z64 + static_cast<size_t>(t) * E + E);
        std::sort(v.begin(), v.end(), std::greater<double>());
        int f = (k < E) && (v[k - 1] - v[k] < eps);
        flag[t] = f;
        n += f;
    }
    return n;
}

// R4: group the T*k pairs p = t*k + j by expert with a stable counting sort.
// offsets[e] = first permuted position of expert e (offsets[E] = T*k);
// perm[pos] = p. Returns -1 if an index is outside [0, E).
int orc_permute(const int32_t* idx, int T, int k, int E, int32_t* offsets, int32_t* perm) {
    const int P = T * k;
    std::vector<int> count(E, 0);
    for (int p = 0; p < P; ++p) {
        if (idx[p] < 0 || idx[p] >= E) return -1;
        count[idx[p]]++;
    }
    offsets[0] = 0;
    for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + count[e];
    std::vector<int> fill(offsets, offsets + E);
    for (int p = 0; p < P; ++p) perm[fill[idx[p]]++] = p;
    return 0;
}

// One expert on one token, in double from the bf16 entry
// [W_gate (I x H) | W_up (I x H) | W_down (H x I)], all row-major:
//   g = W_gate x, u = W_up x, h = silu(g) * u = g / (1 + exp(-g)) * u, y = W_down h.
void orc_expert_ffn(const uint16_t* entry, int H, int I, const uint16_t* x, double* y) {
    const uint16_t* Wg = entry;
    const uint16_t* Wu = entry + static_cast<size_t>(I) * H;
    const uint16_t* Wd = entry + 2 * static_cast<size_t>(I) * H;
    std::vector<double> h(I);
    for (int i = 0; i < I; ++i) {
        double g = 0.0, u = 0.0;
        for (int c = 0; c < H; ++c) {
            double xc = bf16_to_double(x[c]);
            g += bf16_to_double(Wg[static_cast<size_t>(i) * H + c]) * xc;
            u += bf16_to_double(Wu[static_cast<size_t>(i) * H + c]) * xc;
        }
        h[i] = g / (1.0 + std::exp(-g)) * u;
    }
    for (int n = 0; n < H; ++n) {
        double acc = 0.0;
        for (int i = 0; i < I; ++i) acc += bf16_to_double(Wd[static_cast<size_t>(n) * I + i]) * h[i];
        y[n] = acc;
    }
}

// Sparse layer: out[t] = resid[t] + sum_{j<k} w[t,j] * y_{idx[t,j]}(x[t]), summed in j order.
// entries[e] points at expert e's entry of this layer.
void orc_moe_layer(const uint16_t* const* entries, int H, int I, const uint16_t* x, const float* resid,
                   int T, int k, const int32_t* idx, const double* w, double* out) {
    const int P = T * k;
    std::vector<double> y(static_cast<size_t>(P) * H);
#pragma omp parallel for schedule(dynamic, 1)
    for (int p = 0; p < P; ++p) {
        int t = p / k;
        orc_expert_ffn(entries[idx[p]], H, I, x + static_cast<size_t>(t) * H, &y[static_cast<size_t>(p) * H]);
    }
    for (int t = 0; t < T; ++t)
        for (int n = 0; n < H; ++n) {
            double acc = static_cast<double>(resid[static_cast<size_t>(t) * H + n]);
            for (int j = 0; j < k; ++j) acc += w[static_cast<size_t>(t) * k + j] * y[(static_cast<size_t>(t) * k + j) * H + n];
            out[static_cast<size_t>(t) * H + n] = acc;
        }
}

// Dense reference with zero-masked gates: every expert runs on every token and
// out[t] = resid[t] + sum_{e<E} g[t,e] * y_e(x[t]), with g[t,e] = w[t,j] if idx[t,j] == e
// and 0 otherwise. A second route to the same result as orc_moe_layer.
void orc_moe_dense(const uint16_t* const* entries, int H, int I, int E, const uint16_t* x, const float* resid,
                   int T, int k, const int32_t* idx, const double* w, double* out) {
#pragma omp parallel for schedule(static)
    for (int t = 0; t < T; ++t) {
        std::vector<double> y(H), acc(H);
        for (int n = 0; n < H; ++n) acc[n] = static_cast<double>(resid[static_cast<size_t>(t) * H + n]);
        for (int e = 0; e < E; ++e) {
            double g = 0.0;
            for (int j = 0; j < k; ++j)
                if (idx[static_cast<size_t>(t) * k + j] == e) g = w[static_cast<size_t>(t) * k + j];
            orc_expert_ffn(entries[e], H, I, x + static_cast<size_t>(t) * H, y.data());
            for (int n = 0; n < H; ++n) acc[n] += g * y[n];
        }
        for (int n = 0; n < H; ++n) out[static_cast<size_t>(t) * H + n] = acc[n];
    }
}

// MXFP4 weights (OCP Microscaling): element i of a tensor is the E2M1 code in nibble i%2 of
// byte i/2 (low nibble first) -- bit 3 the sign, bits 0-2 the magnitude 0, 0.5, 1, 1.5, 2, 3,
// 4, 6 -- times 2^(s - 127), s the E8M0 byte of its block of 32. Every such value has at most
// two significant bits, so it is written here as an exact bf16 (the caller's entries then
// run through the same bf16 expert FFN). Returns the number of elements that were not
// exactly representable (0 for any scale in the normal bf16 range).
int64_t orc_mxfp4_dequant(const uint8_t* q, const uint8_t* s, int64_t n, uint16_t* out) {
    static const double kMag[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};
    int64_t inexact = 0;
    for (int64_t i = 0; i < n; ++i) {
        const int code = (q[i / 2] >> (4 * (i % 2))) & 15;
        double v = std::ldexp(kMag[code & 7], static_cast<int>(s[i / 32]) - 127);
        if (code & 8) v = -v;
        const float f = static_cast<float>(v);
        uint32_t u;
        std::memcpy(&u, &f, 4);
        if ((u & 0xffffu) != 0 || static_cast<double>(f) != v) ++inexact;
        out[i] = static_cast<uint16_t>(u >> 16);
    }
    return inexact;
}

// NVFP4 weights: element i of a matrix is the E2M1 code in nibble i%2 of byte i/2 (low nibble
// first; bit 3 the sign; bits 2-1 the exponent e with bias 1, bit 0 the mantissa m: value
// m/2 when e = 0, else (1 + m/2) * 2^(e-1)) times the FP8 E4M3 scale of its block of 16
// (exponent field f with bias 7, mantissa m3: m3/8 * 2^-6 when f = 0, else (1 + m3/8) *
// 2^(f-7); sign and the all-ones NaN pattern are never valid scales) times the matrix's fp32
// tensor scale. In double every such product is exact. Returns the number of invalid scales.
static double orc_e2m1_value(int code) {
    const int e = (code >> 1) & 3, m = code & 1;
    const double mag = e == 0 ? 0.5 * m : (1.0 + 0.5 * m) * std::ldexp(1.0, e - 1);
    return (code & 8) ? -mag : mag;
}

static double orc_e4m3_value(int c, bool* ok) {
    const int f = (c >> 3) & 15, m3 = c & 7;
    *ok = !(c & 0x80) && !(f == 15 && m3 == 7);
    return f == 0 ? std::ldexp(m3 / 8.0, -6) : std::ldexp(1.0 + m3 / 8.0, f - 7);
}

int64_t orc_nvfp4_dequant(const uint8_t* q, const uint8_t* s, int64_t n, float tensor_scale, double* out) {
    int64_t invalid = 0;
    for (int64_t b = 0; b < n / 16; ++b) {
        bool ok;
        const double scale = orc_e4m3_value(s[b], &ok) * static_cast<double>(tensor_scale);
        if (!ok) ++invalid;
        for (int64_t i = 16 * b; i < 16 * b + 16; ++i)
            out[i] = orc_e2m1_value((q[i / 2] >> (4 * (i % 2))) & 15) * scale;
    }
    return invalid;
}

// The expert FFN of orc_expert_ffn with the weights given as doubles (W_gate | W_up | W_down,
// row-major), for entries whose values are not bf16 (NVFP4 with its tensor scales).
void orc_expert_ffn_f64(const double* W, int H, int I, const uint16_t* x, double* y) {
    const double* Wg = W;
    const double* Wu = W + static_cast<size_t>(I) * H;
    const double* Wd = W + 2 * static_cast<size_t>(I) * H;
    std::vector<double> h(I);
    for (int i = 0; i < I; ++i) {
        double g = 0.0, u = 0.0;
        for (int c = 0; c < H; ++c) {
            const double xc = bf16_to_double(x[c]);
            g += Wg[static_cast<size_t>(i) * H + c] * xc;
            u += Wu[static_cast<size_t>(i) * H + c] * xc;
        }
        h[i] = g / (1.0 + std::exp(-g)) * u;
    }
    for (int n = 0; n < H; ++n) {
        double acc = 0.0;
        for (int i = 0; i < I; ++i) acc += Wd[static_cast<size_t>(n) * I + i] * h[i];
        y[n] = acc;
    }
}

// orc_moe_layer for entries given as float64 weights (orc_expert_ffn_f64): out[t] = resid[t] +
// sum_{j<k} w[t,j] * y_{idx[t,j]}(x[t]), summed in j order. entries[e] points at expert e's
// weights W_gate | W_up | W_down.
void orc_moe_layer_f64(const double* const* entries, int H, int I, const uint16_t* x, const float* resid, int T,
                       int k, const int32_t* idx, const double* w, double* out) {
    const int P = T * k;
    std::vector<double> y(static_cast<size_t>(P) * H);
#pragma omp parallel for schedule(dynamic, 1)
    for (int p = 0; p < P; ++p) {
        int t = p / k;
        orc_expert_ffn_f64(entries[idx[p]], H, I, x + static_cast<size_t>(t) * H, &y[static_cast<size_t>(p) * H]);
    }
    for (int t = 0; t < T; ++t)
        for (int n = 0; n < H; ++n) {
            double acc = static_cast<double>(resid[static_cast<size_t>(t) * H + n]);
            for (int j = 0; j < k; ++j) acc += w[static_cast<size_t>(t) * k + j] * y[(static_cast<size_t>(t) * k + j) * H + n];
            out[static_cast<size_t>(t) * H + n] = acc;
        }
}

// R5: the distinct experts routed in one layer invocation, in ascending id (the order in
// which the LRU sees them). Returns their number.
int orc_layer_accesses(const int32_t* idx, int T, int k, int E, int32_t* experts) {
    std::vector<char> used(E, 0);
    for (int p = 0; p < T * k; ++p) used[idx[p]] = 1;
    int n = 0;
    for (int e = 0; e < E; ++e)
        if (used[e]) experts[n++] = e;
    return n;
}

// Shared LRU over whole (layer, expert) entries with `capacity` slots, run on a sequence
// of operations; kind_in[i] = 0 for a routed access, 1 for a prefetch of the whole next
// layer, 2 for a change of capacity to expert[i] slots (layer[i] ignored).
// Brute force: a recency list scanned linearly, MRU first.
// A present key is a hit and becomes MRU. An absent key takes the lowest free slot; if
// none is free, the LRU entry is evicted and its slot reused; the key becomes MRU.
// A capacity change keeps the min(n, new) most recently used entries and evicts the others,
// least recent first; the survivors are renumbered 0, 1, ... in the order of their old
// slots, and the slots from the number of survivors up to the new capacity are free.
// Events out, one per access and one per entry evicted by a capacity change:
//   kind 0 HIT, 1 FILL (routed miss), 2 PREFETCH_FILL, 3 PREFETCH_HIT, 4 RESIZE_EVICT;
//   (layer, expert) of the access or of the evicted entry; slot = the entry's slot
//   (for RESIZE_EVICT the slot it held); ev_vl/ev_ve = evicted (layer, expert) or -1/-1.
// Returns the number of events (at most max_events), or -1 for a capacity < 1 or too many
// events.
int orc_lru_run(int capacity, int n, const int32_t* layer, const int32_t* expert, const int32_t* kind_in,
                int max_events, int32_t* ev_kind, int32_t* ev_l, int32_t* ev_e, int32_t* ev_slot, int32_t* ev_vl,
                int32_t* ev_ve) {
    if (capacity < 1) return -1;
    std::vector<std::pair<int, int>> recency;  // front = most recently used
    std::map<std::pair<int, int>, int> slot_of;
    std::set<int> free_slots;
    for (int s = 0; s < capacity; ++s) free_slots.insert(s);
    int m = 0;
    auto emit = [&](int kind, int l, int e, int slot, int vl, int ve) {
        if (m >= max_events) return false;
        ev_kind[m] = kind;
        ev_l[m] = l;
        ev_e[m] = e;
        ev_slot[m] = slot;
        ev_vl[m] = vl;
        ev_ve[m] = ve;
        ++m;
        return true;
    };
    for (int i = 0; i < n; ++i) {
        if (kind_in[i] == 2) {
            const int cap2 = expert[i];
            if (cap2 < 1) return -1;
            while (static_cast<int>(recency.size()) > cap2) {
                std::pair<int, int> victim = recency.back();
                recency.pop_back();
                if (!emit(4, victim.first, victim.second, slot_of[victim], -1, -1)) return -1;
                slot_of.erase(victim);
            }
            // renumber the survivors in the order of their old slots
            std::vector<std::pair<int, std::pair<int, int>>> by_slot;
            for (const auto& kv : slot_of) by_slot.push_back({kv.second, kv.first});
            std::sort(by_slot.begin(), by_slot.end());
            for (size_t r = 0; r < by_slot.size(); ++r) slot_of[by_slot[r].second] = static_cast<int>(r);
            free_slots.clear();
            for (int s = static_cast<int>(by_slot.size()); s < cap2; ++s) free_slots.insert(s);
            capacity = cap2;
            continue;
        }
        std::pair<int, int> key(layer[i], expert[i]);
        bool prefetch = kind_in[i] == 1;
        auto it = std::find(recency.begin(), recency.end(), key);
        if (it != recency.end()) {
            recency.erase(it);
            recency.insert(recency.begin(), key);
            if (!emit(prefetch ? 3 : 0, key.first, key.second, slot_of[key], -1, -1)) return -1;
            continue;
        }
        int slot, vl = -1, ve = -1;
        if (!free_slots.empty()) {
            slot = *free_slots.begin();
            free_slots.erase(free_slots.begin());
        } else {
            std::pair<int, int> victim = recency.back();
            recency.pop_back();
            slot = slot_of[victim];
            slot_of.erase(victim);
            vl = victim.first;
            ve = victim.second;
        }
        recency.insert(recency.begin(), key);
        slot_of[key] = slot;
        if (!emit(prefetch ? 2 : 1, key.first, key.second, slot, vl, ve)) return -1;
    }
    return m;
}

}  // extern "C"
