/*
 * Seeded synthetic inputs for the routed-MoE layer: expert weights, router
 * weights, router bias, activations and forced-routing traces.
 *
 * This file holds no arithmetic of the MoE method itself. It only draws random
 * numbers, so both the CUDA library and the CPU oracle consume identical bytes.
 *
 * Generator: Philox-4x32-10, the counter-based generator of Salmon, Moraes,
 * Dror and Shaw, "Parallel random numbers: as easy as 1, 2, 3" (SC'11),
 * written here from its published definition. Each 64-bit "stream" names one
 * tensor. Element i of a stream takes word i%4 of the block with counter
 * (i/4, stream). Normals use the Box-Muller transform on pairs of words; the
 * arithmetic core lives in normal_core.h, shared with the GPU build gen_gpu.cu
 * so both give the same bits.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include "mxfp4_core.h"
#include "normal_core.h"
#include "nvfp4_core.h"

void mi_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) { mi_philox_10(ctr, key, out); }

static inline void block_of(uint64_t seed, uint64_t stream, uint64_t q, uint32_t out[4]) {
    mi_block(seed, stream, q, out);
}

static inline void normals4(uint64_t seed, uint64_t stream, uint64_t q, double z[4]) {
    mi_normals4(seed, stream, q, z);
}

static inline uint16_t f32_to_bf16_rne(float f) { return mi_bf16_rne(f); }

/* The series logarithm and turn sine/cosine of the normal transform, for the pins. */
double mi_log_unit(double x) { return mi_log(x); }
void mi_sincos_2pi(double u, double* sn, double* cs) { mi_sincos_turn(u, sn, cs); }

uint16_t mi_f32_to_bf16(float f) { return f32_to_bf16_rne(f); }

/* Elements [first, first+n) of stream `stream`, each N(0, stddev) rounded to
 * fp32 and then to bf16 (RNE). */
void mi_normal_bf16(uint64_t seed, uint64_t stream, uint64_t first, uint64_t n, double stddev, uint16_t* out) {
    if (n == 0) return;
    uint64_t q0 = first / 4, q1 = (first + n + 3) / 4;
#pragma omp parallel for schedule(static)
    for (int64_t q = (int64_t)q0; q < (int64_t)q1; ++q) {
        double z[4];
        normals4(seed, stream, (uint64_t)q, z);
        for (int w = 0; w < 4; ++w) {
            uint64_t i = (uint64_t)q * 4 + w;
            if (i < first || i >= first + n) continue;
            out[i - first] = f32_to_bf16_rne((float)(z[w] * stddev));
        }
    }
}

void mi_normal_f32(uint64_t seed, uint64_t stream, uint64_t first, uint64_t n, double stddev, float* out) {
    if (n == 0) return;
    uint64_t q0 = first / 4, q1 = (first + n + 3) / 4;
#pragma omp parallel for schedule(static)
    for (int64_t q = (int64_t)q0; q < (int64_t)q1; ++q) {
        double z[4];
        normals4(seed, stream, (uint64_t)q, z);
        for (int w = 0; w < 4; ++w) {
            uint64_t i = (uint64_t)q * 4 + w;
            if (i < first || i >= first + n) continue;
            out[i - first] = (float)(z[w] * stddev);
        }
    }
}

void mi_uniform_u32(uint64_t seed, uint64_t stream, uint64_t first, uint64_t n, uint32_t* out) {
    for (uint64_t i = first; i < first + n; ++i) {
        uint32_t r[4];
        block_of(seed, stream, i / 4, r);
        out[i - first] = r[i % 4];
    }
}

/* A sequential source of uniform words on one stream. */
typedef struct {
    uint64_t seed, stream, next;
    uint32_t buf[4];
} word_src;

static uint32_t next_word(word_src* s) {
    uint64_t i = s->next++;
    if (i % 4 == 0) block_of(s->seed, s->stream, i / 4, s->buf);
    return s->buf[i % 4];
}

/* integer in [0, n) from one word (multiply-shift) */
static inline uint32_t bounded(uint32_t w, uint32_t n) { return (uint32_t)(((uint64_t)w * n) >> 32); }

/* Zipf(s) probabilities over ranks 1..E, p_r = r^-s / sum_j j^-s. */
static void zipf_probs(int E, double s, double* p) {
    double tot = 0.0;
    for (int r = 1; r <= E; ++r) tot += pow((double)r, -s);
    for (int r = 1; r <= E; ++r) p[r - 1] = pow((double)r, -s) / tot;
}

/*
 * Router bias that gives routing a Zipf(s) preference over experts.
 * A seeded Fisher-Yates shuffle pi maps rank r (0-based) to an expert;
 * bias[pi[r]] = (float) ln p_{r+1}. perm_out[r] = pi[r].
 */
void mi_zipf_bias(uint64_t seed, uint64_t stream, int E, double s, int32_t* perm_out, float* bias_out) {
    word_src src = {seed, stream, 0, {0, 0, 0, 0}};
    for (int r = 0; r < E; ++r) perm_out[r] = r;
    for (int i = E - 1; i > 0; --i) {
        uint32_t j = bounded(next_word(&src), (uint32_t)(i + 1));
        int32_t t = perm_out[i];
        perm_out[i] = perm_out[j];
        perm_out[j] = t;
    }
    double* p = (double*)malloc(sizeof(double) * (size_t)E);
    zipf_probs(E, s, p);
    for (int r = 0; r < E; ++r) bias_out[perm_out[r]] = (float)log(p[r]);
    free(p);
}

/* draw a rank from Zipf(s) by inverse CDF on a (0,1) uniform */
static int zipf_draw(const double* cdf, int E, word_src* src) {
    double u = mi_unit_open(next_word(src));
    int lo = 0, hi = E - 1;
    while (lo < hi) {
        int mid = (lo + hi) / 2;
        if (cdf[mid] >= u) hi = mid; else lo = mid + 1;
    }
    return lo;
}

/*
 * Forced-routing trace with temporal reuse, one persistent stream per batch
 * position b. sets[((step*L + l)*B + b)*k + j] is the j-th pick.
 * Step 0: k Zipf draws (expert = perm[l*E + rank]) without duplicates.
 * Step s>0, each pick j: with probability p_reuse choose uniformly among the
 * experts that position b used at step s-1 in layer l and that are not yet
 * picked (if none are left, fall through); otherwise draw Zipf, rejecting
 * duplicates. perm holds one rank->expert table per layer.
 * Returns 0, or -1 when k > E.
 */
int mi_trace_reuse(uint64_t seed, uint64_t stream, int L, int steps, int B, int E, int k, double s,
                   double p_reuse, const int32_t* perm, int32_t* sets) {
    if (k > E || k <= 0) return -1;
    double* p = (double*)malloc(sizeof(double) * (size_t)E);
    double* cdf = (double*)malloc(sizeof(double) * (size_t)E);
    zipf_probs(E, s, p);
    double acc = 0.0;
    for (int r = 0; r < E; ++r) { acc += p[r]; cdf[r] = acc; }
    cdf[E - 1] = 1.0;
    word_src src = {seed, stream, 0, {0, 0, 0, 0}};
    const uint32_t reuse_thresh = (uint32_t)(p_reuse * 4294967296.0 > 4294967295.0 ? 4294967295.0 : p_reuse * 4294967296.0);
    int32_t cand[1024];
    for (int st = 0; st < steps; ++st)
        for (int l = 0; l < L; ++l)
            for (int b = 0; b < B; ++b) {
                int32_t* cur = sets + (((size_t)st * L + l) * B + b) * k;
                const int32_t* prev = st > 0 ? sets + (((size_t)(st - 1) * L + l) * B + b) * k : NULL;
                for (int j = 0; j < k; ++j) {
                    int chosen = -1;
                    if (prev) {
                        uint32_t w = next_word(&src);
                        if (w < reuse_thresh) {
                            int nc = 0;
                            for (int q = 0; q < k; ++q) {
                                int dup = 0;
                                for (int jj = 0; jj < j; ++jj) dup |= (cur[jj] == prev[q]);
                                if (!dup) cand[nc++] = prev[q];
                            }
                            if (nc > 0) chosen = cand[bounded(next_word(&src), (uint32_t)nc)];
                        }
                    }
                    while (chosen < 0) {
                        int e = perm[(size_t)l * E + zipf_draw(cdf, E, &src)];
                        int dup = 0;
                        for (int jj = 0; jj < j; ++jj) dup |= (cur[jj] == e);
                        if (!dup) chosen = e;
                    }
                    cur[j] = chosen;
                }
            }
    free(p);
    free(cdf);
    return 0;
}


/*
 * Expert entry (layer, expert) in MXFP4: the seeded bf16 entry of stream `stream`
 * (W_gate [I x H] | W_up [I x H] | W_down [H x I]) quantized in blocks of 32 along each row
 * (mxfp4_core.h), the blocks placed in the streaming order of mi_mxfp4_place.
 */
void mi_mxfp4_entry(uint64_t seed, uint64_t stream, int H, int I, uint8_t* out) {
    const uint64_t n = 3ull * H * I;
    uint16_t* w = (uint16_t*)malloc(n * sizeof(uint16_t));
    if (!w) return;
    mi_normal_bf16(seed, stream, 0, n, 0.02, w);
    const uint64_t gate = (uint64_t)I * H;
#pragma omp parallel for schedule(static)
    for (int r = 0; r < 2 * I + H; ++r) {
        const int K = r < 2 * I ? H : I;
        const int mat = r < I ? 0 : (r < 2 * I ? 1 : 2);
        const int row = r < I ? r : (r < 2 * I ? r - I : r - 2 * I);
        const uint64_t elem0 = r < 2 * I ? (uint64_t)r * H : 2 * gate + (uint64_t)(r - 2 * I) * I;
        for (int b = 0; b < K / 32; ++b) {
            uint64_t co, so;
            mi_mxfp4_place(H, I, mat, row, b, &co, &so);
            mi_mxfp4_block(w + elem0 + 32 * b, out + co, out + so);
        }
    }
    free(w);
}

/* One block of 32 bf16 values quantized (for the pins). */
void mi_mxfp4_block32(const uint16_t* x, uint8_t* q16, uint8_t* s1) { mi_mxfp4_block(x, q16, s1); }


/*
 * Expert entry (layer, expert) in NVFP4: the seeded bf16 entry of stream `stream` quantized
 * per matrix (tensor scale) and per block of 16 along each row (nvfp4_core.h), the blocks
 * placed by mi_nvfp4_place, then the three fp32 tensor scales and 4 zero bytes.
 */
void mi_nvfp4_entry(uint64_t seed, uint64_t stream, int H, int I, uint8_t* out) {
    const uint64_t n = 3ull * H * I;
    uint16_t* w = (uint16_t*)malloc(n * sizeof(uint16_t));
    if (!w) return;
    mi_normal_bf16(seed, stream, 0, n, 0.02, w);
    const uint64_t mat_elems = (uint64_t)I * H;
    float t[3];
    for (int m = 0; m < 3; ++m) {
        float amax = 0.0f;
        for (uint64_t i = 0; i < mat_elems; ++i) {
            const float a = mi_bf16_to_f32(w[m * mat_elems + i] & 0x7fff);
            if (a > amax) amax = a;
        }
        t[m] = mi_nvfp4_tensor_scale(amax);
    }
#pragma omp parallel for schedule(static)
    for (int r = 0; r < 2 * I + H; ++r) {
        const int K = r < 2 * I ? H : I;
        const int mat = r < I ? 0 : (r < 2 * I ? 1 : 2);
        const int row = r < I ? r : (r < 2 * I ? r - I : r - 2 * I);
        const uint64_t elem0 = r < 2 * I ? (uint64_t)r * H : 2 * mat_elems + (uint64_t)(r - 2 * I) * I;
        for (int b = 0; b < K / 16; ++b) {
            uint64_t co, so;
            mi_nvfp4_place(H, I, mat, row, b, &co, &so);
            mi_nvfp4_block(w + elem0 + 16 * b, t[mat], out + co, out + so);
        }
    }
    uint8_t* trailer = out + mi_nvfp4_entry_bytes(H, I) - 16;
    memcpy(trailer, t, 12);
    memset(trailer + 12, 0, 4);
    free(w);
}

/* Pieces of the NVFP4 quantizer, for the pins. */
void mi_nvfp4_block16(const uint16_t* x, float t, uint8_t* q8, uint8_t* s1) { mi_nvfp4_block(x, t, q8, s1); }
uint8_t mi_e4m3_encode(float v) { return mi_e4m3_rne(v); }
float mi_e4m3_decode(uint8_t c) { return mi_e4m3_value(c); }
float mi_nvfp4_tscale(float amax) { return mi_nvfp4_tensor_scale(amax); }
uint64_t mi_nvfp4_bytes(int H, int I) { return mi_nvfp4_entry_bytes(H, I); }
