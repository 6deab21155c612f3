/*
 * The arithmetic core of the seeded input generator, shared by its CPU build (gen.c) and
 * its GPU build (gen_gpu.cu) so that both produce the same bits:
 *
 *  - Philox-4x32-10 (Salmon, Moraes, Dror and Shaw, "Parallel random numbers: as easy as
 *    1, 2, 3", SC'11), written from its published definition;
 *  - Box-Muller normals, with the logarithm and the sine/cosine evaluated by this file's
 *    own series in double precision. They use only operations that IEEE 754 rounds
 *    exactly the same way everywhere (+, *, /, sqrt, fused multiply-add, bit moves), in a
 *    fixed order, so a CPU and a GPU give identical results. Both builds must keep the
 *    compiler from contracting a*b+c on its own (gcc -ffp-contract=off, nvcc -fmad=false).
 *
 * Series used (standard analysis, not a library's implementation):
 *  - ln m = 2 atanh(s) = 2 (s + s^3/3 + s^5/5 + ... + s^23/23), s = (m-1)/(m+1), after
 *    reducing x = m * 2^e with m in [sqrt(1/2), sqrt(2)), so |s| <= 0.172 and the first
 *    omitted term is below 1e-19 relative;
 *  - sin a and cos a by their Taylor series to a^25 and a^24 on a in [0, pi/2), after
 *    splitting the turn 2*pi*u into its quadrant; the first omitted term is below 1e-22.
 * This file holds no arithmetic of the MoE method; it only draws random numbers.
 */
#ifndef MOE_INPUTS_NORMAL_CORE_H
#define MOE_INPUTS_NORMAL_CORE_H

#include <math.h>
#include <stdint.h>
#include <string.h>

#ifdef __CUDACC__
#define MI_HD static __host__ __device__ __forceinline__
#else
#define MI_HD static inline
#endif

#define MI_PHILOX_M0 0xD2511F53u
#define MI_PHILOX_M1 0xCD9E8D57u
#define MI_PHILOX_W0 0x9E3779B9u
#define MI_PHILOX_W1 0xBB67AE85u

MI_HD void mi_philox_round(uint32_t c[4], const uint32_t k[2]) {
    const uint64_t p0 = (uint64_t)MI_PHILOX_M0 * c[0];
    const uint64_t p1 = (uint64_t)MI_PHILOX_M1 * c[2];
    const uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
    const uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
    const uint32_t n0 = hi1 ^ c[1] ^ k[0];
    const uint32_t n2 = hi0 ^ c[3] ^ k[1];
    c[0] = n0;
    c[1] = lo1;
    c[2] = n2;
    c[3] = lo0;
}

MI_HD void mi_philox_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
    uint32_t c[4] = {ctr[0], ctr[1], ctr[2], ctr[3]};
    uint32_t k[2] = {key[0], key[1]};
    for (int r = 0; r < 10; ++r) {
        if (r > 0) {
            k[0] += MI_PHILOX_W0;
            k[1] += MI_PHILOX_W1;
        }
        mi_philox_round(c, k);
    }
    out[0] = c[0];
    out[1] = c[1];
    out[2] = c[2];
    out[3] = c[3];
}

/* Block q of stream `stream`: counter (q, stream), key = seed. */
MI_HD void mi_block(uint64_t seed, uint64_t stream, uint64_t q, uint32_t out[4]) {
    const uint32_t ctr[4] = {(uint32_t)q, (uint32_t)(q >> 32), (uint32_t)stream, (uint32_t)(stream >> 32)};
    const uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    mi_philox_10(ctr, key, out);
}

/* (0,1): the word plus one half, scaled by 2^-32 (exact in double) */
MI_HD double mi_unit_open(uint32_t r) { return ((double)r + 0.5) * (1.0 / 4294967296.0); }

/* natural logarithm of x in (0, 1], x normal */
MI_HD double mi_log(double x) {
    uint64_t b;
    memcpy(&b, &x, 8);
    int e = (int)((b >> 52) & 0x7ff) - 1023;
    b = (b & 0x000fffffffffffffull) | 0x3ff0000000000000ull;
    double m;
    memcpy(&m, &b, 8);
    if (m > 0x1.6a09e667f3bcdp+0) { /* sqrt(2) */
        m = m * 0.5;
        e += 1;
    }
    const double s = (m - 1.0) / (m + 1.0);
    const double s2 = s * s;
    double p = 0x1.642c8590b2164p-5; /* 1/23 */
    p = fma(p, s2, 0x1.8618618618618p-5); /* 1/21 */
    p = fma(p, s2, 0x1.af286bca1af28p-5); /* 1/19 */
    p = fma(p, s2, 0x1.e1e1e1e1e1e1ep-5); /* 1/17 */
    p = fma(p, s2, 0x1.1111111111111p-4); /* 1/15 */
    p = fma(p, s2, 0x1.3b13b13b13b14p-4); /* 1/13 */
    p = fma(p, s2, 0x1.745d1745d1746p-4); /* 1/11 */
    p = fma(p, s2, 0x1.c71c71c71c71cp-4); /* 1/9 */
    p = fma(p, s2, 0x1.2492492492492p-3); /* 1/7 */
    p = fma(p, s2, 0x1.999999999999ap-3); /* 1/5 */
    p = fma(p, s2, 0x1.5555555555555p-2); /* 1/3 */
    p = fma(p, s2, 1.0);
    const double lm = (2.0 * s) * p;
    const double de = (double)e;
    /* ln 2 split in a high and a low part */
    return (de * 0x1.abc9e3b39803fp-56 + lm) + de * 0x1.62e42fefa39efp-1;
}

/* sine and cosine of 2*pi*u for u in [0, 1) */
MI_HD void mi_sincos_turn(double u, double* sn, double* cs) {
    const double t = u * 4.0;           /* exact */
    const int q = (int)t;               /* quadrant 0..3 */
    const double r = t - (double)q;     /* exact, in [0, 1) */
    const double a = r * 0x1.921fb54442d18p+0; /* r * pi/2 */
    const double a2 = a * a;
    double ps = 0x1.3f3ccdd165fa9p-84;  /* 1/25! */
    ps = fma(ps, a2, -0x1.761b41316381ap-75);
    ps = fma(ps, a2, 0x1.71b8ef6dcf572p-66);
    ps = fma(ps, a2, -0x1.2f49b46814157p-57);
    ps = fma(ps, a2, 0x1.952c77030ad4ap-49);
    ps = fma(ps, a2, -0x1.ae7f3e733b81fp-41);
    ps = fma(ps, a2, 0x1.6124613a86d09p-33);
    ps = fma(ps, a2, -0x1.ae64567f544e4p-26);
    ps = fma(ps, a2, 0x1.71de3a556c734p-19);
    ps = fma(ps, a2, -0x1.a01a01a01a01ap-13);
    ps = fma(ps, a2, 0x1.1111111111111p-7);
    ps = fma(ps, a2, -0x1.5555555555555p-3);
    ps = fma(ps, a2, 1.0);
    const double sa = a * ps;
    double pc = 0x1.f2cf01972f578p-80;  /* 1/24! */
    pc = fma(pc, a2, -0x1.0ce396db7f853p-70);
    pc = fma(pc, a2, 0x1.e542ba4020225p-62);
    pc = fma(pc, a2, -0x1.6827863b97d97p-53);
    pc = fma(pc, a2, 0x1.ae7f3e733b81fp-45);
    pc = fma(pc, a2, -0x1.93974a8c07c9dp-37);
    pc = fma(pc, a2, 0x1.1eed8eff8d898p-29);
    pc = fma(pc, a2, -0x1.27e4fb7789f5cp-22);
    pc = fma(pc, a2, 0x1.a01a01a01a01ap-16);
    pc = fma(pc, a2, -0x1.6c16c16c16c17p-10);
    pc = fma(pc, a2, 0x1.5555555555555p-5);
    pc = fma(pc, a2, -0x1.0000000000000p-1);
    const double ca = fma(pc, a2, 1.0);
    switch (q) {
        case 0: *sn = sa; *cs = ca; break;
        case 1: *sn = ca; *cs = -sa; break;
        case 2: *sn = -sa; *cs = -ca; break;
        default: *sn = -ca; *cs = sa; break;
    }
}

/* four standard normals from one Philox block (two Box-Muller pairs) */
MI_HD void mi_normals4(uint64_t seed, uint64_t stream, uint64_t q, double z[4]) {
    uint32_t r[4];
    mi_block(seed, stream, q, r);
    for (int h = 0; h < 2; ++h) {
        const double u1 = mi_unit_open(r[2 * h]), u2 = mi_unit_open(r[2 * h + 1]);
        const double rad = sqrt(-2.0 * mi_log(u1));
        double sn, cs;
        mi_sincos_turn(u2, &sn, &cs);
        z[2 * h] = rad * cs;
        z[2 * h + 1] = rad * sn;
    }
}

/* fp32 -> bf16 bits, round to nearest even; NaN maps to a quiet NaN */
MI_HD uint16_t mi_bf16_rne(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu)) return 0x7fc0;
    u += 0x7fffu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

#endif /* MOE_INPUTS_NORMAL_CORE_H */
