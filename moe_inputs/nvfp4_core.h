/*
 * NVFP4 quantization of the seeded bf16 expert weights (input preparation; no arithmetic of the
 * MoE method). Integer operations, comparisons and single IEEE-rounded fp32 operations in a
 * fixed order only, so every build writes the same bytes.
 *
 * Format (NVIDIA's NVFP4, as this library reads it): each run of 16 consecutive elements of a
 * row shares one scale stored as FP8 E4M3 (sign 0, 4 exponent bits with bias 7, 3 mantissa
 * bits, largest finite value 448, no infinities); each element is E2M1 as in MXFP4
 * (magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6, bit 3 the sign), two per byte, the even element in
 * the low nibble; each matrix carries one fp32 tensor scale. An element's value is
 * e2m1 * e4m3(block scale) * tensor scale.
 *
 * Quantization of a matrix with largest magnitude A: tensor scale t = A / 2688 (6 * 448) in
 * fp32, or 1 when A = 0. A block with largest magnitude a gets the E4M3 scale
 * s = rne_e4m3((a / t) / 6), saturating at 448; each element is rne_e2m1(|x| / (e4m3(s) * t))
 * (the fp32 product, then the fp32 quotient), ties to the even mantissa, magnitudes above 6
 * clamped to 6; a block whose scale rounds to 0 stores zero codes (signs kept).
 */
#ifndef MOE_INPUTS_NVFP4_CORE_H
#define MOE_INPUTS_NVFP4_CORE_H

#include <stdint.h>
#include <string.h>

#include "mxfp4_core.h" /* mi_bf16_to_f32, mi_e2m1_code, mi_pow2f */

MI_HD uint32_t mi_f32_bits(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    return u;
}

MI_HD float mi_bits_f32(uint32_t u) {
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* E4M3 code of v >= 0 (finite), round to nearest even, saturating at 448 (code 0x7e). */
MI_HD uint8_t mi_e4m3_rne(float v) {
    if (!(v > 0.0f)) return 0;
    const uint32_t u = mi_f32_bits(v);
    int e = (int)((u >> 23) & 0xff) - 127;
    if (e < -6) {
        /* subnormal range: units of 2^-9; v * 2^9 is exact, then round to an integer */
        const float m = v * 512.0f;
        const uint32_t mu = mi_f32_bits(m);
        const int me = (int)((mu >> 23) & 0xff) - 127; /* m < 8, so me <= 2 */
        if (me < -1) return 0;                         /* m < 0.5 */
        /* m = 1.f * 2^me with me in [-1, 2]: integer part and the dropped fraction */
        const uint32_t mant = (mu & 0x7fffff) | 0x800000;
        const int shift = 23 - me;
        uint32_t q = mant >> shift;
        const uint32_t rem = mant & ((1u << shift) - 1), half = 1u << (shift - 1);
        if (rem > half || (rem == half && (q & 1u))) ++q;
        return (uint8_t)q; /* 8 is the smallest normal (exponent field 1, mantissa 0) */
    }
    uint32_t m3 = (u >> 20) & 7;
    const uint32_t rem = u & 0xfffff, half = 0x80000;
    if (rem > half || (rem == half && (m3 & 1u))) {
        if (++m3 == 8) {
            m3 = 0;
            ++e;
        }
    }
    if (e > 8 || (e == 8 && m3 == 7)) return 0x7e; /* 448 */
    return (uint8_t)(((e + 7) << 3) | m3);
}

/* The value of an E4M3 code (no NaN is ever produced by mi_e4m3_rne). */
MI_HD float mi_e4m3_value(uint8_t c) {
    const int ef = (c >> 3) & 15, m = c & 7;
    if (ef == 0) return (float)m * mi_pow2f(-9);
    return (float)(8 + m) * mi_pow2f(ef - 10); /* (1 + m/8) * 2^(ef-7) */
}

/* Tensor scale of a matrix whose largest magnitude is amax. */
MI_HD float mi_nvfp4_tensor_scale(float amax) { return amax > 0.0f ? amax / 2688.0f : 1.0f; }

/* One block of 16 bf16 values -> 8 bytes of E2M1 pairs and the E4M3 scale byte. */
MI_HD void mi_nvfp4_block(const uint16_t* x, float t, uint8_t* q, uint8_t* s) {
    float amax = 0.0f;
    for (int i = 0; i < 16; ++i) {
        const float a = mi_bf16_to_f32(x[i] & 0x7fff);
        if (a > amax) amax = a;
    }
    const uint8_t sc = mi_e4m3_rne((amax / t) / 6.0f);
    *s = sc;
    const float denom = mi_e4m3_value(sc) * t;
    for (int i = 0; i < 8; ++i) {
        uint32_t byte = 0;
        for (int h = 0; h < 2; ++h) {
            const uint16_t b = x[2 * i + h];
            uint32_t code = 0;
            if (denom > 0.0f) code = mi_e2m1_code(mi_bf16_to_f32(b & 0x7fff) / denom);
            code |= (b & 0x8000) ? 8u : 0u;
            byte |= code << (4 * h);
        }
        q[i] = (uint8_t)byte;
    }
}

/*
 * Place of a 16-block in an NVFP4 expert entry. Stages of 4608 bytes = 4096 bytes of E2M1
 * codes + 512 scale bytes, in the order a decode kernel would stream them:
 *  - W_gate and W_up [I x H]: per 64-row tile t and 64-column slab k (t-major), one stage =
 *    gate rows (64 x 32 bytes), up rows (64 x 32), gate scales (64 x 4), up scales (64 x 4);
 *  - then W_down [H x I]: per 128-row tile and 64-column slab, rows (128 x 32), scales (128 x 4);
 *  - then 16 bytes: the fp32 tensor scales of W_gate, W_up and W_down, and 4 zero bytes.
 * Within a row of a stage, block j (0..3) of the slab takes bytes 8j .. 8j+7 and scale byte
 * 4*row + j. mat: 0 gate, 1 up, 2 down; b: the 16-block index along the row.
 */
MI_HD void mi_nvfp4_place(int H, int I, int mat, int row, int b, uint64_t* code_off, uint64_t* scale_off) {
    const uint64_t stage_bytes = 4608;
    const int k = b / 4, j = b % 4;
    if (mat < 2) {
        const uint64_t stage = ((uint64_t)(row / 64) * (H / 64) + k) * stage_bytes;
        const int rr = row % 64;
        *code_off = stage + (uint64_t)mat * 2048 + rr * 32 + j * 8;
        *scale_off = stage + 4096 + (uint64_t)mat * 256 + rr * 4 + j;
    } else {
        const uint64_t gu = (uint64_t)(I / 64) * (H / 64) * stage_bytes;
        const uint64_t stage = gu + ((uint64_t)(row / 128) * (I / 64) + k) * stage_bytes;
        const int rr = row % 128;
        *code_off = stage + rr * 32 + j * 8;
        *scale_off = stage + 4096 + rr * 4 + j;
    }
}

/* Bytes of an NVFP4 entry: codes, scales and the 16-byte tensor-scale trailer. */
MI_HD uint64_t mi_nvfp4_entry_bytes(int H, int I) {
    return (uint64_t)3 * H * I / 2 + (uint64_t)3 * H * I / 16 + 16;
}

#endif /* MOE_INPUTS_NVFP4_CORE_H */
