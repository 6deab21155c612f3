/*
 * MXFP4 quantization of the seeded bf16 expert weights, shared by the CPU build (gen.c) and
 * the GPU build (gen_gpu.cu) of the input generator so both write the same bytes. Integer
 * and exact floating-point operations only (comparisons, multiplication by powers of two).
 *
 * Format (OCP Microscaling, MXFP4): each run of 32 consecutive elements of a row shares one
 * E8M0 scale byte s (value 2^(s-127)); each element is E2M1 -- sign, 2-bit exponent, 1-bit
 * mantissa -- with magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6 for codes 0..7, bit 3 the sign.
 * Two elements per byte, the even element in the low nibble.
 *
 * Quantization of a block: shared exponent e = floor(log2(max |x|)) - 2 (2 is the largest
 * E2M1 exponent), clamped to [-127, 127]; each element is x / 2^e rounded to the nearest
 * E2M1 magnitude, ties to the even mantissa bit, magnitudes above 6 clamped to 6. An all-zero
 * block gets s = 0. This file holds no arithmetic of the MoE method: it prepares inputs.
 */
#ifndef MOE_INPUTS_MXFP4_CORE_H
#define MOE_INPUTS_MXFP4_CORE_H

#include <stdint.h>
#include <string.h>

#ifndef MI_HD
#ifdef __CUDACC__
#define MI_HD static __host__ __device__ __forceinline__
#else
#define MI_HD static inline
#endif
#endif

MI_HD float mi_bf16_to_f32(uint16_t b) {
    const uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* 2^k as a float, for k in [-126, 127] (exact) */
MI_HD float mi_pow2f(int k) {
    const uint32_t u = (uint32_t)(k + 127) << 23;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* floor(log2(a)) for a finite a > 0 */
MI_HD int mi_ilog2f(float a) {
    uint32_t u;
    memcpy(&u, &a, 4);
    const int ex = (int)((u >> 23) & 0xff);
    if (ex > 0) return ex - 127;
    int e = -127; /* subnormal: find the leading mantissa bit */
    uint32_t m = u & 0x7fffff;
    while (!(m & 0x400000)) {
        m <<= 1;
        --e;
    }
    return e;
}

/* E2M1 magnitude code of a >= 0 (already divided by the block scale), ties to even */
MI_HD uint32_t mi_e2m1_code(float a) {
    if (a <= 0.25f) return 0;
    if (a < 0.75f) return 1;
    if (a <= 1.25f) return 2;
    if (a < 1.75f) return 3;
    if (a <= 2.5f) return 4;
    if (a < 3.5f) return 5;
    if (a <= 5.0f) return 6;
    return 7;
}

/* One block of 32 bf16 values -> 16 bytes of E2M1 pairs and the E8M0 scale byte. */
MI_HD void mi_mxfp4_block(const uint16_t* x, uint8_t* q, uint8_t* s) {
    float amax = 0.0f;
    for (int i = 0; i < 32; ++i) {
        const float a = mi_bf16_to_f32(x[i] & 0x7fff);
        if (a > amax) amax = a;
    }
    int e = -127;
    if (amax > 0.0f) {
        e = mi_ilog2f(amax) - 2;
        if (e < -127) e = -127;
        if (e > 127) e = 127;
    }
    *s = (uint8_t)(e + 127);
    /* x / 2^e = x * 2^-e (exact); 2^-127 (e = 127) is taken as 2^-126 * 2^-1 */
    const int k = -e;
    const float inv_a = k >= -126 ? mi_pow2f(k) : mi_pow2f(-126);
    const float inv_b = k >= -126 ? 1.0f : 0.5f;
    for (int i = 0; i < 16; ++i) {
        uint32_t byte = 0;
        for (int h = 0; h < 2; ++h) {
            const uint16_t b = x[2 * i + h];
            const float a = mi_bf16_to_f32(b & 0x7fff) * inv_a * inv_b;
            const uint32_t code = mi_e2m1_code(a) | ((b & 0x8000) ? 8u : 0u);
            byte |= code << (4 * h);
        }
        q[i] = (uint8_t)byte;
    }
}

/* rows x K bf16 (row-major, K % 32 == 0) -> q [rows x K/2] bytes, s [rows x K/32] bytes */
MI_HD void mi_mxfp4_rows(const uint16_t* x, int rows, int K, uint8_t* q, uint8_t* s) {
    for (int r = 0; r < rows; ++r)
        for (int b = 0; b < K / 32; ++b)
            mi_mxfp4_block(x + (size_t)r * K + 32 * b, q + (size_t)r * (K / 2) + 16 * b, s + (size_t)r * (K / 32) + b);
}

/*
 * Place of a block in an MXFP4 expert entry. The entry is stored in the order the decode
 * kernels stream it, in stages of 4352 bytes = 4096 bytes of E2M1 codes + 256 scale bytes:
 *  - W_gate and W_up [I x H]: for each 64-row tile t and 64-column slab k (t-major), one stage
 *    = gate rows (64 x 32 bytes), up rows (64 x 32 bytes), gate scales (64 x 2), up scales (64 x 2);
 *  - then W_down [H x I]: for each 128-row tile t and 64-column slab k, one stage = the rows
 *    (128 x 32 bytes), then their scales (128 x 2).
 * Within a row of a stage, block `half` (0 or 1) of the slab takes bytes 16*half .. +15 and
 * scale byte 2*row + half. mat: 0 gate, 1 up, 2 down; b: the 32-block index along the row.
 */
MI_HD void mi_mxfp4_place(int H, int I, int mat, int row, int b, uint64_t* code_off, uint64_t* scale_off) {
    const uint64_t stage_bytes = 4352;
    const int k = b / 2, half = b % 2;
    if (mat < 2) {
        const uint64_t stage = ((uint64_t)(row / 64) * (H / 64) + k) * stage_bytes;
        const int rr = row % 64;
        *code_off = stage + (uint64_t)mat * 2048 + rr * 32 + half * 16;
        *scale_off = stage + 4096 + (uint64_t)mat * 128 + rr * 2 + half;
    } else {
        const uint64_t gu = (uint64_t)(I / 64) * (H / 64) * stage_bytes;
        const uint64_t stage = gu + ((uint64_t)(row / 128) * (I / 64) + k) * stage_bytes;
        const int rr = row % 128;
        *code_off = stage + rr * 32 + half * 16;
        *scale_off = stage + 4096 + rr * 2 + half;
    }
}

#endif /* MOE_INPUTS_MXFP4_CORE_H */
