/*
 * GPU build of the seeded input generator: fills host buffers (normally the library's pinned
 * expert pool) with exactly the bits gen.c produces for the same (seed, stream, element), so
 * large pools are written at GPU speed instead of host speed. The arithmetic is the shared
 * core in normal_core.h; this file only schedules it (one thread per Philox block of four
 * elements) and copies the result to the host. It holds no arithmetic of the MoE method.
 * Built with -fmad=false so that no a*b+c outside the core's explicit fma is fused.
 */
#include <cuda_runtime.h>
#include <stdio.h>

#include "mxfp4_core.h"
#include "normal_core.h"
#include "nvfp4_core.h"

__global__ void mi_normal_bf16_kernel(uint64_t seed, uint64_t stream, uint64_t n, double stddev, uint16_t* out) {
    const uint64_t nq = (n + 3) / 4;
    for (uint64_t q = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; q < nq; q += (uint64_t)gridDim.x * blockDim.x) {
        double z[4];
        mi_normals4(seed, stream, q, z);
        for (int w = 0; w < 4; ++w) {
            const uint64_t i = q * 4 + w;
            if (i < n) out[i] = mi_bf16_rne((float)(z[w] * stddev));
        }
    }
}

// One thread per block of 32 weights of a bf16 entry (W_gate [I x H] | W_up [I x H] |
// W_down [H x I]): its E2M1 bytes and scale placed as mi_mxfp4_place says -- the bytes
// mi_mxfp4_entry of gen.c writes.
__global__ void mi_mxfp4_entry_kernel(const uint16_t* w, int H, int I, uint8_t* out) {
    const uint64_t n = 3ull * H * I, gate = (uint64_t)I * H;
    const uint64_t nblk = n / 32;
    for (uint64_t blk = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; blk < nblk;
         blk += (uint64_t)gridDim.x * blockDim.x) {
        const uint64_t elem = blk * 32;
        int mat, row, b;
        if (elem < 2 * gate) {
            mat = (int)(elem / gate);
            const uint64_t within = elem % gate;
            row = (int)(within / H);
            b = (int)((within % H) / 32);
        } else {
            mat = 2;
            const uint64_t within = elem - 2 * gate;
            row = (int)(within / I);
            b = (int)((within % I) / 32);
        }
        uint64_t co, so;
        mi_mxfp4_place(H, I, mat, row, b, &co, &so);
        mi_mxfp4_block(w + elem, out + co, out + so);
    }
}

// Largest magnitude of each of the three matrices of a bf16 entry, as fp32 bit patterns (a
// non-negative float's bits order like the float): amax_bits[m] must start at 0.
__global__ void mi_amax3_kernel(const uint16_t* w, uint64_t mat_elems, unsigned* amax_bits) {
    __shared__ unsigned best[3];
    if (threadIdx.x < 3) best[threadIdx.x] = 0u;
    __syncthreads();
    for (int m = 0; m < 3; ++m) {
        unsigned local = 0u;
        for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < mat_elems;
             i += (uint64_t)gridDim.x * blockDim.x) {
            const unsigned a = (unsigned)(w[m * mat_elems + i] & 0x7fff) << 16;
            local = a > local ? a : local;
        }
        atomicMax(&best[m], local);
    }
    __syncthreads();
    if (threadIdx.x < 3) atomicMax(&amax_bits[threadIdx.x], best[threadIdx.x]);
}

// One thread per block of 16 weights of a bf16 entry: its E2M1 bytes and E4M3 scale placed as
// mi_nvfp4_place says, with the matrix's tensor scale from mi_nvfp4_tensor_scale; thread 0
// also writes the 16-byte trailer -- the bytes mi_nvfp4_entry of gen.c writes.
__global__ void mi_nvfp4_entry_kernel(const uint16_t* w, int H, int I, const unsigned* amax_bits, uint8_t* out) {
    const uint64_t n = 3ull * H * I, gate = (uint64_t)I * H;
    float t[3];
    for (int m = 0; m < 3; ++m) t[m] = mi_nvfp4_tensor_scale(mi_bits_f32(amax_bits[m]));
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        uint8_t* trailer = out + mi_nvfp4_entry_bytes(H, I) - 16;
        memcpy(trailer, t, 12);
        memset(trailer + 12, 0, 4);
    }
    const uint64_t nblk = n / 16;
    for (uint64_t blk = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; blk < nblk;
         blk += (uint64_t)gridDim.x * blockDim.x) {
        const uint64_t elem = blk * 16;
        int mat, row, b;
        if (elem < 2 * gate) {
            mat = (int)(elem / gate);
            const uint64_t within = elem % gate;
            row = (int)(within / H);
            b = (int)((within % H) / 16);
        } else {
            mat = 2;
            const uint64_t within = elem - 2 * gate;
            row = (int)(within / I);
            b = (int)((within % I) / 16);
        }
        uint64_t co, so;
        mi_nvfp4_place(H, I, mat, row, b, &co, &so);
        mi_nvfp4_block(w + elem, t[mat], out + co, out + so);
    }
}

static int report(cudaError_t e, const char* what, char* err, int err_len) {
    if (err && err_len > 0) snprintf(err, err_len, "%s: %s", what, cudaGetErrorString(e));
    return -1;
}

/*
 * For each i < n_streams: host_dst[i][0 .. n) = elements [0, n) of stream streams[i], each
 * N(0, stddev) rounded to fp32 and then to bf16 -- the same bits as mi_normal_bf16 of gen.c.
 * Runs on the current device with two device staging buffers (generation of one stream
 * overlaps the copy-out of the previous). Returns 0, or -1 with a message in err.
 */
extern "C" int mi_gpu_normal_bf16_to_host(uint64_t seed, int n_streams, const uint64_t* streams, uint64_t n,
                                          double stddev, void* const* host_dst, char* err, int err_len) {
    if (n_streams <= 0 || n == 0) return 0;
    uint16_t* buf[2] = {nullptr, nullptr};
    cudaEvent_t done[2] = {nullptr, nullptr};
    cudaStream_t st = nullptr;
    cudaError_t e = cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking);
    if (e != cudaSuccess) return report(e, "stream", err, err_len);
    int rc = 0;
    for (int b = 0; b < 2 && rc == 0; ++b) {
        if ((e = cudaMalloc(&buf[b], n * sizeof(uint16_t))) != cudaSuccess) rc = report(e, "cudaMalloc", err, err_len);
        else if ((e = cudaEventCreateWithFlags(&done[b], cudaEventDisableTiming)) != cudaSuccess)
            rc = report(e, "event", err, err_len);
        else if ((e = cudaEventRecord(done[b], st)) != cudaSuccess) rc = report(e, "event record", err, err_len);
    }
    const uint64_t nq = (n + 3) / 4;
    const unsigned grid = (unsigned)((nq + 255) / 256 < 148 * 16 ? (nq + 255) / 256 : 148 * 16);
    for (int i = 0; i < n_streams && rc == 0; ++i) {
        const int b = i & 1;
        // the buffer's previous copy-out must be done before it is overwritten (stream order)
        mi_normal_bf16_kernel<<<grid, 256, 0, st>>>(seed, streams[i], n, stddev, buf[b]);
        if ((e = cudaGetLastError()) != cudaSuccess) rc = report(e, "generator launch", err, err_len);
        else if ((e = cudaMemcpyAsync(host_dst[i], buf[b], n * sizeof(uint16_t), cudaMemcpyDeviceToHost, st)) !=
                 cudaSuccess)
            rc = report(e, "copy to host", err, err_len);
    }
    if (rc == 0 && (e = cudaStreamSynchronize(st)) != cudaSuccess) rc = report(e, "synchronize", err, err_len);
    for (int b = 0; b < 2; ++b) {
        if (buf[b]) cudaFree(buf[b]);
        if (done[b]) cudaEventDestroy(done[b]);
    }
    cudaStreamDestroy(st);
    return rc;
}

/*
 * MXFP4 entries on the GPU: for each stream, the N(0, stddev) bf16 entry (3*H*I weights) is
 * generated and quantized as gen.c's mi_mxfp4_entry does, and the 3*H*I*17/32 bytes are copied
 * to host_dst[i]. Returns 0, or -1 with a message in err.
 */
extern "C" int mi_gpu_mxfp4_entries_to_host(uint64_t seed, int n_streams, const uint64_t* streams, int H, int I,
                                            double stddev, void* const* host_dst, char* err, int err_len) {
    if (n_streams <= 0) return 0;
    const uint64_t n = 3ull * H * I, bytes = n / 2 + n / 32;
    uint16_t* w = nullptr;
    uint8_t* buf[2] = {nullptr, nullptr};
    cudaStream_t st = nullptr;
    cudaError_t e = cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking);
    if (e != cudaSuccess) return report(e, "stream", err, err_len);
    int rc = 0;
    if ((e = cudaMalloc(&w, n * sizeof(uint16_t))) != cudaSuccess) rc = report(e, "cudaMalloc", err, err_len);
    for (int b = 0; b < 2 && rc == 0; ++b)
        if ((e = cudaMalloc(&buf[b], bytes)) != cudaSuccess) rc = report(e, "cudaMalloc", err, err_len);
    const uint64_t nq = (n + 3) / 4;
    const unsigned grid = (unsigned)((nq + 255) / 256 < 148 * 16 ? (nq + 255) / 256 : 148 * 16);
    const unsigned qgrid = (unsigned)((n / 32 + 255) / 256 < 148 * 16 ? (n / 32 + 255) / 256 : 148 * 16);
    for (int i = 0; i < n_streams && rc == 0; ++i) {
        mi_normal_bf16_kernel<<<grid, 256, 0, st>>>(seed, streams[i], n, stddev, w);
        mi_mxfp4_entry_kernel<<<qgrid, 256, 0, st>>>(w, H, I, buf[i & 1]);
        if ((e = cudaGetLastError()) != cudaSuccess) rc = report(e, "generator launch", err, err_len);
        else if ((e = cudaMemcpyAsync(host_dst[i], buf[i & 1], bytes, cudaMemcpyDeviceToHost, st)) != cudaSuccess)
            rc = report(e, "copy to host", err, err_len);
    }
    if (rc == 0 && (e = cudaStreamSynchronize(st)) != cudaSuccess) rc = report(e, "synchronize", err, err_len);
    if (w) cudaFree(w);
    for (int b = 0; b < 2; ++b)
        if (buf[b]) cudaFree(buf[b]);
    cudaStreamDestroy(st);
    return rc;
}

/*
 * NVFP4 entries on the GPU: for each stream, the N(0, stddev) bf16 entry (3*H*I weights) is
 * generated and quantized as gen.c's mi_nvfp4_entry does (tensor scale per matrix, E4M3 scale
 * per 16 weights, trailer of tensor scales), and the mi_nvfp4_entry_bytes(H, I) bytes are copied
 * to host_dst[i]. Returns 0, or -1 with a message in err.
 */
extern "C" int mi_gpu_nvfp4_entries_to_host(uint64_t seed, int n_streams, const uint64_t* streams, int H, int I,
                                            double stddev, void* const* host_dst, char* err, int err_len) {
    if (n_streams <= 0) return 0;
    const uint64_t n = 3ull * H * I, bytes = mi_nvfp4_entry_bytes(H, I);
    uint16_t* w = nullptr;
    uint8_t* buf[2] = {nullptr, nullptr};
    unsigned* amax = nullptr;
    cudaStream_t st = nullptr;
    cudaError_t e = cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking);
    if (e != cudaSuccess) return report(e, "stream", err, err_len);
    int rc = 0;
    if ((e = cudaMalloc(&w, n * sizeof(uint16_t))) != cudaSuccess) rc = report(e, "cudaMalloc", err, err_len);
    if (rc == 0 && (e = cudaMalloc(&amax, 3 * sizeof(unsigned))) != cudaSuccess)
        rc = report(e, "cudaMalloc", err, err_len);
    for (int b = 0; b < 2 && rc == 0; ++b)
        if ((e = cudaMalloc(&buf[b], bytes)) != cudaSuccess) rc = report(e, "cudaMalloc", err, err_len);
    const uint64_t nq = (n + 3) / 4;
    const unsigned grid = (unsigned)((nq + 255) / 256 < 148 * 16 ? (nq + 255) / 256 : 148 * 16);
    const unsigned qgrid = (unsigned)((n / 16 + 255) / 256 < 148 * 16 ? (n / 16 + 255) / 256 : 148 * 16);
    for (int i = 0; i < n_streams && rc == 0; ++i) {
        mi_normal_bf16_kernel<<<grid, 256, 0, st>>>(seed, streams[i], n, stddev, w);
        if ((e = cudaMemsetAsync(amax, 0, 3 * sizeof(unsigned), st)) != cudaSuccess) {
            rc = report(e, "memset", err, err_len);
            break;
        }
        mi_amax3_kernel<<<148 * 4, 256, 0, st>>>(w, (uint64_t)I * H, amax);
        mi_nvfp4_entry_kernel<<<qgrid, 256, 0, st>>>(w, H, I, amax, buf[i & 1]);
        if ((e = cudaGetLastError()) != cudaSuccess) rc = report(e, "generator launch", err, err_len);
        else if ((e = cudaMemcpyAsync(host_dst[i], buf[i & 1], bytes, cudaMemcpyDeviceToHost, st)) != cudaSuccess)
            rc = report(e, "copy to host", err, err_len);
    }
    if (rc == 0 && (e = cudaStreamSynchronize(st)) != cudaSuccess) rc = report(e, "synchronize", err, err_len);
    if (w) cudaFree(w);
    if (amax) cudaFree(amax);
    for (int b = 0; b < 2; ++b)
        if (buf[b]) cudaFree(buf[b]);
    cudaStreamDestroy(st);
    return rc;
}
