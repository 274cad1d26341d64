// aux_kernels.cu -- small kernels around the fused operators: the MXFP8
// quantiser and the device-side rail decode used to check ticket order.
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "mxfp8.cuh"
#include "launch.h"

namespace kosmos {

__device__ __forceinline__ float bf16_bits_to_float(uint16_t h) { return __uint_as_float(static_cast<uint32_t>(h) << 16); }

// One thread per 32-element block; scale rows beyond the operand (padding of
// the last 128-row atom) get the neutral scale 2^0.
__global__ void mxfp8_quantize_kernel(const uint16_t *__restrict__ x, int64_t rows, int64_t cols, int along_cols,
                                      uint8_t *__restrict__ q, uint8_t *__restrict__ scales) {
    const int64_t srows = along_cols ? rows : cols;       // scale rows
    const int64_t kblocks = along_cols ? cols / 32 : rows / 32;
    const int64_t srows_pad = cdiv(srows, 128) * 128;
    const int64_t nblk = srows_pad * kblocks;
    for (int64_t bi = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; bi < nblk;
         bi += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        int64_t base, step, sidx;
        if (along_cols) {
            const int64_t r = bi / kblocks, kb = bi % kblocks;
            if (r >= rows) {
                scales[sf_tiled_offset(r, kb, kblocks)] = 127;
                continue;
            }
            base = r * cols + kb * 32;
            step = 1;
            sidx = sf_tiled_offset(r, kb, kblocks);
        } else {
            // consecutive threads take consecutive columns of the same 32-row block
            const int64_t kb = bi / srows_pad, c = bi % srows_pad;
            if (c >= cols) {
                scales[sf_tiled_offset(c, kb, kblocks)] = 127;
                continue;
            }
            base = kb * 32 * cols + c;
            step = cols;
            sidx = sf_tiled_offset(c, kb, kblocks);
        }
        float mx = 0.f;
        for (int j = 0; j < 32; ++j) mx = fmaxf(mx, fabsf(bf16_bits_to_float(x[base + j * step])));
        const int e = mx_block_exp(mx);
        const float inv = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);  // 2^-e, a normal float
        scales[sidx] = static_cast<uint8_t>(e + 127);
        for (int j = 0; j < 32; ++j) {
            const float v = bf16_bits_to_float(x[base + j * step]) * inv;  // exact: power-of-two scale
            q[base + j * step] = static_cast<uint8_t>(__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3));
        }
    }
}

kosmos_status launch_mxfp8_quantize(const void *x, int64_t rows, int64_t cols, int along_cols, void *q, void *scales,
                                    cudaStream_t stream) {
    const int64_t nblk = cdiv(along_cols ? rows : cols, 128) * 128 * (along_cols ? cols / 32 : rows / 32);
    int64_t blocks = cdiv(nblk, 256);
    if (blocks > 65535) blocks = 65535;
    if (blocks < 1) blocks = 1;
    mxfp8_quantize_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
        static_cast<const uint16_t *>(x), rows, cols, along_cols, static_cast<uint8_t *>(q),
        static_cast<uint8_t *>(scales));
    return cudaGetLastError() == cudaSuccess ? KOSMOS_OK : KOSMOS_ERR_CUDA;
}

__global__ void rail_decode_kernel(int op, int P, int64_t m, int64_t n, int order, int rank, int rail, int tile_m,
                                   int64_t split, int32_t *out, int64_t count) {
    for (int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; t < count;
         t += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        int32_t *e = out + 4 * t;
        if (op == KOSMOS_OP_AG_GEMM) {
            const AgGeom g = ag_geom(P, m, 64, n, tile_m, split);
            if (rail == 0) {
                int s, j, q;
                ag_decode_transfer(g, static_cast<int>(t), s, j, q);
                e[0] = K_TRANSFER; e[1] = s; e[2] = j; e[3] = q;
            } else {
                int s, i, c;
                const int kind = ag_decode_tile(g, static_cast<int>(t), s, i, c);
                e[0] = kind; e[1] = s; e[2] = i; e[3] = c;
            }
        } else {
            const RsGeom g = rs_geom(P, m, 64, n, tile_m);
            if (rail == 0) {
                int q, c, b, j;
                rs_decode_tile(g, order, static_cast<int>(t), q, c, b, j);
                e[0] = K_TILE; e[1] = q * P + c; e[2] = b; e[3] = j;
            } else {
                int b, j;
                rs_decode_reduce(g, static_cast<int>(t), b, j);
                e[0] = K_REDUCE; e[1] = rank; e[2] = b; e[3] = j;
            }
        }
    }
}

kosmos_status launch_rail_decode(int op, int P, int64_t m, int64_t n, int order, int rank, int rail, int tile_m,
                                 int64_t split, int32_t *out, int64_t count, cudaStream_t stream) {
    int64_t blocks = cdiv(count, 256);
    if (blocks < 1) blocks = 1;
    if (blocks > 4096) blocks = 4096;
    rail_decode_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(op, P, m, n, order, rank, rail, tile_m, split,
                                                                           out, count);
    return cudaGetLastError() == cudaSuccess ? KOSMOS_OK : KOSMOS_ERR_CUDA;
}

}  // namespace kosmos
