// quantize.cu -- load-time weight quantization (Q4_0), the standalone INIT
// stage (Q8_0 of activation rows) and the load-time repack of Q4_0 weights.
//
// One warp per block of 32 values: lane j owns element j, the block's maximum
// magnitude is a warp reduction, and the codes are decided in f32 exactly as
// the block formats define them (IEEE division, roundf, fp16 round-to-even).
#include "gq_common.cuh"
#include "gq_internal.h"

namespace gq {
namespace {

// Q4_0 (llama.cpp PR #1632, "Introduction": src0 of the q_f32 kind is quantized).
__global__ void quantize_q4_0_kernel(const float *__restrict__ w, uint8_t *__restrict__ out,
                                     int64_t nblocks) {
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t b = warp; b < nblocks; b += nwarps) {
        const float x = w[b * QK + lane];          // K % 32 == 0: block b is 32 contiguous floats
        // magnitudes are non-negative, so their bit patterns order like the values
        const unsigned int abits = __float_as_uint(fabsf(x));
        const unsigned int amax = __reduce_max_sync(0xffffffffu, abits);
        const unsigned int first = __ffs(__ballot_sync(0xffffffffu, abits == amax)) - 1;
        float vmax = __shfl_sync(0xffffffffu, x, first);
        if (amax == 0u) vmax = 0.0f;               // no element exceeded zero: the signed max stays +0
        const float d = vmax / -8.0f;
        int q = 8;
        if (d != 0.0f) {
            const int v = (int)roundf(x / d) + 8;
            q = v < 0 ? 0 : (v > 15 ? 15 : v);
        }
        const int qhi = __shfl_down_sync(0xffffffffu, q, 16);
        uint8_t *o = out + b * Q4_0_BYTES;            // 2-byte aligned: 18 * b is even
        if (lane < 16) o[2 + lane] = (uint8_t)(q | (qhi << 4));
        if (lane == 0) *reinterpret_cast<unsigned short *>(o) = __half_as_ushort(__float2half_rn(d));
    }
}

// Q5_0 of weight blocks: one warp per block, lane j holds element j.  d = (signed max) / -16,
// q = clamp(round(x / d) + 16, 0, 31) (16 when d == 0); block = fp16 d, the fifth bits as a
// little-endian word (bit j from lane j), 16 bytes of low nibbles (q_i | q_{i+16} << 4).
__global__ void quantize_q5_0_kernel(const float *__restrict__ w, uint8_t *__restrict__ out, int64_t nblocks) {
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t b = warp; b < nblocks; b += nwarps) {
        const float x = w[b * QK + lane];
        const unsigned int abits = __float_as_uint(fabsf(x));
        const unsigned int amax = __reduce_max_sync(0xffffffffu, abits);
        const unsigned int first = __ffs(__ballot_sync(0xffffffffu, abits == amax)) - 1;
        float vmax = __shfl_sync(0xffffffffu, x, first);
        if (amax == 0u) vmax = 0.0f;
        const float d = vmax / -16.0f;
        int q = 16;
        if (d != 0.0f) {
            const int v = (int)roundf(x / d) + 16;
            q = v < 0 ? 0 : (v > 31 ? 31 : v);
        }
        const unsigned int qh = __ballot_sync(0xffffffffu, (q >> 4) & 1);
        const int qhi = __shfl_down_sync(0xffffffffu, q, 16);
        uint8_t *o = out + b * 22;                         // 2-byte aligned: 22 * b is even
        if (lane < 16) o[6 + lane] = (uint8_t)((q & 0x0F) | ((qhi & 0x0F) << 4));
        if (lane < 4) o[2 + lane] = (uint8_t)(qh >> (8 * lane));
        if (lane == 0) *reinterpret_cast<unsigned short *>(o) = __half_as_ushort(__float2half_rn(d));
    }
}

// Q4_1 of weight blocks: one warp per block.  lo / hi = the first element (in index order)
// equal to the block's minimum / maximum, d = (hi - lo) / 15, q = clamp(round((x - lo) / d), 0, 15)
// (0 when d == 0); block = fp16 d, fp16 lo, 16 bytes q_i | q_{i+16} << 4.
__global__ void quantize_q4_1_kernel(const float *__restrict__ w, uint8_t *__restrict__ out, int64_t nblocks) {
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t b = warp; b < nblocks; b += nwarps) {
        const float x = w[b * QK + lane];
        float mn = x, mx = x;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        }
        // the values equal to the extreme compare equal whatever their zero sign: take the first
        const float lo = __shfl_sync(0xffffffffu, x, __ffs(__ballot_sync(0xffffffffu, x == mn)) - 1);
        const float hi = __shfl_sync(0xffffffffu, x, __ffs(__ballot_sync(0xffffffffu, x == mx)) - 1);
        const float d = (hi - lo) / 15.0f;
        int q = 0;
        if (d != 0.0f) {
            const int v = (int)roundf((x - lo) / d);
            q = v < 0 ? 0 : (v > 15 ? 15 : v);
        }
        const int qhi = __shfl_down_sync(0xffffffffu, q, 16);
        uint8_t *o = out + b * 20;                         // 4-byte aligned: 20 * b
        if (lane < 16) o[4 + lane] = (uint8_t)(q | (qhi << 4));
        if (lane == 0) {
            *reinterpret_cast<unsigned short *>(o) = __half_as_ushort(__float2half_rn(d));
            *reinterpret_cast<unsigned short *>(o + 2) = __half_as_ushort(__float2half_rn(lo));
        }
    }
}

// Q8_0 of activation rows: the INIT stage that produces wdata (Arm China NUMA
// article, "MulMat 算子優化").
__global__ void quantize_rows_q8_0_kernel(const float *__restrict__ x, uint8_t *__restrict__ out,
                                          int64_t nblocks) {
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t b = warp; b < nblocks; b += nwarps) {
        const float v = x[b * QK + lane];
        const unsigned int amax = __reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(v)));
        const float d = __uint_as_float(amax) / 127.0f;
        uint8_t *o = out + b * Q8_0_BYTES;            // 2-byte aligned: 34 * b is even
        o[2 + lane] = (uint8_t)(q8_code_s(v, q8_scale(d)) & 0xff);
        if (lane == 0) *reinterpret_cast<unsigned short *>(o) = __half_as_ushort(__float2half_rn(d));
    }
}

// Load-time repack into the tiled layout documented with gq_repack_q4_0.  One
// thread per 16-byte piece of a tile: 64 pieces of codes (one block-row each)
// and 8 pieces of scales.
__global__ void repack_q4_0_kernel(const uint8_t *__restrict__ q4, uint8_t *__restrict__ rep,
                                   int64_t N, int64_t nb, int64_t NT, int64_t ntiles) {
    pdl_wait();
    const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t tile = tid / 72;
    if (tile >= ntiles) return;
    const int piece = (int)(tid % 72);
    const int64_t g = tile / NT, t = tile % NT;
    uint8_t *dst = rep + tile * TILE_BYTES;
    if (piece < 64) {
        const int j = piece / 16, r = piece % 16;
        const int64_t n = 16 * g + r, b = 4 * t + j;
        uint32_t wv[4] = {0x88888888u, 0x88888888u, 0x88888888u, 0x88888888u};
        if (n < N && b < nb) {
            const uint16_t *src = reinterpret_cast<const uint16_t *>(q4 + (n * nb + b) * Q4_0_BYTES + 2);
            for (int k = 0; k < 4; k++) wv[k] = (uint32_t)src[2 * k] | ((uint32_t)src[2 * k + 1] << 16);
        }
        *reinterpret_cast<uint4 *>(dst + piece * 16) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
    } else {
        const int q = piece - 64;                 // scales 8q .. 8q+7, index r*4 + j
        uint32_t hv[4];
        for (int k = 0; k < 4; k++) {
            uint32_t two = 0;
            for (int e = 0; e < 2; e++) {
                const int idx = 8 * q + 2 * k + e, r = idx / 4, j = idx % 4;
                const int64_t n = 16 * g + r, b = 4 * t + j;
                const uint32_t h = (n < N && b < nb) ? *reinterpret_cast<const uint16_t *>(q4 + (n * nb + b) * Q4_0_BYTES)
                                                     : 0u;
                two |= h << (16 * e);
            }
            hv[k] = two;
        }
        *reinterpret_cast<uint4 *>(dst + TILE_SCALE_OFFSET + q * 16) = make_uint4(hv[0], hv[1], hv[2], hv[3]);
    }
}

// F16 weights [N][K] -> tiles of 16 rows x 32 columns, 64 bytes per row, tile (g, t)
// of row group g and column tile t at (g * NT + t) * 1024.  One thread per 16-byte
// piece (64 per tile); rows past N are zeros.
__global__ void repack_f16_kernel(const uint8_t *__restrict__ w, uint8_t *__restrict__ out, int64_t N, int64_t K,
                                  int64_t NT, int64_t pieces) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < pieces;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t tile = i / 64, pc = i % 64;
        const int64_t g = tile / NT, t = tile % NT;
        const int64_t row = 16 * g + pc / 4, col = 32 * t + 8 * (pc % 4);
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (row < N) v = *reinterpret_cast<const uint4 *>(w + (row * K + col) * 2);
        *reinterpret_cast<uint4 *>(out + i * 16) = v;
    }
}

// Q8_0 blocks [N][nb] x 34 -> tiles of 16 rows x 4 blocks: the 32 codes of block j of row r at
// (j * 16 + r) * 32, then the fp16 scale at 2048 + (r * 4 + j) * 2; tile (g, t) at (g * NT + t) * 2176.
// One thread per (tile, row, block); rows past N and blocks past nb hold codes 0 and scale 0.
__global__ void repack_q8_0_kernel(const uint8_t *__restrict__ q8, uint8_t *__restrict__ out, int64_t N,
                                   int64_t nb, int64_t NT, int64_t items) {
    constexpr int TB = 16 * TILE_BLOCKS * (QK + 2), SC = 16 * TILE_BLOCKS * QK;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < items;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t tile = i / 64, rj = i % 64;
        const int r = (int)(rj / 4), j = (int)(rj % 4);
        const int64_t g = tile / NT, t = tile % NT;
        const int64_t n = 16 * g + r, b = 4 * t + j;
        uint8_t *dt = out + tile * TB;
        uint4 c0 = make_uint4(0u, 0u, 0u, 0u), c1 = c0;
        uint16_t d = 0;
        if (n < N && b < nb) {
            const uint8_t *src = q8 + (n * nb + b) * 34;
            uint32_t w[8];
            for (int k = 0; k < 8; k++)
                w[k] = (uint32_t)src[2 + 4 * k] | ((uint32_t)src[3 + 4 * k] << 8) | ((uint32_t)src[4 + 4 * k] << 16) |
                       ((uint32_t)src[5 + 4 * k] << 24);
            c0 = make_uint4(w[0], w[1], w[2], w[3]);
            c1 = make_uint4(w[4], w[5], w[6], w[7]);
            d = (uint16_t)(src[0] | (src[1] << 8));
        }
        *reinterpret_cast<uint4 *>(dt + (j * 16 + r) * 32) = c0;
        *reinterpret_cast<uint4 *>(dt + (j * 16 + r) * 32 + 16) = c1;
        *reinterpret_cast<uint16_t *>(dt + SC + (r * 4 + j) * 2) = d;
    }
}

// Q5_0 blocks [N][nb] x 22 -> tiles of 16 rows x 4 blocks, 1408 bytes: the 16 nibble bytes of
// block j of row r at (j * 16 + r) * 16, its fifth bits at 1024 + (j * 16 + r) * 4 arranged as
// block_dot_q5 reads them (bit 8b + 7 - s = fifth bit of element b of group s: groups 0..3 are
// elements 4s .., groups 4..7 elements 16 + 4(s - 4) ..), then the fp16 scales at
// 1280 + (r * 4 + j) * 2.  One thread per (tile, row, block); padding holds codes 16 and scale 0.
__global__ void repack_q5_0_kernel(const uint8_t *__restrict__ q5, uint8_t *__restrict__ out, int64_t N,
                                   int64_t nb, int64_t NT, int64_t items) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < items;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t tile = i / 64, rj = i % 64;
        const int r = (int)(rj / 4), j = (int)(rj % 4);
        const int64_t g = tile / NT, t = tile % NT;
        const int64_t n = 16 * g + r, b = 4 * t + j;
        uint8_t *dt = out + tile * 1408;
        uint32_t nib[4] = {0u, 0u, 0u, 0u}, qh = 0xFFFFFFFFu;   // padding: code 16 = nibble 0, fifth bit 1
        uint16_t d = 0;
        if (n < N && b < nb) {
            const uint8_t *src = q5 + (n * nb + b) * 22;
            d = (uint16_t)(src[0] | (src[1] << 8));
            qh = (uint32_t)src[2] | ((uint32_t)src[3] << 8) | ((uint32_t)src[4] << 16) | ((uint32_t)src[5] << 24);
            for (int k = 0; k < 4; k++)
                nib[k] = (uint32_t)src[6 + 4 * k] | ((uint32_t)src[7 + 4 * k] << 8) | ((uint32_t)src[8 + 4 * k] << 16) |
                         ((uint32_t)src[9 + 4 * k] << 24);
        }
        uint32_t h = 0;
        for (int sg = 0; sg < 8; sg++)
            for (int bb = 0; bb < 4; bb++) {
                const int e = sg < 4 ? 4 * sg + bb : 16 + 4 * (sg - 4) + bb;
                h |= ((qh >> e) & 1u) << (8 * bb + 7 - sg);
            }
        *reinterpret_cast<uint4 *>(dt + (j * 16 + r) * 16) = make_uint4(nib[0], nib[1], nib[2], nib[3]);
        *reinterpret_cast<uint32_t *>(dt + 1024 + (j * 16 + r) * 4) = h;
        *reinterpret_cast<uint16_t *>(dt + 1280 + (r * 4 + j) * 2) = d;
    }
}

// Q4_1 blocks [N][nb] x 20 -> tiles of 16 rows x 4 blocks, 1280 bytes: the 16 nibble bytes of
// block j of row r at (j * 16 + r) * 16, the fp16 scales at 1024 + (r * 4 + j) * 2 and the fp16
// minimums at 1152 + (r * 4 + j) * 2.  One thread per (tile, row, block); padding is all zeros.
__global__ void repack_q4_1_kernel(const uint8_t *__restrict__ q41, uint8_t *__restrict__ out, int64_t N,
                                   int64_t nb, int64_t NT, int64_t items) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < items;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t tile = i / 64, rj = i % 64;
        const int r = (int)(rj / 4), j = (int)(rj % 4);
        const int64_t g = tile / NT, t = tile % NT;
        const int64_t n = 16 * g + r, b = 4 * t + j;
        uint8_t *dt = out + tile * 1280;
        uint4 nib = make_uint4(0u, 0u, 0u, 0u);
        uint16_t d = 0, m = 0;
        if (n < N && b < nb) {
            const uint8_t *src = q41 + (n * nb + b) * 20;   // 4-byte aligned
            d = *reinterpret_cast<const uint16_t *>(src);
            m = *reinterpret_cast<const uint16_t *>(src + 2);
            const uint32_t *q = reinterpret_cast<const uint32_t *>(src + 4);
            nib = make_uint4(q[0], q[1], q[2], q[3]);
        }
        *reinterpret_cast<uint4 *>(dt + (j * 16 + r) * 16) = nib;
        *reinterpret_cast<uint16_t *>(dt + 1024 + (r * 4 + j) * 2) = d;
        *reinterpret_cast<uint16_t *>(dt + 1152 + (r * 4 + j) * 2) = m;
    }
}

int grid_for(int64_t work_items, int threads) {
    int64_t blocks = (work_items + threads - 1) / threads;
    const int64_t cap = (int64_t)sm_count() * 16;
    if (blocks > cap) blocks = cap;
    return (int)(blocks < 1 ? 1 : blocks);
}

}  // namespace

gq_status launch_quantize_q4_0(const float *w, void *q4, int64_t N, int64_t K, cudaStream_t s) {
    const int64_t nblocks = N * (K / QK);
    quantize_q4_0_kernel<<<grid_for(nblocks * 32, 256), 256, 0, s>>>(w, (uint8_t *)q4, nblocks);
    return check_cuda(cudaGetLastError(), "quantize_q4_0 launch");
}

gq_status launch_quantize_rows_q8_0(const float *x, void *q8, int64_t M, int64_t K, cudaStream_t s) {
    const int64_t nblocks = M * (K / QK);
    quantize_rows_q8_0_kernel<<<grid_for(nblocks * 32, 256), 256, 0, s>>>(x, (uint8_t *)q8, nblocks);
    return check_cuda(cudaGetLastError(), "quantize_rows_q8_0 launch");
}

gq_status launch_repack_q4_0(const void *q4, void *rep, int64_t N, int64_t K, cudaStream_t s) {
    const int64_t nb = K / QK;
    const int64_t N16 = (N + 15) / 16, NT = (K + TILE_COLS - 1) / TILE_COLS;
    const int64_t ntiles = N16 * NT;
    const int64_t threads = ntiles * 72;
    const int64_t blocks = (threads + 255) / 256;
    repack_q4_0_kernel<<<(unsigned)blocks, 256, 0, s>>>((const uint8_t *)q4, (uint8_t *)rep, N, nb, NT, ntiles);
    return check_cuda(cudaGetLastError(), "repack_q4_0 launch");
}

gq_status launch_quantize_q4_1(const float *w, void *q41, int64_t N, int64_t K, cudaStream_t s) {
    const int64_t nblocks = N * (K / QK);
    quantize_q4_1_kernel<<<grid_for(nblocks * 32, 256), 256, 0, s>>>(w, (uint8_t *)q41, nblocks);
    return check_cuda(cudaGetLastError(), "quantize_q4_1 launch");
}

gq_status launch_repack_q4_1(const void *q41, void *rep, int64_t N, int64_t K, cudaStream_t s) {
    const int64_t nb = K / QK, NT = (nb + TILE_BLOCKS - 1) / TILE_BLOCKS, items = (N + 15) / 16 * NT * 64;
    repack_q4_1_kernel<<<grid_for(items, 256), 256, 0, s>>>((const uint8_t *)q41, (uint8_t *)rep, N, nb, NT, items);
    return check_cuda(cudaGetLastError(), "repack_q4_1 launch");
}

gq_status launch_quantize_q5_0(const float *w, void *q5, int64_t N, int64_t K, cudaStream_t s) {
    const int64_t nblocks = N * (K / QK);
    quantize_q5_0_kernel<<<grid_for(nblocks * 32, 256), 256, 0, s>>>(w, (uint8_t *)q5, nblocks);
    return check_cuda(cudaGetLastError(), "quantize_q5_0 launch");
}

gq_status launch_repack_q5_0(const void *q5, void *rep, int64_t N, int64_t K, cudaStream_t s) {
    const int64_t nb = K / QK, NT = (nb + TILE_BLOCKS - 1) / TILE_BLOCKS, items = (N + 15) / 16 * NT * 64;
    repack_q5_0_kernel<<<grid_for(items, 256), 256, 0, s>>>((const uint8_t *)q5, (uint8_t *)rep, N, nb, NT, items);
    return check_cuda(cudaGetLastError(), "repack_q5_0 launch");
}

gq_status launch_repack_q8_0(const void *q8, void *rep, int64_t N, int64_t K, cudaStream_t s) {
    const int64_t nb = K / QK, NT = (nb + TILE_BLOCKS - 1) / TILE_BLOCKS, items = (N + 15) / 16 * NT * 64;
    repack_q8_0_kernel<<<grid_for(items, 256), 256, 0, s>>>((const uint8_t *)q8, (uint8_t *)rep, N, nb, NT, items);
    return check_cuda(cudaGetLastError(), "repack_q8_0 launch");
}

gq_status launch_repack_f16(const void *w16, void *rep, int64_t N, int64_t K, cudaStream_t s) {
    const int64_t NT = K / 32, pieces = (N + 15) / 16 * NT * 64;
    repack_f16_kernel<<<grid_for(pieces, 256), 256, 0, s>>>((const uint8_t *)w16, (uint8_t *)rep, N, K, NT, pieces);
    return check_cuda(cudaGetLastError(), "repack_f16 launch");
}

}  // namespace gq
