// gemv.cu -- the skinny GEMV family (M <= 16 rows of activations per launch).
//
// The regime where every weight byte is read once and the product is bound by
// HBM (Smallem, "Générer à plusieurs", introduction and section "Où la courbe
// s'aplatit": with B sequences each weight read serves B products; DeepSpeed-
// Inference notes, III.A: small batches are limited by the bandwidth of reading
// the weights).
//
// Work decomposition (one launch):
//   grid = (S, ceil(N16 / 4)), cluster = (S, 1, 1).  A CTA of 4 warps owns 4 row
//   groups of 16 weight rows; CTA `s` of a cluster owns the s-th slice of the
//   K dimension (split-K: Smallem, "La courbe, une première fois": give each
//   block a [begin, end) slice of the common dimension and add the partial sums
//   afterwards; DeepSpeed-Inference notes, III.C.1: tile the output dimension,
//   and the input dimension too when there are too few tiles).
//   Each warp streams its row group's tiles of that slice, and the S partial
//   sums of every output are added in a fixed order through distributed shared
//   memory, so the result does not depend on timing.
//
// Q4_0: the CTA first quantizes its slice of every activation row to Q8_0 in
// shared memory (the INIT stage fused in; Arm China NUMA article, "MulMat
// 算子優化": each node quantizes src1 into its own wdata copy).  Each block
// product is one int8 tensor instruction m16n8k32 giving 16 * sumi exactly
// (16 weight rows x 8 activation rows x 32), then f32 scaling by d4 * d8.
//
// F16: weights stream in 16-byte pieces straight from the row-major matrix;
// activations are rounded to fp16 in shared memory and m16n8k16 instructions
// accumulate in f32.  The order of the K elements inside each 32-column span is
// permuted identically for both operands, which leaves the sum unchanged.
#include <algorithm>

#include "gq_common.cuh"
#include "gq_internal.h"

namespace gq {
namespace {

constexpr int GEMV_WARPS = 4;                 // row groups (of 16 rows) per CTA
constexpr int GEMV_THREADS = GEMV_WARPS * 32;
constexpr int GEMV_ROWS = GEMV_WARPS * 16;    // weight rows per CTA
constexpr int MAX_SPLITS = 8;                 // portable cluster size

struct GemvQ4Params {
    const uint8_t *w;     // repacked Q4_0
    const float *x;       // [M][K]
    float *dst;           // [M][N]
    int M, N, K;
    int nb, N16, NT;      // blocks per row, row groups, tiles per row group
    int tps;              // tiles per split
};

struct GemvF16Params {
    const __half *w;      // [N][K]
    const float *x;
    float *dst;
    int M, N, K;
    int N16, nsp;         // row groups, 32-column spans
    int sps;              // spans per split
};

// Adds the S partial sums of the CTA's outputs (part[MT][GEMV_ROWS] in every
// CTA of the cluster) in rank order and stores the valid ones to dst.
template <int MT>
__device__ __forceinline__ void cluster_reduce_store(float *part, float *dst, int M, int N,
                                                     int row_base, int S) {
    constexpr int TOTAL = MT * GEMV_ROWS;
    if (S == 1) {
        __syncthreads();
        for (int o = threadIdx.x; o < TOTAL; o += GEMV_THREADS) {
            const int m = o / GEMV_ROWS, n = row_base + o % GEMV_ROWS;
            if (m < M && n < N) dst[(size_t)m * N + n] = part[o];
        }
        return;
    }
    cluster_sync();
    const int rank = (int)cluster_ctarank();
    const int chunk = (TOTAL + S - 1) / S;
    const int o_end = min(TOTAL, (rank + 1) * chunk);
    for (int o = rank * chunk + threadIdx.x; o < o_end; o += GEMV_THREADS) {
        const int m = o / GEMV_ROWS, n = row_base + o % GEMV_ROWS;
        if (m < M && n < N) {
            float v = 0.0f;
            for (int q = 0; q < S; q++) v += ld_shared_cluster_f32(map_shared_rank(part + o, (uint32_t)q));
            dst[(size_t)m * N + n] = v;
        }
    }
    cluster_sync();   // no CTA leaves while another still reads its shared memory
}

// ---------------------------------------------------------------------------
// Q4_0 x Q8_0
// ---------------------------------------------------------------------------
__device__ __forceinline__ void load_tile(const uint8_t *tile, int lane, uint4 &q0, uint4 &q1, uint4 &sc) {
    q0 = ldg_stream(tile + lane * 16);
    q1 = ldg_stream(tile + 512 + lane * 16);
    sc = ldg_stream(tile + TILE_SCALE_OFFSET + (lane >> 2) * 16);
}

template <int MT>
__global__ void __launch_bounds__(GEMV_THREADS) gemv_q4_0_kernel(const GemvQ4Params p) {
    extern __shared__ __align__(16) uint8_t smem[];
    const int S = gridDim.x;
    const int s = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = lane >> 2, c = lane & 3;
    const int g = blockIdx.y * GEMV_WARPS + warp;
    const int t0 = s * p.tps;
    const int ntiles = max(0, min(p.NT, t0 + p.tps) - t0);
    const int qstride = 2 * p.tps * 64 + 64;   // bytes per activation row; = 64 (mod 128)
    uint8_t *act_q = smem;                                                  // [MT][qstride]
    float *act_d = reinterpret_cast<float *>(smem + MT * qstride);          // [4*tps][MT]
    float *part = act_d + 4 * p.tps * MT;                                   // [MT][GEMV_ROWS]

    pdl_wait();

    const bool row_ok = g < p.N16;
    const uint8_t *wrow = p.w + ((size_t)g * p.NT + t0) * TILE_BYTES;
    uint4 n0 = make_uint4(0, 0, 0, 0), n1 = n0, nsc = n0;
    if (row_ok && ntiles > 0) load_tile(wrow, lane, n0, n1, nsc);   // in flight during the INIT stage

    // INIT: Q8_0 of this CTA's columns of every activation row.  Eight threads
    // per block, four values each; codes stored per (row, block pair, lane c)
    // in the order the B fragments of the tensor instruction read them.
    const int nblk_slot = 4 * p.tps;
    for (int task = threadIdx.x; task < MT * nblk_slot * 8; task += GEMV_THREADS) {
        const int e = task & 7;
        const int bm = task >> 3;
        const int bl = bm % nblk_slot, m = bm / nblk_slot;
        const int b = 4 * t0 + bl;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (m < p.M && bl < 4 * ntiles && b < p.nb) v = ldg_f4(p.x + (size_t)m * p.K + b * QK + 4 * e);
        float a = absmax4(v);
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 4));
        const float d = a / 127.0f;
        const uint32_t word = pack_q8x4(v, d);
        *reinterpret_cast<uint32_t *>(act_q + m * qstride + (bl >> 1) * 64 + (e & 3) * 16 + (bl & 1) * 8 +
                                      (e >> 2) * 4) = word;
        if (e == 0) act_d[bl * MT + m] = __half2float(__float2half_rn(d)) * 0.0625f;  // 1/16: see nib_*_x16
    }
    __syncthreads();
    pdl_launch_dependents();

    float acc[MT / 8][4];
#pragma unroll
    for (int i = 0; i < MT / 8; i++) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.0f;

    if (row_ok) {
        for (int i = 0; i < ntiles; i++) {
            const uint4 q0 = n0, q1 = n1, sc = nsc;
            if (i + 1 < ntiles) load_tile(wrow + (size_t)(i + 1) * TILE_BYTES, lane, n0, n1, nsc);
            const uint32_t scw[4] = {sc.x, sc.y, sc.z, sc.w};
#pragma unroll
            for (int h = 0; h < 2; h++) {
                const uint4 qh = h ? q1 : q0;
#pragma unroll
                for (int nt = 0; nt < MT / 8; nt++) {
                    const uint4 bq = *reinterpret_cast<const uint4 *>(act_q + (r + 8 * nt) * qstride +
                                                                      (2 * i + h) * 64 + c * 16);
#pragma unroll
                    for (int e = 0; e < 2; e++) {
                        const int j = 2 * h + e;
                        const uint32_t wr = e ? qh.z : qh.x;
                        const uint32_t wr8 = e ? qh.w : qh.y;
                        int32_t dd[4];
                        mma_s8_16x8x32(dd, nib_lo_x16(wr), nib_lo_x16(wr8), nib_hi_x16(wr), nib_hi_x16(wr8),
                                       e ? bq.z : bq.x, e ? bq.w : bq.y);
                        const float2 d8 = *reinterpret_cast<const float2 *>(act_d + (4 * i + j) * MT + 8 * nt + 2 * c);
                        const float d4r = half_lo(scw[j]), d4r8 = half_hi(scw[j]);
                        acc[nt][0] = fmaf(d4r * d8.x, (float)dd[0], acc[nt][0]);
                        acc[nt][1] = fmaf(d4r * d8.y, (float)dd[1], acc[nt][1]);
                        acc[nt][2] = fmaf(d4r8 * d8.x, (float)dd[2], acc[nt][2]);
                        acc[nt][3] = fmaf(d4r8 * d8.y, (float)dd[3], acc[nt][3]);
                    }
                }
            }
        }
    }

    // this warp's partial sums: rows warp*16 + {r, r+8}, activation rows 8nt + 2c + {0, 1}
#pragma unroll
    for (int nt = 0; nt < MT / 8; nt++) {
        const int m0 = 8 * nt + 2 * c;
        part[m0 * GEMV_ROWS + warp * 16 + r] = acc[nt][0];
        part[(m0 + 1) * GEMV_ROWS + warp * 16 + r] = acc[nt][1];
        part[m0 * GEMV_ROWS + warp * 16 + r + 8] = acc[nt][2];
        part[(m0 + 1) * GEMV_ROWS + warp * 16 + r + 8] = acc[nt][3];
    }
    cluster_reduce_store<MT>(part, p.dst, p.M, p.N, blockIdx.y * GEMV_ROWS, S);
}

// ---------------------------------------------------------------------------
// F16 x F32
// ---------------------------------------------------------------------------
template <int MT>
__global__ void __launch_bounds__(GEMV_THREADS) gemv_f16_kernel(const GemvF16Params p) {
    extern __shared__ __align__(16) uint8_t smem[];
    const int S = gridDim.x;
    const int s = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = lane >> 2, c = lane & 3;
    const int g = blockIdx.y * GEMV_WARPS + warp;
    const int sp0 = s * p.sps;
    const int nspans = max(0, min(p.nsp, sp0 + p.sps) - sp0);
    const int hstride = p.sps * 64 + ((p.sps & 1) ? 0 : 64);   // bytes per row; = 64 (mod 128)
    uint8_t *act_h = smem;                                                       // [MT][hstride]
    float *part = reinterpret_cast<float *>(smem + ((MT * hstride + 15) & ~15)); // [MT][GEMV_ROWS]

    pdl_wait();

    const int n0 = 16 * g + r, n1 = n0 + 8;
    const bool ok0 = n0 < p.N, ok1 = n1 < p.N;
    const __half *w0 = p.w + (size_t)n0 * p.K + (size_t)sp0 * 32 + 8 * c;
    const __half *w1 = p.w + (size_t)n1 * p.K + (size_t)sp0 * 32 + 8 * c;
    uint4 a = make_uint4(0, 0, 0, 0), b = a;
    if (nspans > 0) {
        if (ok0) a = ldg_stream(w0);
        if (ok1) b = ldg_stream(w1);
    }

    // activations of this CTA's columns, rounded to fp16
    const int per_row = p.sps * 8;   // float4 groups per activation row slice
    for (int task = threadIdx.x; task < MT * per_row; task += GEMV_THREADS) {
        const int m = task / per_row, q = task % per_row;
        const int col = sp0 * 32 + 4 * q;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (m < p.M && q < nspans * 8) v = ldg_f4(p.x + (size_t)m * p.K + col);
        const __half2 lo = __floats2half2_rn(v.x, v.y), hi = __floats2half2_rn(v.z, v.w);
        uint2 packed;
        packed.x = *reinterpret_cast<const uint32_t *>(&lo);
        packed.y = *reinterpret_cast<const uint32_t *>(&hi);
        *reinterpret_cast<uint2 *>(act_h + m * hstride + q * 8) = packed;
    }
    __syncthreads();
    pdl_launch_dependents();

    float acc[MT / 8][4];
#pragma unroll
    for (int i = 0; i < MT / 8; i++) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.0f;

    for (int i = 0; i < nspans; i++) {
        const uint4 wa = a, wb = b;
        if (i + 1 < nspans) {
            if (ok0) a = ldg_stream(w0 + (size_t)(i + 1) * 32);
            if (ok1) b = ldg_stream(w1 + (size_t)(i + 1) * 32);
        }
#pragma unroll
        for (int nt = 0; nt < MT / 8; nt++) {
            const uint4 xb = *reinterpret_cast<const uint4 *>(act_h + (r + 8 * nt) * hstride + i * 64 + c * 16);
            mma_f16_16x8x16(acc[nt], wa.x, wb.x, wa.y, wb.y, xb.x, xb.y);
            mma_f16_16x8x16(acc[nt], wa.z, wb.z, wa.w, wb.w, xb.z, xb.w);
        }
    }

#pragma unroll
    for (int nt = 0; nt < MT / 8; nt++) {
        const int m0 = 8 * nt + 2 * c;
        part[m0 * GEMV_ROWS + warp * 16 + r] = acc[nt][0];
        part[(m0 + 1) * GEMV_ROWS + warp * 16 + r] = acc[nt][1];
        part[m0 * GEMV_ROWS + warp * 16 + r + 8] = acc[nt][2];
        part[(m0 + 1) * GEMV_ROWS + warp * 16 + r + 8] = acc[nt][3];
    }
    cluster_reduce_store<MT>(part, p.dst, p.M, p.N, blockIdx.y * GEMV_ROWS, S);
}

// ---------------------------------------------------------------------------
// Block dots through the same unpack + int8 tensor instruction, for parity.
// One warp per (row group, block, group of 8 activation rows).
// ---------------------------------------------------------------------------
__global__ void block_dots_q4_0_kernel(const uint8_t *__restrict__ w, const uint8_t *__restrict__ q8,
                                       int32_t *__restrict__ sumi, int M, int N, int nb, int NT,
                                       int64_t nitems) {
    const int lane = threadIdx.x & 31;
    const int64_t item = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (item >= nitems) return;
    const int r = lane >> 2, c = lane & 3;
    const int mgroups = (M + 7) / 8;
    const int mg = (int)(item % mgroups);
    const int64_t gb = item / mgroups;
    const int b = (int)(gb % nb);
    const int64_t g = gb / nb;
    const int t = b / 4, j = b % 4, h = j / 2, e = j % 2;
    const uint8_t *tile = w + ((size_t)g * NT + t) * TILE_BYTES;
    const uint4 qh = *reinterpret_cast<const uint4 *>(tile + h * 512 + lane * 16);
    const uint32_t wr = e ? qh.z : qh.x, wr8 = e ? qh.w : qh.y;
    const int m = 8 * mg + r;
    uint32_t b0 = 0, b1 = 0;
    if (m < M) {
        const uint8_t *blk = q8 + ((size_t)m * nb + b) * Q8_0_BYTES + 2;
        for (int k = 0; k < 4; k++) {
            b0 |= (uint32_t)blk[4 * c + k] << (8 * k);
            b1 |= (uint32_t)blk[16 + 4 * c + k] << (8 * k);
        }
    }
    int32_t dd[4];
    mma_s8_16x8x32(dd, nib_lo_x16(wr), nib_lo_x16(wr8), nib_hi_x16(wr), nib_hi_x16(wr8), b0, b1);
    const int rows[4] = {r, r, r + 8, r + 8};
    for (int i = 0; i < 4; i++) {
        const int mm = 8 * mg + 2 * c + (i & 1);
        const int64_t n = 16 * g + rows[i];
        if (mm < M && n < N) sumi[((size_t)mm * N + n) * nb + b] = dd[i] / 16;   // exact: 16 * sumi
    }
}

template <typename Kernel, typename Params>
gq_status launch_split(Kernel kernel, const Params &p, dim3 grid, size_t smem, cudaStream_t s, const char *what) {
    static_assert(sizeof(Params) < 4096, "kernel parameters");
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return check_cuda(e, what);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(GEMV_THREADS, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attrs[2];
    int na = 0;
    attrs[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[na].val.programmaticStreamSerializationAllowed = 1;
    na++;
    if (grid.x > 1) {
        attrs[na].id = cudaLaunchAttributeClusterDimension;
        attrs[na].val.clusterDim.x = grid.x;
        attrs[na].val.clusterDim.y = 1;
        attrs[na].val.clusterDim.z = 1;
        na++;
    }
    cfg.attrs = attrs;
    cfg.numAttrs = na;
    return check_cuda(cudaLaunchKernelEx(&cfg, kernel, p), what);
}

// Number of K slices: enough CTAs for about four per SM, at most a cluster of 8,
// never more slices than K units.  Depends on N and K only, so every activation
// row is reduced in the same order whatever M is.
int choose_splits(int64_t row_ctas, int64_t kunits) {
    const int64_t target = 4LL * sm_count();
    int S = 1;
    while (S < MAX_SPLITS && 2 * S <= kunits && row_ctas * S < target) S *= 2;
    return S;
}

}  // namespace

gq_status launch_gemv_q4_0(const void *rep, const float *x, float *dst, int64_t M, int64_t N, int64_t K,
                           cudaStream_t s) {
    GemvQ4Params p{};
    p.w = (const uint8_t *)rep;
    p.N = (int)N;
    p.K = (int)K;
    p.nb = (int)(K / QK);
    p.N16 = (int)((N + 15) / 16);
    p.NT = (int)((K + TILE_COLS - 1) / TILE_COLS);
    const int64_t row_ctas = (p.N16 + GEMV_WARPS - 1) / GEMV_WARPS;
    int S = choose_splits(row_ctas, p.NT);
    p.tps = (p.NT + S - 1) / S;
    S = (p.NT + p.tps - 1) / p.tps;
    const dim3 grid((unsigned)S, (unsigned)row_ctas, 1);
    for (int64_t m0 = 0; m0 < M; m0 += 16) {
        p.M = (int)std::min<int64_t>(16, M - m0);
        p.x = x + m0 * K;
        p.dst = dst + m0 * N;
        const int qstride = 2 * p.tps * 64 + 64;
        gq_status st;
        if (p.M <= 8) {
            const size_t smem = 8 * qstride + 4 * p.tps * 8 * 4 + 8 * GEMV_ROWS * 4;
            st = launch_split(gemv_q4_0_kernel<8>, p, grid, smem, s, "gemv_q4_0 launch");
        } else {
            const size_t smem = 16 * qstride + 4 * p.tps * 16 * 4 + 16 * GEMV_ROWS * 4;
            st = launch_split(gemv_q4_0_kernel<16>, p, grid, smem, s, "gemv_q4_0 launch");
        }
        if (st != GQ_OK) return st;
    }
    return GQ_OK;
}

gq_status launch_gemv_f16(const void *w16, const float *x, float *dst, int64_t M, int64_t N, int64_t K,
                          cudaStream_t s) {
    GemvF16Params p{};
    p.w = (const __half *)w16;
    p.N = (int)N;
    p.K = (int)K;
    p.N16 = (int)((N + 15) / 16);
    p.nsp = (int)(K / 32);
    const int64_t row_ctas = (p.N16 + GEMV_WARPS - 1) / GEMV_WARPS;
    int S = choose_splits(row_ctas, p.nsp);
    p.sps = (p.nsp + S - 1) / S;
    S = (p.nsp + p.sps - 1) / p.sps;
    const dim3 grid((unsigned)S, (unsigned)row_ctas, 1);
    const int hstride = p.sps * 64 + ((p.sps & 1) ? 0 : 64);
    for (int64_t m0 = 0; m0 < M; m0 += 16) {
        p.M = (int)std::min<int64_t>(16, M - m0);
        p.x = x + m0 * K;
        p.dst = dst + m0 * N;
        gq_status st;
        if (p.M <= 8) {
            const size_t smem = ((8 * hstride + 15) & ~15) + 8 * GEMV_ROWS * 4;
            st = launch_split(gemv_f16_kernel<8>, p, grid, smem, s, "gemv_f16 launch");
        } else {
            const size_t smem = ((16 * hstride + 15) & ~15) + 16 * GEMV_ROWS * 4;
            st = launch_split(gemv_f16_kernel<16>, p, grid, smem, s, "gemv_f16 launch");
        }
        if (st != GQ_OK) return st;
    }
    return GQ_OK;
}

gq_status launch_block_dots_q4_0(const void *rep, const void *q8, int32_t *sumi, int64_t M, int64_t N,
                                 int64_t K, cudaStream_t s) {
    const int64_t nb = K / QK, N16 = (N + 15) / 16, NT = (K + TILE_COLS - 1) / TILE_COLS;
    const int64_t nitems = N16 * nb * ((M + 7) / 8);
    const int64_t blocks = (nitems * 32 + 255) / 256;
    block_dots_q4_0_kernel<<<(unsigned)blocks, 256, 0, s>>>((const uint8_t *)rep, (const uint8_t *)q8, sumi,
                                                            (int)M, (int)N, (int)nb, (int)NT, nitems);
    return check_cuda(cudaGetLastError(), "block_dots_q4_0 launch");
}

}  // namespace gq
