// gemv.cu -- the F16 skinny GEMV (up to 16 activation rows per launch) and the
// block-dot verification kernel of the Q4_0 path.
//
// The regime where every weight byte is read once and the product is bound by
// HBM (Smallem, "Générer à plusieurs", introduction and section "Où la courbe
// s'aplatit": with B sequences each weight read serves B products; DeepSpeed-
// Inference notes, III.A: small batches are limited by the bandwidth of reading
// the weights).
//
// Work decomposition (one launch):
//   grid = (S, ceil(N16 / W)), cluster = (S, 1, 1).  A CTA of W warps owns W row
//   groups of 16 weight rows; CTA `s` of a cluster owns the s-th slice of the K
//   dimension (split-K: Smallem, "La courbe, une première fois": give each block
//   a [begin, end) slice of the common dimension and add the partial sums
//   afterwards; DeepSpeed-Inference notes, III.C.1: tile the output dimension,
//   and the input dimension too when there are too few tiles).  The S partial
//   sums of every output are added in a fixed order through distributed shared
//   memory, so results do not depend on timing.
//
// Weight streaming: at kernel start one lane of every warp issues bulk (TMA)
// copies of its row group's slice into a ring of shared-memory chunks, so the
// whole slice is requested before any arithmetic; each chunk completes on its
// own mbarrier and is refilled as soon as it has been consumed.
//
// F16: activations are rounded to fp16 in shared memory and m16n8k16
// instructions accumulate in f32.  Inside each 32-column span the K order is
// permuted identically for both operands, which leaves every sum unchanged.
#include <algorithm>

#include "gq_common.cuh"
#include "gq_internal.h"

namespace gq {
namespace {

constexpr int MAX_SPLITS = 8;                 // portable cluster size
constexpr size_t SMEM_PER_SM = 227 * 1024;

struct GemvF16Params {
    const __half *w;      // [N][K]
    const float *x;
    float *dst;
    unsigned int *status;
    int M, N, K;
    int N16, nsp;         // row groups, 32-column spans
    int sps;              // spans per split
    int ch, ns;           // spans per chunk, chunk slots per warp
};

__host__ __device__ constexpr size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Shared memory layout of an F16 GEMV CTA (offsets in bytes).
struct F16Smem {
    size_t bars, wbuf, act_h, part, total;
    int rs, hstride;
    __host__ __device__ F16Smem(int W, int MT, int M, int sps, int ch, int ns) {
        rs = ch * 64 + ((ch & 1) ? 0 : 64);          // = 64 (mod 128): conflict-free fragments
        hstride = sps * 64 + ((sps & 1) ? 0 : 64);
        bars = 0;
        wbuf = align_up((size_t)W * ns * 8, 128);
        act_h = wbuf + (size_t)W * ns * 16 * rs;
        part = align_up(act_h + (size_t)(M + 1) * hstride, 16);
        total = part + (size_t)MT * W * 16 * 4;
    }
};

// Adds the S partial sums of the CTA's outputs (part[MT][rows] in every CTA of
// the cluster) in rank order and stores the valid ones to dst.
template <int MT>
__device__ __forceinline__ void cluster_reduce_store(float *part, float *dst, int M, int N, int row_base,
                                                     int rows, int S) {
    const int total = MT * rows;
    if (S == 1) {
        __syncthreads();
        for (int o = threadIdx.x; o < total; o += blockDim.x) {
            const int m = o / rows, n = row_base + o % rows;
            if (m < M && n < N) dst[(size_t)m * N + n] = part[o];
        }
        return;
    }
    cluster_sync();
    const int rank = (int)cluster_ctarank();
    const int chunk = (total + S - 1) / S;
    const int o_end = min(total, (rank + 1) * chunk);
    for (int o = rank * chunk + threadIdx.x; o < o_end; o += blockDim.x) {
        const int m = o / rows, n = row_base + o % rows;
        if (m < M && n < N) {
            float v = 0.0f;
            for (int q = 0; q < S; q++) v += ld_shared_cluster_f32(map_shared_rank(part + o, (uint32_t)q));
            dst[(size_t)m * N + n] = v;
        }
    }
    cluster_sync();   // no CTA leaves while another still reads its shared memory
}

template <int MT>
__device__ __forceinline__ void store_partials(float *part, const float (&acc)[MT / 8][4], int warp, int rows,
                                               int r, int c) {
#pragma unroll
    for (int nt = 0; nt < MT / 8; nt++) {
        const int m0 = 8 * nt + 2 * c;
        part[m0 * rows + warp * 16 + r] = acc[nt][0];
        part[(m0 + 1) * rows + warp * 16 + r] = acc[nt][1];
        part[m0 * rows + warp * 16 + r + 8] = acc[nt][2];
        part[(m0 + 1) * rows + warp * 16 + r + 8] = acc[nt][3];
    }
}

// ---------------------------------------------------------------------------
// F16 x F32
// ---------------------------------------------------------------------------
template <int MT>
__global__ void __launch_bounds__(128) gemv_f16_kernel(const GemvF16Params p) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int W = blockDim.x >> 5;
    const int S = gridDim.x;
    const int s = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = lane >> 2, c = lane & 3;
    const int g = blockIdx.y * W + warp;
    const int sp0 = s * p.sps;
    const int nspans = max(0, min(p.nsp, sp0 + p.sps) - sp0);
    const int nch = (nspans + p.ch - 1) / p.ch;
    const F16Smem L(W, MT, p.M, p.sps, p.ch, p.ns);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L.bars) + warp * p.ns;
    uint8_t *wbuf = smem + L.wbuf + (size_t)warp * p.ns * 16 * L.rs;
    uint8_t *act_h = smem + L.act_h;
    float *part = reinterpret_cast<float *>(smem + L.part);
    const bool row_ok = g < p.N16;
    const int valid_rows = min(16, p.N - 16 * g);

    if (lane == 0)
        for (int i = 0; i < p.ns; i++) mbar_init(smem_addr(bars + i), 1);
    fence_barrier_init();
    __syncwarp();

    pdl_wait();

    auto issue = [&](int chunk) {   // whole warp: lanes 0..15 copy one row piece each
        const int first = chunk * p.ch;
        const uint32_t piece = (uint32_t)(min(p.ch, nspans - first) * 64);
        const uint32_t bar = smem_addr(bars + chunk % p.ns);
        if (lane == 0) mbar_arrive_expect_tx(bar, piece * (uint32_t)valid_rows);
        __syncwarp();
        if (lane < valid_rows) {
            const __half *src = p.w + (size_t)(16 * g + lane) * p.K + (size_t)(sp0 + first) * 32;
            bulk_g2s(smem_addr(wbuf + ((size_t)(chunk % p.ns) * 16 + lane) * L.rs), src, piece, bar);
        }
    };
    if (row_ok)
        for (int k = 0; k < min(p.ns, nch); k++) issue(k);

    // activations of this CTA's columns, rounded to fp16; rows >= M read a zero row
    const int per_row = p.sps * 8;   // float4 groups per row slice
    for (int task = threadIdx.x; task < p.M * per_row; task += blockDim.x) {
        const int m = task / per_row, q = task % per_row;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (q < nspans * 8) v = ldg_f4(p.x + (size_t)m * p.K + (size_t)sp0 * 32 + 4 * q);
        const __half2 lo = __floats2half2_rn(v.x, v.y), hi = __floats2half2_rn(v.z, v.w);
        uint2 packed;
        packed.x = *reinterpret_cast<const uint32_t *>(&lo);
        packed.y = *reinterpret_cast<const uint32_t *>(&hi);
        *reinterpret_cast<uint2 *>(act_h + m * L.hstride + q * 8) = packed;
    }
    for (int i = threadIdx.x; i < L.hstride / 16; i += blockDim.x)
        reinterpret_cast<uint4 *>(act_h + p.M * L.hstride)[i] = make_uint4(0, 0, 0, 0);
    __syncthreads();
    pdl_launch_dependents();

    float acc[MT / 8][4];
#pragma unroll
    for (int i = 0; i < MT / 8; i++) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.0f;
    const uint8_t *brow[MT / 8];
#pragma unroll
    for (int nt = 0; nt < MT / 8; nt++) brow[nt] = act_h + min(r + 8 * nt, p.M) * L.hstride + c * 16;

    if (row_ok) {
        for (int k = 0; k < nch; k++) {
            const bool landed = mbar_wait(smem_addr(bars + k % p.ns), (uint32_t)((k / p.ns) & 1), p.status);
            if (!__all_sync(0xffffffffu, landed)) break;   // a wait gave up (flagged): stop streaming
            const uint8_t *chunk = wbuf + (size_t)(k % p.ns) * 16 * L.rs;
            const int ns_here = min(p.ch, nspans - k * p.ch);
            for (int si = 0; si < ns_here; si++) {
                const int i = k * p.ch + si;
                const uint4 wa = lds128(chunk + r * L.rs + si * 64 + c * 16);
                const uint4 wb = lds128(chunk + (r + 8) * L.rs + si * 64 + c * 16);
#pragma unroll
                for (int nt = 0; nt < MT / 8; nt++) {
                    const uint4 xb = lds128(brow[nt] + i * 64);
                    mma_f16_16x8x16(acc[nt], wa.x, wb.x, wa.y, wb.y, xb.x, xb.y);
                    mma_f16_16x8x16(acc[nt], wa.z, wb.z, wa.w, wb.w, xb.z, xb.w);
                }
            }
            if (k + p.ns < nch) {
                fence_proxy_async_shared();
                __syncwarp();
                issue(k + p.ns);
            }
        }
    }

    store_partials<MT>(part, acc, warp, W * 16, r, c);
    cluster_reduce_store<MT>(part, p.dst, p.M, p.N, blockIdx.y * W * 16, W * 16, S);
}

// ---------------------------------------------------------------------------
// Block dots through the same unpack + dp4a sequence as the Q4_0 GEMV, for
// parity: one thread per (activation row m, weight row n, block b).
// ---------------------------------------------------------------------------
__global__ void block_dots_q4_0_kernel(const uint8_t *__restrict__ w, const uint8_t *__restrict__ q8,
                                       int32_t *__restrict__ sumi, int M, int N, int nb, int NT) {
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= (int64_t)M * N * nb) return;
    const int b = (int)(idx % nb);
    const int64_t rest = idx / nb;
    const int n = (int)(rest % N), m = (int)(rest / N);
    const uint8_t *tile = w + ((size_t)(n / 16) * NT + b / 4) * TILE_BYTES;
    const uint4 q = *reinterpret_cast<const uint4 *>(tile + ((b % 4) * 16 + n % 16) * 16);
    const uint16_t *codes = reinterpret_cast<const uint16_t *>(q8 + ((size_t)m * nb + b) * Q8_0_BYTES + 2);
    uint32_t a[8];
    int qsum = 0;
    for (int k = 0; k < 8; k++) {
        a[k] = (uint32_t)codes[2 * k] | ((uint32_t)codes[2 * k + 1] << 16);
        for (int e = 0; e < 4; e++) qsum += (int)(int8_t)(a[k] >> (8 * e));
    }
    sumi[idx] = block_dot(q, make_uint4(a[0], a[1], a[2], a[3]), make_uint4(a[4], a[5], a[6], a[7]), -8 * qsum);
}

template <typename Kernel, typename Params>
gq_status launch_split(Kernel kernel, const Params &p, dim3 grid, int warps, size_t smem, cudaStream_t s,
                       const char *what) {
    if (smem > SMEM_PER_SM) return fail(GQ_ERR_INVALID_ARG, "%s: %zu bytes of shared memory needed", what, smem);
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return check_cuda(e, what);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(32 * warps, 1, 1);
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

// Number of K slices (the cluster size): as many as the K extent allows, up to
// 8, which gives each SM several small CTAs to balance.  Depends on K only, so
// every activation row is reduced in the same order whatever M is.
int env_int(const char *name, int dflt);

int choose_splits(int64_t kunits) {
    const char *v = getenv("GQ_GEMV_SPLITS");
    int cap = v && *v ? std::max(1, std::min(MAX_SPLITS, atoi(v))) : MAX_SPLITS;
    int S = 1;
    while (S < cap && 2 * S <= kunits) S *= 2;
    return S;
}

int env_int(const char *name, int dflt) {
    const char *v = getenv(name);
    return v && *v ? atoi(v) : dflt;
}

}  // namespace

gq_status launch_gemv_f16(const void *w16, const float *x, float *dst, int64_t M, int64_t N, int64_t K,
                          cudaStream_t s) {
    GemvF16Params p{};
    p.w = (const __half *)w16;
    p.status = device_status_word();
    if (!p.status) return fail(GQ_ERR_CUDA, "device status word unavailable");
    p.N = (int)N;
    p.K = (int)K;
    p.N16 = (int)((N + 15) / 16);
    p.nsp = (int)(K / 32);
    int S = choose_splits(p.nsp);
    p.sps = (p.nsp + S - 1) / S;
    S = (p.nsp + p.sps - 1) / p.sps;
    p.ch = std::min(p.sps, env_int("GQ_GEMV_F16_CHUNK_SPANS", 5));
    const int nch = (p.sps + p.ch - 1) / p.ch;
    p.ns = std::min(nch, env_int("GQ_GEMV_F16_SLOTS", 4));
    const int W = std::max(1, std::min(4, env_int("GQ_GEMV_WARPS", 2)));
    const dim3 grid((unsigned)S, (unsigned)((p.N16 + W - 1) / W), 1);
    for (int64_t m0 = 0; m0 < M; m0 += 16) {
        p.M = (int)std::min<int64_t>(16, M - m0);
        p.x = x + m0 * K;
        p.dst = dst + m0 * N;
        gq_status st;
        if (p.M <= 8) {
            const F16Smem L(W, 8, p.M, p.sps, p.ch, p.ns);
            st = launch_split(gemv_f16_kernel<8>, p, grid, W, L.total, s, "gemv_f16 launch");
        } else {
            const F16Smem L(W, 16, p.M, p.sps, p.ch, p.ns);
            st = launch_split(gemv_f16_kernel<16>, p, grid, W, L.total, s, "gemv_f16 launch");
        }
        if (st != GQ_OK) return st;
    }
    return GQ_OK;
}

gq_status launch_block_dots_q4_0(const void *rep, const void *q8, int32_t *sumi, int64_t M, int64_t N,
                                 int64_t K, cudaStream_t s) {
    const int64_t nb = K / QK, NT = (K + TILE_COLS - 1) / TILE_COLS;
    const int64_t total = M * N * nb;
    block_dots_q4_0_kernel<<<(unsigned)((total + 255) / 256), 256, 0, s>>>(
        (const uint8_t *)rep, (const uint8_t *)q8, sumi, (int)M, (int)N, (int)nb, (int)NT);
    return check_cuda(cudaGetLastError(), "block_dots_q4_0 launch");
}

}  // namespace gq
