// gemv_m1.cu -- the one-row Q4_0 x Q8_0 product (M = 1): single-token decode.
//
// With one activation row every weight byte feeds one multiply-add, so the
// product is bound by reading the weights once (Smallem, "Générer à plusieurs",
// introduction and "Où la courbe s'aplatit"; DeepSpeed-Inference notes, III.A).
// A product may read its activation row only after the kernel in front of it
// has finished (stream order: the row is usually that kernel's output); that
// wait costs about 0.8 us per product whatever the kernel does.  The kernel is
// shaped so that as little as possible happens after it:
//
//  * Before the wait.  The producer warp copies the CTA's first weight chunks
//    into a ring of shared memory and prefetches the rest of its range into L2
//    as soon as the CTA is resident (when the caller declared its weights
//    static).  The CTA takes at most half of an SM (shared memory, registers),
//    so the CTAs of the next product in the stream are resident beside this
//    one and do the same while this product runs.
//  * INIT after the wait (llama.cpp PR #1632, "Introduction": the q_f32 kind
//    quantizes src1 to Q8_0 before the block dots; Arm China NUMA article,
//    "MulMat 算子優化": every worker reads the wdata).  Each CTA owns whole row
//    groups (16 weight rows), so chunk position p of every row group holds a
//    tile whose column is congruent to p modulo 16, and consumer warp w (which
//    takes position w) only ever meets the columns congruent to w modulo 16.
//    Each warp therefore quantizes just those blocks of the row into the CTA's
//    shared image, and no barrier of the CTA follows.
//  * The block dots.  Lane (b, r) of a warp takes block b of rows r and r + 8
//    of a tile, so the activation codes and scale it loads serve two rows;
//    each block dot is eight dp4a on the unpacked nibbles and the codes, exact
//    in int32, scaled by d4 * d8 into an f32 accumulator per (tile position,
//    row).  A row group's per-position sums stay in registers; every two row
//    groups they are written over the warps' own tiles of the last chunk, and
//    one warp (in rotation) adds the sixteen positions of each row in a fixed
//    order and stores dst while the others go on.  No row group is shared
//    between CTAs, so nothing is combined across CTAs and the result does not
//    depend on timing.
//
// Warp roles: 16 consumer warps, 1 producer warp (bulk copies of 16-tile chunks,
// mbarrier completion).
#include <algorithm>
#include <atomic>

#include "gq_common.cuh"
#include "gq_internal.h"

namespace gq {
namespace {

constexpr int M1_TILES = 16;                         // tiles per chunk = tile positions
constexpr int M1_CW = 16;                            // consumer warps (one tile position each)
constexpr int M1_CHUNK = M1_TILES * TILE_BYTES;      // 18,432 bytes
constexpr int M1_MAX_SLOTS = 6;
constexpr int M1_RED_BARS = 8;                       // batch-end barriers, used in rotation
constexpr int M1_BATCH = 2;                          // row groups whose sums are reduced together
constexpr size_t M1_SMEM_HALF = 113 * 1024;          // two CTAs per SM
constexpr int64_t M1_MAX_K = 32768;                  // the image (K + K/8 bytes) leaves room for 4 slots

struct M1Params {
    const uint8_t *w;        // repacked Q4_0 tiles
    const float *x;          // the activation row [K]
    float *dst;              // [N]
    unsigned int *status;    // device status word
    int N, K, NT, N16;
    int slots;
    int early;               // 1: the weights may be read before the grids in front finished
};

// Shared memory: barriers (full[slots], empty[slots], red[8]), the ring, then the Q8_0 image of
// the row: codes [4 NT blocks][32] (element order), then one word per block, fp16 d8 in the low
// half and -8 * (sum of the codes) in the high half.  A warp fills only the blocks of its own
// tile columns; blocks past K are never read (their weights are padding).
struct M1Layout {
    size_t ring, codes, scales, total;
    __host__ __device__ M1Layout(int NT, int slots) {
        ring = 256;
        codes = ring + (size_t)slots * M1_CHUNK;
        scales = codes + (size_t)NT * TILE_COLS;
        total = scales + (size_t)NT * TILE_BLOCKS * 4;
    }
};

__device__ __forceinline__ void m1_arrive(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ uint4 m1_lds128(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
    return v;
}
__device__ __forceinline__ uint32_t m1_lds32(uint32_t a) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ uint32_t m1_lds16(uint32_t a) {
    uint32_t v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}

// CW consumer warps (each takes 16 / CW tile positions of a chunk) and one producer warp.
template <int CW>
__global__ void __launch_bounds__((CW + 1) * 32, 2) gemv_m1_q4_0_kernel(const M1Params p) {
    constexpr int TPW = M1_TILES / CW;                // tile positions per consumer warp
    constexpr int X_ROUNDS = CW == 8 ? 3 : 1;         // half blocks per lane loaded at once (within the register cap)
    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = (int)gridDim.x, c = (int)blockIdx.x;
    const int g0 = (int)((int64_t)p.N16 * c / G), g1 = (int)((int64_t)p.N16 * (c + 1) / G);   // row groups
    const int nc = (p.NT + M1_TILES - 1) / M1_TILES;                                            // chunks per row group
    const M1Layout L(p.NT, p.slots);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem);
    uint64_t *empty = full + p.slots;
    uint64_t *red = empty + p.slots;

    if (threadIdx.x < 2 * p.slots + M1_RED_BARS)
        mbar_init(smem_addr(full + threadIdx.x), threadIdx.x < p.slots ? 1 : CW);
    fence_barrier_init();
    __syncthreads();
    pdl_launch_dependents();   // the next product's CTAs may become resident beside this one

    // ---------------------------------------------------------------- producer
    if (warp == CW) {
        if (lane != 0) return;
        const int nk = (g1 - g0) * nc;                // chunks of this CTA, row group by row group
        auto chunk_at = [&](int k, const uint8_t *&src, uint32_t &bytes) {
            const int g = g0 + k / nc, u = (k % nc) * M1_TILES;
            src = p.w + ((size_t)g * p.NT + u) * TILE_BYTES;
            bytes = (uint32_t)(min(M1_TILES, p.NT - u) * TILE_BYTES);
        };
        const uint8_t *src;
        uint32_t bytes;
        // L2 prefetch of the chunks past the first ring fill: it moves nothing into the CTA, and
        // L2 is where every access to device memory meets, so it may run before the wait
        auto prefetch_from = [&](int k0) {
            for (int k = k0; k < nk; k++) {
                chunk_at(k, src, bytes);
                bulk_prefetch_l2(src, bytes);
            }
        };
        if (!p.early) {
            prefetch_from(0);
            pdl_wait();   // the weights may still be written by the grid in front
        }
        const uint64_t policy = l2_evict_first_policy();   // every weight byte is read once
        for (int k = 0; k < nk; k++) {
            const int slot = k % p.slots;
            if (k >= p.slots && !mbar_wait(smem_addr(empty + slot), (uint32_t)(((k / p.slots) - 1) & 1), p.status))
                break;
            chunk_at(k, src, bytes);
            GQ_DCHECK(g0 + k / nc < p.N16 && (k % nc) * M1_TILES + (int)(bytes / TILE_BYTES) <= p.NT &&
                          bytes <= (uint32_t)M1_CHUNK,
                      p.status);
            mbar_arrive_expect_tx(smem_addr(full + slot), bytes);
            bulk_g2s_hint(smem_addr(smem + L.ring + (size_t)slot * M1_CHUNK), src, bytes, smem_addr(full + slot),
                          policy);
            if (p.early && k == p.slots - 1) prefetch_from(p.slots);
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    const uint32_t ring_a = smem_addr(smem + L.ring), codes_a = smem_addr(smem + L.codes),
                   scales_a = smem_addr(smem + L.scales);
    pdl_wait();   // src1 is final
    {
        // INIT of this warp's blocks: tile columns t = warp + CW i, blocks 4 t .. 4 t + 3.  Lane
        // pair (2 k, 2 k + 1) takes the two halves (16 values, four float4) of one block.
        const int ntw = (p.NT - warp + CW - 1) / CW;   // tile columns of this warp
        const int nh = 8 * ntw;                       // half blocks of this warp
        const int kb = p.K / QK;
#pragma unroll 1
        for (int h0 = 0; h0 < nh; h0 += 32 * X_ROUNDS) {
            float4 v[X_ROUNDS][4];
#pragma unroll
            for (int r = 0; r < X_ROUNDS; r++) {
                const int h = h0 + lane + 32 * r, b = h >> 1;
                const int blk = 4 * (warp + CW * (b >> 2)) + (b & 3);
                const bool live = h < nh && blk < kb;
                const float *src = p.x + (size_t)blk * QK + 16 * (h & 1);
#pragma unroll
                for (int i = 0; i < 4; i++) v[r][i] = live ? ldg_f4(src + 4 * i) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int r = 0; r < X_ROUNDS; r++) {
                if (h0 + 32 * r >= nh) break;   // warp-uniform: no half block of this round
                const int h = h0 + lane + 32 * r, b = h >> 1;
                const int blk = 4 * (warp + CW * (b >> 2)) + (b & 3);
                float am = fmaxf(fmaxf(absmax4(v[r][0]), absmax4(v[r][1])), fmaxf(absmax4(v[r][2]), absmax4(v[r][3])));
                am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 1));
                const float d = am / 127.0f;
                const Q8Scale q = q8_scale(d);
                uint32_t wq[4];
                pack_q8_words_fast<4>(v[r], q, wq);
                int qs = sum_q8x4(wq[0]) + sum_q8x4(wq[1]) + sum_q8x4(wq[2]) + sum_q8x4(wq[3]);
                qs += __shfl_xor_sync(0xffffffffu, qs, 1);
                if (h < nh) {
                    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(codes_a + blk * QK + 16 * (h & 1)),
                                 "r"(wq[0]), "r"(wq[1]), "r"(wq[2]), "r"(wq[3])
                                 : "memory");
                    if ((h & 1) == 0)
                        asm volatile("st.shared.u32 [%0], %1;" ::"r"(scales_a + 4 * blk),
                                     "r"((uint32_t)__half_as_ushort(__float2half_rn(d)) | ((uint32_t)(-8 * qs) << 16))
                                     : "memory");
                }
            }
        }
        __syncwarp();   // the warp's blocks are in the image (only this warp reads them)
    }

    const int jb = lane >> 3, r0 = lane & 7;   // this lane's block of a tile and rows r0, r0 + 8
    // the tile at chunk position ti (tile column u + ti) into the accumulators of rows r0, r0 + 8
    auto tile_dot = [&](const uint32_t chunk_a, const int u, const int ti, float (&a)[2]) {
        const uint32_t tile_a = chunk_a + ti * TILE_BYTES;
        const int blk = 4 * (u + ti) + jb;
        GQ_DCHECK(ti < M1_TILES && blk < 4 * p.NT, p.status);
        const uint4 a0 = m1_lds128(codes_a + blk * QK), a1 = m1_lds128(codes_a + blk * QK + 16);
        const uint32_t sc = m1_lds32(scales_a + 4 * blk);
        const uint4 q0 = m1_lds128(tile_a + (jb * 16 + r0) * 16);
        const uint4 q1 = m1_lds128(tile_a + (jb * 16 + r0 + 8) * 16);
        const uint32_t h0 = m1_lds16(tile_a + TILE_SCALE_OFFSET + (r0 * 4 + jb) * 2);
        const uint32_t h1 = m1_lds16(tile_a + TILE_SCALE_OFFSET + ((r0 + 8) * 4 + jb) * 2);
        const int corr = (int)(short)(sc >> 16);
        const float d8 = half_lo(sc);
        const int s0 = block_dot(q0, a0, a1, corr), s1 = block_dot(q1, a0, a1, corr);
        a[0] = fmaf(half_lo(h0) * d8, (float)s0, a[0]);
        a[1] = fmaf(half_lo(h1) * d8, (float)s1, a[1]);
    };
    int slot = 0;
    uint32_t phase = 0;
    bool failed = false;
    // Row groups go in batches of M1_BATCH.  A row group's per-position sums stay in registers (the
    // four block lanes of a row added by a butterfly, so every lane holds the row's value); at
    // the end of a batch every warp writes its sums over the first bytes of its own tile of the
    // chunk the batch ended in (only this warp reads that tile) and arrives on the batch's
    // barrier.  One warp, in rotation, waits for all of them, adds positions 0 .. 15 of each row
    // in order, stores the sums and releases that slot for all the consumer warps; the others go
    // on with the next batch at once.
    float part[M1_BATCH][TPW][2];
    const int nbatch = (g1 - g0 + M1_BATCH - 1) / M1_BATCH;
    for (int bi = 0; bi < nbatch; bi++) {
        const int gb = g0 + bi * M1_BATCH, nrg = min(M1_BATCH, g1 - gb);
#pragma unroll
        for (int j = 0; j < M1_BATCH; j++) {
            if (j >= nrg) break;
            float acc[TPW][2];
#pragma unroll
            for (int tw = 0; tw < TPW; tw++) acc[tw][0] = acc[tw][1] = 0.0f;
            uint32_t chunk_a = 0;
            for (int ci = 0; ci < nc; ci++) {
                const int u = ci * M1_TILES;
                // a lane whose wait gave up skips the chunks from here on
                if (!failed) failed = !mbar_wait(smem_addr(full + slot), phase, p.status);
                chunk_a = ring_a + slot * M1_CHUNK;
                const int nt = min(M1_TILES, p.NT - u);
                if (!failed) {
#pragma unroll
                    for (int tw = 0; tw < TPW; tw++)
                        if (warp + CW * tw < nt) tile_dot(chunk_a, u, warp + CW * tw, acc[tw]);
                }
                const bool batch_end = j + 1 == nrg && ci + 1 == nc;
                if (!batch_end) {                    // release the chunk
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_addr(empty + slot));
                    if (++slot == p.slots) {
                        slot = 0;
                        phase ^= 1u;
                    }
                }
            }
#pragma unroll
            for (int tw = 0; tw < TPW; tw++)
#pragma unroll
                for (int h = 0; h < 2; h++) {
                    acc[tw][h] += __shfl_xor_sync(0xffffffffu, acc[tw][h], 8);
                    acc[tw][h] += __shfl_xor_sync(0xffffffffu, acc[tw][h], 16);
                    part[j][tw][h] = acc[tw][h];
                }
            if (j + 1 == nrg) {
                // batch end: the current slot holds the batch's last chunk
                const uint32_t mine = chunk_a + warp * TILE_BYTES;   // [row group j][position tw][row]
                if (lane < 8) {
#pragma unroll
                    for (int jj = 0; jj < M1_BATCH; jj++) {
                        if (jj >= nrg) break;
#pragma unroll
                        for (int tw = 0; tw < TPW; tw++) {
                            const uint32_t a = mine + ((jj * TPW + tw) * 16 + r0) * 4;
                            asm volatile("st.shared.f32 [%0], %1;" ::"r"(a), "f"(part[jj][tw][0]) : "memory");
                            asm volatile("st.shared.f32 [%0], %1;" ::"r"(a + 32), "f"(part[jj][tw][1]) : "memory");
                        }
                    }
                }
                fence_proxy_async_shared();   // a later bulk copy overwrites these bytes
                __syncwarp();
                const uint32_t rbar = smem_addr(red + bi % M1_RED_BARS);
                if (lane == 0) mbar_arrive(rbar);
                if (warp == bi % CW) {
                    // The barrier of batch bi completes once per M1_RED_BARS batches; no warp runs
                    // that far ahead of this one (the ring has fewer slots).
                    if (!failed) failed = !mbar_wait(rbar, (uint32_t)((bi / M1_RED_BARS) & 1), p.status);
                    for (int o = lane; o < 16 * nrg; o += 32) {   // output row o % 16 of row group o / 16
                        const int jj = o >> 4, row = o & 15;
                        float v = 0.0f;
#pragma unroll
                        for (int pos = 0; pos < M1_TILES; pos++) {
                            float t;
                            asm volatile("ld.shared.f32 %0, [%1];"
                                         : "=f"(t)
                                         : "r"(chunk_a + (pos % CW) * TILE_BYTES + ((jj * TPW + pos / CW) * 16 + row) * 4));
                            v += t;
                        }
                        const int n = 16 * (gb + jj) + row;
                        if (n < p.N) p.dst[n] = v;
                    }
                    fence_proxy_async_shared();
                    __syncwarp();
                    if (lane == 0) m1_arrive(smem_addr(empty + slot), CW);
                }
                if (++slot == p.slots) {
                    slot = 0;
                    phase ^= 1u;
                }
            }
        }
    }
}

std::atomic<bool> g_m1_smem_set[64];

template <int CW>
gq_status launch_m1(const M1Params &p, int G, size_t smem, cudaStream_t s) {
    auto kernel = gemv_m1_q4_0_kernel<CW>;
    int dev = 0;
    gq_status st = check_cuda(cudaGetDevice(&dev), "cudaGetDevice");
    if (st != GQ_OK) return st;
    std::atomic<bool> *set = (dev >= 0 && dev < 64) ? &g_m1_smem_set[dev] : nullptr;
    if (!set || !set->load(std::memory_order_acquire)) {
        st = check_cuda(cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)M1_SMEM_HALF),
                        "gemv (one row) shared-memory attribute");
        if (st == GQ_OK)   // all of the unified L1 as shared memory: two CTAs per SM
            st = check_cuda(cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                                 (int)cudaSharedmemCarveoutMaxShared),
                            "gemv (one row) carveout attribute");
        if (st != GQ_OK) return st;
        if (set) set->store(true, std::memory_order_release);
    }
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.gridDim = dim3((unsigned)G, 1, 1);
    cfg.blockDim = dim3((CW + 1) * 32, 1, 1);
    cfg.dynamicSmemBytes = smem;
    return check_cuda(cudaLaunchKernelEx(&cfg, kernel, p), "gemv (one row) launch");
}

}  // namespace

bool gemv_m1_supported(int64_t N, int64_t K) { return N > 0 && K > 0 && K <= M1_MAX_K; }

gq_status launch_gemv_m1_q4_0(const void *rep, const float *x, float *dst, int64_t N, int64_t K, cudaStream_t s) {
    M1Params p{};
    p.w = (const uint8_t *)rep;
    p.x = x;
    p.dst = dst;
    p.status = device_status_word();
    if (!p.status) return fail(GQ_ERR_CUDA, "device status word unavailable");
    p.N = (int)N;
    p.K = (int)K;
    p.NT = (int)((K + TILE_COLS - 1) / TILE_COLS);
    p.N16 = (int)((N + 15) / 16);
    p.early = static_weights() ? 1 : 0;
    const size_t fixed = M1Layout(p.NT, 0).total;
    p.slots = (int)std::min<size_t>(M1_MAX_SLOTS, (M1_SMEM_HALF - std::min(M1_SMEM_HALF, fixed)) / M1_CHUNK);
    if (p.slots < 2) return fail(GQ_ERR_INVALID_ARG, "gemv (one row): K=%lld leaves no room for the ring", (long long)K);
    const size_t smem = M1Layout(p.NT, p.slots).total;
    const int G = std::min(sm_count(), p.N16);   // whole row groups per CTA
    return launch_m1<M1_CW>(p, G, smem, s);
}

}  // namespace gq
