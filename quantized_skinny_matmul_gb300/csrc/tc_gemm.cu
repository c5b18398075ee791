// tc_gemm.cu -- the tensor-core tile kernels for M >= 32 activation rows, where
// the product is a dense contraction (Smallem, "Générer à plusieurs", "Où la
// courbe s'aplatit": past B ~ the ridge point the card computes instead of
// waiting on memory; llama.cpp PR #1632, "Introduction": de-quantization time
// is significant up to M ~ 128, so it is fused into the tile pipeline here
// instead of being a separate pass; Smallem, "La courbe, une première fois":
// converting operands to bf16 cost more than the tensor cores saved there,
// which is why the conversion happens in shared memory on the way in).
//
// One CTA computes a 128 (weight rows) x BN (activation rows, 32 .. 256) tile of
// dst^T = W . X^T over all of K with tcgen05.mma kind::f16 and an f32
// accumulator in tensor memory:
//   warp 0      weight producer: one 2D TMA load per 128-column step of the
//               eight repacked Q4_0 tiles of the CTA's rows (or two TMA loads
//               of the F16 weights straight into the MMA's operand ring);
//   warp 10     activation producer: TMA loads of the fp16 activations;
//   warp 1      allocates tensor memory; one thread issues the MMAs and commits
//               them to the mbarrier that frees the operand stage (one wait and
//               one commit per step: each mbarrier operation of this thread
//               measurably delays the next MMAs);
//   warps 2..9  (Q4_0) de-quantize each 128 x 128 weight tile into fp16,
//               (q - 8) * d rounded once, in the 128-byte-swizzled K-major
//               layout the MMA reads (each warp 32 rows x 64 columns); then
//               they read the accumulators back (tcgen05.ld) and store dst.
// The raw weight bytes have a ring of their own with their own producer, so the
// weight stream from device memory runs as many stages ahead as that ring holds,
// whatever the operand ring (converted weights and activations of one MMA step
// per stage) is waiting for.  The MMAs of a stage rotate over 2 (BN >= 128) or 4
// independent accumulators in tensor memory, so consecutive MMAs do not wait
// for each other's results; the epilogue adds them in a fixed order.
// When the output tiles are too few to occupy the GPU, K is split over a cluster
// of 2, 4 or 8 CTAs along z: each accumulates its K range, and the cluster adds
// the partial tiles in a fixed order through distributed shared memory.
// The activations are quantized first by a small kernel into a workspace copy
// B[m][k] = fp16(q8 * d8) (Q4_0), or rounded to fp16 (F16): the same Q8_0
// values as the GEMV path, each rounded once to fp16, so the result is within
// 2e-3 of sum |terms| of the exact block-dot result.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cstdlib>
#include <mutex>

#include "gq_common.cuh"
#include "gq_internal.h"

namespace gq {
namespace {

constexpr int BM = 128;                          // weight rows per CTA = MMA M = TMEM lanes
constexpr int BK = 128;                          // K per pipeline stage (one repacked tile column)
constexpr int ATOM_BYTES = BM * 128;             // one 128-row x 64-half swizzle atom: 16 KB
constexpr int A_STAGE = BM * BK * 2;             // 32 KB
constexpr int RAW_ROWGROUPS = BM / 16;           // repacked row groups of a CTA
constexpr int RAW_STAGE = RAW_ROWGROUPS * TILE_BYTES;   // 8 row groups of 16 rows x one tile
constexpr int RAW_WORDS = TILE_BYTES / 8;        // a repacked tile in 8-byte TMA elements
constexpr int CONVERTER_WARPS = 8;               // warps 2 .. 9
constexpr int ACT_PRODUCER_WARP = 2 + CONVERTER_WARPS;
constexpr int THREADS = (ACT_PRODUCER_WARP + 1) * 32;
constexpr int MAX_STAGES = 4, MAX_RAW = 4;

// Ring depths and the shared-memory map (offsets from a 1024-aligned base).
// A stage holds the operands of one MMA step: the fp16 weight tile (Q4_0:
// converted from the RAW ring, which holds the repacked bytes as loaded; F16:
// loaded as is) and the activation tile.  Depths fill the 227 KB of an SM.
template <int BN, bool QUANT>
struct TcLayout {
    static constexpr int ST = BN == 256 ? 2 : BN == 128 ? 3 : 4;
    static constexpr int RAW = QUANT ? (BN >= 64 ? 3 : 4) : 0;
    static constexpr int NACC = BN >= 128 ? 2 : 4;          // accumulators in tensor memory
    static constexpr uint32_t TMEM_COLS = NACC * BN;         // 128, 256 or 512: a power of two >= 32
    static constexpr int B_STAGE = BN * BK * 2;
    static constexpr int PSTRIDE = BN + 4;                   // floats per row of a split-K partial
    static constexpr bool CAN_SPLIT = BM * PSTRIDE * 4 <= ST * A_STAGE;   // the partial fits the operand memory
    static constexpr int a = 0;
    static constexpr int b = a + ST * A_STAGE;
    static constexpr int raw = b + ST * B_STAGE;
    static constexpr int bars = raw + RAW * RAW_STAGE;
    static constexpr int total = bars + 256;     // from a 1024-aligned base
    static_assert(ST <= MAX_STAGES && RAW <= MAX_RAW, "barrier table too small");
    static_assert(total + 1024 <= 227 * 1024, "shared memory");
};

struct TcParams {
    float *dst;
    unsigned int *status;
    int M, N, K;
    int NT, N16;             // tiles of 128 columns, row groups of 16
};

// barrier indices.  FULL[s] completes when both operands of stage s are in place:
// the activation producer's arrival with its TMA bytes, and the eight converter
// warps' arrivals (Q4_0) or the weight producer's arrival with its TMA bytes (F16).
// EMPTY[s] completes when the MMAs that read stage s have completed.  The MMA
// thread thus handles one barrier wait and one commit per step.
enum : int {
    RAW_FULL = 0,
    RAW_EMPTY = RAW_FULL + MAX_RAW,
    FULL = RAW_EMPTY + MAX_RAW,
    EMPTY = FULL + MAX_STAGES,
    ACC_FULL = EMPTY + MAX_STAGES,
    NUM_BARS = ACC_FULL + 1
};
static_assert(NUM_BARS * 8 + 4 <= 256, "barrier area");

// ---------------------------------------------------------------------------
// tcgen05 / TMA wrappers
// ---------------------------------------------------------------------------
// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart (stride byte offset), descriptor version 1.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);          // start address
    d |= (uint64_t)1 << 16;                             // leading byte offset (unused for swizzled K-major)
    d |= (uint64_t)(1024 >> 4) << 32;                   // stride byte offset
    d |= (uint64_t)1 << 46;                             // version
    d |= (uint64_t)2 << 61;                             // 128-byte swizzle
    return d;
}

// Instruction descriptor of kind::f16: f16 A and B, f32 D, both K-major.
__host__ __device__ constexpr uint32_t f16_idesc(int m, int n) {
    return (1u << 4) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ void mma_f16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                        uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(tmem_d), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int c0, int c1, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
        ::"r"(dst), "l"(map), "r"(c0), "r"(c1), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void mbar_arrive_plain(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// 32 consecutive f32 columns of this warp's 32 tensor-memory lanes.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; i++) v[i] = __uint_as_float(r[i]);
}

// Waits on a barrier phase unless an earlier wait of this thread gave up.
__device__ __forceinline__ void wait_or_fail(uint32_t bar, uint32_t parity, bool &failed, unsigned int *status) {
    if (!failed && !mbar_wait(bar, parity, status)) failed = true;
}

// Eight Q4_0 codes of bytes [b0..b3] of a word -> two half2 of (q - 8) * d.
__device__ __forceinline__ uint4 dequant8(uint32_t lo_word, uint32_t hi_word, bool high_nibbles, __half2 d2) {
    const __half2 bias = __halves2half2(__ushort_as_half(0x6408), __ushort_as_half(0x6408));   // 1032
    uint32_t out[4];
    const uint32_t words[2] = {lo_word, hi_word};
#pragma unroll
    for (int i = 0; i < 2; i++) {
#pragma unroll
        for (int h = 0; h < 2; h++) {
            uint32_t t = __byte_perm(words[i], 0u, h ? 0x4342u : 0x4140u);   // bytes (2h, 2h+1) -> halves
            if (high_nibbles) t >>= 4;
            t = (t & 0x000F000Fu) | 0x64006400u;                             // 1024 + q
            __half2 v = *reinterpret_cast<__half2 *>(&t);
            v = __hmul2(__hsub2(v, bias), d2);                               // (q - 8) * d, rounded once
            out[2 * i + h] = *reinterpret_cast<uint32_t *>(&v);
        }
    }
    return make_uint4(out[0], out[1], out[2], out[3]);
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
template <int BN, bool QUANT>
__global__ void __launch_bounds__(THREADS, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap map_b, const __grid_constant__ CUtensorMap map_a,
                   const TcParams p) {
    using L = TcLayout<BN, QUANT>;
    constexpr int ST = L::ST, RAW = QUANT ? L::RAW : 1;   // RAW: ring of the Q4_0 path only
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::bars);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + NUM_BARS);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m0 = blockIdx.x * BN, n0 = blockIdx.y * BM;
    // split-K: CTA z of the cluster along z takes k steps [kt0, kt0 + NT) of the p.NT steps
    const int S = (int)gridDim.z, z = (int)blockIdx.z;
    const int kt0 = (int)((int64_t)p.NT * z / S), NT = (int)((int64_t)p.NT * (z + 1) / S) - kt0;
    auto bar = [&](int i) { return smem_addr(bars + i); };

    if (threadIdx.x == 0) {
        for (int i = 0; i < L::RAW; i++) {
            mbar_init(bar(RAW_FULL + i), 1);
            mbar_init(bar(RAW_EMPTY + i), CONVERTER_WARPS);
        }
        for (int i = 0; i < ST; i++) {
            mbar_init(bar(FULL + i), QUANT ? CONVERTER_WARPS + 1 : 2);
            mbar_init(bar(EMPTY + i), 1);
        }
        mbar_init(bar(ACC_FULL), 1);
    }
    fence_barrier_init();
    if (warp == 1) {   // tensor memory: NACC accumulators of BN f32 columns x 128 lanes
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tmem_slot)),
                     "r"(L::TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    pdl_wait();   // weights, activations and dst follow every earlier grid in the stream
    bool failed = false;

    if (warp == 0) {
        // ---------------------------------------------------------- weight producer
        if (lane == 0) {
            for (int kt = 0; kt < NT && !failed; kt++) {
                if (QUANT) {
                    // the eight row groups' tiles of column step kt: one box of 8 x 1152 bytes
                    // (row groups past the matrix are filled with zeros: weight 0 after conversion)
                    const int rs = kt % RAW;
                    GQ_DCHECK(kt0 + kt < p.NT && n0 / 16 < p.N16, p.status);
                    if (kt >= RAW) wait_or_fail(bar(RAW_EMPTY + rs), (uint32_t)((kt / RAW - 1) & 1), failed, p.status);
                    if (failed) break;
                    mbar_arrive_expect_tx(bar(RAW_FULL + rs), (uint32_t)RAW_STAGE);
                    tma_load_2d(smem_addr(smem + L::raw + rs * RAW_STAGE), &map_a, (kt0 + kt) * RAW_WORDS, n0 / 16,
                                bar(RAW_FULL + rs));
                } else {
                    const int st = kt % ST;
                    if (kt >= ST) wait_or_fail(bar(EMPTY + st), (uint32_t)((kt / ST - 1) & 1), failed, p.status);
                    if (failed) break;
                    mbar_arrive_expect_tx(bar(FULL + st), (uint32_t)A_STAGE);
                    tma_load_2d(smem_addr(smem + L::a + st * A_STAGE), &map_a, (kt0 + kt) * BK, n0, bar(FULL + st));
                    tma_load_2d(smem_addr(smem + L::a + st * A_STAGE + ATOM_BYTES), &map_a, (kt0 + kt) * BK + 64, n0,
                                bar(FULL + st));
                }
            }
        }
    } else if (warp == ACT_PRODUCER_WARP) {
        // ---------------------------------------------------------- activation producer
        if (lane == 0) {
            for (int kt = 0; kt < NT && !failed; kt++) {
                const int st = kt % ST;
                if (kt >= ST) wait_or_fail(bar(EMPTY + st), (uint32_t)((kt / ST - 1) & 1), failed, p.status);
                if (failed) break;
                mbar_arrive_expect_tx(bar(FULL + st), (uint32_t)L::B_STAGE);
                tma_load_2d(smem_addr(smem + L::b + st * L::B_STAGE), &map_b, (kt0 + kt) * BK, m0, bar(FULL + st));
                tma_load_2d(smem_addr(smem + L::b + st * L::B_STAGE + BN * 128), &map_b, (kt0 + kt) * BK + 64, m0,
                            bar(FULL + st));
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA issuer
        // The whole warp runs the loop and waits; lane 0 issues the MMAs and commits.
        constexpr uint32_t idesc = f16_idesc(BM, BN);
        for (int kt = 0; kt < NT; kt++) {
            const int st = kt % ST;
            wait_or_fail(bar(FULL + st), (uint32_t)((kt / ST) & 1), failed, p.status);
            if (__any_sync(0xffffffffu, failed)) {
                failed = true;
                break;
            }
            tc_fence_after();
            if (lane == 0) {
                // The descriptors of the stage's operands; a K step of 16 halves inside a swizzle
                // atom moves the start address by 32 bytes, an atom by its size: both are added to
                // the descriptor's start-address field (address / 16, no carry out of the field).
                const uint64_t ad0 = sw128_desc(smem_addr(smem + L::a + st * A_STAGE));
                const uint64_t bd0 = sw128_desc(smem_addr(smem + L::b + st * L::B_STAGE));
#pragma unroll
                for (int kk = 0; kk < BK / 16; kk++) {
                    const uint64_t ad = ad0 + (uint64_t)(((kk >> 2) * ATOM_BYTES + (kk & 3) * 32) >> 4);
                    const uint64_t bd = bd0 + (uint64_t)(((kk >> 2) * (BN * 128) + (kk & 3) * 32) >> 4);
                    // accumulator kk % NACC; its first MMA overwrites it
                    mma_f16(tmem + (uint32_t)((kk % L::NACC) * BN), ad, bd, idesc,
                            (kt > 0 || kk >= L::NACC) ? 1u : 0u);
                }
                mma_commit(bar(EMPTY + st));   // the stage may be refilled once these MMAs completed
            }
            __syncwarp();
        }
        if (lane == 0 && !failed) mma_commit(bar(ACC_FULL));
    } else {
        // ---------------------------------------------------------- converters, then epilogue
        // warp 2 + 4h + i converts rows 32i .. 32i + 31, columns 64h .. 64h + 63 of each stage
        const int ct = threadIdx.x - 64;
        const int t = ct & (BM - 1), h = ct >> 7;   // weight row of the tile 0..127, column half
        if (QUANT) {
            const int gi = t >> 4, rr = t & 15;
            const bool row_ok = n0 + t < p.N;
            for (int kt = 0; kt < NT; kt++) {
                const int rs = kt % RAW, st = kt % ST;
                wait_or_fail(bar(RAW_FULL + rs), (uint32_t)((kt / RAW) & 1), failed, p.status);
                if (kt >= ST) wait_or_fail(bar(EMPTY + st), (uint32_t)((kt / ST - 1) & 1), failed, p.status);
                GQ_DCHECK(gi < RAW_ROWGROUPS && rr < 16 && h < 2, p.status);
                if (!failed) {
                    const uint8_t *tile = smem + L::raw + rs * RAW_STAGE + gi * TILE_BYTES;
                    uint8_t *a_stage = smem + L::a + st * A_STAGE;
                    // scales of blocks 2h and 2h + 1 of row rr
                    const uint32_t dw =
                        row_ok ? *reinterpret_cast<const uint32_t *>(tile + TILE_SCALE_OFFSET + rr * 8 + h * 4) : 0u;
#pragma unroll
                    for (int jj = 0; jj < 2; jj++) {
                        const int j = 2 * h + jj;
                        const uint4 w = row_ok ? lds128(tile + (j * 16 + rr) * 16) : make_uint4(0x88888888u, 0x88888888u,
                                                                                              0x88888888u, 0x88888888u);
                        const __half d = __ushort_as_half((unsigned short)(jj ? (dw >> 16) : (dw & 0xffffu)));
                        const __half2 d2 = __halves2half2(d, d);
                        // chunk u of 8 values: u=0 low nibbles of bytes 0..7, u=1 bytes 8..15, u=2,3 high nibbles
#pragma unroll
                        for (int u = 0; u < 4; u++) {
                            const uint4 v = dequant8((u & 1) ? w.z : w.x, (u & 1) ? w.w : w.y, u >= 2, d2);
                            const int col = 32 * j + 8 * u;              // K position in the stage
                            const int c = (col & 63) >> 3;               // 16-byte chunk in the 128-byte row
                            *reinterpret_cast<uint4 *>(a_stage + (col >> 6) * ATOM_BYTES + (t >> 3) * 1024 +
                                                       (t & 7) * 128 + ((c ^ (t & 7)) << 4)) = v;
                        }
                    }
                }
                fence_proxy_async_shared();   // the MMA (async proxy) reads what these threads wrote
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive_plain(bar(RAW_EMPTY + rs));
                    mbar_arrive_plain(bar(FULL + st));
                }
            }
        }
        // epilogue: this warp reads tensor-memory lanes 32 * (warp % 4) .. + 31, column
        // chunks h, h + 2, ... of 32, and adds the accumulators in order
        wait_or_fail(bar(ACC_FULL), 0u, failed, p.status);
        tc_fence_after();
    }
    const int q = warp & 3, h = (threadIdx.x - 64) >> 7;   // (epilogue warps 2 .. 9)
    const bool epi = warp >= 2 && warp < 2 + CONVERTER_WARPS;
    // the tile's sums of this thread's row (weight row 32 q + lane) for columns c0 .. c0 + 31
    auto read_acc = [&](const int c0, float (&v)[32]) {
        tmem_ld32(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)c0, v);
#pragma unroll 1
        for (int a = 1; a < L::NACC; a++) {
            float u[32];
            tmem_ld32(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(a * BN + c0), u);
#pragma unroll
            for (int i = 0; i < 32; i++) v[i] += u[i];
        }
    };
    if (S == 1) {
        const int row = n0 + 32 * q + lane;
        if (epi && !failed) {
#pragma unroll 1
            for (int c0 = 32 * h; c0 < BN; c0 += 64) {
                float v[32];
                read_acc(c0, v);
                if (row < p.N) {
#pragma unroll
                    for (int i = 0; i < 32; i++) {
                        const int m = m0 + c0 + i;
                        if (m < p.M) p.dst[(size_t)m * p.N + row] = v[i];
                    }
                }
            }
        }
    } else {
        // Split-K: the S CTAs of the cluster each computed the partial sums of one tile over
        // their K ranges.  Once every CTA's MMAs have completed (first cluster barrier: from then
        // on the operand memory of every CTA is free), each CTA sends row r of its partial to CTA
        // r / (128 / S), into that CTA's slot for it: buf[z][r % (128 / S)][columns].  After the
        // second barrier CTA z adds its 128 / S rows over the S partials in the order
        // z' = 0 .. S - 1, from its own shared memory, and stores them.  Every thread of every
        // CTA passes both barriers; no CTA touches another's memory after the second.
        const int R = BM / S;                            // S divides 128
        cluster_sync();
        if (epi && !failed) {
            const int r = 32 * q + lane;
#pragma unroll 1
            for (int c0 = 32 * h; c0 < BN; c0 += 64) {
                float v[32];
                read_acc(c0, v);
                const uint32_t dst_a = map_shared_rank_addr(
                    smem_addr(smem + L::a) + (uint32_t)(((z * R + r % R) * L::PSTRIDE + c0) * 4), (uint32_t)(r / R));
#pragma unroll
                for (int i = 0; i < 32; i += 4)
                    asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(dst_a + 4 * i), "f"(v[i]),
                                 "f"(v[i + 1]), "f"(v[i + 2]), "f"(v[i + 3])
                                 : "memory");
            }
        }
        cluster_sync();
        if (epi && !failed) {
            const int t = threadIdx.x - 64;              // 0 .. 255
            const int rr = t % R, cstep = CONVERTER_WARPS * 32 / R;   // 256 / R column groups
            const float *buf = reinterpret_cast<const float *>(smem + L::a);
            const int n = n0 + R * z + rr;
#pragma unroll 4
            for (int c = t / R; c < BN; c += cstep) {
                float v = 0.0f;
                for (int zz = 0; zz < S; zz++) v += buf[(zz * R + rr) * L::PSTRIDE + c];
                const int m = m0 + c;
                if (m < p.M && n < p.N) p.dst[(size_t)m * p.N + n] = v;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(L::TMEM_COLS) : "memory");
    }
}

// ---------------------------------------------------------------------------
// activation pre-pass: B[m][k] in fp16
// ---------------------------------------------------------------------------
// Q4_0: the Q8_0 value q8 * fp16(d8) of every activation (one warp per block).
__global__ void __launch_bounds__(256) act_q8_f16_kernel(const float *__restrict__ x, __half *__restrict__ b,
                                                          int M, int K) {
    pdl_wait();
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int64_t nblocks = (int64_t)M * (K / QK);
    for (int64_t blk = warp; blk < nblocks; blk += nwarps) {
        const float v = x[blk * QK + lane];
        const unsigned int amax = __reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(v)));
        const float d = __uint_as_float(amax) / 127.0f;
        const float d16 = __half2float(__float2half_rn(d));
        b[blk * QK + lane] = __float2half_rn((float)q8_code_s(v, q8_scale(d)) * d16);   // the product is exact in f32
    }
}

// F16: the activations rounded to fp16.
__global__ void __launch_bounds__(256) act_f16_kernel(const float *__restrict__ x, __half *__restrict__ b,
                                                      int64_t n) {
    pdl_wait();
    pdl_launch_dependents();
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
        b[i] = __float2half_rn(x[i]);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

gq_status encoder(PFN_cuTensorMapEncodeTiled_v12000 *out) {
    std::call_once(g_encode_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    if (!g_encode) return fail(GQ_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
    *out = g_encode;
    return GQ_OK;
}

// fp16 matrix [rows][K], K contiguous; box of 64 K x box_rows with 128-byte swizzle
gq_status f16_map(CUtensorMap *map, const void *base, int64_t rows, int64_t K, int box_rows) {
    PFN_cuTensorMapEncodeTiled_v12000 enc;
    gq_status st = encoder(&enc);
    if (st != GQ_OK) return st;
    const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    const cuuint32_t box[2] = {64u, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1u, 1u};
    const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(GQ_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return GQ_OK;
}

// Repacked Q4_0 weights as a 2D tensor of row groups: row g holds the NT tiles of
// row group g (NT * 1152 bytes), read as 8-byte elements; a box is one tile
// column of 8 row groups.  Row groups past the matrix read as zeros.
gq_status q4_raw_map(CUtensorMap *map, const void *base, int64_t N16, int64_t NT) {
    PFN_cuTensorMapEncodeTiled_v12000 enc;
    gq_status st = encoder(&enc);
    if (st != GQ_OK) return st;
    const cuuint64_t dims[2] = {(cuuint64_t)(NT * RAW_WORDS), (cuuint64_t)N16};
    const cuuint64_t strides[1] = {(cuuint64_t)(NT * TILE_BYTES)};
    const cuuint32_t box[2] = {(cuuint32_t)RAW_WORDS, (cuuint32_t)RAW_ROWGROUPS};
    const cuuint32_t estr[2] = {1u, 1u};
    const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, const_cast<void *>(base), dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(GQ_ERR_CUDA, "cuTensorMapEncodeTiled (repacked weights) failed (%d)", (int)r);
    return GQ_OK;
}

constexpr int MAX_DEV = 64;
std::atomic<bool> g_tc_smem_set[MAX_DEV][8];

template <typename Kernel>
gq_status allow_tc_smem(Kernel kernel, int which, int bytes) {
    int dev = 0;
    gq_status st = check_cuda(cudaGetDevice(&dev), "cudaGetDevice");
    if (st != GQ_OK) return st;
    if (dev >= 0 && dev < MAX_DEV && g_tc_smem_set[dev][which].load(std::memory_order_acquire)) return GQ_OK;
    st = check_cuda(cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes),
                    "tc shared-memory attribute");
    if (st == GQ_OK && dev >= 0 && dev < MAX_DEV) g_tc_smem_set[dev][which].store(true, std::memory_order_release);
    return st;
}

// Split-K factor for a grid of `tiles` output tiles of NT k steps: the largest power of two
// S <= 8 with tiles * S CTAs in one wave (one CTA per SM) and at least 4 k steps per CTA
// (Smallem, "La courbe, une première fois": split the common dimension when the output
// tiles are too few to occupy the GPU; DeepSpeed-Inference notes, III.C.1).  GQ_TC_SPLIT
// (1, 2, 4 or 8), when set, replaces it (a tuning and test switch).
int split_for(int64_t tiles, int NT, bool can_split) {
    if (!can_split) return 1;
    const char *e = getenv("GQ_TC_SPLIT");
    if (e && *e) {
        const int f = atoi(e);
        if (f == 1 || f == 2 || f == 4 || f == 8) return std::min(f, std::max(1, NT));
    }
    int S = 1;
    while (S < 8 && tiles * 2 * S <= sm_count() && NT / (2 * S) >= 4) S *= 2;
    return S;
}

template <int BN, bool QUANT>
gq_status launch_tc(const CUtensorMap &mb, const CUtensorMap &ma, const TcParams &p, cudaStream_t s, int which) {
    using L = TcLayout<BN, QUANT>;
    constexpr int smem = L::total + 1024;
    auto kernel = tc_gemm_kernel<BN, QUANT>;
    gq_status st = allow_tc_smem(kernel, which, smem);
    if (st != GQ_OK) return st;
    const int64_t gx = (p.M + BN - 1) / BN, gy = (p.N + BM - 1) / BM;
    int S = split_for(gx * gy, p.NT, L::CAN_SPLIT);
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(THREADS, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    cfg.attrs = attr;
    for (;;) {
        cfg.gridDim = dim3((unsigned)gx, (unsigned)gy, (unsigned)S);
        attr[1].val.clusterDim.x = 1;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = (unsigned)S;
        cfg.numAttrs = S > 1 ? 2 : 1;
        if (S == 1) break;
        // the clusters of a split are co-scheduled on one GPC: keep the split only if every
        // cluster of the grid is resident at once
        int active = 0;
        if (cudaOccupancyMaxActiveClusters(&active, kernel, &cfg) == cudaSuccess && (int64_t)active >= gx * gy) break;
        cudaGetLastError();
        S /= 2;
    }
    return check_cuda(cudaLaunchKernelEx(&cfg, kernel, mb, ma, p), "tc_gemm launch");
}

// Activation rows per tile, the MMA's N.  Each tcgen05.mma costs about the same
// time up to N = 256 on this GPU, so 256-wide tiles do twice the work per
// instruction; they are taken when 128-wide tiles would need more than one wave
// of CTAs, where the halved grid still fills the SMs.
int tile_n(int64_t M, int64_t N) {
    if (M <= 32) return 32;
    if (M <= 64) return 64;
    if (M <= 128) return 128;
    const int64_t grid128 = ((M + 127) / 128) * ((N + BM - 1) / BM);
    return grid128 > sm_count() ? 256 : 128;
}

gq_status launch_tc_common(bool quant, const void *w, const float *x, float *dst, int64_t M, int64_t N, int64_t K,
                           cudaStream_t s) {
    TcParams p{};
    p.status = device_status_word();
    if (!p.status) return fail(GQ_ERR_CUDA, "device status word unavailable");
    p.M = (int)M;
    p.N = (int)N;
    p.K = (int)K;
    p.NT = (int)((K + BK - 1) / BK);
    p.N16 = (int)((N + 15) / 16);
    p.dst = dst;

    Workspace ws;
    gq_status st = get_workspace(s, 0, tc_workspace_bytes(M, K), &ws);
    if (st != GQ_OK) return st;
    __half *b = reinterpret_cast<__half *>(ws.data);

    // the activations in fp16
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const int64_t n = M * K;
    cfg.gridDim = dim3((unsigned)std::min<int64_t>((n + 255) / 256, 8LL * sm_count()), 1, 1);
    if (quant)
        st = check_cuda(cudaLaunchKernelEx(&cfg, act_q8_f16_kernel, x, b, (int)M, (int)K), "activation pre-pass");
    else
        st = check_cuda(cudaLaunchKernelEx(&cfg, act_f16_kernel, x, b, n), "activation pre-pass");
    if (st != GQ_OK) return st;

    const int bn = tile_n(M, N);
    CUtensorMap mb, ma;
    memset(&ma, 0, sizeof(ma));
    st = f16_map(&mb, b, M, K, bn);
    if (st != GQ_OK) return st;
    st = quant ? q4_raw_map(&ma, w, p.N16, p.NT) : f16_map(&ma, w, N, K, BM);
    if (st != GQ_OK) return st;
    if (quant) {
        if (bn == 32) return launch_tc<32, true>(mb, ma, p, s, 0);
        if (bn == 64) return launch_tc<64, true>(mb, ma, p, s, 1);
        if (bn == 128) return launch_tc<128, true>(mb, ma, p, s, 2);
        return launch_tc<256, true>(mb, ma, p, s, 3);
    }
    if (bn == 32) return launch_tc<32, false>(mb, ma, p, s, 4);
    if (bn == 64) return launch_tc<64, false>(mb, ma, p, s, 5);
    if (bn == 128) return launch_tc<128, false>(mb, ma, p, s, 6);
    return launch_tc<256, false>(mb, ma, p, s, 7);
}

}  // namespace

size_t tc_workspace_bytes(int64_t M, int64_t K) { return (size_t)M * (size_t)K * sizeof(__half); }

gq_status launch_tc_q4_0(const void *rep, const float *x, float *dst, int64_t M, int64_t N, int64_t K,
                         cudaStream_t s) {
    return launch_tc_common(true, rep, x, dst, M, N, K, s);
}

gq_status launch_tc_f16(const void *w16, const float *x, float *dst, int64_t M, int64_t N, int64_t K,
                        cudaStream_t s) {
    return launch_tc_common(false, w16, x, dst, M, N, K, s);
}

constexpr int F16_TILE_COLS_RM = 32;

gq_status f16_tile_map(void *map, const void *base, int64_t N, int64_t K) {
    PFN_cuTensorMapEncodeTiled_v12000 enc;
    gq_status st = encoder(&enc);
    if (st != GQ_OK) return st;
    if (N <= 0 || N > 0xFFFFFFFFLL || K <= 0 || K % F16_TILE_COLS_RM)
        return fail(GQ_ERR_INVALID_ARG, "row-major F16 tensor map of %lld x %lld", (long long)N, (long long)K);
    // element (column c of tile column t, row n) at base + 2 (n K + 32 t + c)
    const cuuint64_t dims[3] = {(cuuint64_t)F16_TILE_COLS_RM, (cuuint64_t)N, (cuuint64_t)(K / F16_TILE_COLS_RM)};
    const cuuint64_t strides[2] = {(cuuint64_t)K * 2, (cuuint64_t)F16_TILE_COLS_RM * 2};
    const cuuint32_t box[3] = {(cuuint32_t)F16_TILE_COLS_RM, 16u, 16u};
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    const CUresult r = enc(reinterpret_cast<CUtensorMap *>(map), CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void *>(base),
                           dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(GQ_ERR_CUDA, "cuTensorMapEncodeTiled (row-major F16 tiles) failed (%d)", (int)r);
    return GQ_OK;
}

gq_status byte_rows_map(void *map, const void *base, int64_t rows, int box_rows) {
    PFN_cuTensorMapEncodeTiled_v12000 enc;
    gq_status st = encoder(&enc);
    if (st != GQ_OK) return st;
    if (rows <= 0 || rows > 0xFFFFFFFFLL) return fail(GQ_ERR_INVALID_ARG, "tensor map of %lld rows", (long long)rows);
    const cuuint64_t dims[2] = {128u, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {128u};
    const cuuint32_t box[2] = {128u, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1u, 1u};
    const CUresult r = enc(reinterpret_cast<CUtensorMap *>(map), CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base),
                           dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(GQ_ERR_CUDA, "cuTensorMapEncodeTiled (byte rows) failed (%d)", (int)r);
    return GQ_OK;
}

}  // namespace gq
