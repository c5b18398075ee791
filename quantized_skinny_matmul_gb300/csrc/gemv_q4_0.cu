// gemv_q4_0.cu -- the persistent GEMV of the weight formats in repacked tiles
// (Q4_0, Q8_0, Q5_0, Q4_1 and F16 tiles) for up to 16 activation rows per
// launch: small-batch decode.  (The one-row Q4_0 product, single-token decode,
// runs the kernel of gemv_m1.cu.)
//
// In this regime every weight byte is read once and the product is bound by
// HBM (Smallem, "Générer à plusieurs", introduction and "Où la courbe
// s'aplatit": with B sequences each weight read serves B products; DeepSpeed-
// Inference notes, III.A: small batches are limited by the bandwidth of reading
// the weights).
//
//  * K slices.  K is cut into S slices so that a CTA's image of the activations
//    fits in shared memory (S depends on K and on the number of rows).  With
//    several activation rows a product runs one launch per slice: every CTA
//    owns whole row groups (16 weight rows) and the launches of later slices
//    add their sums into dst in slice order (split-K for small grids: Smallem,
//    "La courbe, une première fois"; DeepSpeed-Inference notes, III.C.1).  With
//    one row and several slices (very long rows) one launch runs all slices:
//    the tiles of a slice are divided evenly between its CTAs, and a row group
//    that CTAs share is added by a fix-up warp of the CTA that arrives last, in
//    a fixed order.
//  * INIT (llama.cpp PR #1632, "Introduction": the q_f32 kind quantizes src1
//    to Q8_0 before the block dots; Arm China NUMA article, "MulMat 算子優化":
//    every worker reads the wdata).  With one row each consumer warp
//    quantizes the blocks of its own tiles; with several rows the CTA
//    quantizes its slice of the rows into shared memory (up to three load
//    rounds), or, for larger rows, a small kernel (wdata_kernel) writes the
//    images of all slices to the workspace once and the GEMV loads its slice.
//  * COMPUTE, persistent, at most one CTA per SM (two for one row: the CTA of
//    the next product is resident beside this one).  Two producer warps stream
//    the CTA's tiles through a ring of shared-memory chunks with bulk (TMA)
//    copies and keep L2 prefetches ahead of it; with static weights they start
//    before the wait on the grids in front.  8 or 16 consumer warps take the
//    tiles of each chunk by position (two tiles, or one, per warp): up to four
//    rows, eight dp4a per block on
//    the unpacked nibbles and the codes (exact int32) scaled by d4 * d8; eight
//    rows and more, two m16n8k16 fp16 MMAs per block whose f32 result is the
//    exact block dot (the codes and (q - 8) are exact in fp16).  At the end of
//    a row group the positions' partials are added in shared memory in a fixed
//    order (DeepSpeed-Inference notes, III.C.2: make the partials of one
//    output contiguous and reduce them in one pass).
#include <cuda.h>

#include <algorithm>
#include <atomic>

#include "gq_common.cuh"
#include "gq_internal.h"

namespace gq {
namespace {

constexpr int CHUNK_TILES = 16;                    // tiles per chunk = tile positions
constexpr int PRODUCERS = 2;                       // producer warps (bulk-copy issue rate is per warp)

// CTA shapes: 8 consumer warps (one row, with no fix-up warp: two CTAs per SM, so
// the next product's CTA streams its weights beside this one; several rows of a
// block format: one CTA per SM, 128 registers, two tiles of each chunk per warp) or
// 16 (one CTA per SM: F16 tiles of more than 8 rows).  A consumer warp keeps one accumulator per tile position of a chunk,
// and the row-group sum adds the 16 positions in order: every output is the same
// sum, in the same order, for both shapes.  A scheduler holds 16 K registers: five
// warps of 96 (16 + 2 + 2 warps, one CTA), twice over five of 88 (8 + 2 + 0 warps,
// two CTAs), or three of 128 (8 + 2 + 1 warps, one CTA).
template <int CWT, int FIXW = (CWT == 8 ? 1 : 2)>
struct Shape {
    static constexpr int CW = CWT;                          // consumer warps
    static constexpr int TPW = CHUNK_TILES / CWT;           // tile positions per consumer warp
    static constexpr int PRODUCER_WARP = CWT;               // .. + PRODUCERS - 1
    static constexpr int FIXUPS = FIXW;                     // fix-up warps (none: no shared row group)
    static constexpr int FIXUP_WARP = CWT + PRODUCERS;      // .. + FIXUPS - 1
    static constexpr int THREADS = (CWT + PRODUCERS + FIXUPS) * 32;
    static constexpr int CONSUMERS = CWT * 32;
    static constexpr int FUSED_LOADS = 4;                   // float4 per consumer thread and round of the fused INIT
};
// Repacked F16 weights: a tile is 16 rows x 32 columns, 64 bytes per row.
constexpr int F16_TILE_COLS = 32;
constexpr int F16_TILE_BYTES = 16 * F16_TILE_COLS * 2;
// Repacked Q8_0 weights: a tile is 16 rows x 4 blocks like Q4_0; the 32 codes of block j of row r
// at (j * 16 + r) * 32, then the 64 fp16 scales at 2048 + (r * 4 + j) * 2.
constexpr int Q8_TILE_SCALE_OFFSET = 16 * TILE_BLOCKS * QK;
constexpr int Q8_TILE_BYTES = Q8_TILE_SCALE_OFFSET + 16 * TILE_BLOCKS * 2;
// Repacked Q5_0 weights: 16 rows x 4 blocks; the nibble bytes as in Q4_0 (1024 bytes), the fifth
// bits of block j of row r at 1024 + (j * 16 + r) * 4, then the fp16 scales at 1280 + (r * 4 + j) * 2.
constexpr int Q5_TILE_HIGH_OFFSET = TILE_SCALE_OFFSET;
constexpr int Q5_TILE_SCALE_OFFSET = Q5_TILE_HIGH_OFFSET + 16 * TILE_BLOCKS * 4;
constexpr int Q5_TILE_BYTES = Q5_TILE_SCALE_OFFSET + 16 * TILE_BLOCKS * 2;
// Repacked Q4_1 weights: the nibble bytes as in Q4_0, the fp16 scales at 1024 + (r * 4 + j) * 2 and
// the fp16 minimums at 1152 + (r * 4 + j) * 2.
constexpr int Q41_TILE_MIN_OFFSET = TILE_SCALE_OFFSET + 16 * TILE_BLOCKS * 2;
constexpr int Q41_TILE_BYTES = Q41_TILE_MIN_OFFSET + 16 * TILE_BLOCKS * 2;
// weight formats of the kernel
// (WF_F16RM: F16 weights as stored, row-major [N][K]; a 3D tensor copy lands 16 of their
// 16 x 32 tiles in the layout of the repacked F16 tiles, so the kernel is the repacked one's)
enum : int { WF_Q4 = 0, WF_F16 = 1, WF_Q8 = 2, WF_Q5 = 3, WF_Q41 = 4, WF_F16RM = 5 };
__host__ __device__ constexpr bool is_f16(int wf) { return wf == WF_F16 || wf == WF_F16RM; }
// (tile_bytes and Layout spell the F16 test out: the kernels build their Layout from a wf argument,
// and with the call to is_f16 there the one-row 88-register kernels spilled and ran 5-10 % slower)
__host__ __device__ constexpr int tile_bytes(int wf) {
    return wf == WF_F16 || wf == WF_F16RM ? F16_TILE_BYTES
           : wf == WF_Q8 ? Q8_TILE_BYTES
           : wf == WF_Q5 ? Q5_TILE_BYTES
           : wf == WF_Q41 ? Q41_TILE_BYTES
                          : TILE_BYTES;
}
__host__ __device__ constexpr int chunk_bytes(int wf) { return CHUNK_TILES * tile_bytes(wf); }
constexpr int MAX_SLOTS = 12;
constexpr int PART_STRIDE = 16 * 16;               // floats of one partial (16 rows x 16 activation rows)
constexpr int FIX_BATCH = 8;                       // partials one fix-up lane loads before adding them
constexpr int FUSED_ROUNDS = 3;                    // load rounds of the fused INIT (more: a separate INIT is faster)
constexpr size_t ACT_BUDGET = 112 * 1024;          // wdata image of one slice
constexpr size_t SMEM_LIMIT = 227 * 1024;
constexpr size_t SMEM_HALF = 113 * 1024;           // half of the shared memory of an SM
constexpr int MIN_SLOTS_HALF = 4;
constexpr int PF_KB = 160;                         // L2 prefetch distance beyond the ring, per CTA

__host__ __device__ constexpr size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// One slice's wdata image: the Q8_0 codes of M activation rows ([M][4*ntmax
// blocks][32 bytes], element order) and per (row, block) the pair
// (f32 scale fp16(d), int32 -8 * sum of the codes).
struct Image {
    // Rows are padded by 16 bytes (codes) and one float2 (scales) so that the eight
    // activation rows one MMA fragment reads fall in different shared-memory banks.
    // F16 rows take an odd number of 64-byte tiles: the two rows of a quarter warp's
    // 16-byte loads then fill the 128 bytes of the banks once.
    size_t row_bytes, codes, scales, bytes;
    int sc_stride;                                  // float2 per row of scales
    // Q4_0: Q8_0 codes [M][ntmax tiles x 128] then {d8, -8 sum q8} per block;
    // F16: the activations in fp16, [M][ntmax tiles x 32], no scales.
    __host__ __device__ Image(int M, int ntmax, bool f16 = false) {
        row_bytes = f16 ? (size_t)(ntmax | 1) * F16_TILE_COLS * 2 : (size_t)4 * ntmax * 32 + 16;
        sc_stride = f16 ? 0 : 4 * ntmax + 1;
        codes = 0;
        scales = (size_t)M * row_bytes;
        bytes = align_up(scales + (size_t)M * sc_stride * 8, 16);
    }
};

// The tensor map of row-major F16 weights (dims {32, N, K / 32}, box {32, 16, 16}: one chunk),
// a kernel parameter of its own: in the parameters of every kernel, its 128 bytes made the
// 88-register one-row kernels spill (and run 5-7 % slower), so the other kernels take a byte.
template <bool RM>
struct Wmap {
    unsigned char unused;
};
template <>
struct Wmap<true> {
    CUtensorMap map;
};

struct Params {
    const uint8_t *w;        // repacked Q4_0
    const float *x;          // [M][K]
    float *dst;              // [M][N]
    unsigned int *status;    // device status word
    float *part;             // workspace partials [N16][S][2][PART_STRIDE]
    unsigned int *cnt;       // workspace counters [N16], zero between launches
    uint8_t *wdata;          // workspace wdata images [S][image bytes]
    int M, N, K;
    int nb, N16, NT;
    int S, Gs;               // slices, CTAs per slice (grid = S * Gs)
    int slots, ntmax, maxfix;
    int pf;                  // L2 prefetch distance of the producers, in chunks
    int fused;               // 1: no INIT launch, each CTA quantizes its slice of src1
    int early;               // 1: the producers may read the weights before the grids in front finished
    int init_early;          // 1: INIT lets the GEMV start before the grids in front finished (static weights)
    int seq_slice;           // >= 0: this launch takes K slice seq_slice over whole row groups per CTA
                             // (one launch per slice); slices after the first add into dst
};

// Buffers of row-group partials: four for tiles of 2 to 4 rows (the partials of two row groups
// are added after one barrier: 2-4 % faster at M = 2 and 4 on the 7B decode shapes), two otherwise
// (one barrier per row group; four buffers cost a ring slot at M = 8 and measured 5 % slower, and
// the 88-register one-row shape spilled and lost 5-7 % with them).
__host__ __device__ constexpr int red_buffers(int MT) { return MT >= 2 && MT <= 4 ? 4 : 2; }

struct Layout {
    size_t bars, ring, act, red, total;
    __host__ __device__ Layout(int MT, int M, int ntmax, int slots, int maxfix, int wf = WF_Q4) {
        const Image im(M, ntmax, wf == WF_F16 || wf == WF_F16RM);   // Q8_0 weights use the Q4_0 image
        bars = 0;                                         // full[slots], empty[slots], act, fix[maxfix]
        ring = align_up((size_t)(2 * slots + 1 + maxfix) * 8, 128);
        act = ring + (size_t)slots * chunk_bytes(wf);
        red = act + im.bytes;
        total = red + (size_t)red_buffers(MT) * CHUNK_TILES * 16 * MT * 4;   // row groups rotate over them
    }
};

__host__ __device__ inline void slice_of(int NT, int S, int s, int &ts0, int &nts) {
    ts0 = (int)((int64_t)NT * s / S);
    nts = (int)((int64_t)NT * (s + 1) / S) - ts0;
}

// The CTAs of a slice own the consecutive ranges [T*i/Gs, T*(i+1)/Gs) of its T
// tiles.  Index of the CTA whose range holds tile x.
__host__ __device__ inline int owner(int T, int Gs, int x) {
    const int i = (int)(((int64_t)(x + 1) * Gs + T - 1) / T) - 1;
    return i < Gs - 1 ? i : Gs - 1;
}

// Number of CTAs of all slices that hold a part of row group g.
__device__ inline unsigned int contributors(const Params &p, int g) {
    unsigned int n = 0;
    for (int s2 = 0; s2 < p.S; s2++) {
        int t2, n2;
        slice_of(p.NT, p.S, s2, t2, n2);
        const int T2 = p.N16 * n2;
        n += (unsigned)(owner(T2, p.Gs, (g + 1) * n2 - 1) - owner(T2, p.Gs, g * n2) + 1);
    }
    return n;
}

// The row-group segments of a CTA's range [a, b) of slice tiles, in the order
// the CTA processes them: segments shared with another CTA first (all of them
// when S > 1), then the CTA's own row groups in increasing order.
struct Segments {
    int a, b;
    int nts, g0, n;          // first row group, number of segments
    bool head, tail, all_shared;
    int nshared;
    __host__ __device__ Segments(int a_, int b_, int nts_, int S) : a(a_), b(b_), nts(nts_) {
        g0 = (int)(a / nts);
        n = (int)((b - 1) / nts) - g0 + 1;
        head = (a % nts) != 0;
        tail = (b % nts) != 0;
        all_shared = S > 1;
        nshared = all_shared ? n : (int)head + (int)(tail && !(head && n == 1));
    }
    // natural index (0 = first row group of the range) of the j-th processed segment
    __host__ __device__ int natural(int j) const {
        if (all_shared) return j;
        int k = 0;
        if (tail && !(head && n == 1)) {
            if (j == k) return n - 1;
            k++;
        }
        if (head) {
            if (j == k) return 0;
            k++;
        }
        return j - k + (head ? 1 : 0);   // the unshared row groups, ascending
    }
    __host__ __device__ void get(int j, int &g, int &u0, int &u1) const {
        const int nat = natural(j);
        g = g0 + nat;
        const int lo = g * nts, hi = lo + nts;
        u0 = (a > lo ? a : lo) - lo;
        u1 = (b < hi ? b : hi) - lo;
    }
};

template <int CONSUMERS>
__device__ __forceinline__ void consumers_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(CONSUMERS) : "memory");
}

// Release of this thread's (and, through a preceding barrier, its CTA's or
// warp's) earlier writes and acquire of the other arrivals' writes.
__device__ __forceinline__ unsigned int atomic_add_acq_rel_gpu(unsigned int *p, unsigned int v) {
    unsigned int old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

// ---------------------------------------------------------------------------
// INIT: Q8_0 of the activation rows into the wdata images.  One warp per
// (row, block): lane j holds element j; the block goes to the image of the
// slice that holds it.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) wdata_kernel(const Params p) {
    if (p.init_early) pdl_launch_dependents();   // weights are static: the GEMV may stream them at once
    pdl_wait();                 // src1 and the workspace are final: every earlier grid has completed
    pdl_launch_dependents();    // (no-op if already triggered) every grid before INIT is complete
    const Image im(p.M, p.ntmax);
    const int lane = threadIdx.x & 31;
    const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int nblk = 4 * p.NT;                   // blocks including the padding of the last tile
    for (int64_t task = warp; task < (int64_t)p.M * nblk; task += nwarps) {
        const int m = (int)(task / nblk), b = (int)(task % nblk);
        const int t = b / 4;
        int s = 0, ts0 = 0, nts = 0;
        for (; s < p.S; s++) {
            slice_of(p.NT, p.S, s, ts0, nts);
            if (t < ts0 + nts) break;
        }
        const int bl = b - 4 * ts0;
        const float v = b < p.nb ? p.x[(size_t)m * p.K + (size_t)b * QK + lane] : 0.0f;
        const unsigned int amax = __reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(v)));
        const float d = __uint_as_float(amax) / 127.0f;
        const int q = q8_code_s(v, q8_scale(d));
        const int qsum = __reduce_add_sync(0xffffffffu, q);
        uint8_t *img = p.wdata + (size_t)s * im.bytes;
        img[im.codes + (size_t)m * im.row_bytes + (size_t)bl * 32 + lane] = (uint8_t)(q & 0xff);
        if (lane == 0)
            reinterpret_cast<float2 *>(img + im.scales)[(size_t)m * im.sc_stride + bl] =
                make_float2(__half2float(__float2half_rn(d)), __int_as_float(-8 * qsum));
    }
}

// 3D tensor copy of one box into shared memory (completion on an mbarrier, L2 cache hint), and
// its L2 prefetch.  Coordinates are element indices; the innermost one is 0 here (x * 2 bytes
// aligned to 16).
__device__ __forceinline__ void tensor3d_g2s_hint(uint32_t dst, const CUtensorMap *map, int x, int y, int z,
                                                  uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void tensor3d_prefetch_l2(const CUtensorMap *map, int x, int y, int z) {
    asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y), "r"(z)
                 : "memory");
}

// ---------------------------------------------------------------------------
// COMPUTE
// ---------------------------------------------------------------------------
template <int MT, int CWT, int REGS, int WF, int FIXW>
__global__ void __launch_bounds__(Shape<CWT, FIXW>::THREADS) __maxnreg__(REGS)
    gemv_q4_0_kernel(const Params p, const __grid_constant__ Wmap<WF == WF_F16RM> wm) {
    constexpr bool F16W = is_f16(WF), RMW = WF == WF_F16RM, Q8W = WF == WF_Q8, Q5W = WF == WF_Q5, Q41W = WF == WF_Q41;
    constexpr int TB = tile_bytes(WF), CB = chunk_bytes(WF);
    // fp16 scales in a Q4_0 / Q5_0 / Q8_0 tile
    constexpr int SCALES = Q8W ? Q8_TILE_SCALE_OFFSET : Q5W ? Q5_TILE_SCALE_OFFSET : TILE_SCALE_OFFSET;
    using SH = Shape<CWT, FIXW>;
    constexpr int CW = SH::CW, TPW = SH::TPW, CONSUMERS = SH::CONSUMERS, THREADS = SH::THREADS;
    constexpr int PRODUCER_WARP = SH::PRODUCER_WARP, FIXUP_WARP = SH::FIXUP_WARP, FUSED_LOADS = SH::FUSED_LOADS;
    constexpr int FIXUPS = SH::FIXUPS;
    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // one launch per K slice: several activation rows only (the host never asks it of the
    // one-row kernels, which then compile without it)
    const int seq_slice = (F16W || MT > 1) ? p.seq_slice : -1;
    const bool one_slice = p.S == 1 || seq_slice >= 0;   // whole row groups per CTA
    const int s = seq_slice >= 0 ? seq_slice : (int)(blockIdx.x / p.Gs);
    const int ci = seq_slice >= 0 ? (int)blockIdx.x : (int)(blockIdx.x % p.Gs);
    int ts0, nts;
    slice_of(p.NT, p.S, s, ts0, nts);
    const int T = p.N16 * nts;   // tiles of the slice (< 2^31: N * K <= 2^40)
    // one slice per launch: whole row groups per CTA (no shared row group); S > 1 slices in
    // one launch: equal tile ranges
    const Segments seg = one_slice ? Segments((int)((int64_t)p.N16 * ci / p.Gs) * nts,
                                             (int)((int64_t)p.N16 * (ci + 1) / p.Gs) * nts, nts, 1)
                                  : Segments((int)((int64_t)T * ci / p.Gs), (int)((int64_t)T * (ci + 1) / p.Gs), nts,
                                             p.S);
    const Layout L(MT, p.M, p.ntmax, p.slots, p.maxfix, WF);
    const Image im(p.M, p.ntmax, F16W);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.bars);
    uint64_t *empty = full + p.slots;
    uint64_t *actbar = empty + p.slots;
    uint64_t *fixbar = actbar + 1;
    uint8_t *ring = smem + L.ring;
    const int outs = 16 * MT;                        // outputs of a row group: t = m * 16 + row

    // barriers in parallel: full[slots] (1 arrival), empty[slots] (CW), act (1), fix[maxfix] (1)
    for (int i = threadIdx.x; i < 2 * p.slots + 1 + p.maxfix; i += THREADS)
        mbar_init(smem_addr(full + i), (i >= p.slots && i < 2 * p.slots) ? CW : 1);
    fence_barrier_init();
    __syncthreads();
    pdl_launch_dependents();

    // ---------------------------------------------------------------- producers
    // Producer warp pw issues the chunks k = pw (mod PRODUCERS); the ring has an
    // even number of slots, so each producer refills only its own slots.  The ring
    // alone keeps too few bytes in flight for HBM; each producer also keeps L2
    // prefetches of its chunks up to p.pf chunks ahead of its copies, so that the
    // copies are served from L2.  A prefetch moves nothing into the CTA and L2 is
    // where all accesses to device memory meet, so prefetches may run before the
    // grids in front have finished; the copies wait for them when the weights are
    // not declared static.
    if (warp >= PRODUCER_WARP && warp < PRODUCER_WARP + PRODUCERS) {
        const int pw = warp - PRODUCER_WARP;
        // chunk k of this CTA's sequence: source and size (row group g, first tile column t of the
        // slice); false past the last chunk
        auto chunk_at = [&](int k, const uint8_t *&src, uint32_t &bytes, int &g, int &t) -> bool {
            for (int j = 0; j < seg.n; j++) {
                int u0, u1;
                seg.get(j, g, u0, u1);
                const int n = (u1 - u0 + CHUNK_TILES - 1) / CHUNK_TILES;
                if (k < n) {
                    const int u = u0 + k * CHUNK_TILES;
                    t = ts0 + u;
                    src = p.w + ((size_t)g * p.NT + t) * TB;
                    // row-major F16: the whole box, whose tiles past the row group's end are those
                    // of the next K slice (unused) or lie past K (zeros)
                    bytes = RMW ? (uint32_t)CB : (uint32_t)(min(CHUNK_TILES, u1 - u) * TB);
                    return true;
                }
                k -= n;
            }
            return false;
        };
        int kp = p.early ? pw + p.slots : pw;   // next chunk to prefetch (early: the ring's first copies go first)
        auto prefetch_to = [&](int kend) {
            const uint8_t *src;
            uint32_t bytes;
            int g, t;
            for (; kp < kend && chunk_at(kp, src, bytes, g, t); kp += PRODUCERS) {
                if constexpr (RMW) tensor3d_prefetch_l2(&wm.map, 0, 16 * g, t);
                else bulk_prefetch_l2(src, bytes);
            }
        };
        if (!p.early) {
            if (lane == 0) prefetch_to(p.pf);
            pdl_wait();   // the weights may still be written by the grid in front
        }
        if (lane == 0) {
            const uint64_t policy = l2_evict_first_policy();   // every weight byte is read once
            const uint8_t *src;
            uint32_t bytes;
            int g, t;
            for (int k = pw; chunk_at(k, src, bytes, g, t); k += PRODUCERS) {
                const int slot = k % p.slots;
                if (k >= p.slots &&
                    !mbar_wait(smem_addr(empty + slot), (uint32_t)(((k / p.slots) - 1) & 1), p.status))
                    break;
                mbar_arrive_expect_tx(smem_addr(full + slot), bytes);
                if constexpr (RMW)
                    tensor3d_g2s_hint(smem_addr(ring + (size_t)slot * CB), &wm.map, 0, 16 * g, t, smem_addr(full + slot),
                                      policy);
                else
                    bulk_g2s_hint(smem_addr(ring + (size_t)slot * CB), src, bytes, smem_addr(full + slot), policy);
                prefetch_to(k + p.pf);
            }
        }
        return;
    }

    // ---------------------------------------------------------------- fix-up
    if (FIXUPS > 0 && warp >= FIXUP_WARP) {   // (the launch has no shared row group when FIXUPS == 0)
        pdl_wait();
        for (int f = warp - FIXUP_WARP; f < seg.nshared; f += (FIXUPS > 0 ? FIXUPS : 1)) {
            const bool ok = mbar_wait(smem_addr(fixbar + f), 0u, p.status);
            if (!__all_sync(0xffffffffu, ok)) break;
            int g, u0, u1;
            seg.get(f, g, u0, u1);
            unsigned int last = 0;
            if (lane == 0)   // the consumers' partial is in the workspace: release it, count the arrival
                last = (atomic_add_acq_rel_gpu(p.cnt + g, 1u) + 1 == contributors(p, g)) ? 1u : 0u;
            last = __shfl_sync(0xffffffffu, last, 0);
            if (last) {   // add every partial of row group g in a fixed order: slice, then contributor
                // a lane takes four consecutive outputs and has up to FIX_BATCH partials in flight
                for (int tq = lane; tq < outs / 4; tq += 32) {
                    float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
                    for (int i0 = 0; i0 < 2 * p.S; i0 += FIX_BATCH) {
                        float4 v[FIX_BATCH];
                        bool have[FIX_BATCH];
#pragma unroll
                        for (int b = 0; b < FIX_BATCH; b++) {
                            const int s2 = (i0 + b) >> 1, q = (i0 + b) & 1;
                            have[b] = false;
                            if (s2 < p.S) {
                                int t2, n2;
                                slice_of(p.NT, p.S, s2, t2, n2);
                                const int T2 = p.N16 * n2;
                                have[b] = q <= owner(T2, p.Gs, (g + 1) * n2 - 1) - owner(T2, p.Gs, g * n2);
                            }
                            v[b] = have[b] ? __ldcg(reinterpret_cast<const float4 *>(
                                                 p.part + (((size_t)g * p.S + s2) * 2 + q) * PART_STRIDE) + tq)
                                           : make_float4(0.f, 0.f, 0.f, 0.f);
                        }
#pragma unroll
                        for (int b = 0; b < FIX_BATCH; b++)
                            if (have[b]) {
                                sum.x += v[b].x;
                                sum.y += v[b].y;
                                sum.z += v[b].z;
                                sum.w += v[b].w;
                            }
                    }
                    const int m = (4 * tq) / 16, n0 = 16 * g + (4 * tq) % 16;
                    if (m < p.M) {
                        float *o = p.dst + (size_t)m * p.N + n0;
                        if (n0 + 0 < p.N) o[0] = sum.x;
                        if (n0 + 1 < p.N) o[1] = sum.y;
                        if (n0 + 2 < p.N) o[2] = sum.z;
                        if (n0 + 3 < p.N) o[3] = sum.w;
                    }
                }
                if (lane == 0) atomicExch(p.cnt + g, 0u);
            }
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int tid = threadIdx.x;   // 0 .. CONSUMERS-1
    const int n = lane & 15, jh = lane >> 4;   // this lane's row of the tile and first block (jh, jh + 2)
    uint8_t *act = smem + L.act;
    const float2 *act_sc = reinterpret_cast<const float2 *>(act + im.scales);
    float *red = reinterpret_cast<float *>(smem + L.red);
    const int sc_stride = im.sc_stride;

    pdl_wait();                                      // src1, or INIT's wdata, is complete
    // One activation row and one K slice (whole row groups, every segment starts at tile 0):
    // the tile at position warp + CW * tw of a chunk has index t = warp (mod CW), so each
    // consumer warp reads only the Q8_0 blocks of its own tiles.  It quantizes them itself,
    // all its loads issued at once, and no barrier of the CTA is needed.  For the chunk
    // starting at tile u, lane (tw, jb, q) takes the eight values 8q .. 8q+7 of block jb of
    // the tile u + warp + CW * tw.
    constexpr bool LAZY = !F16W && MT == 1;
    const bool lazy = LAZY && p.S == 1 && p.fused;
    const int lz_tw = lane >> 4, lz_jb = (lane >> 2) & 3, lz_q = lane & 3;
    auto lz_load = [&](const int u, float4 (&v)[2]) {
        const int t = u + warp + CW * lz_tw, blk = 4 * t + lz_jb;
        const bool live = t < p.NT && blk < p.nb;
        const float *src = p.x + (size_t)blk * QK + 8 * lz_q;
        v[0] = live ? ldg_f4(src) : make_float4(0.f, 0.f, 0.f, 0.f);
        v[1] = live ? ldg_f4(src + 4) : make_float4(0.f, 0.f, 0.f, 0.f);
    };
    auto lz_quant = [&](const int u, const float4 (&v)[2]) {
        const int t = u + warp + CW * lz_tw, blk = 4 * t + lz_jb;
        float am = fmaxf(absmax4(v[0]), absmax4(v[1]));
        am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 1));
        am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 2));
        const float d = am / 127.0f;
        uint32_t w[2];
        pack_q8_words<2>(v, q8_scale(d), w);
        int qs = sum_q8x4(w[0]) + sum_q8x4(w[1]);
        qs += __shfl_xor_sync(0xffffffffu, qs, 1);
        qs += __shfl_xor_sync(0xffffffffu, qs, 2);
        if (t < p.NT) {
            *reinterpret_cast<uint2 *>(act + im.codes + (size_t)blk * 32 + 8 * lz_q) = make_uint2(w[0], w[1]);
            if (lz_q == 0)
                reinterpret_cast<float2 *>(act + im.scales)[blk] =
                    make_float2(__half2float(__float2half_rn(d)), __int_as_float(-8 * qs));
        }
    };
    if (lazy) {
        constexpr int LZ_BATCH = 2;                      // chunks whose values are loaded at once
        const int nchunk = (p.NT + CHUNK_TILES - 1) / CHUNK_TILES;
#pragma unroll 1
        for (int c0 = 0; c0 < nchunk; c0 += LZ_BATCH) {
            float4 v[LZ_BATCH][2];
#pragma unroll
            for (int c = 0; c < LZ_BATCH; c++) lz_load((c0 + c) * CHUNK_TILES, v[c]);   // past NT: zeros
#pragma unroll
            for (int c = 0; c < LZ_BATCH; c++)
                if (c0 + c < nchunk) lz_quant((c0 + c) * CHUNK_TILES, v[c]);        // warp-uniform
        }
        __syncwarp();
    } else if constexpr (F16W) {
        // INIT in the CTA: this slice's columns of the M activation rows in fp16 (round to
        // nearest even), eight float4 loads in flight per thread
        const int per_row = nts * (F16_TILE_COLS / 4);   // float4 of one row's slice
        const int nf = p.M * per_row;
#pragma unroll 1
        for (int f0 = 0; f0 < nf; f0 += 8 * CONSUMERS) {
            float4 v[8];
#pragma unroll
            for (int i = 0; i < 8; i++) {
                const int f = f0 + tid + CONSUMERS * i, m = f / per_row, c4 = f % per_row;
                v[i] = f < nf ? ldg_f4(p.x + (size_t)m * p.K + (size_t)ts0 * F16_TILE_COLS + 4 * c4)
                              : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int i = 0; i < 8; i++) {
                const int f = f0 + tid + CONSUMERS * i, m = f / per_row, c4 = f % per_row;
                if (f < nf) {
                    const __half2 lo = __floats2half2_rn(v[i].x, v[i].y), hi = __floats2half2_rn(v[i].z, v[i].w);
                    *reinterpret_cast<uint2 *>(act + (size_t)m * im.row_bytes + 8 * c4) =
                        make_uint2(*reinterpret_cast<const uint32_t *>(&lo), *reinterpret_cast<const uint32_t *>(&hi));
                }
            }
        }
    } else if (p.fused) {
        // INIT in the CTA: Q8_0 of this slice's columns of the M activation rows.
        // Every load of a round is issued first (one round trip).  A thread holds half a
        // block (16 values, four float4) and the neighbouring lane the other
        // half, so a block needs one exchange for its maximum and one for its
        // code sum.
        constexpr int HALVES = FUSED_LOADS / 4;          // half blocks per thread
        const int per_row = nts * 8;                     // half blocks of one row's slice
        const int nh = p.M * per_row;
#pragma unroll 1
        for (int h0 = 0; h0 < nh; h0 += HALVES * CONSUMERS) {   // at most FUSED_ROUNDS rounds
        float4 v[HALVES][4];
#pragma unroll
        for (int i = 0; i < HALVES; i++) {
            const int h = h0 + tid + CONSUMERS * i, m = h / per_row, col = ts0 * TILE_COLS + (h % per_row) * 16;
            const bool live = h < nh && col < p.K;       // K is a multiple of 32: halves are whole
            const float *src = p.x + (size_t)m * p.K + col;
#pragma unroll
            for (int k = 0; k < 4; k++) v[i][k] = live ? ldg_f4(src + 4 * k) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int i = 0; i < HALVES; i++) {
            const int h = h0 + tid + CONSUMERS * i;
            if (h0 + CONSUMERS * i >= nh) break;         // no half of this step is live (CTA-uniform)
            float am = fmaxf(fmaxf(absmax4(v[i][0]), absmax4(v[i][1])), fmaxf(absmax4(v[i][2]), absmax4(v[i][3])));
            am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 1));
            const float d = am / 127.0f;
            const Q8Scale q = q8_scale(d);
            uint32_t w[4];
            pack_q8x16(v[i], q, w);
            int qs = sum_q8x4(w[0]) + sum_q8x4(w[1]) + sum_q8x4(w[2]) + sum_q8x4(w[3]);
            qs += __shfl_xor_sync(0xffffffffu, qs, 1);
            if (h < nh) {
                const int m = h / per_row, hb = h % per_row, bl = hb >> 1;
                *reinterpret_cast<uint4 *>(act + im.codes + (size_t)m * im.row_bytes + (size_t)hb * 16) =
                    make_uint4(w[0], w[1], w[2], w[3]);
                if ((hb & 1) == 0)
                    reinterpret_cast<float2 *>(act + im.scales)[m * im.sc_stride + bl] =
                        make_float2(__half2float(__float2half_rn(d)), __int_as_float(-8 * qs));
            }
        }
        }
    } else {   // plain coalesced loads of the slice's wdata image (the bulk-copy queue carries the weights),
               // eight per thread in flight at a time
        const uint4 *src = reinterpret_cast<const uint4 *>(p.wdata + (size_t)s * im.bytes);
        uint4 *dsts = reinterpret_cast<uint4 *>(act);
        const int n16 = (int)(im.bytes / 16);
#pragma unroll 1
        for (int i0 = 0; i0 < n16; i0 += 8 * CONSUMERS) {
            uint4 v[8];
#pragma unroll
            for (int b = 0; b < 8; b++) {
                const int i = i0 + b * CONSUMERS + tid;
                if (i < n16) v[b] = __ldcg(src + i);
            }
#pragma unroll
            for (int b = 0; b < 8; b++) {
                const int i = i0 + b * CONSUMERS + tid;
                if (i < n16) dsts[i] = v[b];
            }
        }
    }
    if (!lazy) consumers_sync<CONSUMERS>();
    bool failed = false;

    // dp4a path (up to four rows): one accumulator per tile position this warp owns and row.
    // MMA path (eight rows and more): per position, block parity (even / odd blocks, the
    // two halves the dp4a path keeps in lanes jh = 0, 1), activation-row tile and fragment
    // element; the same sums in the same order.
    constexpr bool MMA = F16W || MT >= 8;
    constexpr int NTL = MMA ? MT / 8 : 1;
    float acc[TPW][MMA ? 1 : MT];
    float hacc[MMA ? TPW : 1][2][NTL][4];
#pragma unroll
    for (int tw = 0; tw < TPW; tw++)
#pragma unroll
        for (int m = 0; m < (MMA ? 1 : MT); m++) acc[tw][m] = 0.0f;
#pragma unroll
    for (int tw = 0; tw < (MMA ? TPW : 1); tw++)
#pragma unroll
        for (int e = 0; e < 2; e++)
#pragma unroll
            for (int nt = 0; nt < NTL; nt++)
#pragma unroll
                for (int i = 0; i < 4; i++) hacc[tw][e][nt][i] = 0.0f;
    const int fg = lane >> 2, ft = lane & 3;           // m16n8k16 fragment coordinates

    int slot = 0;
    uint32_t phase = 0;
    constexpr int NRB = red_buffers(MT), BATCH = NRB / 2;   // row groups added after one barrier
    int pend = 0, gprev = 0;   // row groups written but not yet added (0 .. BATCH - 1); the last one's g
    for (int j = 0; j < seg.n; j++) {
        int g, u0, u1;
        seg.get(j, g, u0, u1);
        for (int u = u0; u < u1; u += CHUNK_TILES) {
            // a lane whose wait gave up skips the chunks from here on; nothing below needs the whole warp
            if (!failed) failed = !mbar_wait(smem_addr(full + slot), phase, p.status);
            // the tile at position ti of the chunk, into the accumulators of position tw
            auto tile_dot = [&](const int tw, const int ti) {
                const int tl = u + ti;
                GQ_DCHECK(tl < p.NT && ti < CHUNK_TILES, p.status);                         // tile index within the slice
                const uint8_t *tile = ring + (size_t)slot * CB + ti * TB;
                const uint2 d4w = *reinterpret_cast<const uint2 *>(tile + SCALES + n * 8);
                const uint2 m4w = Q41W ? *reinterpret_cast<const uint2 *>(tile + Q41_TILE_MIN_OFFSET + n * 8) : d4w;
#pragma unroll
                for (int jj = 0; jj < 2; jj++) {
                    const int jb = jh + 2 * jj;                // block of the tile
                    // Q4_0: the 16 code bytes of row n, block jb; Q8_0: its 32 codes
                    const uint4 q = lds128(tile + (jb * 16 + n) * (Q8W ? 32 : 16));
                    const uint4 q_hi = Q8W ? lds128(tile + (jb * 16 + n) * 32 + 16) : q;
                    const uint32_t dw = jb & 2 ? d4w.y : d4w.x;
                    const float d4 = (jb & 1) ? half_hi(dw) : half_lo(dw);
                    const uint32_t mw = jb & 2 ? m4w.y : m4w.x;
                    const float m4 = (jb & 1) ? half_hi(mw) : half_lo(mw);   // Q4_1: the block minimum
                    const int blk = 4 * tl + jb;
                    const uint8_t *a = act + im.codes + (size_t)blk * 32;
#pragma unroll
                    for (int m = 0; m < MT; m++) {
                        // up to four rows, rows past M repeat row M-1 (no branch; their sums are
                        // never stored); with more rows the rows past M are skipped
                        if (MT > 4 && m >= p.M) continue;
                        const int mm = MT > 4 ? m : min(m, p.M - 1);
                        const uint4 a0 = lds128(a + mm * im.row_bytes);
                        const uint4 a1 = lds128(a + mm * im.row_bytes + 16);
                        const float2 sc = act_sc[mm * sc_stride + blk];
                        const int sumi =
                            Q8W   ? block_dot_s8(q, q_hi, a0, a1)
                            : Q5W ? block_dot_q5(q, *reinterpret_cast<const uint32_t *>(tile + Q5_TILE_HIGH_OFFSET +
                                                                                     (jb * 16 + n) * 4),
                                                 a0, a1, 2 * __float_as_int(sc.y))   // -16 sum of the codes
                            : Q41W ? block_dot(q, a0, a1, 0)                  // sum_j q_j q8_j
                                   : block_dot(q, a0, a1, __float_as_int(sc.y));
                        acc[tw][MMA ? 0 : m] = fmaf(d4 * sc.x, (float)sumi, acc[tw][MMA ? 0 : m]);
                        if constexpr (Q41W)   // + m d8 sum_j q8_j (the image holds -8 sum_j q8_j)
                            acc[tw][MMA ? 0 : m] =
                                fmaf(m4 * sc.x, (float)(-(__float_as_int(sc.y) >> 3)), acc[tw][MMA ? 0 : m]);
                    }
                }
            };
            // The same tile with tensor-core MMAs (m16n8k16, fp16 in, f32 out).  Weight rows are
            // the MMA rows, activation rows its columns.  Thread (fg, ft) takes code word ft of
            // rows fg and fg + 8: its low nibbles are elements 4ft .. 4ft+3 of the block, the
            // k slots 2ft, 2ft+1, 2ft+8, 2ft+9 of the first MMA; the high nibbles (elements
            // 16 + 4ft ..) fill the same slots of the second.  The activation fragments take the
            // matching elements, so the two MMAs add all 32 products.  (q - 8) and the Q8_0
            // codes are exact in fp16 and every partial sum is an integer below 2^24, so the
            // f32 result is the exact block dot sumi.
            auto tile_mma = [&](const int tw, const int ti) {
                const int tl = u + ti;
                GQ_DCHECK(tl < p.NT && ti < CHUNK_TILES, p.status);
                const uint8_t *tile = ring + (size_t)slot * CB + ti * TB;
                const uint2 s0 = *reinterpret_cast<const uint2 *>(tile + SCALES + fg * 8);
                const uint2 s1 = *reinterpret_cast<const uint2 *>(tile + SCALES + (fg + 8) * 8);
                const uint2 mn0 = Q41W ? *reinterpret_cast<const uint2 *>(tile + Q41_TILE_MIN_OFFSET + fg * 8) : s0;
                const uint2 mn1 = Q41W ? *reinterpret_cast<const uint2 *>(tile + Q41_TILE_MIN_OFFSET + (fg + 8) * 8) : s1;
#pragma unroll
                for (int jb = 0; jb < 4; jb++) {
                    uint32_t alo[4], ahi[4];
                    if constexpr (Q8W) {   // elements 4ft .. 4ft+3 (word ft) and 16 + 4ft .. (word ft + 4)
                        const uint8_t *r0 = tile + (jb * 16 + fg) * 32 + 4 * ft, *r1 = r0 + 8 * 32;
                        q8_to_f16x2(*reinterpret_cast<const uint32_t *>(r0), alo[0], alo[2]);
                        q8_to_f16x2(*reinterpret_cast<const uint32_t *>(r1), alo[1], alo[3]);
                        q8_to_f16x2(*reinterpret_cast<const uint32_t *>(r0 + 16), ahi[0], ahi[2]);
                        q8_to_f16x2(*reinterpret_cast<const uint32_t *>(r1 + 16), ahi[1], ahi[3]);
                    } else if constexpr (Q41W) {   // the codes q themselves (the minimum term is added below)
                        const uint32_t w0 = *reinterpret_cast<const uint32_t *>(tile + (jb * 16 + fg) * 16 + 4 * ft);
                        const uint32_t w1 = *reinterpret_cast<const uint32_t *>(tile + (jb * 16 + fg + 8) * 16 + 4 * ft);
                        q4u_to_f16x2(w0 & 0x0F0F0F0Fu, alo[0], alo[2]);
                        q4u_to_f16x2(w1 & 0x0F0F0F0Fu, alo[1], alo[3]);
                        q4u_to_f16x2((w0 >> 4) & 0x0F0F0F0Fu, ahi[0], ahi[2]);
                        q4u_to_f16x2((w1 >> 4) & 0x0F0F0F0Fu, ahi[1], ahi[3]);
                    } else if constexpr (Q5W) {   // word ft of rows fg, fg + 8 with their fifth bits
                        const uint32_t w0 = *reinterpret_cast<const uint32_t *>(tile + (jb * 16 + fg) * 16 + 4 * ft);
                        const uint32_t w1 = *reinterpret_cast<const uint32_t *>(tile + (jb * 16 + fg + 8) * 16 + 4 * ft);
                        const uint32_t h0 = *reinterpret_cast<const uint32_t *>(tile + Q5_TILE_HIGH_OFFSET + (jb * 16 + fg) * 4);
                        const uint32_t h1 = *reinterpret_cast<const uint32_t *>(tile + Q5_TILE_HIGH_OFFSET + (jb * 16 + fg + 8) * 4);
                        // the group shift depends on ft: lo bits of group ft at 8b + 7 - ft, hi at 8b + 3 - ft
                        const uint32_t l0 = (w0 & 0x0F0F0F0Fu) | (((h0 << ft) >> 3) & 0x10101010u);
                        const uint32_t l1 = (w1 & 0x0F0F0F0Fu) | (((h1 << ft) >> 3) & 0x10101010u);
                        const uint32_t u0 = ((w0 >> 4) & 0x0F0F0F0Fu) | ((h0 << (1 + ft)) & 0x10101010u);
                        const uint32_t u1 = ((w1 >> 4) & 0x0F0F0F0Fu) | ((h1 << (1 + ft)) & 0x10101010u);
                        q5_to_f16x2(l0, alo[0], alo[2]);
                        q5_to_f16x2(l1, alo[1], alo[3]);
                        q5_to_f16x2(u0, ahi[0], ahi[2]);
                        q5_to_f16x2(u1, ahi[1], ahi[3]);
                    } else {
                        const uint32_t w0 = *reinterpret_cast<const uint32_t *>(tile + (jb * 16 + fg) * 16 + 4 * ft);
                        const uint32_t w1 = *reinterpret_cast<const uint32_t *>(tile + (jb * 16 + fg + 8) * 16 + 4 * ft);
                        q4_to_f16x2(w0 & 0x0F0F0F0Fu, alo[0], alo[2]);
                        q4_to_f16x2(w1 & 0x0F0F0F0Fu, alo[1], alo[3]);
                        q4_to_f16x2((w0 >> 4) & 0x0F0F0F0Fu, ahi[0], ahi[2]);
                        q4_to_f16x2((w1 >> 4) & 0x0F0F0F0Fu, ahi[1], ahi[3]);
                    }
                    const uint32_t sw0 = jb & 2 ? s0.y : s0.x, sw1 = jb & 2 ? s1.y : s1.x;
                    const float d4r0 = (jb & 1) ? half_hi(sw0) : half_lo(sw0);   // row fg
                    const float d4r1 = (jb & 1) ? half_hi(sw1) : half_lo(sw1);   // row fg + 8
                    const uint32_t mw0 = jb & 2 ? mn0.y : mn0.x, mw1 = jb & 2 ? mn1.y : mn1.x;
                    const float m4r0 = (jb & 1) ? half_hi(mw0) : half_lo(mw0);   // Q4_1 minimums
                    const float m4r1 = (jb & 1) ? half_hi(mw1) : half_lo(mw1);
                    const int blk = 4 * tl + jb;
#pragma unroll
                    for (int nt = 0; nt < NTL; nt++) {
                        // rows past M repeat row M-1: no branch, and their sums are never stored
                        const int mb = min(8 * nt + fg, p.M - 1);
                        const uint8_t *ab = act + im.codes + (size_t)mb * im.row_bytes + (size_t)blk * 32 + 4 * ft;
                        uint32_t blo[2], bhi[2];
                        q8_to_f16x2(*reinterpret_cast<const uint32_t *>(ab), blo[0], blo[1]);
                        q8_to_f16x2(*reinterpret_cast<const uint32_t *>(ab + 16), bhi[0], bhi[1]);
                        float d[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                        mma_f16_16x8x16(d, alo[0], alo[1], alo[2], alo[3], blo[0], blo[1]);
                        mma_f16_16x8x16(d, ahi[0], ahi[1], ahi[2], ahi[3], bhi[0], bhi[1]);
                        const int mc0 = min(8 * nt + 2 * ft, p.M - 1), mc1 = min(8 * nt + 2 * ft + 1, p.M - 1);
                        const float d8c0 = act_sc[mc0 * sc_stride + blk].x, d8c1 = act_sc[mc1 * sc_stride + blk].x;
                        float *h = hacc[MMA ? tw : 0][jb & 1][nt];
                        h[0] = fmaf(d4r0 * d8c0, d[0], h[0]);   // row fg,     activation row 2ft
                        h[1] = fmaf(d4r0 * d8c1, d[1], h[1]);   // row fg,     activation row 2ft + 1
                        h[2] = fmaf(d4r1 * d8c0, d[2], h[2]);   // row fg + 8, activation row 2ft
                        h[3] = fmaf(d4r1 * d8c1, d[3], h[3]);   // row fg + 8, activation row 2ft + 1
                        if constexpr (Q41W) {   // + m d8 sum_j q8_j, as in the dp4a path
                            const float sx0 = (float)(-(__float_as_int(act_sc[mc0 * sc_stride + blk].y) >> 3));
                            const float sx1 = (float)(-(__float_as_int(act_sc[mc1 * sc_stride + blk].y) >> 3));
                            h[0] = fmaf(m4r0 * d8c0, sx0, h[0]);
                            h[1] = fmaf(m4r0 * d8c1, sx1, h[1]);
                            h[2] = fmaf(m4r1 * d8c0, sx0, h[2]);
                            h[3] = fmaf(m4r1 * d8c1, sx1, h[3]);
                        }
                    }
                }
            };
            // F16 weights: the tile is 16 rows x 32 columns as stored, 64 bytes per row.  Thread
            // (fg, ft) takes elements 8ft .. 8ft+7 of rows fg and fg + 8 and of its activation
            // row: the first four fill k slots 2ft, 2ft+1, 2ft+8, 2ft+9 of one MMA, the last four
            // those of a second, so the two MMAs add the 32 products of the tile.
            auto tile_f16 = [&](const int tw, const int ti) {
                const int tl = u + ti;
                GQ_DCHECK(tl < p.NT && ti < CHUNK_TILES, p.status);
                const uint8_t *tile = ring + (size_t)slot * CB + ti * TB;
                const uint4 wa = lds128(tile + fg * 64 + 16 * ft);
                const uint4 wb = lds128(tile + (fg + 8) * 64 + 16 * ft);
#pragma unroll
                for (int nt = 0; nt < NTL; nt++) {
                    const int mb = min(8 * nt + fg, p.M - 1);   // rows past M repeat row M-1
                    const uint4 xb = lds128(act + (size_t)mb * im.row_bytes + (size_t)tl * 64 + 16 * ft);
                    float *h = hacc[MMA ? tw : 0][0][nt];
                    mma_f16_16x8x16(*reinterpret_cast<float(*)[4]>(h), wa.x, wb.x, wa.y, wb.y, xb.x, xb.y);
                    mma_f16_16x8x16(*reinterpret_cast<float(*)[4]>(h), wa.z, wb.z, wa.w, wb.w, xb.z, xb.w);
                }
            };
            auto tile = [&](const int tw, const int ti) {
                if constexpr (F16W) tile_f16(tw, ti);
                else if constexpr (MMA) tile_mma(tw, ti);
                else tile_dot(tw, ti);
            };
            if (!failed) {
                if (u1 - u >= CHUNK_TILES) {                   // a full chunk: no per-tile test
#pragma unroll
                    for (int tw = 0; tw < TPW; tw++) tile(tw, warp + CW * tw);
                } else {
#pragma unroll
                    for (int tw = 0; tw < TPW; tw++)
                        if (warp + CW * tw < u1 - u) tile(tw, warp + CW * tw);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_addr(empty + slot));   // this warp is done with the chunk
            if (++slot == p.slots) {
                slot = 0;
                phase ^= 1u;
            }
        }

        // ---- row group g of this slice is complete: add the partials of the 16 tile positions.
        // Row group j's partials go to buffer j % NRB.  After a barrier the consumer threads add
        // those of the row groups written since the last one (at most BATCH; a row group shared
        // with another CTA is added at once, for the fix-up).  Before a buffer is written again,
        // every row group that used it has been added: the threads that add a batch do so before
        // they reach the next barrier, which the writers of the batch after next have passed.
        float *redb = red + (j % NRB) * CHUNK_TILES * outs;
        if constexpr (MMA) {
#pragma unroll
            for (int tw = 0; tw < TPW; tw++)
#pragma unroll
                for (int nt = 0; nt < NTL; nt++)
#pragma unroll
                    for (int i = 0; i < 4; i++) {
                        const int row = fg + 8 * (i >> 1), m = 8 * nt + 2 * ft + (i & 1);
                        redb[(warp + CW * tw) * outs + m * 16 + row] = hacc[tw][0][nt][i] + hacc[tw][1][nt][i];
                        hacc[tw][0][nt][i] = 0.0f;
                        hacc[tw][1][nt][i] = 0.0f;
                    }
        } else {
#pragma unroll
            for (int tw = 0; tw < TPW; tw++)
#pragma unroll
                for (int m = 0; m < MT; m++) {
                    const float other = __shfl_down_sync(0xffffffffu, acc[tw][m], 16);   // blocks jh+1 of the row
                    if (lane < 16) redb[(warp + CW * tw) * outs + m * 16 + n] = acc[tw][m] + other;
                    acc[tw][m] = 0.0f;
                }
        }
        const bool shared_rg = j < seg.nshared;
        if constexpr (BATCH == 1) {   // one row group per barrier
            consumers_sync<CONSUMERS>();
            if (tid < outs) {
                float v = 0.0f;
#pragma unroll
                for (int pos = 0; pos < CHUNK_TILES; pos++) v += redb[pos * outs + tid];
                if (shared_rg) {                       // this CTA's part of a shared row group
                    const int slot_i = ci == owner(T, p.Gs, g * nts) ? 0 : 1;
                    p.part[(((size_t)g * p.S + s) * 2 + slot_i) * PART_STRIDE + tid] = v;
                } else {
                    const int m = tid / 16, row = 16 * g + tid % 16;
                    if (m < p.M && row < p.N) {   // a later slice's launch adds to the earlier ones' sum
                        float *dp = p.dst + (size_t)m * p.N + row;
                        *dp = seq_slice > 0 ? *dp + v : v;
                    }
                }
            }
            if (shared_rg) {                           // the partial is written: the fix-up may read it
                consumers_sync<CONSUMERS>();
                if (tid == 0) mbar_arrive(smem_addr(fixbar + j));
            }
            continue;
        }
        if (!shared_rg && pend + 1 < BATCH && j + 1 < seg.n && j + 1 >= seg.nshared) {
            pend++;                                    // added with the next row group
            gprev = g;
            continue;
        }
        consumers_sync<CONSUMERS>();
        const int nb = pend + 1;                       // row groups j - pend .. j
        for (int t = tid; t < nb * outs; t += CONSUMERS) {
            const int k = t / outs, o = t % outs, jj = j - pend + k;
            const int gg = k == pend ? g : gprev;      // BATCH <= 2: an earlier row group is the previous one
            const float *rbuf = red + (jj % NRB) * CHUNK_TILES * outs;
            float v = 0.0f;
#pragma unroll
            for (int pos = 0; pos < CHUNK_TILES; pos++) v += rbuf[pos * outs + o];
            if (shared_rg) {                           // this CTA's part of a shared row group
                const int slot_i = ci == owner(T, p.Gs, gg * nts) ? 0 : 1;
                p.part[(((size_t)gg * p.S + s) * 2 + slot_i) * PART_STRIDE + o] = v;
            } else {
                const int m = o / 16, row = 16 * gg + o % 16;
                if (m < p.M && row < p.N) {   // a later slice's launch adds to the earlier ones' sum
                    float *dp = p.dst + (size_t)m * p.N + row;
                    *dp = seq_slice > 0 ? *dp + v : v;
                }
            }
        }
        pend = 0;
        if (shared_rg) {                               // the partial is written: the fix-up may read it
            consumers_sync<CONSUMERS>();
            if (tid == 0) mbar_arrive(smem_addr(fixbar + j));
        }
    }
}

// K slices for M activation rows: the fewest (a power of two) whose images fit the budget.
int slices_for(int NT, int M, bool f16) {
    int S = 1;
    while (S < 8 && 2 * S <= NT && Image(M, (NT + S - 1) / S, f16).bytes > ACT_BUDGET) S *= 2;
    return S;
}

int env_int(const char *name, int dflt) {
    const char *v = getenv(name);
    return v && *v ? atoi(v) : dflt;
}

// The dynamic shared-memory limit is raised once per (device, kernel).
constexpr int MAX_DEV = 64;
constexpr int MAX_VARIANTS = 32;
std::atomic<bool> g_smem_set[MAX_DEV][MAX_VARIANTS];

template <typename Kernel>
gq_status allow_smem(Kernel kernel, int which) {
    int dev = 0;
    gq_status st = check_cuda(cudaGetDevice(&dev), "cudaGetDevice");
    if (st != GQ_OK) return st;
    if (dev >= 0 && dev < MAX_DEV && g_smem_set[dev][which].load(std::memory_order_acquire)) return GQ_OK;
    st = check_cuda(cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)(SMEM_LIMIT - 1024)),
                    "gemv_q4_0 shared-memory attribute");
    if (st == GQ_OK)   // all of the unified L1 as shared memory: two CTAs of the 8-warp shape fit
        st = check_cuda(cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                             (int)cudaSharedmemCarveoutMaxShared),
                        "gemv_q4_0 carveout attribute");
    if (st == GQ_OK && dev >= 0 && dev < MAX_DEV) g_smem_set[dev][which].store(true, std::memory_order_release);
    return st;
}

struct Plan {
    int S, ntmax, Gs, maxfix;
};

Plan plan(int N16, int NT, int M, bool f16 = false) {
    Plan q;
    q.S = slices_for(NT, M, f16);
    q.ntmax = (NT + q.S - 1) / q.S;
    q.Gs = std::max(1, std::min(sm_count() / q.S, N16));   // S == 1: every CTA gets >= 1 row group
    // row groups a CTA touches: at most ceil(N16 / Gs) + 2 (one mbarrier each)
    q.maxfix = q.S > 1 ? (N16 + q.Gs - 1) / q.Gs + 2 : 2;
    return q;
}

// Instantiated kernels: activation rows per tile (MT), consumer warps (CW), the
// register cap and the fix-up warps.  The one-row 8-warp shape without fix-up
// warps (one K slice: no row group is shared) runs two CTAs per SM, each with half
// of the shared memory, so that the CTAs of the next product in the stream are
// resident and stream their weights while this product finishes; with several K
// slices in its one launch it keeps one fix-up warp and runs one CTA per SM.
// Several rows take one launch per K slice and never share a row group.  The
// 16-warp shape (20 warps) runs one CTA per SM at 96 registers, the 8-warp shape
// of several rows of a block format one at 128.
struct Variant {
    int mt, cw, regs;
    int wf;
    int fixw;
    int consumers, threads, fused_loads;
    const void *kernel;   // gemv_q4_0_kernel<...>(Params, Wmap<wf == WF_F16RM>)
};

template <int MT, int CW, int REGS, int WF, int FIXW>
Variant variant() {
    using SH = Shape<CW, FIXW>;
    return {MT, CW, REGS, WF, FIXW, SH::CONSUMERS, SH::THREADS, SH::FUSED_LOADS,
            reinterpret_cast<const void *>(gemv_q4_0_kernel<MT, CW, REGS, WF, FIXW>)};
}

const Variant VARIANTS[] = {
    variant<1, 8, 88, WF_Q4, 0>(),    variant<1, 8, 88, WF_Q4, 1>(),    variant<2, 8, 128, WF_Q4, 0>(),
    variant<4, 8, 128, WF_Q4, 0>(),   variant<8, 8, 128, WF_Q4, 0>(),   variant<16, 8, 128, WF_Q4, 0>(),
    variant<8, 8, 88, WF_F16, 0>(),   variant<16, 16, 96, WF_F16, 2>(),
    variant<8, 8, 88, WF_F16RM, 0>(), variant<16, 16, 96, WF_F16RM, 2>(),
    variant<1, 8, 88, WF_Q8, 0>(),    variant<1, 8, 88, WF_Q8, 1>(),    variant<2, 8, 128, WF_Q8, 0>(),
    variant<4, 8, 128, WF_Q8, 0>(),   variant<8, 8, 128, WF_Q8, 0>(),   variant<16, 8, 128, WF_Q8, 0>(),
    variant<1, 8, 88, WF_Q5, 0>(),    variant<1, 8, 88, WF_Q5, 1>(),    variant<2, 8, 128, WF_Q5, 0>(),
    variant<4, 8, 128, WF_Q5, 0>(),   variant<8, 8, 128, WF_Q5, 0>(),   variant<16, 8, 128, WF_Q5, 0>(),
    variant<1, 8, 88, WF_Q41, 0>(),   variant<1, 8, 88, WF_Q41, 1>(),   variant<2, 8, 128, WF_Q41, 0>(),
    variant<4, 8, 128, WF_Q41, 0>(),  variant<8, 8, 128, WF_Q41, 0>(),  variant<16, 8, 128, WF_Q41, 0>()};
constexpr int N_VARIANTS = sizeof(VARIANTS) / sizeof(VARIANTS[0]);
static_assert(N_VARIANTS <= MAX_VARIANTS, "one shared-memory flag per variant");

// Consumer warps and register cap.  Block formats: 8 warps, at 88 registers for one activation
// row (two CTAs per SM) and at 128 for several (each warp taking two tiles of a chunk).  Against
// 16 warps at 96 registers, several Q4_0 rows measured 2-16 % faster at M = 2 (where the 8-warp
// shape also takes the separate INIT at K = 11008), 4-11 % at M = 4, 13-16 % at M = 8 and 2-5 %
// at M = 16 on the 7B decode shapes; Q5_0 and Q4_1 at [11008, 4096] 2-17 %; Q8_0 3-5 % from M = 4
// (2.5 % slower at M = 2).  F16 tiles: 8 warps at 88 registers for up to 8 rows, 16 at 96 above.
int consumer_warps_for(int M, int wf) { return is_f16(wf) ? (M <= 8 ? 8 : 16) : 8; }

int regs_for(int cw, int M, int wf) { return cw == 16 ? 96 : M > 1 && !is_f16(wf) ? 128 : 88; }

const Variant *variant_for(int mt, int cw, int regs, int wf, int fixw) {
    for (int i = 0; i < N_VARIANTS; i++)
        if (VARIANTS[i].mt == mt && VARIANTS[i].cw == cw && VARIANTS[i].regs == regs && VARIANTS[i].wf == wf &&
            VARIANTS[i].fixw == fixw)
            return &VARIANTS[i];
    return nullptr;
}

}  // namespace

void gemv_workspace(int wf, int64_t N, int64_t K, size_t *counter_bytes, size_t *data_bytes) {
    const bool f16 = is_f16(wf);
    const int N16 = (int)((N + 15) / 16);
    const int NT = f16 ? (int)(K / F16_TILE_COLS) : (int)((K + TILE_COLS - 1) / TILE_COLS);
    size_t db = 0;
    for (int M = 1; M <= 16; M++) {
        const Plan q = plan(N16, NT, M, f16);
        const size_t parts = (size_t)N16 * q.S * 2 * PART_STRIDE * sizeof(float);
        const size_t images = f16 ? 0 : (size_t)q.S * Image(M, q.ntmax).bytes;   // F16: INIT is always in the CTA
        db = std::max(db, align_up(parts, 256) + images);
    }
    *counter_bytes = (size_t)N16 * sizeof(unsigned int);
    *data_bytes = db;
}

int gemv_q4_0_slices(int64_t N, int64_t K, int64_t M) {
    const int N16 = (int)((N + 15) / 16);
    const int NT = (int)((K + TILE_COLS - 1) / TILE_COLS);
    return plan(N16, NT, (int)std::min<int64_t>(16, std::max<int64_t>(1, M))).S;
}

void gemv_q4_0_workspace(int64_t N, int64_t K, size_t *counter_bytes, size_t *data_bytes) {
    gemv_workspace(WF_Q4, N, K, counter_bytes, data_bytes);
}

void gemv_f16r_workspace(int64_t N, int64_t K, size_t *counter_bytes, size_t *data_bytes) {
    gemv_workspace(WF_F16, N, K, counter_bytes, data_bytes);
}

namespace {

gq_status launch_gemv_with(int wf, const void *rep, const float *x, float *dst, int64_t M, int64_t N, int64_t K,
                           const Workspace &ws, cudaStream_t s) {
    const bool f16 = is_f16(wf);
    Params p{};
    p.w = (const uint8_t *)rep;
    p.status = device_status_word();
    if (!p.status) return fail(GQ_ERR_CUDA, "device status word unavailable");
    p.N = (int)N;
    p.K = (int)K;
    p.nb = (int)(K / QK);
    p.N16 = (int)((N + 15) / 16);
    p.NT = f16 ? (int)(K / F16_TILE_COLS) : (int)((K + TILE_COLS - 1) / TILE_COLS);

    gq_status st = GQ_OK;
    Wmap<true> wmap{};       // row-major F16 only
    Wmap<false> no_wmap{};
    if (wf == WF_F16RM) {
        st = f16_tile_map(&wmap.map, rep, N, K);
        if (st != GQ_OK) return st;
    }
    p.cnt = reinterpret_cast<unsigned int *>(ws.counters);

    for (int64_t m0 = 0; m0 < M; m0 += 16) {
        p.M = (int)std::min<int64_t>(16, M - m0);
        p.x = x + m0 * K;
        p.dst = dst + m0 * N;
        if (p.M == 1 && wf == WF_Q4 && gemv_m1_supported(N, K) && env_int("GQ_GEMV_M1", 1) != 0) {
            st = launch_gemv_m1_q4_0(rep, p.x, p.dst, N, K, s);   // one row: its own kernel, no workspace
            if (st != GQ_OK) return st;
            continue;
        }
        // F16: tensor-core tiles of 8 or 16 activation rows
        const int MT = f16 ? (p.M <= 8 ? 8 : 16) : p.M <= 1 ? 1 : p.M <= 2 ? 2 : p.M <= 4 ? 4 : p.M <= 8 ? 8 : 16;
        const Plan q = plan(p.N16, p.NT, p.M, f16);   // the images hold p.M rows
        p.S = q.S;
        p.ntmax = q.ntmax;
        p.Gs = q.Gs;
        p.maxfix = q.maxfix;
        // Several K slices with several activation rows: one launch per slice, each CTA (one per
        // SM, at most one per row group) owning whole row groups and the later slices adding into
        // dst, instead of one launch whose S groups of CTAs share row groups and add partials
        // across CTAs (measured about twice as slow).  One activation row keeps the single launch.
        const bool seq = q.S > 1 && (f16 || MT > 1);
        p.seq_slice = -1;
        if (seq) p.Gs = std::max(1, std::min(sm_count(), p.N16));
        const int cw = consumer_warps_for(f16 ? MT : p.M, wf);
        const int consumers = cw == 8 ? Shape<8>::CONSUMERS : Shape<16>::CONSUMERS;
        const int fused_loads = cw == 8 ? Shape<8>::FUSED_LOADS : Shape<16>::FUSED_LOADS;
        // fuse INIT when each consumer thread loads a few float4 (F16: always)
        // (one row and one K slice: each warp quantizes its own blocks as it goes, any K)
        p.fused = f16 || (MT == 1 && q.S == 1) ||
                          (int64_t)p.M * p.ntmax * 32 <= (int64_t)consumers * fused_loads * FUSED_ROUNDS
                      ? 1
                      : 0;
        // one K slice, or one launch per slice: no shared row group, no fix-up warp (the 16-warp
        // shape has its two either way)
        const int fixw = cw == 16 ? 2 : q.S == 1 || seq ? 0 : 1;
        const Variant *kvp = variant_for(MT, cw, regs_for(cw, p.M, wf), wf, fixw);
        if (!kvp) return fail(GQ_ERR_INVALID_ARG, "gemv: no kernel for M=%d", p.M);
        const Variant &kv = *kvp;
        // behind INIT (which waited for every earlier grid) the weights are final; otherwise only
        // a caller that declared its weights static lets the producers start before the wait
        p.early = (!p.fused || static_weights()) ? 1 : 0;
        // INIT itself triggers the GEMV before its own wait only for static weights; otherwise the
        // GEMV starts once INIT has waited for every earlier grid
        p.init_early = static_weights() ? 1 : 0;
        p.part = reinterpret_cast<float *>(ws.data);
        p.wdata = ws.data + align_up((size_t)p.N16 * p.S * 2 * PART_STRIDE * sizeof(float), 256);
        const size_t fixed = Layout(MT, p.M, p.ntmax, 0, p.maxfix, wf).total;
        auto slots_for = [&](size_t budget) {
            return (int)std::min<size_t>(MAX_SLOTS,
                                         (budget - std::min(budget, fixed + 256)) / (chunk_bytes(wf) + 16));
        };
        // the 8-warp Q4_0 / Q4_1 / Q5_0 shape keeps a ring of half the shared memory (MIN_SLOTS_HALF chunks at
        // least): two CTAs per SM without fix-up warps; with one, a half ring measured faster than
        // a full one.  F16 and Q8_0 tiles (more bytes per weight; 34 KB Q8_0 chunks would leave
        // two slots in half the shared memory) keep a full ring.
        // (The 128-register shape of several rows never fits twice in an SM's registers.)
        p.slots = kv.cw == 8 && kv.regs == 88 && (wf == WF_Q4 || wf == WF_Q5 || wf == WF_Q41)
                      ? slots_for(SMEM_HALF - 1024)
                      : 0;
        if (p.slots < MIN_SLOTS_HALF) p.slots = slots_for(SMEM_LIMIT - 1024);
        const int slots_env = env_int("GQ_GEMV_SLOTS", 0);   // tuning: ring slots, up to what fits
        if (slots_env > 0) p.slots = std::min(slots_env, slots_for(SMEM_LIMIT - 1024));
        p.slots &= ~(PRODUCERS - 1);
        if (p.slots < 2)
            return fail(GQ_ERR_INVALID_ARG, "gemv: N=%lld K=%lld leaves no room for the weight ring",
                        (long long)N, (long long)K);
        const int pf_kb = env_int("GQ_GEMV_PF_KB", PF_KB);   // tuning; negative: no L2 prefetch
        p.pf = pf_kb < 0 ? 0 : p.slots + pf_kb * 1024 / chunk_bytes(wf);
        const size_t smem = Layout(MT, p.M, p.ntmax, p.slots, p.maxfix, wf).total;
        st = allow_smem(kv.kernel, (int)(&kv - VARIANTS));
        if (st != GQ_OK) return st;
        const int threads = kv.threads;

        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cudaLaunchConfig_t cfg = {};
        cfg.stream = s;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        const int64_t warps = (int64_t)p.M * 4 * p.NT;
        cfg.gridDim = dim3((unsigned)std::max<int64_t>(1, std::min<int64_t>((warps + 7) / 8, 2LL * sm_count())), 1, 1);
        cfg.blockDim = dim3(256, 1, 1);
        cfg.dynamicSmemBytes = 0;
        if (!p.fused) {
            st = check_cuda(cudaLaunchKernelEx(&cfg, wdata_kernel, p), "gemv_q4_0 INIT launch");
            if (st != GQ_OK) return st;
        }
        cfg.gridDim = dim3((unsigned)(seq ? p.Gs : p.S * p.Gs), 1, 1);
        cfg.blockDim = dim3((unsigned)threads, 1, 1);
        cfg.dynamicSmemBytes = smem;
        for (int sl = 0; sl < (seq ? p.S : 1); sl++) {
            if (seq) p.seq_slice = sl;
            void *args[] = {(void *)&p, wf == WF_F16RM ? (void *)&wmap : (void *)&no_wmap};
            st = check_cuda(cudaLaunchKernelExC(&cfg, kv.kernel, args), "gemv launch");
            if (st != GQ_OK) return st;
        }
    }
    return GQ_OK;
}

}  // namespace

gq_status launch_gemv_q4_0_with(const void *rep, const float *x, float *dst, int64_t M, int64_t N, int64_t K,
                                const Workspace &ws, cudaStream_t s) {
    return launch_gemv_with(WF_Q4, rep, x, dst, M, N, K, ws, s);
}

gq_status launch_gemv_f16r(const void *rep, const float *x, float *dst, int64_t M, int64_t N, int64_t K,
                           cudaStream_t s) {
    size_t cb, db;
    gemv_f16r_workspace(N, K, &cb, &db);
    Workspace ws;
    gq_status st = get_workspace(s, cb, db, &ws);
    if (st != GQ_OK) return st;
    return launch_gemv_with(WF_F16, rep, x, dst, M, N, K, ws, s);
}

gq_status launch_gemv_f16_rowmajor(const void *w16, const float *x, float *dst, int64_t M, int64_t N, int64_t K,
                                   cudaStream_t s) {
    size_t cb, db;
    gemv_f16r_workspace(N, K, &cb, &db);
    Workspace ws;
    gq_status st = get_workspace(s, cb, db, &ws);
    if (st != GQ_OK) return st;
    return launch_gemv_with(WF_F16RM, w16, x, dst, M, N, K, ws, s);
}

gq_status launch_gemv_q4_0(const void *rep, const float *x, float *dst, int64_t M, int64_t N, int64_t K,
                           cudaStream_t s) {
    size_t cb, db;
    gemv_q4_0_workspace(N, K, &cb, &db);
    Workspace ws;
    gq_status st = get_workspace(s, cb, db, &ws);
    if (st != GQ_OK) return st;
    return launch_gemv_q4_0_with(rep, x, dst, M, N, K, ws, s);
}

gq_status launch_gemv_q8_0(const void *rep, const float *x, float *dst, int64_t M, int64_t N, int64_t K,
                           cudaStream_t s) {
    size_t cb, db;
    gemv_workspace(WF_Q8, N, K, &cb, &db);
    Workspace ws;
    gq_status st = get_workspace(s, cb, db, &ws);
    if (st != GQ_OK) return st;
    return launch_gemv_with(WF_Q8, rep, x, dst, M, N, K, ws, s);
}

gq_status launch_gemv_q5_0(const void *rep, const float *x, float *dst, int64_t M, int64_t N, int64_t K,
                           cudaStream_t s) {
    size_t cb, db;
    gemv_workspace(WF_Q5, N, K, &cb, &db);
    Workspace ws;
    gq_status st = get_workspace(s, cb, db, &ws);
    if (st != GQ_OK) return st;
    return launch_gemv_with(WF_Q5, rep, x, dst, M, N, K, ws, s);
}

gq_status launch_gemv_q4_1(const void *rep, const float *x, float *dst, int64_t M, int64_t N, int64_t K,
                           cudaStream_t s) {
    size_t cb, db;
    gemv_workspace(WF_Q41, N, K, &cb, &db);
    Workspace ws;
    gq_status st = get_workspace(s, cb, db, &ws);
    if (st != GQ_OK) return st;
    return launch_gemv_with(WF_Q41, rep, x, dst, M, N, K, ws, s);
}

}  // namespace gq
