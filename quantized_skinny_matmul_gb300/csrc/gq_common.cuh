// gq_common.cuh -- device helpers shared by the CUDA sources of libgq.
//
// Built for sm_103a only.  Compiled without fast-math so that the divisions
// x / d of the quantizers are IEEE round-to-nearest, matching the block
// formats' definition (no flush-to-zero either).
#pragma once

#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "gq.h"

namespace gq {

constexpr int QK = 32;                 // values per block
constexpr int Q4_0_BYTES = 18;
constexpr int Q8_0_BYTES = 34;
constexpr int TILE_ROWS = 16;          // rows of a repacked tile
constexpr int TILE_BLOCKS = 4;         // blocks (of 32 columns) of a repacked tile
constexpr int TILE_COLS = TILE_BLOCKS * QK;   // 128 columns
constexpr int TILE_BYTES = 1152;       // 16 rows x 4 blocks x 18 bytes
constexpr int TILE_SCALE_OFFSET = 1024;

// Kernels with bounded waits receive the address of the device's sticky
// status word (owned by gq_api.cu, read and cleared by gq_last_error).
constexpr unsigned int STATUS_TIMEOUT = 1u;
constexpr unsigned int STATUS_RANGE = 2u;     // a length or position read on the device was out of range
constexpr unsigned int STATUS_CHECK = 4u;     // a GQ_DEBUG bounds check failed

// GQ_DEBUG builds (see _build.py) check the indices the kernels derive from their arguments and
// record a failure in the device status word; they never trap.  Other builds compile the checks out.
#ifdef GQ_DEBUG
#define GQ_DCHECK(cond, status)                                      \
    do {                                                             \
        if (!(cond)) atomicOr((status), ::gq::STATUS_CHECK);         \
    } while (0)
#else
#define GQ_DCHECK(cond, status) \
    do {                        \
    } while (0)
#endif
__device__ __forceinline__ void flag_timeout(unsigned int *status) { atomicOr(status, STATUS_TIMEOUT); }

// ---------------------------------------------------------------------------
// Programmatic dependent launch: wait for the grids this launch depends on
// before touching global memory; let the next launch start its prologue.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------------------
// Loads that bypass L1 (each weight byte is used once per launch).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint4 ldg_stream(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ float4 ldg_f4(const float *p) {
    return __ldg(reinterpret_cast<const float4 *>(p));
}

// ---------------------------------------------------------------------------
// Q8_0 code of one activation given the block's f32 scale d (the quantizer's
// decision is taken in f32: IEEE division, then roundf, ties away from zero).
// ---------------------------------------------------------------------------
__device__ __forceinline__ int q8_code(float x, float d) {
    if (d == 0.0f) return 0;
    int v = (int)roundf(x / d);
    return v < -127 ? -127 : (v > 127 ? 127 : v);
}

// The same code without a division.  With r within one ulp of 1/d
// (rcp.approx.f32), y = x * r is within a relative 2^-22 of the quotient, and
// |x / d| <= 127 (1 + 2^-23) for a normal d (below 191 for a subnormal one,
// whose rounding is coarser), so the two differ by less than 3.5e-5: they
// round to the same integer unless y lies within 2^-14 (6.1e-5) of a
// half-integer.  Away from
// half-integers every round-to-nearest agrees with roundf, so the nearest
// integer of y (rintf) is the code.
//
// Near the half-integer h = k + 1/2 (k = floor|y|), roundf(x / d) is k + 1 in
// magnitude iff the IEEE quotient rounds to h or above, i.e. iff |x| / d lies
// above the midpoint m = h - u/2 between h and its predecessor (u = h minus
// that predecessor), or on it when h has an even significand.  The sign of
// |x| - m d decides: e = |x| - h d is exact in f32 (|x| and h d agree to 14
// bits and both are multiples of ulp(d)/2), and fmaf(u/2, d, e) rounds the
// exact |x| - m d once, which keeps its sign and its zero.
//
// Both codes are formed for every value and one is selected, without a
// branch.  Scales below 2^-60 are first multiplied, with x, by 2^64: the
// quotient is unchanged, r stays finite and u/2 * d cannot underflow.
struct Q8Scale {
    float d;   // the block scale, multiplied by s
    float r;   // approximately 1 / d (0 when d = 0)
    float s;   // 1, or 2^64 for a tiny scale
};

__device__ __forceinline__ Q8Scale q8_scale(float d) {
    Q8Scale q;
    q.s = d < 0x1p-60f ? 0x1p64f : 1.0f;
    q.d = d * q.s;
    float r;
    asm("rcp.approx.f32 %0, %1;" : "=f"(r) : "f"(q.d));
    q.r = d == 0.0f ? 0.0f : r;
    return q;
}

// y is within 2^-14 of a half-integer (the quotient is within 3.5e-5 of y)
__device__ __forceinline__ bool q8_near_half(float y, float n) { return !(fabsf(y - n) < 0.5f - 0x1p-14f); }

__device__ __forceinline__ int q8_code_s(float x, const Q8Scale &q) {
    const float xs = x * q.s;
    const float y = xs * q.r;
    const float n = rintf(y);
    const bool away = !q8_near_half(y, n);
    const float ax = fabsf(xs);
    const float k = floorf(fabsf(y));
    const float h = k + 0.5f;
    const float u = h - __int_as_float(__float_as_int(h) - 1);
    const float t = fmaf(0.5f * u, q.d, fmaf(-h, q.d, ax));
    const bool up = t > 0.0f || (t == 0.0f && (__float_as_int(h) & 1) == 0);
    int c = (int)k + (up ? 1 : 0);
    c = xs < 0.0f ? -c : c;
    c = away ? (int)n : c;
    return c < -127 ? -127 : (c > 127 ? 127 : c);   // |x / d| exceeds 127 only for a subnormal d
}

// Four Q8_0 codes packed into a little-endian word (code of x.x in the low byte).
__device__ __forceinline__ uint32_t pack_bytes(int c0, int c1, int c2, int c3) {
    const uint32_t lo = __byte_perm((uint32_t)c0, (uint32_t)c1, 0x0040);
    const uint32_t hi = __byte_perm((uint32_t)c2, (uint32_t)c3, 0x0040);
    return __byte_perm(lo, hi, 0x5410);
}

__device__ __forceinline__ uint32_t pack_q8x4(float4 x, const Q8Scale &q) {
    return pack_bytes(q8_code_s(x.x, q), q8_code_s(x.y, q), q8_code_s(x.z, q), q8_code_s(x.w, q));
}

// The codes of 4N values (N = 4: a half block) into N words.  The nearest
// integers are formed first; only if some lane of the warp has a value near a
// half-integer (a few percent of warps) does the warp form the full codes.
__device__ __forceinline__ int q8_nearest(float x, const Q8Scale &q, bool &near) {
    const float y = (x * q.s) * q.r;
    const float n = rintf(y);
    near = q8_near_half(y, n);
    const int c = (int)n;
    return c < -127 ? -127 : (c > 127 ? 127 : c);
}

template <int N>
__device__ __forceinline__ void pack_q8_words(const float4 (&x)[N], const Q8Scale &q, uint32_t (&w)[N]) {
    bool any = false;
#pragma unroll
    for (int k = 0; k < N; k++) {
        bool n0, n1, n2, n3;
        const int c0 = q8_nearest(x[k].x, q, n0), c1 = q8_nearest(x[k].y, q, n1);
        const int c2 = q8_nearest(x[k].z, q, n2), c3 = q8_nearest(x[k].w, q, n3);
        w[k] = pack_bytes(c0, c1, c2, c3);
        any |= n0 | n1 | n2 | n3;
    }
    if (__any_sync(0xffffffffu, any))   // warp-uniform
#pragma unroll
        for (int k = 0; k < N; k++) w[k] = pack_q8x4(x[k], q);
}

// The codes of 4N values.  The nearest integer of y = x * (1/d) comes from the low mantissa
// bits of y + 1.5 * 2^23 (|y| <= 127.5 here, so that byte is the code in two's complement);
// only if some lane of the warp has a value whose y lies within 2^-14 of a half-integer
// does the warp form the exact codes instead (one warp-uniform branch, rarely taken).
template <int N>
__device__ __forceinline__ void pack_q8_words_fast(const float4 (&x)[N], const Q8Scale &q, uint32_t (&w)[N]) {
    bool near = false;
    auto one = [&](float v) {
        const float y = (v * q.s) * q.r;
        const float t = y + 12582912.0f;
        near |= q8_near_half(y, t - 12582912.0f);
        return (int)__float_as_uint(t);
    };
#pragma unroll
    for (int k = 0; k < N; k++) w[k] = pack_bytes(one(x[k].x), one(x[k].y), one(x[k].z), one(x[k].w));
    if (__any_sync(0xffffffffu, near))
#pragma unroll
        for (int k = 0; k < N; k++) w[k] = pack_q8x4(x[k], q);
}

__device__ __forceinline__ void pack_q8x16(const float4 (&x)[4], const Q8Scale &q, uint32_t (&w)[4]) {
    pack_q8_words<4>(x, q, w);
}

// Sum of the four signed codes of a packed word.
__device__ __forceinline__ int sum_q8x4(uint32_t word) { return __dp4a((int)word, 0x01010101, 0); }

__device__ __forceinline__ float absmax4(float4 v) {
    return fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
}

// ---------------------------------------------------------------------------
// The integer block dot of the q_f32 kind with dp4a.  A Q4_0 block's 16 code
// bytes hold q_i in the low nibble and q_{i+16} in the high nibble of byte i.
// With the activation codes a[0..31] (int8, element order) and
// corr = -8 * sum(a):
//     sum_j (q_j - 8) * a_j = corr + sum_j q_j * a_j        (exact in int32)
// The low nibbles are masked in place (bytes 0..15); the high nibbles are
// masked in place too, as 16 q (bytes 0..240, unsigned), so their dot product
// is 16 times the wanted one and an arithmetic shift by 4 recovers it exactly.
// Two independent dp4a chains; no shifts of the code words.
// ---------------------------------------------------------------------------
__device__ __forceinline__ int dp4a_u8s8(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// w: the 16 code bytes of a block; a0: activation codes 0..15, a1: codes 16..31
__device__ __forceinline__ int block_dot(uint4 w, uint4 a0, uint4 a1, int corr) {
    int lo = corr, hi = 0;
    lo = dp4a_u8s8(w.x & 0x0F0F0F0Fu, a0.x, lo);
    hi = dp4a_u8s8(w.x & 0xF0F0F0F0u, a1.x, hi);
    lo = dp4a_u8s8(w.y & 0x0F0F0F0Fu, a0.y, lo);
    hi = dp4a_u8s8(w.y & 0xF0F0F0F0u, a1.y, hi);
    lo = dp4a_u8s8(w.z & 0x0F0F0F0Fu, a0.z, lo);
    hi = dp4a_u8s8(w.z & 0xF0F0F0F0u, a1.z, hi);
    lo = dp4a_u8s8(w.w & 0x0F0F0F0Fu, a0.w, lo);
    hi = dp4a_u8s8(w.w & 0xF0F0F0F0u, a1.w, hi);
    return lo + (hi >> 4);
}

// Q8_0 weights: w0, w1 the 32 signed codes of a block, a0, a1 the activation codes (exact int32).
__device__ __forceinline__ int block_dot_s8(uint4 w0, uint4 w1, uint4 a0, uint4 a1) {
    int s0 = 0, s1 = 0;
    s0 = __dp4a((int)w0.x, (int)a0.x, s0);
    s1 = __dp4a((int)w1.x, (int)a1.x, s1);
    s0 = __dp4a((int)w0.y, (int)a0.y, s0);
    s1 = __dp4a((int)w1.y, (int)a1.y, s1);
    s0 = __dp4a((int)w0.z, (int)a0.z, s0);
    s1 = __dp4a((int)w1.z, (int)a1.z, s1);
    s0 = __dp4a((int)w0.w, (int)a0.w, s0);
    s1 = __dp4a((int)w1.w, (int)a1.w, s1);
    return s0 + s1;
}

// Q5_0 weights in a repacked tile: w the 16 nibble bytes of a block (the Q4_0 order), h the
// block's 32 fifth bits arranged so that bit 8b + 7 - s holds the fifth bit of element b of group
// s (groups 0..3: elements 4s .. 4s+3, the low nibbles of word s; groups 4..7: elements
// 16 + 4(s-4) .., the high nibbles).  The five-bit codes of word w then are
// (w & 0x0F) | ((h >> (3 - w)) & 0x10) per byte (low) and ((w >> 4) & 0x0F) | ((h << (1 + w)) & 0x10)
// (high).  corr = -16 * sum of the activation codes; the result is sum_j (q5_j - 16) q8_j.
__device__ __forceinline__ uint32_t q5_lo(uint32_t w, uint32_t h, int word) {
    return (w & 0x0F0F0F0Fu) | ((h >> (3 - word)) & 0x10101010u);
}
__device__ __forceinline__ uint32_t q5_hi(uint32_t w, uint32_t h, int word) {
    return ((w >> 4) & 0x0F0F0F0Fu) | ((h << (1 + word)) & 0x10101010u);
}
__device__ __forceinline__ int block_dot_q5(uint4 w, uint32_t h, uint4 a0, uint4 a1, int corr) {
    int lo = corr, hi = 0;
    lo = dp4a_u8s8(q5_lo(w.x, h, 0), a0.x, lo);
    hi = dp4a_u8s8(q5_hi(w.x, h, 0), a1.x, hi);
    lo = dp4a_u8s8(q5_lo(w.y, h, 1), a0.y, lo);
    hi = dp4a_u8s8(q5_hi(w.y, h, 1), a1.y, hi);
    lo = dp4a_u8s8(q5_lo(w.z, h, 2), a0.z, lo);
    hi = dp4a_u8s8(q5_hi(w.z, h, 2), a1.z, hi);
    lo = dp4a_u8s8(q5_lo(w.w, h, 3), a0.w, lo);
    hi = dp4a_u8s8(q5_hi(w.w, h, 3), a1.w, hi);
    return lo + hi;
}

// D(16x8, f32) += A(16x16, f16, row) . B(16x8, f16, col)
__device__ __forceinline__ void mma_f16_16x8x16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                                uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Four codes 0..15 (one per byte) -> two half2 of q itself, exact (as q4_to_f16x2, bias 1024).
__device__ __forceinline__ void q4u_to_f16x2(uint32_t v, uint32_t &h01, uint32_t &h23) {
    const __half2 bias = __halves2half2(__ushort_as_half(0x6400), __ushort_as_half(0x6400));   // 1024
    uint32_t a = __byte_perm(v, 0x64646464u, 0x4140u), b = __byte_perm(v, 0x64646464u, 0x4342u);
    __half2 x = __hsub2(*reinterpret_cast<__half2 *>(&a), bias), y = __hsub2(*reinterpret_cast<__half2 *>(&b), bias);
    h01 = *reinterpret_cast<uint32_t *>(&x);
    h23 = *reinterpret_cast<uint32_t *>(&y);
}

// Four codes 0..31 (one per byte) -> two half2 of (q - 16), exact (as q4_to_f16x2, bias 1040).
__device__ __forceinline__ void q5_to_f16x2(uint32_t v, uint32_t &h01, uint32_t &h23) {
    const __half2 bias = __halves2half2(__ushort_as_half(0x6410), __ushort_as_half(0x6410));   // 1040
    uint32_t a = __byte_perm(v, 0x64646464u, 0x4140u), b = __byte_perm(v, 0x64646464u, 0x4342u);
    __half2 x = __hsub2(*reinterpret_cast<__half2 *>(&a), bias), y = __hsub2(*reinterpret_cast<__half2 *>(&b), bias);
    h01 = *reinterpret_cast<uint32_t *>(&x);
    h23 = *reinterpret_cast<uint32_t *>(&y);
}

// Four codes 0..15 (one per byte) -> two half2 of (q - 8), exact: the bytes become the
// low mantissa bits of 1024 + q, and 1032 is subtracted.
__device__ __forceinline__ void q4_to_f16x2(uint32_t v, uint32_t &h01, uint32_t &h23) {
    const __half2 bias = __halves2half2(__ushort_as_half(0x6408), __ushort_as_half(0x6408));   // 1032
    uint32_t a = __byte_perm(v, 0x64646464u, 0x4140u), b = __byte_perm(v, 0x64646464u, 0x4342u);
    __half2 x = __hsub2(*reinterpret_cast<__half2 *>(&a), bias), y = __hsub2(*reinterpret_cast<__half2 *>(&b), bias);
    h01 = *reinterpret_cast<uint32_t *>(&x);
    h23 = *reinterpret_cast<uint32_t *>(&y);
}

// Four int8 codes -> two half2, exact: the bytes plus 128 become 1024 + 128 + q, less 1152.
__device__ __forceinline__ void q8_to_f16x2(uint32_t v, uint32_t &h01, uint32_t &h23) {
    const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));   // 1152
    v ^= 0x80808080u;
    uint32_t a = __byte_perm(v, 0x64646464u, 0x4140u), b = __byte_perm(v, 0x64646464u, 0x4342u);
    __half2 x = __hsub2(*reinterpret_cast<__half2 *>(&a), bias), y = __hsub2(*reinterpret_cast<__half2 *>(&b), bias);
    h01 = *reinterpret_cast<uint32_t *>(&x);
    h23 = *reinterpret_cast<uint32_t *>(&y);
}

__device__ __forceinline__ float half_lo(uint32_t w) { return __half2float(__ushort_as_half((unsigned short)(w & 0xffffu))); }
__device__ __forceinline__ float half_hi(uint32_t w) { return __half2float(__ushort_as_half((unsigned short)(w >> 16))); }

// ---------------------------------------------------------------------------
// Thread-block clusters: distributed shared memory for split-K partial sums.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Address of the same shared variable in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t map_shared_rank(const void *smem_ptr, uint32_t rank) {
    uint32_t a = (uint32_t)__cvta_generic_to_shared(smem_ptr);
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
    return r;
}

// The same, from a shared-memory address of this CTA.
__device__ __forceinline__ uint32_t map_shared_rank_addr(uint32_t saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}

__device__ __forceinline__ float ld_shared_cluster_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

// ---------------------------------------------------------------------------
// mbarriers and bulk (TMA) copies global -> shared.
// ---------------------------------------------------------------------------
constexpr uint32_t WAIT_LIMIT = 1u << 22;   // try_wait polls before a wait gives up

__device__ __forceinline__ uint32_t smem_addr(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Makes barrier initialisation visible to the asynchronous (TMA) proxy.
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Orders this thread's generic-proxy shared-memory accesses before later
// asynchronous-proxy writes (a refill of a buffer that was just read).
__device__ __forceinline__ void fence_proxy_async_shared() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// 1-D bulk copy; dst, src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(dst), "l"(src), "r"(bytes), "r"(bar) : "memory");
}

// An L2 policy for data read once (streamed weights): their lines are the first to be
// evicted, so they do not push out what is read again (activations, outputs).
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// bulk_g2s with an L2 cache policy.
__device__ __forceinline__ void bulk_g2s_hint(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar,
                                              uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
        ::"r"(dst), "l"(src), "r"(bytes), "r"(bar), "l"(policy) : "memory");
}

// Brings [src, src + bytes) into L2 (a hint: no data moves to the SM, nothing waits for it).
// L2 is where every access to device memory meets, so this never makes a later read stale.
__device__ __forceinline__ void bulk_prefetch_l2(const void *src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    return ok != 0;
}

// Waits for the phase with the given parity; gives up after `limit` polls, records the
// timeout in the device status word and returns false.  The product kernels use the
// fixed WAIT_LIMIT: a shorter limit inside a pipeline would let a consumer give up on a
// copy that is still landing.  The wait-timeout probe passes its own limit.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, unsigned int *status,
                                          uint32_t limit = WAIT_LIMIT) {
    for (uint32_t i = 0; i < limit; i++)
        if (mbar_try_wait(bar, parity)) return true;
    flag_timeout(status);
    return false;
}

__device__ __forceinline__ uint4 lds128(const uint8_t *p) { return *reinterpret_cast<const uint4 *>(p); }

}  // namespace gq
