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

// Four Q8_0 codes packed into a little-endian word (code of x.x in the low byte).
__device__ __forceinline__ uint32_t pack_q8x4(float4 x, float d) {
    uint32_t b0 = (uint32_t)(q8_code(x.x, d) & 0xff);
    uint32_t b1 = (uint32_t)(q8_code(x.y, d) & 0xff);
    uint32_t b2 = (uint32_t)(q8_code(x.z, d) & 0xff);
    uint32_t b3 = (uint32_t)(q8_code(x.w, d) & 0xff);
    return b0 | (b1 << 8) | (b2 << 16) | (b3 << 24);
}

__device__ __forceinline__ float absmax4(float4 v) {
    return fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
}

// ---------------------------------------------------------------------------
// Nibble unpacking for the int8 tensor instruction.  A word holds the codes of
// four consecutive bytes; the low nibbles are elements 4c..4c+3 of a block and
// the high nibbles elements 16+4c..16+4c+3.  Each code q in 0..15 becomes the
// int8 16*(q-8) = (q ^ 8) << 4, so the product is 16 * sumi exactly.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t nib_lo_x16(uint32_t w) { return ((w << 4) & 0xF0F0F0F0u) ^ 0x80808080u; }
__device__ __forceinline__ uint32_t nib_hi_x16(uint32_t w) { return (w & 0xF0F0F0F0u) ^ 0x80808080u; }

// D(16x8, s32) = A(16x32, s8, row) . B(32x8, s8, col)
__device__ __forceinline__ void mma_s8_16x8x32(int32_t (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%10, %11, %12, %13};"
        : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "r"(0), "r"(0), "r"(0), "r"(0));
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

__device__ __forceinline__ float ld_shared_cluster_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

}  // namespace gq
