// gq_internal.h -- host-side interface between the translation units of libgq.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "gq.h"

namespace gq {

// Records the message returned by gq_last_error_message() for this thread.
gq_status fail(gq_status s, const char *fmt, ...);
// Clears that message and returns GQ_OK.
gq_status ok();
// Argument checks shared by the entry points (they never touch the GPU).
gq_status check_sizes(int64_t M, int64_t N, int64_t K);
gq_status check_ptr(const void *p, const char *name);
// GQ_ERR_UNSUPPORTED_DEVICE unless the current device is sm_103.
gq_status check_device();
// Maps a CUDA error to GQ_ERR_CUDA (with its text), cudaSuccess to GQ_OK.
gq_status check_cuda(cudaError_t e, const char *what);

// Number of SMs of the current device (cached per device).
int sm_count();
// Whether callers declared that work in front of a product never writes its weights.
bool static_weights();
// Device address of the current device's sticky status word (nullptr on error).
unsigned int *device_status_word();

// Per-(device, stream) workspace: a zeroed counter region and a data region.
struct Workspace {
    uint8_t *counters;
    uint8_t *data;
};
gq_status get_workspace(cudaStream_t s, size_t counter_bytes, size_t data_bytes, Workspace *out);
gq_status reset_workspace_counters();
// Per-(device, stream) device staging buffer of at least `bytes` bytes (grows on demand).
gq_status get_staging(cudaStream_t s, size_t bytes, uint8_t **out);

// Launchers (arguments already validated by the entry points).
gq_status launch_quantize_q4_0(const float *w, void *q4, int64_t N, int64_t K, cudaStream_t s);
gq_status launch_quantize_rows_q8_0(const float *x, void *q8, int64_t M, int64_t K, cudaStream_t s);
gq_status launch_repack_q4_0(const void *q4, void *rep, int64_t N, int64_t K, cudaStream_t s);

gq_status launch_gemv_q4_0(const void *rep, const float *x, float *dst, int64_t M, int64_t N,
                           int64_t K, cudaStream_t s);
// K slices the Q4_0 GEMV runs for M (up to 16) activation rows of an [N][K] weight (one launch
// per slice for several rows).
int gemv_q4_0_slices(int64_t N, int64_t K, int64_t M);
// Workspace bytes (counters, data) the Q4_0 GEMV needs for an [N][K] weight.
void gemv_q4_0_workspace(int64_t N, int64_t K, size_t *counter_bytes, size_t *data_bytes);
// The Q4_0 GEMV on a given workspace (counters zero on entry, left at zero).
gq_status launch_gemv_q4_0_with(const void *rep, const float *x, float *dst, int64_t M, int64_t N, int64_t K,
                                const Workspace &ws, cudaStream_t s);
// The one-row Q4_0 product (whole row groups per CTA, no workspace): whether it serves
// [N][K], and its launch.
bool gemv_m1_supported(int64_t N, int64_t K);
gq_status launch_gemv_m1_q4_0(const void *rep, const float *x, float *dst, int64_t N, int64_t K, cudaStream_t s);
// F16 weights repacked into 16 x 32 tiles: the repack, and the GEMV on them (the Q4_0
// GEMV's pipeline with fp16 MMAs on the tiles as stored).
gq_status launch_repack_f16(const void *w16, void *rep, int64_t N, int64_t K, cudaStream_t s);
void gemv_f16r_workspace(int64_t N, int64_t K, size_t *counter_bytes, size_t *data_bytes);
gq_status launch_gemv_f16r(const void *rep, const float *x, float *dst, int64_t M, int64_t N, int64_t K,
                           cudaStream_t s);
// Q8_0 weights: the repack into 16-row x 4-block tiles (2176 bytes) and the GEMV on them.
gq_status launch_repack_q8_0(const void *q8, void *rep, int64_t N, int64_t K, cudaStream_t s);
gq_status launch_gemv_q8_0(const void *rep, const float *x, float *dst, int64_t M, int64_t N, int64_t K,
                           cudaStream_t s);
// Q5_0 weights: the quantizer, the repack into 16-row x 4-block tiles (1408 bytes), the GEMV.
gq_status launch_quantize_q5_0(const float *w, void *q5, int64_t N, int64_t K, cudaStream_t s);
gq_status launch_repack_q5_0(const void *q5, void *rep, int64_t N, int64_t K, cudaStream_t s);
gq_status launch_gemv_q5_0(const void *rep, const float *x, float *dst, int64_t M, int64_t N, int64_t K,
                           cudaStream_t s);
// Q4_1 weights: the quantizer, the repack into 16-row x 4-block tiles (1280 bytes), the GEMV.
gq_status launch_quantize_q4_1(const float *w, void *q41, int64_t N, int64_t K, cudaStream_t s);
gq_status launch_repack_q4_1(const void *q41, void *rep, int64_t N, int64_t K, cudaStream_t s);
gq_status launch_gemv_q4_1(const void *rep, const float *x, float *dst, int64_t M, int64_t N, int64_t K,
                           cudaStream_t s);
// Tensor-core tiles (tcgen05) for M >= 32; workspace: the fp16 activations.
size_t tc_workspace_bytes(int64_t M, int64_t K);
gq_status launch_tc_q4_0(const void *rep, const float *x, float *dst, int64_t M, int64_t N, int64_t K,
                         cudaStream_t s);
gq_status launch_tc_f16(const void *w16, const float *x, float *dst, int64_t M, int64_t N, int64_t K,
                        cudaStream_t s);
// INT8 KV cache: rows of D values to codes and f32 scales; one token per sequence into
// the cache at pos[b]; the decode attention over the cache (D 128 with Hq / Hkv 1 .. 8, or D 64
// with Hq / Hkv 1, 2, 4, 8).
gq_status launch_kv_quantize_i8(const float *x, int8_t *q, float *scale, int64_t rows, int64_t D, cudaStream_t s);
gq_status launch_kv_append_i8(const float *x, int8_t *q, float *scale, const int32_t *pos, int64_t B, int64_t Hkv,
                              int64_t Tcap, int64_t D, cudaStream_t s);
gq_status launch_attn_decode_i8(const float *q, const int8_t *k, const float *ks, const int8_t *v, const float *vs,
                                const int32_t *lens, float *out, int64_t B, int64_t Hq, int64_t Hkv, int64_t Tcap,
                                int64_t D, float softmax_scale, cudaStream_t s);
// A 2D tensor map (`map` points to a 64-byte-aligned CUtensorMap) over `rows` rows of 128
// bytes at `base`: boxes of 128 bytes x box_rows rows, 128-byte swizzle, rows past the end
// read as zeros.
gq_status byte_rows_map(void *map, const void *base, int64_t rows, int box_rows);
// A 3D tensor map (`map` as above) over row-major F16 weights [N][K] (K a multiple of 32):
// dimensions {32 columns, N rows, K / 32 tile columns}, boxes {32, 16, 16}: one box is 16
// consecutive 16 x 32 tiles of a row group, each stored as 16 rows of 64 bytes, one tile after
// the other (the repacked F16 layout).  Rows past N and columns past K read as zeros.
gq_status f16_tile_map(void *map, const void *base, int64_t N, int64_t K);
// The F16 product over row-major weights through the GEMV pipeline of the repacked tiles.
gq_status launch_gemv_f16_rowmajor(const void *w16, const float *x, float *dst, int64_t M, int64_t N, int64_t K,
                                   cudaStream_t s);
gq_status launch_block_dots_q4_0(const void *rep, const void *q8, int32_t *sumi, int64_t M,
                                 int64_t N, int64_t K, cudaStream_t s);

}  // namespace gq
