/*
 * gq.h -- C ABI of the GB300 quantized skinny MUL_MAT library (libgq.so).
 *
 * The operation is llama.cpp's MUL_MAT for decode and small-batch serving:
 *
 *     dst[M][N] = src1[M][K] . src0[N][K]^T        dst[m][n] = sum_k src0[n][k] * src1[m][k]
 *
 * in the two kinds named in llama.cpp pull request #1632, "Introduction":
 * mul_mat_q_f32 (src0 block-quantized, here Q4_0) and mul_mat_f16_f32 (src0
 * F16); src1 is F32 in both.  For the q_f32 kind, src1 is quantized row by row
 * to Q8_0 (the "wdata" buffer of the Arm China NUMA article, section
 * "MulMat 算子優化": dst = src0 * wdata) and the product is formed from exact
 * int32 block dot products scaled by the two fp16 block scales.
 *
 * Conventions shared by every entry point
 *   - All matrices are row-major with the last index contiguous: src0 [N][K],
 *     src1 [M][K], dst [M][N].  Sizes are element counts (int64_t).
 *   - Every pointer is a DEVICE pointer on the current CUDA device.  The caller
 *     owns every buffer; the library keeps no pointer after a call returns.
 *   - Work is enqueued on `stream` (0 = the legacy default stream) and the call
 *     returns without waiting for it.  Results are defined once the stream has
 *     reached that point.
 *   - K must be a positive multiple of 32 (the block size); M and N positive.
 *   - Every pointer must be 16-byte aligned.
 *   - dst is overwritten, never accumulated into.
 *   - Inputs are assumed finite; NaN or Inf inputs give unspecified outputs.
 *   - Errors: GQ_ERR_INVALID_ARG (bad size, null pointer) and GQ_ERR_MISALIGNED
 *     are returned before anything is launched; GQ_ERR_UNSUPPORTED_DEVICE when
 *     the current device is not compute capability 10.3 (GB300);
 *     GQ_ERR_CUDA when a CUDA call or launch failed (see gq_last_error_message);
 *     a kernel-side wait that gave up is reported later by gq_last_error().
 *     No C++ exception crosses this interface.
 *   - Thread safety: every entry point may be called from several host threads.
 *
 * Block formats (the pages name Q4_0 and Q8_0 without defining them; these are
 * the ggml layouts as this library reads them):
 *   Q4_0, 18 bytes per 32 weights: fp16 d (little endian), then 16 bytes whose
 *     byte i holds code q_i in the low nibble and q_{i+16} in the high nibble.
 *     Weight j is (q_j - 8) * d.  Quantization of x[0..31]: m = the element of
 *     largest magnitude (the first on a tie), d = m / -8 (f32),
 *     q_j = clamp(roundf(x_j / d) + 8, 0, 15), or 8 when d == 0; the stored
 *     scale is d rounded to fp16 (nearest even).
 *   Q8_0, 34 bytes per 32 values: fp16 d, then 32 int8 codes.  d = amax / 127
 *     (f32), q_j = roundf(x_j / d), or 0 when d == 0; stored scale fp16(d).
 */
#ifndef GQ_H
#define GQ_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define GQ_ABI_VERSION 1

typedef enum gq_status {
    GQ_OK = 0,
    GQ_ERR_INVALID_ARG = 1,        /* size <= 0, K % 32 != 0, null pointer, bad enum */
    GQ_ERR_MISALIGNED = 2,         /* a pointer is not 16-byte aligned */
    GQ_ERR_UNSUPPORTED_DEVICE = 3, /* the current device is not sm_103 */
    GQ_ERR_CUDA = 4,               /* a CUDA runtime call or a launch failed */
    GQ_ERR_TIMEOUT = 5,            /* a bounded in-kernel wait gave up (gq_last_error) */
    GQ_ERR_NO_MEMORY = 6,          /* the stream-ordered workspace could not be allocated */
    GQ_ERR_DEVICE_CHECK = 7        /* a bounds check of a GQ_DEBUG build failed (gq_last_error) */
} gq_status;

/* Which kernel family serves a product. */
typedef enum gq_path {
    GQ_PATH_AUTO = 0,   /* the shape's dispatch profile, if one is set; else M <= threshold:
                           the GEMV family, above it the tensor-core tiles (Q4_0 rows also
                           take the tiles when the GEMV would need several K slices for them) */
    GQ_PATH_GEMV = 1,   /* the skinny GEMV kernels (any M; M > 16 runs in 16-row slices) */
    GQ_PATH_TC = 2      /* the tcgen05 tensor-core tile kernels (any M) */
} gq_path;

/* ---- library information and errors ------------------------------------ */

int gq_abi_version(void);                      /* GQ_ABI_VERSION of the built library */
const char *gq_status_string(gq_status status); /* static text, never NULL */

/* Text of the last error returned to this host thread (static storage of the
 * thread, valid until its next call).  "" when the last call succeeded. */
const char *gq_last_error_message(void);

/* Sticky device-side status of the current device: GQ_ERR_TIMEOUT if a kernel
 * gave up a bounded wait since the last call, else GQ_ERR_DEVICE_CHECK if a
 * bounds check of a GQ_DEBUG build failed (a library bug; those builds check the
 * indices the kernels derive from their arguments and never trap), else
 * GQ_ERR_INVALID_ARG if a length or position read on the device was out of range
 * (the INT8 KV-cache calls), else GQ_OK; reading clears it and, after a timeout, re-zeroes the
 * workspace counters of the device.  Synchronizes the current device first. */
gq_status gq_last_error(void);

/* ---- buffer sizes --------------------------------------------------------- */

size_t gq_q4_0_bytes(int64_t N, int64_t K);          /* N * K / 32 * 18 */
size_t gq_q8_0_bytes(int64_t M, int64_t K);          /* M * K / 32 * 34 */
size_t gq_q4_0_repacked_bytes(int64_t N, int64_t K); /* ceil(N/16) * ceil(K/128) * 1152 */

/* ---- load-time preparation of the weights ---------------------------------- */

/* Quantize F32 weights w [N][K] into canonical Q4_0 blocks q4_blocks
 * [N][K/32] (gq_q4_0_bytes(N, K) bytes), byte-exact to the format above.
 * llama.cpp PR #1632, "Introduction": src0 of the q_f32 kind is quantized. */
gq_status gq_quantize_q4_0(const float *w, void *q4_blocks, int64_t N, int64_t K,
                           cudaStream_t stream);

/* Permute canonical Q4_0 blocks into the layout the product kernels stream
 * (done once when the weights are loaded).  q4_repacked must hold
 * gq_q4_0_repacked_bytes(N, K) bytes and must not overlap q4_blocks.
 *
 * Repacked layout (a pure byte permutation plus padding): rows are grouped by
 * 16 (N16 = ceil(N/16) groups) and columns by 128 (NT = ceil(K/128) tiles of 4
 * blocks).  Tile (g, t) occupies the 1152 bytes at offset (g*NT + t)*1152:
 *   bytes [(j*16 + r)*16, +16), j in 0..3, r in 0..15: the 16 code bytes of
 *       (row 16g+r, block 4t+j), in their canonical order;
 *   bytes [1024 + (r*4 + j)*2, +2): the fp16 scale of (row 16g+r, block 4t+j).
 * Rows >= N and blocks >= K/32 are padding: nibble bytes 0x88 and scale +0.
 * Each row group's tiles are contiguous, so a slice of K streams as one block
 * of bytes (DeepSpeed-Inference notes, section III.C.3: rearrange the weights
 * once at initialisation so that loads fill whole cache lines). */
gq_status gq_repack_q4_0(const void *q4_blocks, void *q4_repacked, int64_t N, int64_t K,
                         cudaStream_t stream);

/* ---- the INIT stage on its own ------------------------------------------------- */

/* Quantize F32 activations x [M][K] into Q8_0 blocks q8_blocks [M][K/32]
 * (gq_q8_0_bytes(M, K) bytes), byte-exact to the format above.  The product
 * entry points do this themselves (fused); this entry exists for callers that
 * keep wdata and for verification.  Arm China NUMA article, "MulMat 算子優化". */
gq_status gq_quantize_rows_q8_0(const float *x, void *q8_blocks, int64_t M, int64_t K,
                                cudaStream_t stream);

/* ---- the products ---------------------------------------------------------------- */

/* dst[M][N] = Q8_0(src1)[M][K] . Q4_0(src0)[N][K]^T with src0 given in the
 * repacked layout of gq_repack_q4_0.  src1 is quantized to Q8_0 inside the call;
 * each output is sum_b fp16(d4_b) * fp16(d8_b) * sumi_b with the exact int32
 * block dots sumi_b, accumulated in f32 on the GEMV path (M <= threshold) and,
 * on the tensor-core path, from fp16-rounded de-quantized operands with f32
 * accumulation (relative error <= 2e-3 of sum |terms|).  Uses the stream's
 * workspace (see gq_reserve_workspace); results do not depend on timing. */
gq_status gq_mul_mat_q4_0_f32(const void *q4_repacked, const float *src1, float *dst,
                              int64_t M, int64_t N, int64_t K, cudaStream_t stream);

/* dst[M][N] = src1[M][K] . src0[N][K]^T with F16 weights src0 (IEEE binary16,
 * row-major).  Activations are rounded to fp16 for the tensor instructions and
 * the sums are accumulated in f32 (relative error <= 2e-3 of sum |terms|).  On
 * the GEMV path (M <= threshold) tensor copies read the row-major weights as
 * 16 x 32 tiles, the unit of gq_mul_mat_f16r_f32, whose kernel it shares.  Uses
 * the stream's workspace (see gq_reserve_workspace); results do not depend on
 * timing. */
gq_status gq_mul_mat_f16_f32(const void *src0_f16, const float *src1, float *dst,
                             int64_t M, int64_t N, int64_t K, cudaStream_t stream);

/* The Q4_0 product of gq_mul_mat_q4_0_f32 with src1 ([M][K] f32) and dst ([M][N]
 * f32) in HOST memory.  The call enqueues on `stream` the transfer of src1 to a
 * device staging buffer, the product, and the transfer of dst back to the host,
 * and returns; dst_host holds the result once the stream has reached that point
 * (cudaStreamSynchronize).  src1_host and dst_host are plain host pointers with
 * no alignment rule.  Page-locked memory that the device maps (cudaHostAlloc,
 * cudaHostRegister with mapping; 16-byte aligned) is moved by the kernels
 * themselves: a small kernel stages src1 and the product stores dst straight into
 * host memory, with no copy-engine transfer.  Other host memory is copied with
 * cudaMemcpyAsync (synchronous for the host when it is pageable).  (Reading src1
 * in place in the product was slower: every CTA would read all of src1 across the
 * host link.)  The staging buffer belongs to the stream and grows like the
 * workspace (GQ_ERR_NO_MEMORY while the stream is captured); calls on one stream
 * use it in stream order.  Results equal gq_mul_mat_q4_0_f32's bit for bit.  (An
 * interface of this library: one call per decode step from host data.) */
gq_status gq_mul_mat_q4_0_f32_host(const void *q4_repacked, const float *src1_host, float *dst_host,
                                   int64_t M, int64_t N, int64_t K, cudaStream_t stream);

/* F16 weights for decode.  gq_repack_f16 copies row-major F16 weights [N][K]
 * into tiles of 16 rows x 32 columns (64 bytes per row, tile (g, t) of rows
 * 16g.. and columns 32t.. at byte (g * K/32 + t) * 1024, rows past N zero):
 * gq_f16_repacked_bytes(N, K) = ceil(N/16) * (K/32) * 1024 bytes, allocated by
 * the caller, not overlapping src0_f16 (GQ_ERR_INVALID_ARG).  A 16-row tile is
 * one contiguous kilobyte, the unit the GEMV streams.  gq_mul_mat_f16r_f32 is
 * the product of gq_mul_mat_f16_f32 on that layout, for any M (16 activation
 * rows per launch): the activations are rounded to fp16 and the f32 sums come
 * from fp16 tensor instructions (relative error <= 2e-3 of sum |terms|; the
 * results do not depend on timing).  It uses the stream's workspace like the
 * other products.  (llama.cpp PR #1632, "Introduction": MUL_MAT with F16
 * weights; the tile layout is this library's.) */
size_t gq_f16_repacked_bytes(int64_t N, int64_t K);   /* 0 if N <= 0, K <= 0 or K % 32 */
gq_status gq_repack_f16(const void *src0_f16, void *f16_repacked, int64_t N, int64_t K,
                        cudaStream_t stream);
gq_status gq_mul_mat_f16r_f32(const void *f16_repacked, const float *src1, float *dst,
                              int64_t M, int64_t N, int64_t K, cudaStream_t stream);

/* Q8_0 weights (llama.cpp PR #1632, "Introduction": src0 of the q_f32 kind may be
 * any quantized type; "Results": Q8_0 is among the types measured on 7B).  The
 * weights use the activations' Q8_0 block format: quantize them with
 * gq_quantize_rows_q8_0 ([N][K/32] x 34 bytes), then copy them once with
 * gq_repack_q8_0 into tiles of 16 rows x 4 blocks, 2176 bytes each: the 32 codes
 * of block j of row r at (j * 16 + r) * 32, then the fp16 scale of (r, j) at
 * 2048 + (r * 4 + j) * 2; tile (g, t) at (g * ceil(K/128) + t) * 2176; padding
 * holds codes 0 and scale 0.  gq_q8_0_repacked_bytes(N, K) = ceil(N/16) *
 * ceil(K/128) * 2176 bytes (0 if N <= 0, K <= 0 or K % 32); q8_repacked must not
 * overlap q8_blocks (GQ_ERR_INVALID_ARG).  gq_mul_mat_q8_0_f32 computes
 * dst[M][N] = Q8_0(src1) . Q8_0(src0)^T: each output is
 * sum_b fp16(dw_b) * fp16(dx_b) * sumi_b with the exact int32 block dots
 * sumi_b = sum_j qw_j * qx_j, accumulated in f32, by the GEMV family for every M
 * (16 activation rows per launch); it uses the stream's workspace like the other
 * products and its results do not depend on timing. */
size_t gq_q8_0_repacked_bytes(int64_t N, int64_t K);
gq_status gq_repack_q8_0(const void *q8_blocks, void *q8_repacked, int64_t N, int64_t K,
                         cudaStream_t stream);
gq_status gq_mul_mat_q8_0_f32(const void *q8_repacked, const float *src1, float *dst,
                              int64_t M, int64_t N, int64_t K, cudaStream_t stream);

/* Q4_1 weights (llama.cpp PR #1632, "Introduction": named beside Q4_0 as a src0
 * type of the q_f32 kind; the pages do not define it, and this library reads it
 * as a scale and a minimum per block).  Block (20 bytes): fp16 d, fp16 m, then 16
 * bytes with q_i in the low nibble and q_{i+16} in the high nibble of byte i;
 * lo / hi = the first element equal to the block's minimum / maximum,
 * d = (hi - lo) / 15, m = lo, q_j = clamp(round((x_j - lo) / d), 0, 15) (0 when
 * d == 0), all in f32; the weight is q_j * fp16(d) + fp16(m).  gq_quantize_q4_1
 * writes gq_q4_1_bytes(N, K) = N * K/32 * 20 bytes, byte-exact;
 * gq_repack_q4_1 copies them once into tiles of 16 rows x 4 blocks, 1280 bytes
 * each: the nibble bytes of block j of row r at (j * 16 + r) * 16, the fp16
 * scales at 1024 + (r * 4 + j) * 2, the fp16 minimums at 1152 + (r * 4 + j) * 2;
 * tile (g, t) at (g * ceil(K/128) + t) * 1280; padding is zero.
 * gq_q4_1_repacked_bytes(N, K) = ceil(N/16) * ceil(K/128) * 1280.
 * gq_mul_mat_q4_1_f32: dst[M][N] = Q8_0(src1) . Q4_1(src0)^T, each output
 * sum_b (fp16(d_b) fp16(d8_b) sumi_b + fp16(m_b) fp16(d8_b) sx_b) with the exact
 * int32 sums sumi_b = sum_j q_j q8_j and sx_b = sum_j q8_j, accumulated in f32
 * (the GEMV family for every M; the stream's workspace as for the other products). */
size_t gq_q4_1_bytes(int64_t N, int64_t K);            /* 0 if N <= 0, K <= 0 or K % 32 */
size_t gq_q4_1_repacked_bytes(int64_t N, int64_t K);
gq_status gq_quantize_q4_1(const float *w, void *q41_blocks, int64_t N, int64_t K, cudaStream_t stream);
gq_status gq_repack_q4_1(const void *q41_blocks, void *q41_repacked, int64_t N, int64_t K,
                         cudaStream_t stream);
gq_status gq_mul_mat_q4_1_f32(const void *q41_repacked, const float *src1, float *dst,
                              int64_t M, int64_t N, int64_t K, cudaStream_t stream);

/* Q5_0 weights (llama.cpp PR #1632, "Results": Q5_0 is among the types measured
 * on 7B; the pages do not define it, and this library reads it as Q4_0 with
 * five-bit codes).  Block (22 bytes): fp16 d, a little-endian 32-bit word whose
 * bit j is bit 4 of q_j, then 16 bytes with the low four bits of q_i in the low
 * nibble and those of q_{i+16} in the high nibble of byte i; m = the element of
 * largest magnitude (the first one on a tie), d = m / -16,
 * q_j = clamp(round(x_j / d) + 16, 0, 31) (16 when d == 0), the weight is
 * (q_j - 16) * fp16(d).  gq_quantize_q5_0 writes gq_q5_0_bytes(N, K) =
 * N * K/32 * 22 bytes, byte-exact; gq_repack_q5_0 copies them once into tiles of
 * 16 rows x 4 blocks, 1408 bytes each: the nibble bytes of block j of row r at
 * (j * 16 + r) * 16, its fifth bits at 1024 + (j * 16 + r) * 4 (bit 8b + 7 - s
 * holds the fifth bit of element b of group s; groups 0..3 are elements
 * 4s .. 4s+3, groups 4..7 elements 16 + 4(s-4) ..), then the fp16 scales at
 * 1280 + (r * 4 + j) * 2; tile (g, t) at (g * ceil(K/128) + t) * 1408; padding
 * holds code 16 and scale 0.  gq_q5_0_repacked_bytes(N, K) = ceil(N/16) *
 * ceil(K/128) * 1408.  gq_mul_mat_q5_0_f32: dst[M][N] = Q8_0(src1) . Q5_0(src0)^T,
 * each output sum_b fp16(d5_b) * fp16(d8_b) * sumi_b with the exact int32 block
 * dots sumi_b = sum_j (q5_j - 16) * q8_j, accumulated in f32 (the GEMV family for
 * every M, 16 rows per launch; the stream's workspace as for the other products). */
size_t gq_q5_0_bytes(int64_t N, int64_t K);            /* 0 if N <= 0, K <= 0 or K % 32 */
size_t gq_q5_0_repacked_bytes(int64_t N, int64_t K);
gq_status gq_quantize_q5_0(const float *w, void *q5_blocks, int64_t N, int64_t K, cudaStream_t stream);
gq_status gq_repack_q5_0(const void *q5_blocks, void *q5_repacked, int64_t N, int64_t K,
                         cudaStream_t stream);
gq_status gq_mul_mat_q5_0_f32(const void *q5_repacked, const float *src1, float *dst,
                              int64_t M, int64_t N, int64_t K, cudaStream_t stream);

/* Workspace.  The products keep a small device workspace per (device, stream):
 * partial sums of weight rows that several CTAs share, with per-row counters
 * that every launch leaves at zero, and (tensor-core path) the quantized
 * activations.  It is allocated with cudaMalloc the first time a stream needs it
 * and grows when a larger problem comes (at least doubling); growth synchronizes
 * that stream, and the replaced buffer stays allocated until the process exits,
 * so launches and graphs that took its address remain valid.  A
 * call that would grow it while the stream is being captured into a CUDA graph
 * returns GQ_ERR_NO_MEMORY: reserve it first with this call, on the stream that
 * will be captured, for the largest M, N, K it will run.  A growth whose
 * cudaMalloc fails returns GQ_ERR_NO_MEMORY and leaves the current workspace in
 * place (smaller problems keep running on it).  Graphs captured on a
 * stream use that stream's workspace: do not replay them concurrently with
 * other work on that stream's workspace. */
gq_status gq_reserve_workspace(int64_t M, int64_t N, int64_t K, cudaStream_t stream);

/* The same two products with the kernel family chosen by the caller. */
gq_status gq_mul_mat_q4_0_f32_path(const void *q4_repacked, const float *src1, float *dst,
                                   int64_t M, int64_t N, int64_t K, gq_path path,
                                   cudaStream_t stream);
gq_status gq_mul_mat_f16_f32_path(const void *src0_f16, const float *src1, float *dst,
                                  int64_t M, int64_t N, int64_t K, gq_path path,
                                  cudaStream_t stream);

/* M threshold of GQ_PATH_AUTO: M <= threshold runs the GEMV family.  Default 16
 * (Smallem, "Générer à plusieurs", section "La courbe, une première fois": the
 * narrow kernel serves products of at most 16 rows, the tiles the rest).  Q4_0
 * products of 2 .. threshold rows whose activation image needs several K slices
 * (one GEMV launch per slice, for example 9 to 16 rows at K = 11008) take the
 * tiles, which split K within one launch.  F16 products take the GEMV only when
 * N < 64 x the number of SMs and M * K * 2 <= 64 KiB (the fp16 activations);
 * otherwise the tiles, which read fp16 weights straight into the tensor cores
 * and measured faster there (for example [11008, 4096] at every M, [4096, 11008]
 * from 3 rows, [4096, 4096] from 9).
 * Process-wide; GQ_ERR_INVALID_ARG if t < 0.  The environment variable
 * GQ_M_THRESHOLD, read when the library loads, replaces the default when it
 * holds a non-negative decimal integer (other values are ignored). */
gq_status gq_set_m_threshold(int64_t t);
int64_t gq_get_m_threshold(void);

/* Per-shape dispatch profiles (llama.cpp PR #1632, "Solutions", item 4: the
 * shape is matched by N and K, the time of every kernel profile is estimated for
 * the given M by interpolating between benched M, and the fastest is taken).  A
 * profile holds, for one weight kind and one (N, K), the benched times of the
 * GEMV family and of the tile family at `count` values of M (strictly increasing,
 * positive; the times finite and non-negative, in any unit).  GQ_PATH_AUTO then
 * runs, for M rows, the family whose time is smaller when each curve is taken as
 * linear through its two benched points around M (the two end points outside the
 * benched range); shapes without a profile use the M threshold.  A new profile
 * for a shape replaces the old one.  Process-wide, thread-safe; no GPU work.
 * gq_choose_path reports the family GQ_PATH_AUTO would run.  The Python helper
 * tune_dispatch() benches both families on the current device and installs the
 * profile. */
typedef enum { GQ_KIND_Q4_0 = 0, GQ_KIND_F16 = 1 } gq_weight_kind;
gq_status gq_set_dispatch_profile(int kind, int64_t N, int64_t K, const int64_t *Ms, const double *t_gemv,
                                  const double *t_tc, int64_t count);
gq_status gq_clear_dispatch_profiles(void);
gq_path gq_choose_path(int kind, int64_t N, int64_t K, int64_t M);

/* The Q4_0 product of gq_mul_mat_q4_0_f32, for callers that cannot let a library
 * allocate device memory: serving processes whose own pooling allocator has
 * reserved the device memory up front (for example for a KV cache) and must
 * account for every byte, plug-ins loaded by a runtime that forbids them to
 * allocate, and latency-bound loops in which cudaMalloc (which can synchronize
 * the device) may not run.
 * (The pages have no counterpart: this is an interface of this library.)
 * All scratch space comes from one static device array of 4 MiB that every
 * device loading the library holds until the process exits; nothing is ever
 * allocated or freed.  It always runs the GEMV family (any M, 16 rows per
 * launch).  GQ_ERR_INVALID_ARG when [N][K] needs more scratch than 4 MiB (for
 * example N = 11008 with K up to 11008 fits).  The first call on a device
 * resolves the array's device address (cudaGetSymbolAddress) and keeps it for
 * the life of the process: make that call before any stream capture, and do not
 * use this entry point on a device after cudaDeviceReset.  Each call re-zeroes the array's counters on `stream`
 * (cudaMemsetAsync) and then uses the whole array: calls that overlap on the
 * GPU, from any streams, race on it and give wrong results. */
gq_status gq_mul_mat_q4_0_f32_noalloc(const void *q4_repacked, const float *src1, float *dst,
                                      int64_t M, int64_t N, int64_t K, cudaStream_t stream);

/* Static weights.  A product launch may start before the kernel in front of it
 * in the stream has finished (programmatic dependent launch), so that its
 * weight stream overlaps the tail of that kernel; it waits for it before it
 * reads src1 or writes dst.  With enable = 1 the caller declares that the work
 * enqueued right before a product never writes that product's weights (true in
 * a decode loop, where weights are written once at load time); the GEMV then
 * reads the weights before that wait.  Default 0: weights are read only after
 * every earlier kernel in the stream has finished.  Process-wide. */
gq_status gq_set_static_weights(int enable);
int gq_get_static_weights(void);

/* ---- INT8 KV cache and the decode attention over it -------------------------------
 *
 * xFasterTransformer (arXiv 2407.07304), "2.2 Effective KV cache Optimization":
 * the KV cache is stored as INT8 with its own scale for each token and each head,
 * and after the first token attention is a pair of memory-bound GEMVs whose INT8
 * operand is widened to FP32 before the multiply-add.  Section "2.1 LLM
 * Optimization" (SlimAttention) fixes the order for a query row: all its scores,
 * the softmax over them, then their product with the values.
 *
 * Scale (the page does not give its formula; this library reads it like Q8_0's):
 * for the D values x[0..D-1] of one token and one head, s = amax / 127 in f32,
 * kept as f32; q_j = roundf(x_j / s) (IEEE f32 division, ties away from zero),
 * or 0 when s == 0.  The cached value is q_j * s.
 *
 * Layouts (row-major, last index contiguous; all DEVICE pointers, 16-byte aligned):
 *   cache codes  int8  [B][Hkv][Tcap][D]   (one array for K, one for V)
 *   cache scales float [B][Hkv][Tcap]
 *   queries      float [B][Hq][D], Hq = G * Hkv; query head h reads KV head h / G
 *   lens, pos    int32 [B]
 *   output       float [B][Hq][D]
 * Sizes: D is 64 or 128; G is 1 to 8 for D = 128, and 1, 2, 4 or 8 for D = 64;
 * B, Hkv, Tcap positive with
 * B * Hkv * Tcap * D < 2^40 and Tcap < 2^30.  Other sizes: GQ_ERR_INVALID_ARG. */

/* Quantizes `rows` rows of D f32 values x [rows][D] into codes q [rows][D] and
 * scales scale [rows] (for example a prefill's K or V, laid out as the cache). */
gq_status gq_kv_quantize_i8(const float *x, int8_t *q, float *scale, int64_t rows, int64_t D,
                            cudaStream_t stream);

/* Appends one token per sequence: row (b, h) of x [B][Hkv][D] is quantized into
 * position pos[b] of the cache (codes [B][Hkv][Tcap][D], scales [B][Hkv][Tcap]).
 * pos is read on the device; a pos[b] outside [0, Tcap) skips that sequence and
 * makes the next gq_last_error() return GQ_ERR_INVALID_ARG. */
gq_status gq_kv_append_i8(const float *x, int8_t *q, float *scale, const int32_t *pos,
                          int64_t B, int64_t Hkv, int64_t Tcap, int64_t D, cudaStream_t stream);

/* Decode attention of one query row per (sequence, query head) over the INT8 cache:
 * for query head h of sequence b, over the tokens t < lens[b] of KV head h / G,
 *     score_t = softmax_scale * ks_t * sum_j q_j * k_tj
 *     out_j   = sum_t softmax(score)_t * vs_t * v_tj
 * with f32 arithmetic (INT8 widened exactly to f32) and a softmax that subtracts
 * the row's maximum.  lens[b] == 0 gives a zero row.  lens is read on the
 * device: a value outside [0, Tcap] is taken as 0 and makes the next
 * gq_last_error() return GQ_ERR_INVALID_ARG.  Long caches, or too few
 * (sequence, KV head) pairs to fill the GPU, split a sequence's tokens over
 * several CTAs whose parts are merged in a fixed order in the stream's
 * workspace (grown on demand, as for the products; GQ_ERR_NO_MEMORY if that
 * fails).  Results are deterministic. */
gq_status gq_attn_decode_i8(const float *q, const int8_t *k, const float *k_scale,
                            const int8_t *v, const float *v_scale, const int32_t *lens,
                            float *out, int64_t B, int64_t Hq, int64_t Hkv, int64_t Tcap,
                            int64_t D, float softmax_scale, cudaStream_t stream);

/* ---- verification --------------------------------------------------------------- */

/* The integer block dots of the GEMV instruction sequence, for parity tests:
 * sumi[M][N][K/32] (int32) = sum_j (q4_j - 8) * q8_j for every (row m of the
 * Q8_0 blocks q8_blocks [M][K/32], row n of the repacked Q4_0 weights, block b).
 * Not a product entry point: it writes M*N*K/32 int32 values. */
gq_status gq_debug_block_dots_q4_0(const void *q4_repacked, const void *q8_blocks,
                                   int32_t *sumi, int64_t M, int64_t N, int64_t K,
                                   cudaStream_t stream);

/* dp4a throughput probe, for the benchmark's ALU roofline: `blocks` CTAs of 256 threads,
 * each thread 8 * iters independent dp4a (int8 x4 dot with int32 accumulate); writes one
 * int per thread to sink [blocks * 256].  Not a product entry point. */
gq_status gq_debug_dp4a_probe(int64_t iters, int *sink, int64_t blocks, cudaStream_t stream);

/* The failure path of the bounded in-kernel waits, for tests: launches one warp that
 * waits, `limit` polls at most (1 .. 2^22), on an mbarrier that nothing completes and
 * that no copy signals, so the wait gives up and the kernel returns.  The next
 * gq_last_error() then returns GQ_ERR_TIMEOUT (and clears it); nothing else is
 * touched, and the products that follow on the device run as before.  Not a product
 * entry point. */
gq_status gq_debug_wait_timeout(uint32_t limit, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* GQ_H */
