// gq_api.cu -- the C entry points of libgq: argument checks, device checks,
// error reporting and the M-threshold dispatch between the kernel families.
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <algorithm>
#include <cmath>
#include <mutex>
#include <vector>

#include "gq_common.cuh"
#include "gq_internal.h"

namespace gq {

// Sticky device-side status word of each device (bit STATUS_TIMEOUT).
__device__ unsigned int g_status_word;

namespace {

thread_local char t_message[512];

constexpr int MAX_DEVICES = 64;
std::atomic<int> g_arch_ok[MAX_DEVICES];      // 0 unknown, 1 sm_103, -1 other
std::atomic<int> g_sm_count[MAX_DEVICES];
std::atomic<unsigned int *> g_status_ptr[MAX_DEVICES];
std::atomic<int64_t> g_m_threshold{16};

// GQ_M_THRESHOLD, when set to a non-negative decimal integer, replaces the default M
// threshold at load time (for dispatch experiments without code changes); any other
// value is ignored.
struct ThresholdFromEnvironment {
    ThresholdFromEnvironment() {
        const char *v = getenv("GQ_M_THRESHOLD");
        if (!v || !*v) return;
        char *end = nullptr;
        const long long t = strtoll(v, &end, 10);
        if (end && *end == '\0' && t >= 0) g_m_threshold.store((int64_t)t);
    }
} g_threshold_from_environment;
std::atomic<int> g_static_weights{0};

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

gq_status current_device(int *dev) {
    cudaError_t e = cudaGetDevice(dev);
    if (e != cudaSuccess) return check_cuda(e, "cudaGetDevice");
    if (*dev < 0 || *dev >= MAX_DEVICES) return fail(GQ_ERR_UNSUPPORTED_DEVICE, "device index %d", *dev);
    return GQ_OK;
}

#define GQ_TRY(expr)                       \
    do {                                   \
        gq_status _st = (expr);            \
        if (_st != GQ_OK) return _st;      \
    } while (0)

}  // namespace

// The kernels are built for sm_103a only: refuse other devices up front.
gq_status check_device() {
    int dev;
    gq_status st = current_device(&dev);
    if (st != GQ_OK) return st;
    int known = g_arch_ok[dev].load(std::memory_order_relaxed);
    if (known == 0) {
        int major = 0, minor = 0;
        cudaError_t e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        if (e != cudaSuccess) return check_cuda(e, "cudaDeviceGetAttribute");
        known = (major == 10 && minor == 3) ? 1 : -1;
        g_arch_ok[dev].store(known, std::memory_order_relaxed);
        if (known < 0)
            return fail(GQ_ERR_UNSUPPORTED_DEVICE, "device %d is sm_%d%d; libgq is built for sm_103a only",
                        dev, major, minor);
    }
    if (known < 0) return fail(GQ_ERR_UNSUPPORTED_DEVICE, "device %d is not sm_103", dev);
    return GQ_OK;
}

gq_status check_sizes(int64_t M, int64_t N, int64_t K) {
    if (M <= 0 || N <= 0 || K <= 0) return fail(GQ_ERR_INVALID_ARG, "sizes must be positive (M=%lld N=%lld K=%lld)",
                                                (long long)M, (long long)N, (long long)K);
    if (K % QK != 0) return fail(GQ_ERR_INVALID_ARG, "K=%lld is not a multiple of 32", (long long)K);
    // 32-bit index arithmetic inside the kernels
    if (N > (1LL << 30) || K > (1LL << 30) || M > (1LL << 30) || N * K > (1LL << 40))
        return fail(GQ_ERR_INVALID_ARG, "sizes too large (M=%lld N=%lld K=%lld)", (long long)M, (long long)N,
                    (long long)K);
    return GQ_OK;
}

gq_status check_ptr(const void *p, const char *name) {
    if (p == nullptr) return fail(GQ_ERR_INVALID_ARG, "%s is NULL", name);
    if (!aligned16(p)) return fail(GQ_ERR_MISALIGNED, "%s (%p) is not 16-byte aligned", name, p);
    return GQ_OK;
}

gq_status ok() {
    t_message[0] = '\0';
    return GQ_OK;
}

gq_status fail(gq_status s, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(t_message, sizeof(t_message), fmt, ap);
    va_end(ap);
    return s;
}

gq_status check_cuda(cudaError_t e, const char *what) {
    if (e == cudaSuccess) return GQ_OK;
    return fail(GQ_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorString(e), cudaGetErrorName(e));
}

bool static_weights() { return g_static_weights.load(std::memory_order_relaxed) != 0; }

int sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) return 148;
    int n = g_sm_count[dev].load(std::memory_order_relaxed);
    if (n == 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
        g_sm_count[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

// Kernels receive this address as an argument: the symbol itself is a host-side
// stand-in, so it is resolved once per device, with that device current.
unsigned int *device_status_word() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) return nullptr;
    unsigned int *p = g_status_ptr[dev].load(std::memory_order_acquire);
    if (p == nullptr) {
        void *a = nullptr;
        if (cudaGetSymbolAddress(&a, g_status_word) != cudaSuccess) return nullptr;
        p = static_cast<unsigned int *>(a);
        g_status_ptr[dev].store(p, std::memory_order_release);
    }
    return p;
}

}  // namespace gq

using namespace gq;

extern "C" {

int gq_abi_version(void) { return GQ_ABI_VERSION; }

const char *gq_status_string(gq_status s) {
    switch (s) {
        case GQ_OK: return "ok";
        case GQ_ERR_INVALID_ARG: return "invalid argument";
        case GQ_ERR_MISALIGNED: return "pointer not 16-byte aligned";
        case GQ_ERR_UNSUPPORTED_DEVICE: return "unsupported device (sm_103 required)";
        case GQ_ERR_CUDA: return "CUDA error";
        case GQ_ERR_TIMEOUT: return "a kernel gave up a bounded wait";
        case GQ_ERR_NO_MEMORY: return "workspace allocation failed";
        case GQ_ERR_DEVICE_CHECK: return "a device-side bounds check failed";
    }
    return "unknown status";
}

const char *gq_last_error_message(void) { return t_message; }

gq_status gq_last_error(void) {
    GQ_TRY(check_device());
    GQ_TRY(check_cuda(cudaDeviceSynchronize(), "cudaDeviceSynchronize"));
    unsigned int word = 0, zero = 0;
    GQ_TRY(check_cuda(cudaMemcpyFromSymbol(&word, g_status_word, sizeof(word)), "read device status"));
    GQ_TRY(check_cuda(cudaMemcpyToSymbol(g_status_word, &zero, sizeof(zero)), "clear device status"));
    if (word & STATUS_TIMEOUT) {
        reset_workspace_counters();
        return fail(GQ_ERR_TIMEOUT, "a kernel gave up a bounded wait");
    }
    if (word & STATUS_CHECK) return fail(GQ_ERR_DEVICE_CHECK, "a device-side bounds check (GQ_DEBUG build) failed");
    if (word & STATUS_RANGE) return fail(GQ_ERR_INVALID_ARG, "a length or position read on the device was out of range");
    return ok();
}

size_t gq_q4_0_bytes(int64_t N, int64_t K) {
    if (N <= 0 || K <= 0 || K % QK) return 0;
    return (size_t)N * (size_t)(K / QK) * Q4_0_BYTES;
}

size_t gq_q8_0_bytes(int64_t M, int64_t K) {
    if (M <= 0 || K <= 0 || K % QK) return 0;
    return (size_t)M * (size_t)(K / QK) * Q8_0_BYTES;
}

size_t gq_q4_0_repacked_bytes(int64_t N, int64_t K) {
    if (N <= 0 || K <= 0 || K % QK) return 0;
    return (size_t)((N + 15) / 16) * (size_t)((K + TILE_COLS - 1) / TILE_COLS) * TILE_BYTES;
}

gq_status gq_quantize_q4_0(const float *w, void *q4_blocks, int64_t N, int64_t K, cudaStream_t stream) {
    GQ_TRY(check_sizes(1, N, K));
    GQ_TRY(check_ptr(w, "w"));
    GQ_TRY(check_ptr(q4_blocks, "q4_blocks"));
    GQ_TRY(check_device());
    GQ_TRY(launch_quantize_q4_0(w, q4_blocks, N, K, stream));
    return ok();
}

gq_status gq_quantize_rows_q8_0(const float *x, void *q8_blocks, int64_t M, int64_t K, cudaStream_t stream) {
    GQ_TRY(check_sizes(M, 1, K));
    GQ_TRY(check_ptr(x, "x"));
    GQ_TRY(check_ptr(q8_blocks, "q8_blocks"));
    GQ_TRY(check_device());
    GQ_TRY(launch_quantize_rows_q8_0(x, q8_blocks, M, K, stream));
    return ok();
}

gq_status gq_repack_q4_0(const void *q4_blocks, void *q4_repacked, int64_t N, int64_t K, cudaStream_t stream) {
    GQ_TRY(check_sizes(1, N, K));
    GQ_TRY(check_ptr(q4_blocks, "q4_blocks"));
    GQ_TRY(check_ptr(q4_repacked, "q4_repacked"));
    const uintptr_t a = (uintptr_t)q4_blocks, b = (uintptr_t)q4_repacked;
    if (a < b + gq_q4_0_repacked_bytes(N, K) && b < a + gq_q4_0_bytes(N, K))
        return fail(GQ_ERR_INVALID_ARG, "q4_blocks and q4_repacked overlap");
    GQ_TRY(check_device());
    GQ_TRY(launch_repack_q4_0(q4_blocks, q4_repacked, N, K, stream));
    return ok();
}

gq_status gq_reserve_workspace(int64_t M, int64_t N, int64_t K, cudaStream_t stream) {
    GQ_TRY(check_sizes(M, N, K));
    GQ_TRY(check_device());
    size_t cb = 0, db = 0;
    gemv_q4_0_workspace(N, K, &cb, &db);
    size_t cb16 = 0, db16 = 0;
    gemv_f16r_workspace(N, K, &cb16, &db16);
    cb = std::max(cb, cb16);
    db = std::max(db, db16);
    // the tile path's activations: whatever the dispatcher picks for M (a tuned profile may send M
    // rows to the tile path below the threshold), the reserve covers it
    db = std::max(db, tc_workspace_bytes(M, K));
    Workspace ws;
    GQ_TRY(get_workspace(stream, cb, db, &ws));
    return ok();
}

gq_status gq_set_m_threshold(int64_t t) {
    if (t < 0) return fail(GQ_ERR_INVALID_ARG, "threshold %lld < 0", (long long)t);
    g_m_threshold.store(t);
    return ok();
}

int64_t gq_get_m_threshold(void) { return g_m_threshold.load(); }

gq_status gq_set_static_weights(int enable) {
    g_static_weights.store(enable ? 1 : 0);
    return ok();
}

int gq_get_static_weights(void) { return g_static_weights.load(); }

static gq_status check_path(gq_path path) {
    if (path != GQ_PATH_AUTO && path != GQ_PATH_GEMV && path != GQ_PATH_TC)
        return fail(GQ_ERR_INVALID_ARG, "unknown path %d", (int)path);
    return GQ_OK;
}

// Per-shape dispatch profiles: benched times of both kernel families at a few M
// (llama.cpp PR #1632, "Solutions", item 4: match the shape by N and K, estimate
// the time of every profile for the given M by interpolating between the benched
// M -- the M-time curve is close to linear -- and take the fastest).
namespace {
struct Profile {
    int kind;
    int64_t N, K;
    std::vector<int64_t> Ms;
    std::vector<double> t_gemv, t_tc;
};
std::mutex g_prof_mutex;
std::vector<Profile> g_profiles;

// Linear through the two benched points around M (the two end points outside the range).
double interpolate(const std::vector<int64_t> &Ms, const std::vector<double> &t, int64_t M) {
    const size_t n = Ms.size();
    if (n == 1) return t[0];
    size_t i = 0;
    while (i + 2 < n && Ms[i + 1] <= M) i++;
    return t[i] + (t[i + 1] - t[i]) * (double)(M - Ms[i]) / (double)(Ms[i + 1] - Ms[i]);
}
}  // namespace

// Which family serves M rows: a benched profile of the shape when there is one, else
// the M threshold (Smallem, "La courbe, une première fois": the narrow kernel up to 16
// rows, tiles above; llama.cpp PR #1632, "Introduction": the M >= 32 rule and how
// sensitive the choice is around it).
//
// Without a profile, Q4_0 rows also go to the tiles when the GEMV would need several K slices
// for them (one launch per slice: measured slower than the split-K tiles, for example
// 4096 x 11008 at M = 16: 28.0 against 20.9 us).  One row always takes the GEMV.
static gq_path choose_path(int kind, int64_t N, int64_t K, int64_t M) {
    {
        std::lock_guard<std::mutex> lock(g_prof_mutex);
        for (const Profile &pr : g_profiles)
            if (pr.kind == kind && pr.N == N && pr.K == K)
                return interpolate(pr.Ms, pr.t_tc, M) < interpolate(pr.Ms, pr.t_gemv, M) ? GQ_PATH_TC : GQ_PATH_GEMV;
    }
    if (M > g_m_threshold.load()) return GQ_PATH_TC;
    if (kind == GQ_KIND_Q4_0 && M > 1 && gemv_q4_0_slices(N, K, M) > 1) return GQ_PATH_TC;
    // F16: the tiles stream fp16 weights into the MMAs with nothing to convert, and measured faster
    // than the GEMV once their grid has enough row tiles (N >= 64 per SM: [11008, 4096] at every M)
    // or once the GEMV's fp16 image of the activations passes 64 KiB ([4096, 11008] from 3 rows,
    // [4096, 4096] from 9)
    if (kind == GQ_KIND_F16 && (N >= 64 * (int64_t)sm_count() || M * K * 2 > 64 * 1024)) return GQ_PATH_TC;
    return GQ_PATH_GEMV;
}

static gq_path resolve(gq_path path, int kind, int64_t M, int64_t N, int64_t K) {
    if (path != GQ_PATH_AUTO) return path;
    return choose_path(kind, N, K, M);
}

gq_status gq_set_dispatch_profile(int kind, int64_t N, int64_t K, const int64_t *Ms, const double *t_gemv,
                                  const double *t_tc, int64_t count) {
    if (kind != GQ_KIND_Q4_0 && kind != GQ_KIND_F16) return fail(GQ_ERR_INVALID_ARG, "unknown weight kind %d", kind);
    if (N <= 0 || K <= 0 || K % QK) return fail(GQ_ERR_INVALID_ARG, "N and K must be positive, K a multiple of 32");
    if (count < 1 || !Ms || !t_gemv || !t_tc) return fail(GQ_ERR_INVALID_ARG, "a profile needs at least one point");
    Profile pr{kind, N, K, {}, {}, {}};
    for (int64_t i = 0; i < count; i++) {
        if (Ms[i] <= 0 || (i > 0 && Ms[i] <= Ms[i - 1]))
            return fail(GQ_ERR_INVALID_ARG, "the M of a profile must be positive and increasing");
        if (!std::isfinite(t_gemv[i]) || !std::isfinite(t_tc[i]) || t_gemv[i] < 0 || t_tc[i] < 0)
            return fail(GQ_ERR_INVALID_ARG, "profile times must be finite and non-negative");
        pr.Ms.push_back(Ms[i]);
        pr.t_gemv.push_back(t_gemv[i]);
        pr.t_tc.push_back(t_tc[i]);
    }
    std::lock_guard<std::mutex> lock(g_prof_mutex);
    for (Profile &old : g_profiles)
        if (old.kind == kind && old.N == N && old.K == K) {
            old = pr;
            return ok();
        }
    g_profiles.push_back(pr);
    return ok();
}

gq_status gq_clear_dispatch_profiles(void) {
    std::lock_guard<std::mutex> lock(g_prof_mutex);
    g_profiles.clear();
    return ok();
}

gq_path gq_choose_path(int kind, int64_t N, int64_t K, int64_t M) { return choose_path(kind, N, K, M); }

gq_status gq_mul_mat_q4_0_f32_path(const void *q4_repacked, const float *src1, float *dst, int64_t M, int64_t N,
                                   int64_t K, gq_path path, cudaStream_t stream) {
    GQ_TRY(check_sizes(M, N, K));
    GQ_TRY(check_path(path));
    GQ_TRY(check_ptr(q4_repacked, "q4_repacked"));
    GQ_TRY(check_ptr(src1, "src1"));
    GQ_TRY(check_ptr(dst, "dst"));
    GQ_TRY(check_device());
    if (resolve(path, GQ_KIND_Q4_0, M, N, K) == GQ_PATH_TC)
        GQ_TRY(launch_tc_q4_0(q4_repacked, src1, dst, M, N, K, stream));
    else
        GQ_TRY(launch_gemv_q4_0(q4_repacked, src1, dst, M, N, K, stream));
    return ok();
}

gq_status gq_mul_mat_f16_f32_path(const void *src0_f16, const float *src1, float *dst, int64_t M, int64_t N,
                                  int64_t K, gq_path path, cudaStream_t stream) {
    GQ_TRY(check_sizes(M, N, K));
    GQ_TRY(check_path(path));
    GQ_TRY(check_ptr(src0_f16, "src0_f16"));
    GQ_TRY(check_ptr(src1, "src1"));
    GQ_TRY(check_ptr(dst, "dst"));
    GQ_TRY(check_device());
    if (resolve(path, GQ_KIND_F16, M, N, K) == GQ_PATH_TC)
        GQ_TRY(launch_tc_f16(src0_f16, src1, dst, M, N, K, stream));
    else
        GQ_TRY(launch_gemv_f16_rowmajor(src0_f16, src1, dst, M, N, K, stream));
    return ok();
}

gq_status gq_mul_mat_q4_0_f32(const void *q4_repacked, const float *src1, float *dst, int64_t M, int64_t N,
                              int64_t K, cudaStream_t stream) {
    return gq_mul_mat_q4_0_f32_path(q4_repacked, src1, dst, M, N, K, GQ_PATH_AUTO, stream);
}

}  // extern "C"

namespace gq {
namespace {
// The device address of page-locked host memory mapped into the device's address space, or
// nullptr (pageable memory, or memory this device cannot address).
void *mapped_host(const void *p) {
    cudaPointerAttributes a{};
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();   // clear the error of an unknown pointer
        return nullptr;
    }
    return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
}
}  // namespace

// Copies n float4 from mapped host memory into device memory, after every earlier grid in the
// stream (the previous product may still read the destination).
__global__ void host_stage_kernel(const float4 *__restrict__ src, float4 *__restrict__ dst, int64_t n) {
    pdl_wait();
    pdl_launch_dependents();
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
        dst[i] = src[i];
}
}  // namespace gq

extern "C" {

gq_status gq_mul_mat_q4_0_f32_host(const void *q4_repacked, const float *src1_host, float *dst_host, int64_t M,
                                   int64_t N, int64_t K, cudaStream_t stream) {
    GQ_TRY(check_sizes(M, N, K));
    GQ_TRY(check_ptr(q4_repacked, "q4_repacked"));
    if (!src1_host) return fail(GQ_ERR_INVALID_ARG, "src1_host is NULL");
    if (!dst_host) return fail(GQ_ERR_INVALID_ARG, "dst_host is NULL");
    GQ_TRY(check_device());
    const size_t xb = (size_t)M * (size_t)K * sizeof(float), ob = (size_t)M * (size_t)N * sizeof(float);
    const size_t xs = (xb + 255) / 256 * 256;
    // Page-locked buffers that the device addresses are read and written by the kernels
    // themselves: a small kernel stages src1 (no copy engine), and the product stores dst into
    // host memory. Other host memory goes through copies on the stream.
    void *hx = mapped_host(src1_host), *hd = mapped_host(dst_host);
    const bool stage_x = hx != nullptr && aligned16(hx), direct_dst = hd != nullptr && aligned16(hd);
    uint8_t *stage = nullptr;
    GQ_TRY(get_staging(stream, xs + (direct_dst ? 0 : ob), &stage));
    float *dx = reinterpret_cast<float *>(stage), *dd = direct_dst ? static_cast<float *>(hd)
                                                                   : reinterpret_cast<float *>(stage + xs);
    if (stage_x) {
        const int64_t n4 = (int64_t)(xb / 16);   // K is a multiple of 32: whole float4
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3((unsigned)std::min<int64_t>((n4 + 255) / 256, 64));
        cfg.blockDim = dim3(256);
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        GQ_TRY(check_cuda(cudaLaunchKernelEx(&cfg, host_stage_kernel, static_cast<const float4 *>(hx),
                                             reinterpret_cast<float4 *>(dx), n4),
                          "src1 staging kernel"));
    } else {
        GQ_TRY(check_cuda(cudaMemcpyAsync(dx, src1_host, xb, cudaMemcpyHostToDevice, stream), "src1 copy to the device"));
    }
    if (resolve(GQ_PATH_AUTO, GQ_KIND_Q4_0, M, N, K) == GQ_PATH_TC)
        GQ_TRY(launch_tc_q4_0(q4_repacked, dx, dd, M, N, K, stream));
    else
        GQ_TRY(launch_gemv_q4_0(q4_repacked, dx, dd, M, N, K, stream));
    if (!direct_dst)
        GQ_TRY(check_cuda(cudaMemcpyAsync(dst_host, dd, ob, cudaMemcpyDeviceToHost, stream), "dst copy to the host"));
    return ok();
}

gq_status gq_mul_mat_f16_f32(const void *src0_f16, const float *src1, float *dst, int64_t M, int64_t N, int64_t K,
                             cudaStream_t stream) {
    return gq_mul_mat_f16_f32_path(src0_f16, src1, dst, M, N, K, GQ_PATH_AUTO, stream);
}

size_t gq_q4_1_bytes(int64_t N, int64_t K) {
    if (N <= 0 || K <= 0 || K % QK) return 0;
    return (size_t)N * (size_t)(K / QK) * 20;
}

size_t gq_q4_1_repacked_bytes(int64_t N, int64_t K) {
    if (N <= 0 || K <= 0 || K % QK) return 0;
    return (size_t)((N + 15) / 16) * (size_t)((K / QK + TILE_BLOCKS - 1) / TILE_BLOCKS) * 1280;
}

gq_status gq_quantize_q4_1(const float *w, void *q41_blocks, int64_t N, int64_t K, cudaStream_t stream) {
    GQ_TRY(check_sizes(1, N, K));
    GQ_TRY(check_ptr(w, "w"));
    GQ_TRY(check_ptr(q41_blocks, "q41_blocks"));
    GQ_TRY(check_device());
    GQ_TRY(launch_quantize_q4_1(w, q41_blocks, N, K, stream));
    return ok();
}

gq_status gq_repack_q4_1(const void *q41_blocks, void *q41_repacked, int64_t N, int64_t K, cudaStream_t stream) {
    GQ_TRY(check_sizes(1, N, K));
    GQ_TRY(check_ptr(q41_blocks, "q41_blocks"));
    GQ_TRY(check_ptr(q41_repacked, "q41_repacked"));
    const uintptr_t a = (uintptr_t)q41_blocks, b = (uintptr_t)q41_repacked;
    if (a < b + gq_q4_1_repacked_bytes(N, K) && b < a + gq_q4_1_bytes(N, K))
        return fail(GQ_ERR_INVALID_ARG, "q41_blocks and q41_repacked overlap");
    GQ_TRY(check_device());
    GQ_TRY(launch_repack_q4_1(q41_blocks, q41_repacked, N, K, stream));
    return ok();
}

gq_status gq_mul_mat_q4_1_f32(const void *q41_repacked, const float *src1, float *dst, int64_t M, int64_t N,
                              int64_t K, cudaStream_t stream) {
    GQ_TRY(check_sizes(M, N, K));
    GQ_TRY(check_ptr(q41_repacked, "q41_repacked"));
    GQ_TRY(check_ptr(src1, "src1"));
    GQ_TRY(check_ptr(dst, "dst"));
    GQ_TRY(check_device());
    GQ_TRY(launch_gemv_q4_1(q41_repacked, src1, dst, M, N, K, stream));
    return ok();
}

size_t gq_q5_0_bytes(int64_t N, int64_t K) {
    if (N <= 0 || K <= 0 || K % QK) return 0;
    return (size_t)N * (size_t)(K / QK) * 22;
}

size_t gq_q5_0_repacked_bytes(int64_t N, int64_t K) {
    if (N <= 0 || K <= 0 || K % QK) return 0;
    return (size_t)((N + 15) / 16) * (size_t)((K / QK + TILE_BLOCKS - 1) / TILE_BLOCKS) * 1408;
}

gq_status gq_quantize_q5_0(const float *w, void *q5_blocks, int64_t N, int64_t K, cudaStream_t stream) {
    GQ_TRY(check_sizes(1, N, K));
    GQ_TRY(check_ptr(w, "w"));
    GQ_TRY(check_ptr(q5_blocks, "q5_blocks"));
    GQ_TRY(check_device());
    GQ_TRY(launch_quantize_q5_0(w, q5_blocks, N, K, stream));
    return ok();
}

gq_status gq_repack_q5_0(const void *q5_blocks, void *q5_repacked, int64_t N, int64_t K, cudaStream_t stream) {
    GQ_TRY(check_sizes(1, N, K));
    GQ_TRY(check_ptr(q5_blocks, "q5_blocks"));
    GQ_TRY(check_ptr(q5_repacked, "q5_repacked"));
    const uintptr_t a = (uintptr_t)q5_blocks, b = (uintptr_t)q5_repacked;
    if (a < b + gq_q5_0_repacked_bytes(N, K) && b < a + gq_q5_0_bytes(N, K))
        return fail(GQ_ERR_INVALID_ARG, "q5_blocks and q5_repacked overlap");
    GQ_TRY(check_device());
    GQ_TRY(launch_repack_q5_0(q5_blocks, q5_repacked, N, K, stream));
    return ok();
}

gq_status gq_mul_mat_q5_0_f32(const void *q5_repacked, const float *src1, float *dst, int64_t M, int64_t N,
                              int64_t K, cudaStream_t stream) {
    GQ_TRY(check_sizes(M, N, K));
    GQ_TRY(check_ptr(q5_repacked, "q5_repacked"));
    GQ_TRY(check_ptr(src1, "src1"));
    GQ_TRY(check_ptr(dst, "dst"));
    GQ_TRY(check_device());
    GQ_TRY(launch_gemv_q5_0(q5_repacked, src1, dst, M, N, K, stream));
    return ok();
}

size_t gq_q8_0_repacked_bytes(int64_t N, int64_t K) {
    if (N <= 0 || K <= 0 || K % QK) return 0;
    return (size_t)((N + 15) / 16) * (size_t)((K / QK + TILE_BLOCKS - 1) / TILE_BLOCKS) * 2176;
}

gq_status gq_repack_q8_0(const void *q8_blocks, void *q8_repacked, int64_t N, int64_t K, cudaStream_t stream) {
    GQ_TRY(check_sizes(1, N, K));
    GQ_TRY(check_ptr(q8_blocks, "q8_blocks"));
    GQ_TRY(check_ptr(q8_repacked, "q8_repacked"));
    const uintptr_t a = (uintptr_t)q8_blocks, b = (uintptr_t)q8_repacked;
    if (a < b + gq_q8_0_repacked_bytes(N, K) && b < a + gq_q8_0_bytes(N, K))
        return fail(GQ_ERR_INVALID_ARG, "q8_blocks and q8_repacked overlap");
    GQ_TRY(check_device());
    GQ_TRY(launch_repack_q8_0(q8_blocks, q8_repacked, N, K, stream));
    return ok();
}

gq_status gq_mul_mat_q8_0_f32(const void *q8_repacked, const float *src1, float *dst, int64_t M, int64_t N,
                              int64_t K, cudaStream_t stream) {
    GQ_TRY(check_sizes(M, N, K));
    GQ_TRY(check_ptr(q8_repacked, "q8_repacked"));
    GQ_TRY(check_ptr(src1, "src1"));
    GQ_TRY(check_ptr(dst, "dst"));
    GQ_TRY(check_device());
    GQ_TRY(launch_gemv_q8_0(q8_repacked, src1, dst, M, N, K, stream));
    return ok();
}

size_t gq_f16_repacked_bytes(int64_t N, int64_t K) {
    if (N <= 0 || K <= 0 || K % QK) return 0;
    return (size_t)((N + 15) / 16) * (size_t)(K / 32) * 1024;
}

gq_status gq_repack_f16(const void *src0_f16, void *f16_repacked, int64_t N, int64_t K, cudaStream_t stream) {
    GQ_TRY(check_sizes(1, N, K));
    GQ_TRY(check_ptr(src0_f16, "src0_f16"));
    GQ_TRY(check_ptr(f16_repacked, "f16_repacked"));
    const uintptr_t a = (uintptr_t)src0_f16, b = (uintptr_t)f16_repacked;
    if (a < b + gq_f16_repacked_bytes(N, K) && b < a + (size_t)N * (size_t)K * 2)
        return fail(GQ_ERR_INVALID_ARG, "src0_f16 and f16_repacked overlap");
    GQ_TRY(check_device());
    GQ_TRY(launch_repack_f16(src0_f16, f16_repacked, N, K, stream));
    return ok();
}

gq_status gq_mul_mat_f16r_f32(const void *f16_repacked, const float *src1, float *dst, int64_t M, int64_t N,
                              int64_t K, cudaStream_t stream) {
    GQ_TRY(check_sizes(M, N, K));
    GQ_TRY(check_ptr(f16_repacked, "f16_repacked"));
    GQ_TRY(check_ptr(src1, "src1"));
    GQ_TRY(check_ptr(dst, "dst"));
    GQ_TRY(check_device());
    GQ_TRY(launch_gemv_f16r(f16_repacked, src1, dst, M, N, K, stream));
    return ok();
}

gq_status gq_debug_block_dots_q4_0(const void *q4_repacked, const void *q8_blocks, int32_t *sumi, int64_t M,
                                   int64_t N, int64_t K, cudaStream_t stream) {
    GQ_TRY(check_sizes(M, N, K));
    GQ_TRY(check_ptr(q4_repacked, "q4_repacked"));
    GQ_TRY(check_ptr(q8_blocks, "q8_blocks"));
    GQ_TRY(check_ptr(sumi, "sumi"));
    GQ_TRY(check_device());
    GQ_TRY(launch_block_dots_q4_0(q4_repacked, q8_blocks, sumi, M, N, K, stream));
    return ok();
}

}  // extern "C"

// ---- the wait-timeout probe (verification) --------------------------------------------

namespace gq {
// One warp waits, with the given poll limit, on an mbarrier that nothing arrives on and
// no copy signals: phase 0 never completes, so every wait gives up, records the timeout
// in the device status word and returns; the kernel then invalidates the barrier and ends.
__global__ void wait_probe_kernel(unsigned int *status, uint32_t limit) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(smem_addr(&bar), 1);
        fence_barrier_init();
    }
    __syncthreads();
    mbar_wait(smem_addr(&bar), 0u, status, limit);
    __syncthreads();
    if (threadIdx.x == 0) asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(smem_addr(&bar)) : "memory");
}
}  // namespace gq

namespace gq {
// dp4a throughput probe: every thread runs `iters` rounds of 8 independent dp4a chains and
// stores one sum (so that nothing is optimized away).  8 * iters dp4a per thread.
__global__ void dp4a_probe_kernel(int64_t iters, int *sink) {
    int a[8];
    const int x = (int)threadIdx.x * 0x01010101, y = (int)blockIdx.x | 0x03050709;
#pragma unroll
    for (int j = 0; j < 8; j++) a[j] = j;
    for (int64_t i = 0; i < iters; i++) {
#pragma unroll
        for (int j = 0; j < 8; j++) a[j] = __dp4a(x + j, y, a[j]);
    }
    int t = 0;
#pragma unroll
    for (int j = 0; j < 8; j++) t += a[j];
    sink[(size_t)blockIdx.x * blockDim.x + threadIdx.x] = t;
}
}  // namespace gq

extern "C" gq_status gq_debug_dp4a_probe(int64_t iters, int *sink, int64_t blocks, cudaStream_t stream) {
    if (iters <= 0 || blocks <= 0 || blocks > (1LL << 20))
        return fail(GQ_ERR_INVALID_ARG, "iters and blocks must be positive (blocks <= 2^20)");
    GQ_TRY(check_ptr(sink, "sink"));
    GQ_TRY(check_device());
    dp4a_probe_kernel<<<(unsigned)blocks, 256, 0, stream>>>(iters, sink);
    GQ_TRY(check_cuda(cudaGetLastError(), "dp4a probe launch"));
    return ok();
}

extern "C" gq_status gq_debug_wait_timeout(uint32_t limit, cudaStream_t stream) {
    if (limit == 0 || limit > WAIT_LIMIT)
        return fail(GQ_ERR_INVALID_ARG, "limit must be in [1, %u] (got %u)", WAIT_LIMIT, limit);
    GQ_TRY(check_device());
    unsigned int *status = device_status_word();
    if (!status) return fail(GQ_ERR_CUDA, "device status word unavailable");
    wait_probe_kernel<<<1, 32, 0, stream>>>(status, limit);
    GQ_TRY(check_cuda(cudaGetLastError(), "wait probe launch"));
    return ok();
}

// ---- INT8 KV cache ------------------------------------------------------------------

namespace {
gq_status check_kv(int64_t B, int64_t Hkv, int64_t Tcap, int64_t D) {
    if (B <= 0 || Hkv <= 0 || Tcap <= 0)
        return fail(GQ_ERR_INVALID_ARG, "sizes must be positive (B=%lld Hkv=%lld Tcap=%lld)", (long long)B,
                    (long long)Hkv, (long long)Tcap);
    if (D != 64 && D != 128) return fail(GQ_ERR_INVALID_ARG, "head size D must be 64 or 128 (got %lld)", (long long)D);
    if (Tcap >= (1LL << 30) || B >= (1LL << 30) || Hkv >= (1LL << 30) || B * Hkv >= (1LL << 31) ||
        (double)B * (double)Hkv * (double)Tcap * (double)D >= 1099511627776.0)
        return fail(GQ_ERR_INVALID_ARG, "sizes too large (B=%lld Hkv=%lld Tcap=%lld D=%lld)", (long long)B,
                    (long long)Hkv, (long long)Tcap, (long long)D);
    return GQ_OK;
}
}  // namespace

extern "C" {

gq_status gq_kv_quantize_i8(const float *x, int8_t *q, float *scale, int64_t rows, int64_t D, cudaStream_t stream) {
    if (rows <= 0 || rows >= (1LL << 34))
        return fail(GQ_ERR_INVALID_ARG, "rows must be in [1, 2^34) (got %lld)", (long long)rows);
    GQ_TRY(check_kv(1, 1, 1, D));
    GQ_TRY(check_ptr(x, "x"));
    GQ_TRY(check_ptr(q, "q"));
    GQ_TRY(check_ptr(scale, "scale"));
    GQ_TRY(check_device());
    GQ_TRY(launch_kv_quantize_i8(x, q, scale, rows, D, stream));
    return ok();
}

gq_status gq_kv_append_i8(const float *x, int8_t *q, float *scale, const int32_t *pos, int64_t B, int64_t Hkv,
                          int64_t Tcap, int64_t D, cudaStream_t stream) {
    GQ_TRY(check_kv(B, Hkv, Tcap, D));
    GQ_TRY(check_ptr(x, "x"));
    GQ_TRY(check_ptr(q, "q"));
    GQ_TRY(check_ptr(scale, "scale"));
    GQ_TRY(check_ptr(pos, "pos"));
    GQ_TRY(check_device());
    GQ_TRY(launch_kv_append_i8(x, q, scale, pos, B, Hkv, Tcap, D, stream));
    return ok();
}

gq_status gq_attn_decode_i8(const float *q, const int8_t *k, const float *k_scale, const int8_t *v,
                            const float *v_scale, const int32_t *lens, float *out, int64_t B, int64_t Hq,
                            int64_t Hkv, int64_t Tcap, int64_t D, float softmax_scale, cudaStream_t stream) {
    GQ_TRY(check_kv(B, Hkv, Tcap, D));
    if (Hq <= 0 || Hq % Hkv != 0)
        return fail(GQ_ERR_INVALID_ARG, "Hq=%lld is not a positive multiple of Hkv=%lld", (long long)Hq,
                    (long long)Hkv);
    const int64_t G = Hq / Hkv;
    if (D == 128 ? (G < 1 || G > 8) : (G != 1 && G != 2 && G != 4 && G != 8))
        return fail(GQ_ERR_INVALID_ARG, "query heads per KV head must be 1 .. 8 (D = 128) or 1, 2, 4, 8 (D = 64); got %lld",
                    (long long)G);
    if (!std::isfinite(softmax_scale)) return fail(GQ_ERR_INVALID_ARG, "softmax_scale is not finite");
    GQ_TRY(check_ptr(q, "q"));
    GQ_TRY(check_ptr(k, "k"));
    GQ_TRY(check_ptr(k_scale, "k_scale"));
    GQ_TRY(check_ptr(v, "v"));
    GQ_TRY(check_ptr(v_scale, "v_scale"));
    GQ_TRY(check_ptr(lens, "lens"));
    GQ_TRY(check_ptr(out, "out"));
    GQ_TRY(check_device());
    GQ_TRY(launch_attn_decode_i8(q, k, k_scale, v, v_scale, lens, out, B, Hq, Hkv, Tcap, D, softmax_scale, stream));
    return ok();
}

}  // extern "C"
