// noalloc.cu -- the Q4_0 product for callers that cannot allocate device memory.
//
// gq_mul_mat_q4_0_f32 takes its scratch space (per-row counters, partial sums,
// quantized activations) from a per-stream workspace that the library obtains
// with cudaMalloc the first time a stream needs it.  Some callers cannot let a
// library call cudaMalloc: serving processes whose pooling allocator reserved
// the device memory up front and must account for every byte, plug-ins hosted
// by a runtime that forbids them to allocate, and latency-bound loops in which
// cudaMalloc (which can synchronize the device) may not run.  This entry point
// gives them the same product with all of its scratch space in one statically
// sized device array that is part of the loaded library, so nothing is
// allocated, ever.
#include <mutex>

#include "gq_common.cuh"
#include "gq_internal.h"

namespace gq {
namespace {

// Upper bound of the scratch this entry point may use.  Every device that loads
// the library holds this array until the process exits.
constexpr size_t NOALLOC_SCRATCH_BYTES = 4u << 20;

static __device__ __align__(256) uint8_t g_noalloc_scratch[NOALLOC_SCRATCH_BYTES];

constexpr int MAX_DEVICES = 64;
std::mutex g_mutex;
uint8_t *g_scratch_addr[MAX_DEVICES];

// In host code the array's name only stands for the device variable; kernels
// need its device address, which is resolved once per device with that device
// current.
gq_status scratch_address(uint8_t **out) {
    int dev = 0;
    gq_status st = check_cuda(cudaGetDevice(&dev), "cudaGetDevice");
    if (st != GQ_OK) return st;
    if (dev < 0 || dev >= MAX_DEVICES) return fail(GQ_ERR_UNSUPPORTED_DEVICE, "device index %d", dev);
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_scratch_addr[dev] == nullptr) {
        void *p = nullptr;
        st = check_cuda(cudaGetSymbolAddress(&p, g_noalloc_scratch), "cudaGetSymbolAddress (no-alloc scratch)");
        if (st != GQ_OK) return st;
        g_scratch_addr[dev] = static_cast<uint8_t *>(p);
    }
    *out = g_scratch_addr[dev];
    return GQ_OK;
}

size_t align256(size_t v) { return (v + 255) / 256 * 256; }

}  // namespace
}  // namespace gq

using namespace gq;

extern "C" gq_status gq_mul_mat_q4_0_f32_noalloc(const void *q4_repacked, const float *src1, float *dst,
                                                 int64_t M, int64_t N, int64_t K, cudaStream_t stream) {
    gq_status st = check_sizes(M, N, K);
    if (st != GQ_OK) return st;
    if ((st = check_ptr(q4_repacked, "q4_repacked")) != GQ_OK) return st;
    if ((st = check_ptr(src1, "src1")) != GQ_OK) return st;
    if ((st = check_ptr(dst, "dst")) != GQ_OK) return st;
    size_t counter_bytes = 0, data_bytes = 0;
    gemv_q4_0_workspace(N, K, &counter_bytes, &data_bytes);
    const size_t need = align256(counter_bytes) + data_bytes;
    if (need > NOALLOC_SCRATCH_BYTES)
        return fail(GQ_ERR_INVALID_ARG,
                    "N=%lld K=%lld needs %zu bytes of scratch; the allocation-free entry point has %zu",
                    (long long)N, (long long)K, need, NOALLOC_SCRATCH_BYTES);
    if ((st = check_device()) != GQ_OK) return st;
    uint8_t *base = nullptr;
    if ((st = scratch_address(&base)) != GQ_OK) return st;
    // the array keeps whatever the last call left: the row counters must start at zero
    st = check_cuda(cudaMemsetAsync(base, 0, align256(counter_bytes), stream), "no-alloc counter reset");
    if (st != GQ_OK) return st;
    Workspace ws;
    ws.counters = base;
    ws.data = base + align256(counter_bytes);
    st = launch_gemv_q4_0_with(q4_repacked, src1, dst, M, N, K, ws, stream);
    if (st != GQ_OK) return st;
    return ok();
}
