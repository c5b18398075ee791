// workspace.cu -- device workspace of the product kernels, one per (device, stream).
//
// The persistent GEMV adds partial sums of row groups that two CTAs share
// through a small global buffer and a per-row-group arrival counter; the
// tensor-core path stages its quantized activations there.  Counters start at
// zero and every launch leaves them at zero again, so the buffer is reused as it
// is.  A stream's workspace grows on demand: growth allocates a new buffer
// (cudaMalloc), zeroes its counters and synchronizes that stream, so it must not
// happen while the stream is being captured into a graph; gq_reserve_workspace
// lets a caller size it beforehand.  A growth that fails leaves the current
// buffer in use.  A replaced buffer is retired, not freed: another host thread may
// have taken its address for a launch on the same stream just before the growth,
// and that launch (or a CUDA graph captured with the old address) must still find
// valid memory.  Each growth at least doubles the data part, so the retired
// buffers of a stream hold less than its current one.
#include <mutex>
#include <vector>

#include "gq_common.cuh"
#include "gq_internal.h"

namespace gq {
namespace {

struct Entry {
    int device;
    cudaStream_t stream;
    uint8_t *ptr;
    size_t counter_bytes;   // zeroed prefix
    size_t bytes;           // total
};

std::mutex g_mutex;
std::vector<Entry> g_entries;
std::vector<uint8_t *> g_retired;   // replaced buffers, kept until the process exits

}  // namespace

gq_status get_workspace(cudaStream_t stream, size_t counter_bytes, size_t data_bytes, Workspace *out) {
    counter_bytes = (counter_bytes + 255) / 256 * 256;
    data_bytes = (data_bytes + 255) / 256 * 256;
    int dev = 0;
    gq_status st = check_cuda(cudaGetDevice(&dev), "cudaGetDevice");
    if (st != GQ_OK) return st;
    std::lock_guard<std::mutex> lock(g_mutex);
    Entry *e = nullptr;
    for (auto &x : g_entries)
        if (x.device == dev && x.stream == stream) e = &x;
    if (e && e->counter_bytes >= counter_bytes && e->bytes - e->counter_bytes >= data_bytes) {
        out->counters = e->ptr;
        out->data = e->ptr + e->counter_bytes;
        return GQ_OK;
    }
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    st = check_cuda(cudaStreamIsCapturing(stream, &cap), "cudaStreamIsCapturing");
    if (st != GQ_OK) return st;
    if (cap != cudaStreamCaptureStatusNone)
        return fail(GQ_ERR_NO_MEMORY,
                    "the stream's workspace must grow (%zu + %zu bytes) while the stream is being captured; "
                    "call gq_reserve_workspace before capturing", counter_bytes, data_bytes);
    size_t cb = counter_bytes, db = data_bytes;
    if (e) {
        cb = std::max(cb, e->counter_bytes);
        db = std::max(db, 2 * (e->bytes - e->counter_bytes));   // at least double (see above)
    }
    // The new buffer is allocated and its counters zeroed first; the entry changes only once
    // both succeeded, so a failed growth leaves the stream's current workspace in place.
    uint8_t *p = nullptr;
    if (cudaMalloc(&p, cb + db) != cudaSuccess) {
        cudaGetLastError();
        return fail(GQ_ERR_NO_MEMORY, "cudaMalloc of a %zu-byte workspace failed", cb + db);
    }
    st = check_cuda(cudaMemsetAsync(p, 0, cb, stream), "workspace counter reset");
    if (st == GQ_OK && e) st = check_cuda(cudaStreamSynchronize(stream), "cudaStreamSynchronize (workspace growth)");
    if (st != GQ_OK) {
        cudaFree(p);
        return st;
    }
    if (e) {
        g_retired.push_back(e->ptr);
    } else {
        g_entries.push_back(Entry{dev, stream, nullptr, 0, 0});
        e = &g_entries.back();
    }
    e->ptr = p;
    e->counter_bytes = cb;
    e->bytes = cb + db;
    out->counters = p;
    out->data = p + cb;
    return GQ_OK;
}

// Staging buffers of the host-pointer entry points (src1 and dst on the device), one
// per (device, stream), grown like the workspace.
namespace {
struct Staging {
    int device;
    cudaStream_t stream;
    uint8_t *ptr;
    size_t bytes;
};
std::vector<Staging> g_staging;
}  // namespace

gq_status get_staging(cudaStream_t stream, size_t bytes, uint8_t **out) {
    bytes = (bytes + 255) / 256 * 256;
    int dev = 0;
    gq_status st = check_cuda(cudaGetDevice(&dev), "cudaGetDevice");
    if (st != GQ_OK) return st;
    std::lock_guard<std::mutex> lock(g_mutex);
    Staging *e = nullptr;
    for (auto &x : g_staging)
        if (x.device == dev && x.stream == stream) e = &x;
    if (e && e->bytes >= bytes) {
        *out = e->ptr;
        return GQ_OK;
    }
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    st = check_cuda(cudaStreamIsCapturing(stream, &cap), "cudaStreamIsCapturing");
    if (st != GQ_OK) return st;
    if (cap != cudaStreamCaptureStatusNone)
        return fail(GQ_ERR_NO_MEMORY, "the stream's staging buffer must grow (%zu bytes) while the stream is "
                    "being captured", bytes);
    if (e) {
        bytes = std::max(bytes, 2 * e->bytes);   // at least double, as for the workspace
        st = check_cuda(cudaStreamSynchronize(stream), "cudaStreamSynchronize (staging growth)");
        if (st != GQ_OK) return st;
        g_retired.push_back(e->ptr);   // as for the workspace: a concurrent launch may still use it
        e->ptr = nullptr;
        e->bytes = 0;
    }
    uint8_t *p = nullptr;
    if (cudaMalloc(&p, bytes) != cudaSuccess) {
        cudaGetLastError();
        return fail(GQ_ERR_NO_MEMORY, "cudaMalloc of a %zu-byte staging buffer failed", bytes);
    }
    if (!e) {
        g_staging.push_back(Staging{dev, stream, nullptr, 0});
        e = &g_staging.back();
    }
    e->ptr = p;
    e->bytes = bytes;
    *out = p;
    return GQ_OK;
}

// Zeroes the counters of every workspace of the current device (after a kernel
// gave up a wait, counters may be left mid-count).
gq_status reset_workspace_counters() {
    int dev = 0;
    gq_status st = check_cuda(cudaGetDevice(&dev), "cudaGetDevice");
    if (st != GQ_OK) return st;
    std::lock_guard<std::mutex> lock(g_mutex);
    for (auto &x : g_entries)
        if (x.device == dev && x.ptr) {
            st = check_cuda(cudaMemset(x.ptr, 0, x.counter_bytes), "workspace counter reset");
            if (st != GQ_OK) return st;
        }
    return GQ_OK;
}

}  // namespace gq
