// block_dots.cu -- the integer block dots of the Q4_0 GEMV, for parity tests: the
// same nibble unpack and dp4a sequence as the product's dp4a path, one thread per
// (activation row, weight row, block), so that every exact int32 block dot the
// product forms can be compared with the oracle's.
#include "gq_common.cuh"
#include "gq_internal.h"

namespace gq {
namespace {

__global__ void block_dots_q4_0_kernel(const uint8_t *__restrict__ w, const uint8_t *__restrict__ q8,
                                       int32_t *__restrict__ sumi, int M, int N, int nb, int NT) {
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= (int64_t)M * N * nb) return;
    const int b = (int)(idx % nb);
    const int64_t rest = idx / nb;
    const int n = (int)(rest % N), m = (int)(rest / N);
    const uint8_t *tile = w + ((size_t)(n / 16) * NT + b / 4) * TILE_BYTES;
    const uint4 q = *reinterpret_cast<const uint4 *>(tile + ((b % 4) * 16 + n % 16) * 16);
    const uint16_t *codes = reinterpret_cast<const uint16_t *>(q8 + ((size_t)m * nb + b) * Q8_0_BYTES + 2);
    uint32_t a[8];
    int qsum = 0;
    for (int k = 0; k < 8; k++) {
        a[k] = (uint32_t)codes[2 * k] | ((uint32_t)codes[2 * k + 1] << 16);
        for (int e = 0; e < 4; e++) qsum += (int)(int8_t)(a[k] >> (8 * e));
    }
    sumi[idx] = block_dot(q, make_uint4(a[0], a[1], a[2], a[3]), make_uint4(a[4], a[5], a[6], a[7]), -8 * qsum);
}

}  // namespace

gq_status launch_block_dots_q4_0(const void *rep, const void *q8, int32_t *sumi, int64_t M, int64_t N,
                                 int64_t K, cudaStream_t s) {
    const int64_t nb = K / QK, NT = (K + TILE_COLS - 1) / TILE_COLS;
    const int64_t total = M * N * nb;
    block_dots_q4_0_kernel<<<(unsigned)((total + 255) / 256), 256, 0, s>>>(
        (const uint8_t *)rep, (const uint8_t *)q8, sumi, (int)M, (int)N, (int)nb, (int)NT);
    return check_cuda(cudaGetLastError(), "block_dots_q4_0 launch");
}

}  // namespace gq
