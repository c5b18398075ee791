// kv_attn.cu -- the INT8 KV cache and the decode attention that reads it.
//
// xFasterTransformer (arXiv 2407.07304), "2.2 Effective KV cache Optimization":
// after the first token, attention over the cache is a pair of GEMVs bound by
// memory bandwidth; the cache is stored as INT8 with one scale for each token and
// each head, and the INT8 operand is widened to FP32 before the multiply-add.
// Section "2.1 LLM Optimization" (SlimAttention) gives the order for one query
// row: the whole row of scores, then the softmax over it, then its product with
// the values.  The scale's formula is not given; it is read like Q8_0's:
// s = amax / 127 (f32, kept as f32), q = roundf(x / s) (IEEE division).
//
// Layouts: codes int8 [B][Hkv][Tcap][D] (a head's tokens are contiguous, so one
// (sequence, head) pair streams as one run of bytes), scales f32 [B][Hkv][Tcap],
// queries f32 [B][Hq][D] with Hq = G * Hkv (query head h reads KV head h / G),
// lens int32 [B], output f32 [B][Hq][D].
//
// The decode kernel takes one (sequence, KV head, token range) per CTA.  A
// producer warp streams the range's K rows and then its V rows through a ring of
// shared-memory slots with bulk copies (the cache is read once: L2 evict-first);
// the consumer warps take whole slots in turn:
//   scores  each lane widens 16 int8 of a token to f32 (a byte placed in the
//           mantissa of 2^23 and the offset subtracted: exact, no conversion
//           instruction), multiplies them with the matching query values in
//           packed f32x2 FMAs, and the lanes of a token add their partials; the
//           score, times the token's scale and the softmax scale in base-2
//           units, goes to a shared-memory row of scores;
//   softmax the consumer warps take the row's maximum, replace each score by
//           exp2(score - max) times the token's value scale, and add the
//           exponentials (the denominator), in a fixed order;
//   values  each lane widens 16 (8 when G = 8) int8 of a token's value row and
//           accumulates weight x value into registers; lanes and then warps are
//           added in a fixed order and divided by the denominator.
// A range longer than the shared-memory row of scores holds, or a grid too small
// to fill the GPU, splits a sequence's tokens over several CTAs; each writes its
// unnormalised output with its maximum and denominator, and a second kernel merges
// the parts in order.  Every result is deterministic.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cuda.h>
#include <cuda_runtime.h>

#include "gq_common.cuh"
#include "gq_internal.h"

namespace gq {
namespace {

// The ring and the consumer warps.  With one or two query heads per KV head a consumer
// does little arithmetic per byte, so eight consumer warps on 4 KB slots keep enough
// bytes in flight; with four or eight, four warps (their registers hold G accumulators)
// on 8 KB slots.  SLOTS is a multiple of W: the warp that takes a slot's chunk also
// takes the next chunk in that slot.
template <int G>
struct AtCfg {
    static constexpr int W = G <= 2 ? 8 : 4;                 // consumer warps
    static constexpr int CHUNK = G <= 2 ? 4096 : 8192;       // bytes per ring slot
    static constexpr int SLOTS = G <= 2 ? 16 : 8;
    static constexpr int THREADS = (W + 1) * 32;
    static constexpr int CONSUMERS = W * 32;
};
constexpr size_t AT_SMEM_MAX = 113 * 1024;     // two CTAs per SM
constexpr float LOG2E = 1.4426950408889634f;
constexpr uint32_t MAGIC = 0x4B000000u;        // 2^23 as f32 bits
constexpr float MAGIC_OFFSET = 8388736.0f;     // 2^23 + 128

#define KV_TRY(expr)                  \
    do {                              \
        gq_status _st = (expr);       \
        if (_st != GQ_OK) return _st; \
    } while (0)

struct AttnParams {
    const float *q;
    const int8_t *k, *v;
    const float *ks, *vs;
    const int32_t *lens;
    float *out;
    float *part;                // [B][Hq][S][D + 2] when S > 1
    unsigned int *status;
    int Hkv, Tcap, S, TR;
    float c2;                   // softmax scale times log2(e)
};

struct AttnLayout {
    size_t bars, qs, ring, ksc, vsc, sc, wred, total;
};

template <int D, int G>
__host__ __device__ constexpr size_t attn_fixed_bytes() {
    using C = AtCfg<G>;
    return 256 + (size_t)G * D * 4 + (size_t)C::SLOTS * C::CHUNK + 2 * C::W * G * 4 + 128;
}

template <int D, int G>
__host__ __device__ AttnLayout attn_layout(int TR) {
    using C = AtCfg<G>;
    AttnLayout L{};
    L.bars = 0;                                          // full[SLOTS], empty[SLOTS]
    L.qs = 256;                                          // the G query rows, f32
    L.ring = L.qs + (size_t)G * D * 4;                   // 128-byte aligned (D * 4 is)
    L.ksc = L.ring + (size_t)C::SLOTS * C::CHUNK;        // key scale x c2, per token
    L.vsc = L.ksc + (size_t)TR * 4;                      // value scale, per token
    L.sc = L.vsc + (size_t)TR * 4;                       // scores [TR][G]
    L.wred = L.sc + (size_t)TR * G * 4;                  // per-warp maxima and sums [2][W][G]
    L.total = L.wred + 2 * C::W * G * 4;
    return L;
}

// Shared-memory accesses with the state space explicit (a generic access to shared memory
// costs an address-space check and waits on the long scoreboard).
__device__ __forceinline__ uint4 sh_ld128(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
    return v;
}
__device__ __forceinline__ uint2 sh_ld64(uint32_t a) {
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
    return v;
}
__device__ __forceinline__ float sh_ldf(uint32_t a) {
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ void sh_stf(uint32_t a, float v) {
    asm volatile("st.shared.f32 [%0], %1;" ::"r"(a), "f"(v) : "memory");
}

template <int N>
__device__ __forceinline__ void consumer_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ uint64_t pack2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void unpack2(uint64_t r, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(r));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// The four int8 of a word as f32 pairs (bytes 0, 1) and (2, 3).  With u = k + 128 the
// biased byte, the f32 whose bits are 0x4B0000uu is 2^23 + u exactly, and subtracting
// 2^23 + 128 is exact too.
__device__ __forceinline__ void widen4(uint32_t w, uint64_t &p01, uint64_t &p23) {
    const uint32_t u = w ^ 0x80808080u;
    const uint64_t off = pack2(-MAGIC_OFFSET, -MAGIC_OFFSET);
    // result bytes, low to high: byte i of u, then bytes 0, 1 and 3 of MAGIC (0x00, 0x00, 0x4B)
    p01 = add2(pack2(__uint_as_float(__byte_perm(u, MAGIC, 0x7540)), __uint_as_float(__byte_perm(u, MAGIC, 0x7541))), off);
    p23 = add2(pack2(__uint_as_float(__byte_perm(u, MAGIC, 0x7542)), __uint_as_float(__byte_perm(u, MAGIC, 0x7543))), off);
}

// Sums v[0..HG) over the LPT lanes of a token (xor masks LPT/2 .. 1).  While a lane
// holds more than one head, each exchange halves them: the lane with the mask bit set
// keeps the upper half.  On return v[0] is the full sum of head (lane % LPT) / (LPT / HG).
template <int HG, int LPT>
__device__ __forceinline__ float reduce_heads(float (&v)[HG], int lane) {
    static_assert(HG <= LPT, "more heads than lanes per token");
    int nh = HG;
#pragma unroll
    for (int m = LPT / 2; m >= 1; m >>= 1) {
        if (nh > 1) {
            const int half = nh / 2;
            const bool up = (lane & m) != 0;
#pragma unroll
            for (int i = 0; i < HG / 2; i++) {
                if (i < half) {
                    const float send = up ? v[i] : v[i + half];
                    const float keep = up ? v[i + half] : v[i];
                    v[i] = keep + __shfl_xor_sync(0xffffffffu, send, m);
                }
            }
            nh = half;
        } else {
            v[0] += __shfl_xor_sync(0xffffffffu, v[0], m);
        }
    }
    return v[0];
}

template <int D, int G>
__global__ void __launch_bounds__(AtCfg<G>::THREADS, 2) attn_decode_i8_kernel(const AttnParams p) {
    constexpr int W = AtCfg<G>::W, SLOTS = AtCfg<G>::SLOTS, CHUNK = AtCfg<G>::CHUNK;
    constexpr int THREADS = AtCfg<G>::THREADS, CONSUMERS = AtCfg<G>::CONSUMERS;
    constexpr int CT = CHUNK / D;          // tokens per slot
    constexpr int LPT = D / 16;            // score phase: lanes per token, 16 bytes each
    constexpr int TPW = 32 / LPT;          // tokens per warp step
    constexpr int HG = G < 4 ? G : 4;      // heads per pass of the score phase
    constexpr int VB = G >= 8 ? 8 : 16;    // value phase: bytes per lane
    constexpr int LPV = D / VB;
    constexpr int TPV = 32 / LPV;
    static_assert(D % 16 == 0 && 32 % LPT == 0 && 32 % LPV == 0, "head size");

    extern __shared__ __align__(128) uint8_t smem[];
    const AttnLayout L = attn_layout<D, G>(p.TR);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.bars);
    uint64_t *empty = full + SLOTS;
    float *qs = reinterpret_cast<float *>(smem + L.qs);
    float *ksc = reinterpret_cast<float *>(smem + L.ksc);
    float *vsc = reinterpret_cast<float *>(smem + L.vsc);
    float *sc = reinterpret_cast<float *>(smem + L.sc);
    float *wmax = reinterpret_cast<float *>(smem + L.wred);
    float *wsum = wmax + W * G;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int z = blockIdx.x % p.S, bh = blockIdx.x / p.S;   // bh = b * Hkv + hk
    const int b = bh / p.Hkv, hk = bh % p.Hkv;
    const int Hq = p.Hkv * G;

    pdl_launch_dependents();
    pdl_wait();   // the cache, the queries and the lengths may come from the grid in front

    int len = p.lens[b];
    if (len < 0 || len > p.Tcap) {
        if (threadIdx.x == 0) atomicOr(p.status, STATUS_RANGE);
        len = 0;
    }
    const int t0 = z * p.TR;
    const int nt = max(0, min(len, t0 + p.TR) - t0);
    const size_t orow = ((size_t)b * Hq + (size_t)hk * G) * D;   // first output row of this CTA

    if (nt == 0) {   // an empty range: a zero output, or an empty part
        for (int i = threadIdx.x; i < G * D; i += THREADS) {
            if (p.S == 1) {
                p.out[orow + i] = 0.0f;
            } else {
                const int g = i / D, d = i % D;
                float *pp = p.part + (((size_t)b * Hq + (size_t)hk * G + g) * p.S + z) * (D + 2);
                pp[d] = 0.0f;
                if (d == 0) {
                    pp[D] = -INFINITY;
                    pp[D + 1] = 0.0f;
                }
            }
        }
        return;
    }
    const int nc = (nt + CT - 1) / CT;   // slots per phase
    GQ_DCHECK(nt <= p.TR && t0 + nt <= p.Tcap, p.status);

    if (threadIdx.x == 0) {
        for (int s = 0; s < SLOTS; s++) {
            mbar_init(smem_addr(full + s), 1);
            mbar_init(smem_addr(empty + s), 1);
        }
        fence_barrier_init();
    }
    __syncthreads();

    // ---------------------------------------------------------------- producer
    if (warp == W) {
        if (lane != 0) return;
        const size_t row0 = (size_t)bh * p.Tcap + t0;
        const int8_t *kbase = p.k + row0 * D, *vbase = p.v + row0 * D;
        const uint64_t policy = l2_evict_first_policy();
        int issued = 0;
        for (int i = 0; i < 2 * nc; i++) {
            const int slot = i % SLOTS;
            if (i >= SLOTS && !mbar_wait(smem_addr(empty + slot), (uint32_t)(((i / SLOTS) - 1) & 1), p.status))
                break;
            const int c = i < nc ? i : i - nc;
            const uint32_t bytes = (uint32_t)(min(CT, nt - c * CT) * D);
            GQ_DCHECK(c * CT < nt && bytes <= (uint32_t)CHUNK, p.status);
            mbar_arrive_expect_tx(smem_addr(full + slot), bytes);
            bulk_g2s_hint(smem_addr(smem + L.ring + (size_t)slot * CHUNK), (i < nc ? kbase : vbase) + (size_t)c * CT * D,
                          bytes, smem_addr(full + slot), policy);
            issued = i + 1;
        }
        // Stay until every copy issued has landed, so that the CTA never ends with a bulk
        // copy in flight (the last copy into each slot completes that slot's last phase).
        for (int i = max(0, issued - SLOTS); i < issued; i++)
            mbar_wait(smem_addr(full + i % SLOTS), (uint32_t)((i / SLOTS) & 1), p.status);
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int ctid = threadIdx.x;   // 0 .. CONSUMERS - 1
    {
        // staging in batches of SB loads per thread, all issued before any is stored, so that
        // the batch costs one memory latency (the producer streams keys meanwhile)
        constexpr int SB = 8;
        const float *qg = p.q + orow;   // the G query rows of KV head hk are contiguous
        for (int i0 = 0; i0 < G * D; i0 += SB * CONSUMERS) {
            float a[SB];
#pragma unroll
            for (int j = 0; j < SB; j++) {
                const int i = i0 + j * CONSUMERS + ctid;
                a[j] = i < G * D ? __ldg(qg + i) : 0.0f;
            }
#pragma unroll
            for (int j = 0; j < SB; j++) {
                const int i = i0 + j * CONSUMERS + ctid;
                if (i < G * D) qs[i] = a[j];
            }
        }
        const float *ksg = p.ks + (size_t)bh * p.Tcap + t0, *vsg = p.vs + (size_t)bh * p.Tcap + t0;
        for (int i0 = 0; i0 < nt; i0 += SB * CONSUMERS) {
            float a[SB], c[SB];
#pragma unroll
            for (int j = 0; j < SB; j++) {
                const int i = i0 + j * CONSUMERS + ctid;
                a[j] = i < nt ? __ldg(ksg + i) : 0.0f;
                c[j] = i < nt ? __ldg(vsg + i) : 0.0f;
            }
#pragma unroll
            for (int j = 0; j < SB; j++) {
                const int i = i0 + j * CONSUMERS + ctid;
                if (i < nt) {
                    ksc[i] = a[j] * p.c2;
                    vsc[i] = c[j];
                }
            }
        }
    }
    consumer_sync<CONSUMERS>();

    const uint32_t ring_a = smem_addr(smem + L.ring), sc_a = smem_addr(sc), ksc_a = smem_addr(ksc),
                   qs_a = smem_addr(qs);
    bool failed = false;
    auto wait_slot = [&](int i) {
        const bool ok = mbar_wait(smem_addr(full + i % SLOTS), (uint32_t)((i / SLOTS) & 1), p.status);
        failed |= !__all_sync(0xffffffffu, ok);
    };
    auto release_slot = [&](int i) {
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(empty + i % SLOTS));
    };

    // ---- scores: slot c of the key phase goes to warp c % W
    const int sl = lane % LPT;   // this lane's 16-byte column of a token row
    for (int c = warp; c < nc; c += W) {
        wait_slot(c);
        if (!failed) {
            const uint32_t chunk = ring_a + (uint32_t)((c % SLOTS) * CHUNK);
            const int ntok = min(CT, nt - c * CT);
            GQ_DCHECK(ntok > 0 && c * CT + ntok <= nt, p.status);
#pragma unroll 1
            for (int pass = 0; pass < G / HG; pass++) {
                uint64_t qv[HG][8];
#pragma unroll
                for (int h = 0; h < HG; h++) {
                    const uint32_t qrow = qs_a + (uint32_t)(((pass * HG + h) * D + sl * 16) * 4);
#pragma unroll
                    for (int j = 0; j < 4; j++) {
                        const uint4 f = sh_ld128(qrow + 16 * j);
                        qv[h][2 * j] = pack2(__uint_as_float(f.x), __uint_as_float(f.y));
                        qv[h][2 * j + 1] = pack2(__uint_as_float(f.z), __uint_as_float(f.w));
                    }
                }
#pragma unroll 4
                for (int it = 0; it < ntok; it += TPW) {
                    const int tok = it + lane / LPT;
                    uint4 w = make_uint4(0u, 0u, 0u, 0u);
                    if (tok < ntok) w = sh_ld128(chunk + (uint32_t)(tok * D + sl * 16));
                    uint64_t kf[8];
                    widen4(w.x, kf[0], kf[1]);
                    widen4(w.y, kf[2], kf[3]);
                    widen4(w.z, kf[4], kf[5]);
                    widen4(w.w, kf[6], kf[7]);
                    float part[HG];
#pragma unroll
                    for (int h = 0; h < HG; h++) {
                        uint64_t a = fma2(qv[h][0], kf[0], 0ull);
#pragma unroll
                        for (int j = 1; j < 8; j++) a = fma2(qv[h][j], kf[j], a);
                        float lo, hi;
                        unpack2(a, lo, hi);
                        part[h] = lo + hi;
                    }
                    const float s = reduce_heads<HG, LPT>(part, lane);
                    if (tok < ntok && (sl % (LPT / HG)) == 0) {
                        const int t = c * CT + tok, h = pass * HG + sl / (LPT / HG);
                        sh_stf(sc_a + 4u * (uint32_t)(t * G + h), s * sh_ldf(ksc_a + 4u * (uint32_t)t));
                    }
                }
            }
        }
        release_slot(c);
    }
    consumer_sync<CONSUMERS>();

    // ---- softmax over the row: thread ctid takes entries ctid, ctid + 128, ... (head ctid % G)
    const int gh = ctid % G;
    {
        float mx = -INFINITY;
        for (int i = ctid; i < nt * G; i += CONSUMERS) mx = fmaxf(mx, sc[i]);
#pragma unroll
        for (int m = 16; m >= G; m >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, m));
        if (lane < G) wmax[warp * G + lane] = mx;
        consumer_sync<CONSUMERS>();
        float M = wmax[gh];
#pragma unroll
        for (int w = 1; w < W; w++) M = fmaxf(M, wmax[w * G + gh]);
        float l = 0.0f;
        for (int i = ctid; i < nt * G; i += CONSUMERS) {
            const float e = exp2f(sc[i] - M);
            l += e;
            sc[i] = e * vsc[i / G];
        }
#pragma unroll
        for (int m = 16; m >= G; m >>= 1) l += __shfl_xor_sync(0xffffffffu, l, m);
        if (lane < G) wsum[warp * G + lane] = l;
    }
    consumer_sync<CONSUMERS>();

    // ---- values: slot nc + c goes to warp c % W
    uint64_t acc[G][VB / 2];
#pragma unroll
    for (int g = 0; g < G; g++)
#pragma unroll
        for (int j = 0; j < VB / 2; j++) acc[g][j] = 0ull;
    const int vl = lane % LPV;
    for (int c = warp; c < nc; c += W) {
        wait_slot(nc + c);
        if (!failed) {
            const uint32_t chunk = ring_a + (uint32_t)(((nc + c) % SLOTS) * CHUNK);
            const int ntok = min(CT, nt - c * CT);
#pragma unroll 4
            for (int it = 0; it < ntok; it += TPV) {
                const int tok = it + lane / LPV;
                const bool live = tok < ntok;
                uint32_t wv[VB / 4];
                if constexpr (VB == 16) {
                    const uint4 w = live ? sh_ld128(chunk + (uint32_t)(tok * D + vl * 16)) : make_uint4(0u, 0u, 0u, 0u);
                    wv[0] = w.x;
                    wv[1] = w.y;
                    wv[2] = w.z;
                    wv[3] = w.w;
                } else {
                    const uint2 w = live ? sh_ld64(chunk + (uint32_t)(tok * D + vl * 8)) : make_uint2(0u, 0u);
                    wv[0] = w.x;
                    wv[1] = w.y;
                }
                uint64_t vf[VB / 2];
#pragma unroll
                for (int j = 0; j < VB / 4; j++) widen4(wv[j], vf[2 * j], vf[2 * j + 1]);
                const int t = c * CT + (live ? tok : 0);
#pragma unroll
                for (int g = 0; g < G; g++) {
                    const float wt = live ? sh_ldf(sc_a + 4u * (uint32_t)(t * G + g)) : 0.0f;
                    const uint64_t w2 = pack2(wt, wt);
#pragma unroll
                    for (int j = 0; j < VB / 2; j++) acc[g][j] = fma2(w2, vf[j], acc[g][j]);
                }
            }
        }
        release_slot(nc + c);
    }

    // ---- add the token lanes of each warp, then the warps (in order), and scale
#pragma unroll
    for (int m = LPV; m < 32; m <<= 1)
#pragma unroll
        for (int g = 0; g < G; g++)
#pragma unroll
            for (int j = 0; j < VB / 2; j++) {
                float lo, hi;
                unpack2(acc[g][j], lo, hi);
                lo += __shfl_xor_sync(0xffffffffu, lo, m);
                hi += __shfl_xor_sync(0xffffffffu, hi, m);
                acc[g][j] = pack2(lo, hi);
            }
    consumer_sync<CONSUMERS>();   // every warp is done with the ring: it holds the per-warp sums now
    float *red = reinterpret_cast<float *>(smem + L.ring);   // [W][G][D]
    if (lane < LPV) {
#pragma unroll
        for (int g = 0; g < G; g++)
#pragma unroll
            for (int j = 0; j < VB / 2; j++) {
                float lo, hi;
                unpack2(acc[g][j], lo, hi);
                red[((size_t)warp * G + g) * D + vl * VB + 2 * j] = lo;
                red[((size_t)warp * G + g) * D + vl * VB + 2 * j + 1] = hi;
            }
    }
    consumer_sync<CONSUMERS>();
    for (int i = ctid; i < G * D; i += CONSUMERS) {
        const int g = i / D, d = i % D;
        float o = red[(size_t)g * D + d];
#pragma unroll
        for (int w = 1; w < W; w++) o += red[((size_t)w * G + g) * D + d];
        float l = wsum[g], M = wmax[g];
#pragma unroll
        for (int w = 1; w < W; w++) {
            l += wsum[w * G + g];
            M = fmaxf(M, wmax[w * G + g]);
        }
        if (p.S == 1) {
            p.out[orow + i] = o / l;
        } else {
            float *pp = p.part + (((size_t)b * Hq + (size_t)hk * G + g) * p.S + z) * (D + 2);
            pp[d] = o;
            if (d == 0) {
                pp[D] = M;
                pp[D + 1] = l;
            }
        }
    }
}

// ---------------------------------------------------------------------------
// The same attention on the tensor cores (D = 128).  With G query rows per KV head the two
// products are [G x D] . [D x T] and [G x T] . [T x D]: G multiply-adds per cached byte, which
// the FP32 lanes cannot issue at the memory rate once G reaches about four.  Here both run as
// m16n8k16 fp16 MMAs with f32 accumulation:
//   * the int8 codes become exact fp16 values (the byte, biased by 128, in the mantissa of
//     1024, then 1152 subtracted);
//   * the query (scores) and the softmax weights (values) are f32 values split into two fp16
//     terms, hi = fp16(x) and lo = fp16(x - hi), after a power-of-two scaling that puts the
//     largest in [2^14, 2^15): hi + lo carries x to within 2^-22 of its magnitude, and each
//     fp16 x fp16 product is exact, so the products keep f32 accuracy;
//   * the cache comes in through 2D tensor copies with the 128-byte swizzle (16-byte chunk c of
//     row r lands at chunk c ^ (r mod 8)), which keeps the fragment loads free of bank
//     conflicts.
// Scores: MMA rows are 16 tokens, columns (head, hi / lo) pairs; the k order inside each 16
// steps is permuted the same way for both operands (lane t takes the 16 bytes of chunk 2t + h
// of its two rows).  Values: MMA rows are 16 of the 128 value positions, columns (head,
// hi / lo) pairs, k the 16 tokens of a step; the hi and lo columns of a head sit in one lane.
template <int G>
struct AmCfg {
    static constexpr int D = 128;
    static constexpr int W = G <= 2 ? 8 : 4;          // consumer warps
    static constexpr int CT = 32;                      // tokens per slot
    static constexpr int CHUNK = CT * D;               // 4 KB
    static constexpr int SLOTS = 16;                   // a multiple of W
    static constexpr int THREADS = (W + 1) * 32;
    static constexpr int CONSUMERS = W * 32;
    static constexpr int NN = G <= 4 ? 1 : 2;          // column tiles of the score MMA (2G columns)
    static constexpr int ROWS = 2 * G;                 // (head, hi / lo) rows of the value MMA
    // five to eight heads: the weights replace the scores in place ([token][head] pairs of fp16),
    // which halves the shared memory per token and so the number of CTAs a sequence is split
    // over; fewer heads: the weights go to rows of their own ([2G][token] fp16), one 32-bit load
    // per pair of tokens in the value steps
    static constexpr bool INPLACE = G > 4;
    static constexpr int PER_TOKEN = 8 + 4 * G + (INPLACE ? 0 : 4 * G);   // shared bytes per token
};

struct AmLayout {
    size_t bars, ring, qf, hsc, ksc, vsc, sc, sp, wred, total;
    int trp;   // fp16 entries per row of sp: TR padded so that the rows start in different banks
};

template <int G>
__host__ __device__ AmLayout am_layout(int TR) {
    using C = AmCfg<G>;
    AmLayout L{};
    L.bars = 0;                                                 // full[16], empty[16]
    L.ring = 1024;                                              // 1024-byte aligned slots (swizzle)
    L.qf = L.ring + (size_t)C::SLOTS * C::CHUNK;                // the query split: [2G][128] fp16
    L.hsc = L.qf + (size_t)C::ROWS * C::D * 2;                  // per head: 1 / its scaling
    L.ksc = L.hsc + 64;                                         // key scale x c2, per token
    L.vsc = L.ksc + (size_t)TR * 4;                             // value scale, per token
    L.sc = L.vsc + (size_t)TR * 4;                              // scores [TR][G] f32 (then weights, in place)
    L.trp = TR + 8;
    L.sp = L.sc + (size_t)TR * G * 4;                           // weights [2G][trp] fp16 (not in place)
    L.wred = L.sp + (C::INPLACE ? 0 : (((size_t)C::ROWS * L.trp * 2 + 15) & ~(size_t)15));   // [W][G] max, sum; [W]
    L.total = L.wred + (2 * C::W * G + C::W + 4) * 4;
    return L;
}

template <int G>
__host__ __device__ constexpr size_t am_fixed_bytes() {
    using C = AmCfg<G>;
    return 1024 + (size_t)C::SLOTS * C::CHUNK + (size_t)C::ROWS * C::D * 2 + 64 +
           (C::INPLACE ? 0 : (size_t)C::ROWS * 8 * 2 + 16) + (2 * C::W * G + C::W + 4) * 4 +
           1024;   // + the alignment of the dynamic base
}

__device__ __forceinline__ void tma_rows(uint32_t dst, const CUtensorMap *map, int row, uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(row), "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void sh_sth(uint32_t a, __half v) {
    asm volatile("st.shared.u16 [%0], %1;" ::"r"(a), "h"(__half_as_ushort(v)) : "memory");
}

__device__ __forceinline__ uint32_t sh_ldu16(uint32_t a) {
    uint32_t v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}

__device__ __forceinline__ uint32_t sh_ld32(uint32_t a) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}

// The four int8 of a word as two exact fp16 pairs: bytes (0, 1) and (2, 3).
__device__ __forceinline__ void i8x4_to_f16x2(uint32_t w, uint32_t &p01, uint32_t &p23) {
    const uint32_t u = w ^ 0x80808080u;
    const __half2 off = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));   // 1152
    uint32_t a = __byte_perm(u, 0x64646464u, 0x4140), b = __byte_perm(u, 0x64646464u, 0x4342);
    __half2 ha = __hsub2(*reinterpret_cast<__half2 *>(&a), off), hb = __hsub2(*reinterpret_cast<__half2 *>(&b), off);
    p01 = *reinterpret_cast<uint32_t *>(&ha);
    p23 = *reinterpret_cast<uint32_t *>(&hb);
}

// Byte j of x and byte j of y as one exact fp16 pair (x_j, y_j), for j = 0 .. 3 of the two words.
__device__ __forceinline__ void i8x4_pairs_to_f16x2(uint32_t x, uint32_t y, uint32_t (&o)[4]) {
    const uint32_t ux = x ^ 0x80808080u, uy = y ^ 0x80808080u;
    const uint32_t i01 = __byte_perm(ux, uy, 0x5140), i23 = __byte_perm(ux, uy, 0x7362);   // x0 y0 x1 y1, x2 y2 x3 y3
    const __half2 off = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));
    uint32_t t[4] = {__byte_perm(i01, 0x64646464u, 0x4140), __byte_perm(i01, 0x64646464u, 0x4342),
                     __byte_perm(i23, 0x64646464u, 0x4140), __byte_perm(i23, 0x64646464u, 0x4342)};
#pragma unroll
    for (int i = 0; i < 4; i++) {
        __half2 h = __hsub2(*reinterpret_cast<__half2 *>(&t[i]), off);
        o[i] = *reinterpret_cast<uint32_t *>(&h);
    }
}

template <int G>
__global__ void __launch_bounds__(AmCfg<G>::THREADS, 2)
    attn_mma_i8_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                       const AttnParams p) {
    using C = AmCfg<G>;
    constexpr int D = C::D, W = C::W, CT = C::CT, CHUNK = C::CHUNK, SLOTS = C::SLOTS, NN = C::NN;
    constexpr int THREADS = C::THREADS, CONSUMERS = C::CONSUMERS, ROWS = C::ROWS;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const AmLayout L = am_layout<G>(p.TR);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.bars);
    uint64_t *empty = full + SLOTS;
    float *hsc = reinterpret_cast<float *>(smem + L.hsc);
    float *ksc = reinterpret_cast<float *>(smem + L.ksc);
    float *vsc = reinterpret_cast<float *>(smem + L.vsc);
    float *sc = reinterpret_cast<float *>(smem + L.sc);
    float *wmax = reinterpret_cast<float *>(smem + L.wred);
    float *wsum = wmax + W * G;
    float *wvmax = wsum + W * G;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int z = blockIdx.x % p.S, bh = blockIdx.x / p.S;   // bh = b * Hkv + hk
    const int b = bh / p.Hkv, hk = bh % p.Hkv;
    const int Hq = p.Hkv * G;

    pdl_launch_dependents();
    pdl_wait();   // the cache, the queries and the lengths may come from the grid in front

    int len = p.lens[b];
    if (len < 0 || len > p.Tcap) {
        if (threadIdx.x == 0) atomicOr(p.status, STATUS_RANGE);
        len = 0;
    }
    const int t0 = z * p.TR;
    const int nt = max(0, min(len, t0 + p.TR) - t0);
    const size_t orow = ((size_t)b * Hq + (size_t)hk * G) * D;

    if (nt == 0) {   // an empty range: a zero output, or an empty part
        for (int i = threadIdx.x; i < G * D; i += THREADS) {
            if (p.S == 1) {
                p.out[orow + i] = 0.0f;
            } else {
                const int g = i / D, d = i % D;
                float *pp = p.part + (((size_t)b * Hq + (size_t)hk * G + g) * p.S + z) * (D + 2);
                pp[d] = 0.0f;
                if (d == 0) {
                    pp[D] = -INFINITY;
                    pp[D + 1] = 0.0f;
                }
            }
        }
        return;
    }
    const int nc = (nt + CT - 1) / CT;   // slots per phase
    GQ_DCHECK(nt <= p.TR && t0 + nt <= p.Tcap, p.status);

    if (threadIdx.x == 0) {
        for (int s = 0; s < SLOTS; s++) {
            mbar_init(smem_addr(full + s), 1);
            mbar_init(smem_addr(empty + s), 1);
        }
        fence_barrier_init();
    }
    __syncthreads();

    // ---------------------------------------------------------------- producer
    if (warp == W) {
        if (lane != 0) return;
        const int row0 = bh * p.Tcap + t0;   // first cache row of the range (rows of 128 bytes)
        const uint64_t policy = l2_evict_first_policy();
        int issued = 0;
        for (int i = 0; i < 2 * nc; i++) {
            const int slot = i % SLOTS;
            if (i >= SLOTS && !mbar_wait(smem_addr(empty + slot), (uint32_t)(((i / SLOTS) - 1) & 1), p.status)) break;
            const int c = i < nc ? i : i - nc;
            GQ_DCHECK(c * CT < nt && t0 + c * CT < p.Tcap, p.status);
            // a whole box every time: rows past the range belong to the next range or lie past the
            // tensor (read as zeros); their scores are not stored and their weights are zero
            mbar_arrive_expect_tx(smem_addr(full + slot), (uint32_t)CHUNK);
            tma_rows(smem_addr(smem + L.ring + (size_t)slot * CHUNK), i < nc ? &kmap : &vmap, row0 + c * CT,
                     smem_addr(full + slot), policy);
            issued = i + 1;
        }
        // stay until every copy issued has landed: the CTA never ends with a copy in flight
        for (int i = max(0, issued - SLOTS); i < issued; i++)
            mbar_wait(smem_addr(full + i % SLOTS), (uint32_t)((i / SLOTS) & 1), p.status);
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int ctid = threadIdx.x;
    const uint32_t qf_a = smem_addr(smem + L.qf), ring_a = smem_addr(smem + L.ring), sp_a = smem_addr(smem + L.sp),
                   sc_a = smem_addr(sc), ksc_a = smem_addr(ksc), vsc_a = smem_addr(vsc), hsc_a = smem_addr(hsc);
    {
        // the query rows, scaled by a power of two per head and split into fp16 hi / lo
        for (int g = warp; g < G; g += W) {
            const float4 v = __ldg(reinterpret_cast<const float4 *>(p.q + orow + (size_t)g * D) + lane);
            float am = absmax4(v);
#pragma unroll
            for (int m = 16; m >= 1; m >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, m));
            int ex = 0;
            if (am > 0.0f) frexpf(am, &ex);                      // am = f 2^ex, f in [0.5, 1)
            const float scale = am > 0.0f ? ldexpf(1.0f, 15 - ex) : 1.0f;
            const float xs[4] = {v.x * scale, v.y * scale, v.z * scale, v.w * scale};
            __half hi[4], lo[4];
#pragma unroll
            for (int i = 0; i < 4; i++) {
                hi[i] = __float2half_rn(xs[i]);
                lo[i] = __float2half_rn(xs[i] - __half2float(hi[i]));
            }
            __half *qh = reinterpret_cast<__half *>(smem + L.qf) + (2 * g) * D + 4 * lane;
            __half *ql = qh + D;
#pragma unroll
            for (int i = 0; i < 4; i++) {
                qh[i] = hi[i];
                ql[i] = lo[i];
            }
            if (lane == 0) hsc[g] = am > 0.0f ? ldexpf(1.0f, ex - 15) : 1.0f;
        }
        // the token scales, in batches of SB loads per thread issued before any is stored
        constexpr int SB = 8;
        const float *ksg = p.ks + (size_t)bh * p.Tcap + t0, *vsg = p.vs + (size_t)bh * p.Tcap + t0;
        float vmax = 0.0f;
        for (int i0 = 0; i0 < nt; i0 += SB * CONSUMERS) {
            float a[SB], c[SB];
#pragma unroll
            for (int j = 0; j < SB; j++) {
                const int i = i0 + j * CONSUMERS + ctid;
                a[j] = i < nt ? __ldg(ksg + i) : 0.0f;
                c[j] = i < nt ? __ldg(vsg + i) : 0.0f;
            }
#pragma unroll
            for (int j = 0; j < SB; j++) {
                const int i = i0 + j * CONSUMERS + ctid;
                if (i < nt) {
                    ksc[i] = a[j] * p.c2;
                    vsc[i] = c[j];
                    vmax = fmaxf(vmax, fabsf(c[j]));
                }
            }
        }
#pragma unroll
        for (int m = 16; m >= 1; m >>= 1) vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, m));
        if (lane == 0) wvmax[warp] = vmax;
    }
    consumer_sync<CONSUMERS>();

    const int g8 = lane >> 2, t = lane & 3;   // m16n8k16 fragment coordinates
    bool failed = false;
    auto wait_slot = [&](int i) {
        const bool ok = mbar_wait(smem_addr(full + i % SLOTS), (uint32_t)((i / SLOTS) & 1), p.status);
        failed |= !__all_sync(0xffffffffu, ok);
    };
    auto release_slot = [&](int i) {
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(empty + i % SLOTS));
    };

    // ---- scores.  B fragments of the query split: column n = 8 nn + g8 is row n of qf (head n / 2,
    // hi for even n, lo for odd); k-step (h, s) takes positions 16 (2t + h) + 4s + {0, 1} and {2, 3}.
    uint32_t qb[NN][2][4][2];
#pragma unroll
    for (int nn = 0; nn < NN; nn++)
#pragma unroll
        for (int h = 0; h < 2; h++)
#pragma unroll
            for (int s = 0; s < 4; s++) {
                const int n = 8 * nn + g8, d0 = 16 * (2 * t + h) + 4 * s;
                const bool live = n < ROWS;
                qb[nn][h][s][0] = live ? sh_ld32(qf_a + (uint32_t)((n * D + d0) * 2)) : 0u;
                qb[nn][h][s][1] = live ? sh_ld32(qf_a + (uint32_t)((n * D + d0 + 2) * 2)) : 0u;
            }
    for (int c = warp; c < nc; c += W) {
        wait_slot(c);
        if (!failed) {
            const uint32_t chunk = ring_a + (uint32_t)((c % SLOTS) * CHUNK);
            const int ntok = min(CT, nt - c * CT);
            GQ_DCHECK(ntok > 0 && c * CT + ntok <= nt, p.status);
#pragma unroll
            for (int mt = 0; mt < CT / 16; mt++) {
                if (16 * mt >= ntok) break;
                float acc[NN][4];
#pragma unroll
                for (int nn = 0; nn < NN; nn++) acc[nn][0] = acc[nn][1] = acc[nn][2] = acc[nn][3] = 0.0f;
                const int ra = 16 * mt + g8;   // rows ra and ra + 8 of the slot: both are g8 mod 8
#pragma unroll
                for (int h = 0; h < 2; h++) {
                    const uint32_t ch = (uint32_t)(((2 * t + h) ^ g8) * 16);
                    const uint4 wa = sh_ld128(chunk + (uint32_t)(ra * D) + ch);
                    const uint4 wb = sh_ld128(chunk + (uint32_t)((ra + 8) * D) + ch);
                    const uint32_t av[4] = {wa.x, wa.y, wa.z, wa.w}, bv[4] = {wb.x, wb.y, wb.z, wb.w};
#pragma unroll
                    for (int s = 0; s < 4; s++) {
                        uint32_t a0, a2, a1, a3;
                        i8x4_to_f16x2(av[s], a0, a2);
                        i8x4_to_f16x2(bv[s], a1, a3);
#pragma unroll
                        for (int nn = 0; nn < NN; nn++)
                            mma_f16_16x8x16(acc[nn], a0, a1, a2, a3, qb[nn][h][s][0], qb[nn][h][s][1]);
                    }
                }
#pragma unroll
                for (int nn = 0; nn < NN; nn++) {
                    const int head = 4 * nn + t;   // columns 2t, 2t + 1 of tile nn: (head, hi), (head, lo)
                    if (head < G) {
                        const int ta = c * CT + ra;
                        const float hs = sh_ldf(hsc_a + 4u * (uint32_t)head);
                        if (ra < ntok)
                            sh_stf(sc_a + 4u * (uint32_t)(ta * G + head),
                                   (acc[nn][0] + acc[nn][1]) * hs * sh_ldf(ksc_a + 4u * (uint32_t)ta));
                        if (ra + 8 < ntok)
                            sh_stf(sc_a + 4u * (uint32_t)((ta + 8) * G + head),
                                   (acc[nn][2] + acc[nn][3]) * hs * sh_ldf(ksc_a + 4u * (uint32_t)(ta + 8)));
                    }
                }
            }
        }
        release_slot(c);
    }
    consumer_sync<CONSUMERS>();

    // ---- softmax over the row, per head
    const int gh = ctid % G;
    float vscale;   // weights are scaled by this power of two so that the largest is below 2^15
    {
        float vm = wvmax[0];
#pragma unroll
        for (int w = 1; w < W; w++) vm = fmaxf(vm, wvmax[w]);
        int ex = 0;
        if (vm > 0.0f) frexpf(vm, &ex);
        vscale = vm > 0.0f ? ldexpf(1.0f, 14 - ex) : 1.0f;   // e vs vscale < 2^15 (e <= 1)
        // each entry (token, head) becomes its weight as two fp16 terms: in place (the thread that
        // reads an entry is the one that writes it), or into rows 2 head (hi) and 2 head + 1 (lo)
        auto put = [&](int i, int tok, int g, float wv) {
            const __half hi = __float2half_rn(wv), lo = __float2half_rn(wv - __half2float(hi));
            if constexpr (C::INPLACE) {
                sh_stf(sc_a + 4u * (uint32_t)i,
                       __uint_as_float((uint32_t)__half_as_ushort(hi) | ((uint32_t)__half_as_ushort(lo) << 16)));
            } else {
                sh_sth(sp_a + 2u * (uint32_t)((2 * g) * L.trp + tok), hi);
                sh_sth(sp_a + 2u * (uint32_t)((2 * g + 1) * L.trp + tok), lo);
            }
        };
        if constexpr (32 % G == 0) {
            // entries ctid, ctid + CONSUMERS, ... all belong to head ctid % G
            float mx = -INFINITY;
            for (int i = ctid; i < nt * G; i += CONSUMERS) mx = fmaxf(mx, sh_ldf(sc_a + 4u * (uint32_t)i));
#pragma unroll
            for (int m = 16; m >= G; m >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, m));
            if (lane < G) wmax[warp * G + lane] = mx;
            consumer_sync<CONSUMERS>();
            float M = wmax[gh];
#pragma unroll
            for (int w = 1; w < W; w++) M = fmaxf(M, wmax[w * G + gh]);
            float l = 0.0f;
            for (int i = ctid; i < nt * G; i += CONSUMERS) {
                const int tok = i / G;
                const float e = exp2f(sh_ldf(sc_a + 4u * (uint32_t)i) - M);
                l += e;
                put(i, tok, gh, e * sh_ldf(vsc_a + 4u * (uint32_t)tok) * vscale);
            }
#pragma unroll
            for (int m = 16; m >= G; m >>= 1) l += __shfl_xor_sync(0xffffffffu, l, m);
            if (lane < G) wsum[warp * G + lane] = l;
        } else {
            // other head counts: each thread takes whole tokens (all G heads of each)
            float mx[G], l[G];
#pragma unroll
            for (int g = 0; g < G; g++) mx[g] = -INFINITY;
            for (int tok = ctid; tok < nt; tok += CONSUMERS)
#pragma unroll
                for (int g = 0; g < G; g++) mx[g] = fmaxf(mx[g], sh_ldf(sc_a + 4u * (uint32_t)(tok * G + g)));
#pragma unroll
            for (int g = 0; g < G; g++) {
#pragma unroll
                for (int m = 16; m >= 1; m >>= 1) mx[g] = fmaxf(mx[g], __shfl_xor_sync(0xffffffffu, mx[g], m));
                if (lane == 0) wmax[warp * G + g] = mx[g];
            }
            consumer_sync<CONSUMERS>();
#pragma unroll
            for (int g = 0; g < G; g++) {
                float M = wmax[g];
#pragma unroll
                for (int w = 1; w < W; w++) M = fmaxf(M, wmax[w * G + g]);
                mx[g] = M;
                l[g] = 0.0f;
            }
            for (int tok = ctid; tok < nt; tok += CONSUMERS) {
                const float vsv = sh_ldf(vsc_a + 4u * (uint32_t)tok) * vscale;
#pragma unroll
                for (int g = 0; g < G; g++) {
                    const int i = tok * G + g;
                    const float e = exp2f(sh_ldf(sc_a + 4u * (uint32_t)i) - mx[g]);
                    l[g] += e;
                    put(i, tok, g, e * vsv);
                }
            }
#pragma unroll
            for (int g = 0; g < G; g++) {
#pragma unroll
                for (int m = 16; m >= 1; m >>= 1) l[g] += __shfl_xor_sync(0xffffffffu, l[g], m);
                if (lane == 0) wsum[warp * G + g] = l[g];
            }
        }
        // the tokens of the last 16-token step past the range weigh nothing
        const int pad = ((nt + 15) & ~15) - nt;
        if constexpr (C::INPLACE) {
            for (int i = nt * G + ctid; i < (nt + pad) * G; i += CONSUMERS) sh_stf(sc_a + 4u * (uint32_t)i, 0.0f);
        } else {
            for (int i = ctid; i < ROWS * pad; i += CONSUMERS)
                sh_sth(sp_a + 2u * (uint32_t)((i / pad) * L.trp + nt + i % pad), __float2half_rn(0.0f));
        }
    }
    consumer_sync<CONSUMERS>();

    // ---- values: D[position][column] = sum_t V[t][position] P[column][t], the MMA rows being
    // 16 value positions (row g8 of row tile m is position 16 g8 + 2m, row g8 + 8 the next one:
    // the 16 bytes a lane loads from each token row serve its rows of all 8 row tiles), the
    // columns (head, hi / lo) pairs, k the 16 tokens of a step.
    constexpr int NV = G <= 4 ? 1 : 2;   // column tiles of the value MMA
    float acc[8][NV][4];
#pragma unroll
    for (int m = 0; m < 8; m++)
#pragma unroll
        for (int nv = 0; nv < NV; nv++) acc[m][nv][0] = acc[m][nv][1] = acc[m][nv][2] = acc[m][nv][3] = 0.0f;
    for (int c = warp; c < nc; c += W) {
        wait_slot(nc + c);
        if (!failed) {
            const uint32_t chunk = ring_a + (uint32_t)(((nc + c) % SLOTS) * CHUNK);
            const int ntok = min(CT, nt - c * CT);
#pragma unroll
            for (int mt = 0; mt < CT / 16; mt++) {
                if (16 * mt >= ntok) break;
                const int tk = c * CT + 16 * mt;   // first token of the step in the range
                GQ_DCHECK(tk + 16 <= ((nt + 15) & ~15) && tk + 16 <= p.TR, p.status);
                // B: the weights of column n = 8 nv + g8 (head n / 2, hi for even n, lo for odd) at tokens
                // 2t, 2t + 1 and 2t + 8, 2t + 9: the fp16 at byte 2 (n % 2) of entry (token, head)
                uint32_t pb[NV][2];
#pragma unroll
                for (int nv = 0; nv < NV; nv++) {
                    const int n = 8 * nv + g8;
                    if (n >= ROWS) {
                        pb[nv][0] = pb[nv][1] = 0u;
                    } else if constexpr (C::INPLACE) {
                        const uint32_t a = sc_a + (uint32_t)(((tk + 2 * t) * G + (n >> 1)) * 4 + (n & 1) * 2);
                        const uint32_t rowb = (uint32_t)(G * 4);   // bytes per token
                        pb[nv][0] = sh_ldu16(a) | (sh_ldu16(a + rowb) << 16);
                        pb[nv][1] = sh_ldu16(a + 8 * rowb) | (sh_ldu16(a + 9 * rowb) << 16);
                    } else {
                        const uint32_t a = sp_a + (uint32_t)((n * L.trp + tk + 2 * t) * 2);
                        pb[nv][0] = sh_ld32(a);
                        pb[nv][1] = sh_ld32(a + 16);
                    }
                }
                // A: positions 16 g8 .. 16 g8 + 15 (chunk g8) of slot rows r, r + 1, r + 8, r + 9
                const int r = 16 * mt + 2 * t;
                const uint4 v0 = sh_ld128(chunk + (uint32_t)(r * D) + (uint32_t)((g8 ^ (r & 7)) * 16));
                const uint4 v1 = sh_ld128(chunk + (uint32_t)((r + 1) * D) + (uint32_t)((g8 ^ ((r + 1) & 7)) * 16));
                const uint4 v8 = sh_ld128(chunk + (uint32_t)((r + 8) * D) + (uint32_t)((g8 ^ ((r + 8) & 7)) * 16));
                const uint4 v9 = sh_ld128(chunk + (uint32_t)((r + 9) * D) + (uint32_t)((g8 ^ ((r + 9) & 7)) * 16));
                const uint32_t x0[4] = {v0.x, v0.y, v0.z, v0.w}, x1[4] = {v1.x, v1.y, v1.z, v1.w};
                const uint32_t x8[4] = {v8.x, v8.y, v8.z, v8.w}, x9[4] = {v9.x, v9.y, v9.z, v9.w};
#pragma unroll
                for (int q = 0; q < 4; q++) {
                    uint32_t p01[4], p89[4];   // byte 4q + i of tokens (r, r + 1) and (r + 8, r + 9)
                    i8x4_pairs_to_f16x2(x0[q], x1[q], p01);
                    i8x4_pairs_to_f16x2(x8[q], x9[q], p89);
#pragma unroll
                    for (int i2 = 0; i2 < 2; i2++) {
                        const int m = 2 * q + i2;   // row tile: positions 16 g8 + 2m (row g8), + 1 (row g8 + 8)
#pragma unroll
                        for (int nv = 0; nv < NV; nv++)
                            mma_f16_16x8x16(acc[m][nv], p01[2 * i2], p01[2 * i2 + 1], p89[2 * i2], p89[2 * i2 + 1],
                                            pb[nv][0], pb[nv][1]);
                    }
                }
            }
        }
        release_slot(nc + c);
    }

    // ---- hi + lo (columns 2t and 2t + 1 of this lane), then the warps in order, then scale
    consumer_sync<CONSUMERS>();   // every warp is done with the ring: it holds the per-warp sums now
    float *red = reinterpret_cast<float *>(smem + L.ring);   // [W][G][D]
#pragma unroll
    for (int nv = 0; nv < NV; nv++) {
        const int head = 4 * nv + t;
        if (head < G) {
            const uint32_t o = smem_addr(red) + 4u * (uint32_t)((warp * G + head) * D + 16 * g8);
#pragma unroll
            for (int m = 0; m < 8; m++) {
                sh_stf(o + 8u * m, acc[m][nv][0] + acc[m][nv][1]);
                sh_stf(o + 8u * m + 4u, acc[m][nv][2] + acc[m][nv][3]);
            }
        }
    }
    consumer_sync<CONSUMERS>();
    const float inv_vscale = 1.0f / vscale;   // a power of two: exact
    for (int i = ctid; i < G * D; i += CONSUMERS) {
        const int g = i / D, d = i % D;
        float o = red[(size_t)g * D + d];
#pragma unroll
        for (int w = 1; w < W; w++) o += red[((size_t)w * G + g) * D + d];
        o *= inv_vscale;
        float l = wsum[g], M = wmax[g];
#pragma unroll
        for (int w = 1; w < W; w++) {
            l += wsum[w * G + g];
            M = fmaxf(M, wmax[w * G + g]);
        }
        if (p.S == 1) {
            p.out[orow + i] = o / l;
        } else {
            float *pp = p.part + (((size_t)b * Hq + (size_t)hk * G + g) * p.S + z) * (D + 2);
            pp[d] = o;
            if (d == 0) {
                pp[D] = M;
                pp[D + 1] = l;
            }
        }
    }
}

// Merges the S parts of each output row in order: with M the largest part maximum,
// out = sum_z 2^(m_z - M) o_z / sum_z 2^(m_z - M) l_z, both sums over z in increasing order.
// One CTA per row.  Two forms: one thread per column walks the parts one by one (few parts);
// or (many parts: a long cache split over many CTAs) the maxima, weights and sums of MERGE_CHUNK
// parts at a time are read in parallel into shared memory, and MERGE_GROUPS groups of one thread
// per column each add every MERGE_GROUPS-th part (MERGE_BATCH value loads in flight per thread),
// then the groups are added in order, so that no chain of dependent loads runs over all the
// parts.  Both orders are fixed: results are deterministic.
constexpr int MERGE_CHUNK = 256, MERGE_BATCH = 8, MERGE_WIDE_FROM = 16, MERGE_GROUPS = 4;

__global__ void attn_merge_kernel(const float *part, float *out, int S, int D) {
    pdl_wait();
    const float *pp = part + (size_t)blockIdx.x * S * (D + 2);
    const int d = threadIdx.x;
    if (d >= D) return;
    float M = -INFINITY;
    for (int z = 0; z < S; z++) M = fmaxf(M, pp[(size_t)z * (D + 2) + D]);
    float o = 0.0f, l = 0.0f;
    if (M != -INFINITY) {
        for (int z = 0; z < S; z++) {
            const float *pz = pp + (size_t)z * (D + 2);
            const float a = exp2f(pz[D] - M);
            o += a * pz[d];
            l += a * pz[D + 1];
        }
    }
    out[(size_t)blockIdx.x * D + d] = l > 0.0f ? o / l : 0.0f;
}

__global__ void attn_merge_wide_kernel(const float *part, float *out, int S, int D) {
    __shared__ float sa[MERGE_CHUNK], sl[MERGE_CHUNK], sred[32], so[MERGE_GROUPS][128];
    pdl_wait();
    const float *pp = part + (size_t)blockIdx.x * S * (D + 2);
    const int tid = threadIdx.x, d = tid % D, grp = tid / D;   // MERGE_GROUPS groups of D threads
    const int lane = tid & 31, wid = tid >> 5, nw = (int)(blockDim.x >> 5);
    // M: every thread takes the parts tid, tid + blockDim.x, ...; then the warps, then the CTA
    float M = -INFINITY;
    for (int z = tid; z < S; z += blockDim.x) M = fmaxf(M, pp[(size_t)z * (D + 2) + D]);
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, m));
    if (lane == 0) sred[wid] = M;
    __syncthreads();
    M = sred[0];
    for (int w = 1; w < nw; w++) M = fmaxf(M, sred[w]);
    if (M == -INFINITY) {   // every part is empty
        if (grp == 0) out[(size_t)blockIdx.x * D + d] = 0.0f;
        return;
    }
    float o = 0.0f, l = 0.0f;
    for (int z0 = 0; z0 < S; z0 += MERGE_CHUNK) {
        const int nz = min(MERGE_CHUNK, S - z0);
        __syncthreads();   // the previous chunk's weights are no longer read (and sred, M, by all)
        for (int i = tid; i < nz; i += blockDim.x) {
            const float *pz = pp + (size_t)(z0 + i) * (D + 2);
            sa[i] = exp2f(pz[D] - M);
            sl[i] = pz[D + 1];
        }
        __syncthreads();
        if (tid == 0)
            for (int i = 0; i < nz; i++) l += sa[i] * sl[i];
        // group grp adds the parts grp, grp + MERGE_GROUPS, ... of the chunk, in increasing order
        for (int i0 = grp; i0 < nz; i0 += MERGE_GROUPS * MERGE_BATCH) {
            float v[MERGE_BATCH];
#pragma unroll
            for (int jj = 0; jj < MERGE_BATCH; jj++) {
                const int i = i0 + jj * MERGE_GROUPS;
                v[jj] = i < nz ? pp[(size_t)(z0 + i) * (D + 2) + d] : 0.0f;
            }
#pragma unroll
            for (int jj = 0; jj < MERGE_BATCH; jj++) {
                const int i = i0 + jj * MERGE_GROUPS;
                if (i < nz) o += sa[i] * v[jj];
            }
        }
    }
    so[grp][d] = o;
    if (tid == 0) sred[0] = l;
    __syncthreads();
    if (grp == 0) {   // the groups in order
        float t = so[0][d];
        for (int q = 1; q < MERGE_GROUPS; q++) t += so[q][d];
        const float lt = sred[0];
        out[(size_t)blockIdx.x * D + d] = lt > 0.0f ? t / lt : 0.0f;
    }
}

// One warp per row of D values: the row's f32 scale amax / 127 and its int8 codes.
__device__ __forceinline__ void quantize_row(const float *x, int8_t *q, float *scale, int D, int lane) {
    float amax = 0.0f;
    for (int j = 4 * lane; j < D; j += 128) {
        const float4 v = *reinterpret_cast<const float4 *>(x + j);
        amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
    }
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, m));
    const float s = amax / 127.0f;
    auto code = [&](float v) -> int {
        if (s == 0.0f) return 0;
        const int c = (int)roundf(v / s);
        return c < -127 ? -127 : (c > 127 ? 127 : c);
    };
    for (int j = 4 * lane; j < D; j += 128) {
        const float4 v = *reinterpret_cast<const float4 *>(x + j);
        *reinterpret_cast<uint32_t *>(q + j) = pack_bytes(code(v.x), code(v.y), code(v.z), code(v.w));
    }
    if (lane == 0) *scale = s;
}

__global__ void kv_quantize_i8_kernel(const float *x, int8_t *q, float *scale, int64_t rows, int D) {
    const int64_t r = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    pdl_wait();
    pdl_launch_dependents();
    if (r >= rows) return;
    quantize_row(x + r * D, q + r * D, scale + r, D, threadIdx.x & 31);
}

// Row (b, h) of x [B][Hkv][D] goes to position pos[b] of the cache [B][Hkv][Tcap][D].
__global__ void kv_append_i8_kernel(const float *x, int8_t *q, float *scale, const int32_t *pos, int64_t rows,
                                    int Hkv, int Tcap, int D, unsigned int *status) {
    const int64_t r = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    pdl_wait();
    pdl_launch_dependents();
    if (r >= rows) return;
    const int t = pos[r / Hkv];
    if (t < 0 || t >= Tcap) {
        if ((threadIdx.x & 31) == 0) atomicOr(status, STATUS_RANGE);
        return;
    }
    const int64_t cr = r * Tcap + t;
    quantize_row(x + r * D, q + cr * D, scale + cr, D, threadIdx.x & 31);
}

gq_status pdl_launch(const void *fn, dim3 grid, dim3 block, size_t smem, cudaStream_t s, void **args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return check_cuda(cudaLaunchKernelExC(&cfg, fn, args), "INT8 KV-cache kernel launch");
}

template <int D, int G>
gq_status launch_attn_dg(const AttnParams &base, int64_t B, int64_t Tcap, cudaStream_t s) {
    constexpr int CT = AtCfg<G>::CHUNK / D;
    auto kernel = attn_decode_i8_kernel<D, G>;
    // tokens per CTA: what the shared-memory row of scores holds, and few enough that
    // (sequence, KV head, range) work items fill the GPU twice over
    const int64_t per_token = 4 * (2 + G);
    const int64_t room = (int64_t)(AT_SMEM_MAX - attn_fixed_bytes<D, G>());
    const int64_t tr_max = std::max<int64_t>(CT, room / per_token / CT * CT);
    const int64_t items = B * base.Hkv;
    const int64_t want = (2 * (int64_t)sm_count() + items - 1) / items;
    int64_t S = std::max<int64_t>((Tcap + tr_max - 1) / tr_max, std::min<int64_t>(want, (Tcap + CT - 1) / CT));
    int64_t TR = ((Tcap + S - 1) / S + CT - 1) / CT * CT;
    TR = std::min(TR, tr_max);
    S = (Tcap + TR - 1) / TR;
    if (items * S > INT32_MAX) return fail(GQ_ERR_INVALID_ARG, "attention grid too large");
    AttnParams p = base;
    p.S = (int)S;
    p.TR = (int)TR;
    float *out = p.out;
    if (S > 1) {
        Workspace ws{};
        KV_TRY(get_workspace(s, 0, (size_t)B * base.Hkv * G * S * (D + 2) * sizeof(float), &ws));
        p.part = reinterpret_cast<float *>(ws.data);
    }
    const size_t smem = attn_layout<D, G>((int)TR).total;
    if (smem > AT_SMEM_MAX) return fail(GQ_ERR_INVALID_ARG, "attention layout of %zu bytes", smem);
    static std::atomic<bool> smem_set[64];   // per device: the opt-in to AT_SMEM_MAX bytes
    int dev = 0;
    KV_TRY(check_cuda(cudaGetDevice(&dev), "cudaGetDevice"));
    if (dev < 0 || dev >= 64) return fail(GQ_ERR_UNSUPPORTED_DEVICE, "device index %d", dev);
    if (!smem_set[dev].load(std::memory_order_acquire)) {
        KV_TRY(check_cuda(cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)AT_SMEM_MAX),
                          "attention shared-memory attribute"));
        smem_set[dev].store(true, std::memory_order_release);
    }
    void *args[] = {(void *)&p};
    KV_TRY(pdl_launch((const void *)kernel, dim3((unsigned)(items * S)), dim3(AtCfg<G>::THREADS), smem, s, args));
    if (S > 1) {
        const float *part = p.part;
        int Si = (int)S, Di = D;
        void *margs[] = {(void *)&part, (void *)&out, (void *)&Si, (void *)&Di};
        KV_TRY(pdl_launch(S >= MERGE_WIDE_FROM ? (const void *)attn_merge_wide_kernel : (const void *)attn_merge_kernel,
                          dim3((unsigned)(B * base.Hkv * G)), dim3(S >= MERGE_WIDE_FROM ? D * MERGE_GROUPS : D), 0, s,
                                   margs));
    }
    return GQ_OK;
}

template <int G>
gq_status launch_attn_mma(const AttnParams &base, int64_t B, int64_t Tcap, cudaStream_t s) {
    using C = AmCfg<G>;
    constexpr int CT = C::CT;
    auto kernel = attn_mma_i8_kernel<G>;
    const int64_t per_token = C::PER_TOKEN;
    const int64_t room = (int64_t)AT_SMEM_MAX - (int64_t)am_fixed_bytes<G>();
    const int64_t tr_max = std::max<int64_t>(CT, room / per_token / CT * CT);
    const int64_t items = B * base.Hkv;
    const int64_t want = (2 * (int64_t)sm_count() + items - 1) / items;
    int64_t S = std::max<int64_t>((Tcap + tr_max - 1) / tr_max, std::min<int64_t>(want, (Tcap + CT - 1) / CT));
    int64_t TR = ((Tcap + S - 1) / S + CT - 1) / CT * CT;
    TR = std::min(TR, tr_max);
    S = (Tcap + TR - 1) / TR;
    if (items * S > INT32_MAX) return fail(GQ_ERR_INVALID_ARG, "attention grid too large");
    AttnParams p = base;
    p.S = (int)S;
    p.TR = (int)TR;
    float *out = p.out;
    if (S > 1) {
        Workspace ws{};
        KV_TRY(get_workspace(s, 0, (size_t)B * base.Hkv * G * S * (C::D + 2) * sizeof(float), &ws));
        p.part = reinterpret_cast<float *>(ws.data);
    }
    const size_t smem = am_layout<G>((int)TR).total + 1024;   // + the alignment of the dynamic base
    if (smem > AT_SMEM_MAX + 1024) return fail(GQ_ERR_INVALID_ARG, "attention layout of %zu bytes", smem);
    static std::atomic<bool> smem_set[64];
    int dev = 0;
    KV_TRY(check_cuda(cudaGetDevice(&dev), "cudaGetDevice"));
    if (dev < 0 || dev >= 64) return fail(GQ_ERR_UNSUPPORTED_DEVICE, "device index %d", dev);
    if (!smem_set[dev].load(std::memory_order_acquire)) {
        KV_TRY(check_cuda(cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)(AT_SMEM_MAX + 1024)),
                          "attention shared-memory attribute"));
        smem_set[dev].store(true, std::memory_order_release);
    }
    alignas(64) CUtensorMap kmap, vmap;
    const int64_t rows = B * base.Hkv * Tcap;
    KV_TRY(byte_rows_map(&kmap, base.k, rows, CT));
    KV_TRY(byte_rows_map(&vmap, base.v, rows, CT));
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)(items * S));
    cfg.blockDim = dim3(C::THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    KV_TRY(check_cuda(cudaLaunchKernelEx(&cfg, kernel, kmap, vmap, p), "attention (tensor cores) launch"));
    if (S > 1) {
        const float *part = p.part;
        int Si = (int)S, Di = C::D;
        void *margs[] = {(void *)&part, (void *)&out, (void *)&Si, (void *)&Di};
        KV_TRY(pdl_launch(S >= MERGE_WIDE_FROM ? (const void *)attn_merge_wide_kernel : (const void *)attn_merge_kernel,
                          dim3((unsigned)(B * base.Hkv * G)), dim3(S >= MERGE_WIDE_FROM ? C::D * MERGE_GROUPS : C::D), 0,
                          s, margs));
    }
    return GQ_OK;
}

template <int D>
gq_status launch_attn_d(const AttnParams &p, int64_t B, int64_t G, int64_t Tcap, cudaStream_t s) {
    switch (G) {
        case 1: return launch_attn_dg<D, 1>(p, B, Tcap, s);
        case 2: return launch_attn_dg<D, 2>(p, B, Tcap, s);
        case 4: return launch_attn_dg<D, 4>(p, B, Tcap, s);
        case 8: return launch_attn_dg<D, 8>(p, B, Tcap, s);
    }
    return fail(GQ_ERR_INVALID_ARG, "query heads per KV head must be 1, 2, 4 or 8 (got %lld)", (long long)G);
}

}  // namespace

gq_status launch_attn_decode_i8(const float *q, const int8_t *k, const float *ks, const int8_t *v, const float *vs,
                                const int32_t *lens, float *out, int64_t B, int64_t Hq, int64_t Hkv, int64_t Tcap,
                                int64_t D, float softmax_scale, cudaStream_t s) {
    AttnParams p{};
    p.q = q;
    p.k = k;
    p.v = v;
    p.ks = ks;
    p.vs = vs;
    p.lens = lens;
    p.out = out;
    p.status = device_status_word();
    if (!p.status) return fail(GQ_ERR_CUDA, "device status word unavailable");
    p.Hkv = (int)Hkv;
    p.Tcap = (int)Tcap;
    p.c2 = softmax_scale * LOG2E;
    const int64_t G = Hq / Hkv;
    if (D == 64) return launch_attn_d<64>(p, B, G, Tcap, s);
    // D = 128: the tensor-core kernel (its tensor maps address at most 2^32 - 1 rows), unless
    // GQ_ATTN_FP32 asks for the FP32 one (a test and tuning switch)
    const char *e = getenv("GQ_ATTN_FP32");
    const bool fp32_g = G == 1 || G == 2 || G == 4 || G == 8;   // the group sizes the FP32 kernel takes
    if (B * Hkv * Tcap <= 0xFFFFFFFFLL && !(fp32_g && e && *e && atoi(e) != 0)) {
        switch (G) {
            case 1: return launch_attn_mma<1>(p, B, Tcap, s);
            case 2: return launch_attn_mma<2>(p, B, Tcap, s);
            case 3: return launch_attn_mma<3>(p, B, Tcap, s);
            case 4: return launch_attn_mma<4>(p, B, Tcap, s);
            case 5: return launch_attn_mma<5>(p, B, Tcap, s);
            case 6: return launch_attn_mma<6>(p, B, Tcap, s);
            case 7: return launch_attn_mma<7>(p, B, Tcap, s);
            case 8: return launch_attn_mma<8>(p, B, Tcap, s);
        }
    }
    if (!fp32_g)
        return fail(GQ_ERR_INVALID_ARG, "%lld query heads per KV head need the tensor-core kernel (at most 2^32 - 1 "
                    "cache rows)", (long long)G);
    return launch_attn_d<128>(p, B, G, Tcap, s);
}

gq_status launch_kv_quantize_i8(const float *x, int8_t *q, float *scale, int64_t rows, int64_t D, cudaStream_t s) {
    const int64_t blocks = (rows + 7) / 8;
    int Di = (int)D;
    void *args[] = {(void *)&x, (void *)&q, (void *)&scale, (void *)&rows, (void *)&Di};
    return pdl_launch((const void *)kv_quantize_i8_kernel, dim3((unsigned)blocks), dim3(256), 0, s, args);
}

gq_status launch_kv_append_i8(const float *x, int8_t *q, float *scale, const int32_t *pos, int64_t B, int64_t Hkv,
                              int64_t Tcap, int64_t D, cudaStream_t s) {
    unsigned int *status = device_status_word();
    if (!status) return fail(GQ_ERR_CUDA, "device status word unavailable");
    int64_t rows = B * Hkv;
    const int64_t blocks = (rows + 7) / 8;
    int Hi = (int)Hkv, Ti = (int)Tcap, Di = (int)D;
    void *args[] = {(void *)&x, (void *)&q, (void *)&scale, (void *)&pos, (void *)&rows,
                    (void *)&Hi, (void *)&Ti, (void *)&Di, (void *)&status};
    return pdl_launch((const void *)kv_append_i8_kernel, dim3((unsigned)blocks), dim3(256), 0, s, args);
}

}  // namespace gq
