// gemv.cuh -- the CUDA-core GEMV building blocks of the decode kernels: bf16 (or fp32)
// weight rows from shared memory times fp32 activation rows, fp32 accumulation, and a
// transposing warp reduction.  Used by the persistent decode kernel and by the cluster
// decode kernel.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "device_common.cuh"

namespace slm {

// Shared-memory position of element k of a staged activation row.  With bf16 weights
// a lane multiplies the 8 elements 8p..8p+7 of piece p; storing elements 8p+e at plane
// e/4, offset 4p + e%4 makes every lane's two float4 reads contiguous across the warp
// (no bank conflicts).  fp32 weights keep the natural order.
__device__ __forceinline__ int xpos(int k, int KBp, bool perm) {
    return perm ? ((k & 4) ? (KBp >> 1) : 0) + ((k >> 3) << 2) + (k & 3) : k;
}

template <int V> struct Log2 {
    static constexpr int value = V >= 32 ? 5 : V >= 16 ? 4 : V >= 8 ? 3 : V >= 4 ? 2 : V >= 2 ? 1 : 0;
};

// Sum each of the V per-lane values over the warp (V a power of two <= 32) with a
// transposing butterfly: V - 1 + 5 - log2(V) shuffles instead of 5 V.  Afterwards lane
// l holds the total of value (l >> (5 - log2 V)).
template <int V>
__device__ __forceinline__ float reduce_scatter(float (&v)[V]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int half = V / 2, off = 16; half >= 1; half >>= 1, off >>= 1) {
        const bool upper = (lane & off) != 0;
#pragma unroll
        for (int i = 0; i < half; i++) {
            const float send = upper ? v[i] : v[i + half];
            const float keep = upper ? v[i + half] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
        }
    }
#pragma unroll
    for (int off = 16 >> Log2<V>::value; off >= 1; off >>= 1) v[0] += __shfl_xor_sync(0xffffffffu, v[0], off);
    return v[0];
}

// Independent accumulator chains per (row, batch row): enough to keep the FMA pipe and
// the shared-memory loads busy with two warps per scheduler.
template <int NB, int RG> struct Unroll {
    static constexpr int value = RG * NB >= 8 ? 1 : RG * NB >= 4 ? 2 : 3;
};

// A lane's first U pieces of each of a group's RG weight rows, held in registers: for
// the layer phases they are loaded before the input vector is polled.
template <int NB, int RG, bool WBF16>
struct GroupW {
    static constexpr int U = Unroll<NB, RG>::value;
    uint4 w[U][RG];
};

// Row r of the group at base + r * rowbytes; rows >= nr read as zero.
template <int NB, int RG, bool WBF16>
__device__ __forceinline__ void load_pieces(uint4 (&w)[Unroll<NB, RG>::value][RG], const uint8_t *base, size_t rowbytes,
                                            int nr, int p0, int pieces) {
#pragma unroll
    for (int u = 0; u < Unroll<NB, RG>::value; u++)
#pragma unroll
        for (int r = 0; r < RG; r++) {
            const int p = p0 + 32 * u;
            w[u][r] = (p < pieces && r < nr) ? ((const uint4 *)(base + (size_t)r * rowbytes))[p] : make_uint4(0, 0, 0, 0);
        }
}

// acc[u][r * NB + b] += piece (p0 + 32 u) of row r . the same piece of staged row b.
template <int NB, int RG, bool WBF16>
__device__ __forceinline__ void fma_pieces(const uint4 (&w)[Unroll<NB, RG>::value][RG], int p0, int pieces,
                                           const float *xs, int KBp, int batch,
                                           float (&acc)[Unroll<NB, RG>::value][RG * NB]) {
    constexpr int U = Unroll<NB, RG>::value;
    constexpr int EPP = WBF16 ? 8 : 4;
    (void)EPP;
#pragma unroll
    for (int u = 0; u < U; u++) {
        const int p = p0 + 32 * u;
        if (p >= pieces) break;
#pragma unroll
        for (int b = 0; b < NB; b++) {
            if (NB > 1 && b >= batch) break;
            float x[EPP];
            if constexpr (WBF16) {
                const float *xr = xs + (size_t)b * KBp + p * 4;  // planes of xpos()
                const float4 x0 = *(const float4 *)xr, x1 = *(const float4 *)(xr + (KBp >> 1));
                x[0] = x0.x; x[1] = x0.y; x[2] = x0.z; x[3] = x0.w;
                x[4] = x1.x; x[5] = x1.y; x[6] = x1.z; x[7] = x1.w;
            } else {
                const float4 x0 = *(const float4 *)(xs + (size_t)b * KBp + p * 4);
                x[0] = x0.x; x[1] = x0.y; x[2] = x0.z; x[3] = x0.w;
            }
#pragma unroll
            for (int r = 0; r < RG; r++) {
                const uint4 q = w[u][r];
                float &a = acc[u][r * NB + b];
                if constexpr (WBF16) {
                    a = fmaf(bf16_lo(q.x), x[0], a);
                    a = fmaf(bf16_hi(q.x), x[1], a);
                    a = fmaf(bf16_lo(q.y), x[2], a);
                    a = fmaf(bf16_hi(q.y), x[3], a);
                    a = fmaf(bf16_lo(q.z), x[4], a);
                    a = fmaf(bf16_hi(q.z), x[5], a);
                    a = fmaf(bf16_lo(q.w), x[6], a);
                    a = fmaf(bf16_hi(q.w), x[7], a);
                } else {
                    a = fmaf(__uint_as_float(q.x), x[0], a);
                    a = fmaf(__uint_as_float(q.y), x[1], a);
                    a = fmaf(__uint_as_float(q.z), x[2], a);
                    a = fmaf(__uint_as_float(q.w), x[3], a);
                }
            }
        }
    }
}

// Dots of RG weight rows with every staged batch row: the lane's first U pieces per row
// come from G, the rest from shared memory.  Value index r * NB + b.
template <int NB, int RG, bool WBF16>
__device__ __forceinline__ void rows_dot(const GroupW<NB, RG, WBF16> &G, const uint8_t *base, size_t rowbytes, int nr,
                                         const float *xs, int KBp, int batch, float (&out)[RG * NB]) {
    constexpr int U = Unroll<NB, RG>::value;
    const int lane = threadIdx.x & 31;
    const int pieces = KBp / (WBF16 ? 8 : 4);
    float acc[U][RG * NB];
#pragma unroll
    for (int u = 0; u < U; u++)
#pragma unroll
        for (int v = 0; v < RG * NB; v++) acc[u][v] = 0.f;
    fma_pieces<NB, RG, WBF16>(G.w, lane, pieces, xs, KBp, batch, acc);
#pragma unroll 1
    for (int p0 = lane + 32 * U; p0 < pieces; p0 += 32 * U) {
        uint4 w[U][RG];
        load_pieces<NB, RG, WBF16>(w, base, rowbytes, nr, p0, pieces);
        fma_pieces<NB, RG, WBF16>(w, p0, pieces, xs, KBp, batch, acc);
    }
#pragma unroll
    for (int v = 0; v < RG * NB; v++) {
        float t = acc[0][v];
#pragma unroll
        for (int u = 1; u < U; u++) t += acc[u][v];
        out[v] = t;
    }
}

}  // namespace slm
