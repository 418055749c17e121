// gemv.cuh -- the CUDA-core GEMV building blocks of the decode kernels: weight rows
// from shared memory (fp32, bf16, or block-quantised int8) times fp32 activation rows,
// fp32 accumulation, and a transposing warp reduction.  Used by the persistent decode
// kernel and by the cluster decode kernel.
//
// Weight types WT: kWF32 (pieces of 4 elements, 16 bytes), kWBF16 (8 elements, 16
// bytes), kWQ8 (8 int8 elements, 8 bytes; a stored row is its KBp int8 values followed by
// one fp32 scale per block of 32, and an element is scale * value).
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

template <int WT> struct Piece {
    static constexpr int elems = WT == kWF32 ? 4 : 8;  // elements per piece
    static constexpr int bytes = WT == kWQ8 ? 8 : 16;
};

// 8 int8 weights (two words) to floats: each byte, sign bit flipped, becomes the low
// mantissa byte of 1.5 * 2^23 (exact for 0..255), and subtracting 1.5 * 2^23 + 128
// leaves the signed value.
__device__ __forceinline__ void q8_unpack(uint32_t lo, uint32_t hi, float (&v)[8]) {
    const uint32_t a = lo ^ 0x80808080u, b = hi ^ 0x80808080u;
    const float off = 12583040.0f;  // 1.5 * 2^23 + 128
    v[0] = __uint_as_float(__byte_perm(a, 0x4B400000u, 0x7650)) - off;
    v[1] = __uint_as_float(__byte_perm(a, 0x4B400000u, 0x7651)) - off;
    v[2] = __uint_as_float(__byte_perm(a, 0x4B400000u, 0x7652)) - off;
    v[3] = __uint_as_float(__byte_perm(a, 0x4B400000u, 0x7653)) - off;
    v[4] = __uint_as_float(__byte_perm(b, 0x4B400000u, 0x7650)) - off;
    v[5] = __uint_as_float(__byte_perm(b, 0x4B400000u, 0x7651)) - off;
    v[6] = __uint_as_float(__byte_perm(b, 0x4B400000u, 0x7652)) - off;
    v[7] = __uint_as_float(__byte_perm(b, 0x4B400000u, 0x7653)) - off;
}

// A lane's first U pieces of each of a group's RG weight rows, held in registers: for
// the layer phases they are loaded before the input vector is polled.  (int8 weights:
// with each piece's block scale.)
template <int NB, int RG, int WT>
struct GroupW {
    static constexpr int U = Unroll<NB, RG>::value;
    uint4 w[U][RG];
    float sc[WT == kWQ8 ? U : 1][WT == kWQ8 ? RG : 1];
};

// Row r of the group at base + r * rowbytes; rows >= nr read as zero.  kbp: elements
// per stored row (where an int8 row's scales start).
template <int NB, int RG, int WT>
__device__ __forceinline__ void load_pieces(GroupW<NB, RG, WT> &G, const uint8_t *base, size_t rowbytes, int nr, int p0,
                                            int pieces, int kbp) {
#pragma unroll
    for (int u = 0; u < Unroll<NB, RG>::value; u++)
#pragma unroll
        for (int r = 0; r < RG; r++) {
            const int p = p0 + 32 * u;
            const bool on = p < pieces && r < nr;
            const uint8_t *row = base + (size_t)r * rowbytes;
            if constexpr (WT == kWQ8) {
                const uint2 q = on ? ((const uint2 *)row)[p] : make_uint2(0, 0);
                G.w[u][r] = make_uint4(q.x, q.y, 0, 0);
                G.sc[u][r] = on ? ((const float *)(row + kbp))[p >> 2] : 0.f;
            } else {
                G.w[u][r] = on ? ((const uint4 *)row)[p] : make_uint4(0, 0, 0, 0);
            }
        }
}

// acc[u][r * NB + b] += piece (p0 + 32 u) of row r . the same piece of staged row b.
template <int NB, int RG, int WT>
__device__ __forceinline__ void fma_pieces(const GroupW<NB, RG, WT> &G, int p0, int pieces, const float *xs, int KBp,
                                           int batch, float (&acc)[Unroll<NB, RG>::value][RG * NB]) {
    constexpr int U = Unroll<NB, RG>::value;
    constexpr bool WBF16 = WT != kWF32;  // 8-element pieces, activations in xpos() planes
    constexpr int EPP = Piece<WT>::elems;
    const auto &w = G.w;
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
                if constexpr (WT == kWQ8) {
                    float v[8];
                    q8_unpack(q.x, q.y, v);
                    float t = v[0] * x[0];
#pragma unroll
                    for (int e = 1; e < 8; e++) t = fmaf(v[e], x[e], t);
                    a = fmaf(G.sc[u][r], t, a);
                } else if constexpr (WBF16) {
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
template <int NB, int RG, int WT>
__device__ __forceinline__ void rows_dot(const GroupW<NB, RG, WT> &G, const uint8_t *base, size_t rowbytes, int nr,
                                         const float *xs, int KBp, int batch, float (&out)[RG * NB]) {
    constexpr int U = Unroll<NB, RG>::value;
    const int lane = threadIdx.x & 31;
    const int pieces = KBp / Piece<WT>::elems;
    float acc[U][RG * NB];
#pragma unroll
    for (int u = 0; u < U; u++)
#pragma unroll
        for (int v = 0; v < RG * NB; v++) acc[u][v] = 0.f;
    fma_pieces<NB, RG, WT>(G, lane, pieces, xs, KBp, batch, acc);
#pragma unroll 1
    for (int p0 = lane + 32 * U; p0 < pieces; p0 += 32 * U) {
        GroupW<NB, RG, WT> w;
        load_pieces<NB, RG, WT>(w, base, rowbytes, nr, p0, pieces, KBp);
        fma_pieces<NB, RG, WT>(w, p0, pieces, xs, KBp, batch, acc);
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
