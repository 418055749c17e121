// attention.cuh -- split-K GQA decode attention over one chunk of cached positions
// (flash-decoding).  Shared by the decode kernel and the stand-alone attention op.
// q arrives with RoPE applied; the cache holds rotated keys.
//
// softmax(q K^T / sqrt(d_head)) V for the G query heads that read one kv head
// (kasahare 0.4.0 / simple-llm, "Architecture": GQA with n_kv_heads <= n_heads).  The
// chunk's keys and values are read once for all G heads; each head keeps an online
// softmax (running max, sum and weighted V) in the log2 domain; lanes, then warps, then
// chunks are merged by rescaling to a common max.  The CTA that finishes a (row, kv
// head) last merges the chunks' partial states.
#pragma once

#include "device_common.cuh"

namespace slm {

// Eight consecutive elements of a cached key or value row (global or shared memory).
__device__ __forceinline__ void load8(const uint8_t *row, int d0, bool kvbf16, float (&v)[8]) {
    if (kvbf16) {
        uint4 u = *(const uint4 *)(row + d0 * 2);
        v[0] = bf16_lo(u.x); v[1] = bf16_hi(u.x); v[2] = bf16_lo(u.y); v[3] = bf16_hi(u.y);
        v[4] = bf16_lo(u.z); v[5] = bf16_hi(u.z); v[6] = bf16_lo(u.w); v[7] = bf16_hi(u.w);
    } else {
        float4 a = *(const float4 *)(row + d0 * 4);
        float4 b = *(const float4 *)(row + d0 * 4 + 16);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    }
}

__device__ __forceinline__ float kv_round(float v, bool bf16) {
    return bf16 ? __bfloat162float(__float2bfloat16_rn(v)) : v;
}

// Online-softmax merge of (m, l, o) pairs in the log2 domain.
__device__ __forceinline__ void merge_state(float &m, float &l, float (&o)[8], float m2, float l2,
                                            const float (&o2)[8]) {
    float M = fmaxf(m, m2);
    float a = (m == -INFINITY) ? 0.f : exp2f(m - M);
    float b = (m2 == -INFINITY) ? 0.f : exp2f(m2 - M);
    l = l * a + l2 * b;
#pragma unroll
    for (int d = 0; d < 8; d++) o[d] = o[d] * a + o2[d] * b;
    m = M;
}


// One work item: G query heads x positions [t0, t1) of one (row, kv head).
struct AttnTask {
    const float *q;              // query rows of the group, head j at q + j * hd, RoPE applied;
                                 //   complete before the call
    bool q_ready;                // q already multiplied by log2(e) / sqrt(hd) and in shared
                                 //   memory; otherwise scaled here into the scratch
    bool kv_bf16;                // cache element type: bf16 or fp32
    const uint8_t *kbase;        // keys of the (row, kv head): position t at t * hd elements
    const uint8_t *vbase;        //   (global cache, or a shared-memory copy of the chunk
                                 //   addressed as if it started at position 0)
    const uint8_t *tail_k;       // position tail_t is read from these rows instead (the
    const uint8_t *tail_v;       //   step's own key and value); tail_t = -1: none
    int tail_t;
    float *out;                  // final output rows: head j at out + j * hd
    float *part;                 // partials: head j, chunk c at (j * kMaxChunksPerSeq + c) * (hd + 2)
    int *counter;                // arrivals of this (row, kv head)'s chunks
    uint64_t *ll_part;           // if set: publish this chunk's states as tagged words
                                 //   (head j at (j * ncap + c) * (hd + 2)); no merge here
    uint64_t *ll_out;            // if set: publish the merged output as tagged words
    uint32_t tag;
    int ncap;                    // chunk capacity of ll_part
    int hd, G, t0, t1, nc, c;
};

// All kComputeThreads threads of the CTA call this.  `scratch` holds
// kMaxGroupPass * hd + kComputeWarps * kMaxGroupPass * (hd + 2) floats; `flag` one int.
__device__ __forceinline__ void attn_core(const AttnTask &T, float *scratch, int *flag) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int hd = T.hd, G = T.G;
    const int t0 = T.t0, t1 = T.t1, nc = T.nc, c = T.c;
    const bool kvbf16 = T.kv_bf16;
    const size_t rowbytes = (size_t)hd * (kvbf16 ? 2 : 4);
    const uint8_t *kbase = T.kbase, *vbase = T.vbase;
    const float qscale = rsqrtf((float)hd) * 1.4426950408889634f;  // scores in log2 units
    float *qs = scratch;
    float *ws = scratch + kMaxGroupPass * hd;
    const int LP = hd / 8;           // lanes holding data for one position
    int LPP = 1;                     // lanes per position, rounded up to a power of two
    while (LPP < LP) LPP <<= 1;
    const int PP = 32 / LPP;         // positions per warp pass
    const int grp = lane / LPP, sub = lane % LPP;
    const bool lane_on = sub < LP;   // lanes past head_dim / 8 carry zeros
    const int d0 = sub * 8;

    for (int jp = 0; jp < G; jp += kMaxGroupPass) {
        const int Gp = min(kMaxGroupPass, G - jp);
        const float *qsrc = T.q + (size_t)jp * hd;
        if (jp > 0 || !T.q_ready) compute_sync();  // previous users of qs / ws are done
        if (!T.q_ready) {
            for (int e = tid; e < Gp * hd; e += kComputeThreads) qs[e] = qsrc[e] * qscale;  // q may be global
            compute_sync();
            qsrc = qs;
        }
        float qv[kMaxGroupPass][8];
#pragma unroll
        for (int j = 0; j < kMaxGroupPass; j++)
#pragma unroll
            for (int d = 0; d < 8; d++) qv[j][d] = (j < Gp && lane_on) ? qsrc[j * hd + d0 + d] : 0.f;
        float mx[kMaxGroupPass], ls[kMaxGroupPass], o[kMaxGroupPass][8];
#pragma unroll
        for (int j = 0; j < kMaxGroupPass; j++) {
            mx[j] = -INFINITY;
            ls[j] = 0.f;
#pragma unroll
            for (int d = 0; d < 8; d++) o[j][d] = 0.f;
        }
        for (int tb = t0 + warp * PP; tb < t1; tb += kComputeWarps * PP) {
            const int t = tb + grp;
            const bool valid = t < t1;
            float kv8[8], vv8[8];
            if (valid && lane_on) {
                const bool tl = t == T.tail_t;
                load8(tl ? T.tail_k : kbase + (size_t)t * rowbytes, d0, kvbf16, kv8);
                load8(tl ? T.tail_v : vbase + (size_t)t * rowbytes, d0, kvbf16, vv8);
            } else {
#pragma unroll
                for (int d = 0; d < 8; d++) kv8[d] = vv8[d] = 0.f;
            }
#pragma unroll
            for (int j = 0; j < kMaxGroupPass; j++) {
                if (j >= Gp) break;
                float s = 0.f;
#pragma unroll
                for (int d = 0; d < 8; d++) s = fmaf(qv[j][d], kv8[d], s);
                for (int off = 1; off < LPP; off <<= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
                if (valid) {
                    float mn = fmaxf(mx[j], s);
                    float corr = exp2f(mx[j] - mn);  // exp2(-inf) = 0 on the first position
                    float p = exp2f(s - mn);
                    ls[j] = ls[j] * corr + p;
#pragma unroll
                    for (int d = 0; d < 8; d++) o[j][d] = fmaf(p, vv8[d], o[j][d] * corr);
                    mx[j] = mn;
                }
            }
        }
        // merge the position groups of this warp (lanes with the same `sub`)
#pragma unroll
        for (int j = 0; j < kMaxGroupPass; j++) {
            if (j >= Gp) break;
            for (int off = LPP; off < LPP * PP; off <<= 1) {
                float m2 = __shfl_xor_sync(0xffffffffu, mx[j], off);
                float l2 = __shfl_xor_sync(0xffffffffu, ls[j], off);
                float o2[8];
#pragma unroll
                for (int d = 0; d < 8; d++) o2[d] = __shfl_xor_sync(0xffffffffu, o[j][d], off);
                merge_state(mx[j], ls[j], o[j], m2, l2, o2);
            }
            if (grp == 0 && lane_on) {
                float *w = ws + ((size_t)warp * kMaxGroupPass + j) * (hd + 2);
#pragma unroll
                for (int d = 0; d < 8; d++) w[2 + d0 + d] = o[j][d];
                if (sub == 0) {
                    w[0] = mx[j];
                    w[1] = ls[j];
                }
            }
        }
        compute_sync();
        // merge the warps: thread e handles (head j, dim d)
        for (int e = tid; e < Gp * hd; e += kComputeThreads) {
            int j = e / hd, d = e - j * hd;
            float M = -INFINITY;
            for (int w = 0; w < kComputeWarps; w++)
                M = fmaxf(M, ws[((size_t)w * kMaxGroupPass + j) * (hd + 2)]);
            float L = 0.f, O = 0.f;
            for (int w = 0; w < kComputeWarps; w++) {
                const float *st = ws + ((size_t)w * kMaxGroupPass + j) * (hd + 2);
                if (st[0] == -INFINITY) continue;
                float sc = exp2f(st[0] - M);
                L = fmaf(st[1], sc, L);
                O = fmaf(st[2 + d], sc, O);
            }
            if (T.ll_part) {
                uint64_t *pp = T.ll_part + ((size_t)(jp + j) * T.ncap + c) * (hd + 2);
                ll_store(pp + 2 + d, O, T.tag);
                if (d == 0) {
                    ll_store(pp, M, T.tag);
                    ll_store(pp + 1, L, T.tag);
                }
            } else if (nc == 1) {
                if (T.ll_out)
                    ll_store(T.ll_out + (size_t)(jp + j) * hd + d, O / L, T.tag);
                else
                    T.out[(size_t)(jp + j) * hd + d] = O / L;
            } else {
                float *pp = T.part + ((size_t)(jp + j) * kMaxChunksPerSeq + c) * (hd + 2);
                pp[2 + d] = O;
                if (d == 0) {
                    pp[0] = M;
                    pp[1] = L;
                }
            }
        }
    }
    if (T.ll_part || nc == 1) return;
    // split-K: the last CTA to finish a (row, kv head) merges its chunks
    compute_sync();
    if (tid == 0) {
        __threadfence();
        int prev = atomicAdd(T.counter, 1);
        *flag = (prev == nc - 1);
    }
    compute_sync();
    if (!*flag) return;
    __threadfence();
    for (int e = tid; e < G * hd; e += kComputeThreads) {
        int j = e / hd, d = e - j * hd;
        const float *pp = T.part + (size_t)j * kMaxChunksPerSeq * (hd + 2);
        float M = -INFINITY;
        for (int cc = 0; cc < nc; cc++) M = fmaxf(M, __ldcg(pp + (size_t)cc * (hd + 2)));
        float L = 0.f, O = 0.f;
        for (int cc = 0; cc < nc; cc++) {
            const float *st = pp + (size_t)cc * (hd + 2);
            float mc = __ldcg(st);
            if (mc == -INFINITY) continue;
            float sc = exp2f(mc - M);
            L = fmaf(__ldcg(st + 1), sc, L);
            O = fmaf(__ldcg(st + 2 + d), sc, O);
        }
        if (T.ll_out)
            ll_store(T.ll_out + (size_t)j * hd + d, O / L, T.tag);
        else
            T.out[(size_t)j * hd + d] = O / L;
    }
    if (tid == 0) *(volatile int *)T.counter = 0;
}


}  // namespace slm
