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
                                 //   addressed as if it started at position 0); with
    const int *pages;            //   pages: position t at pages[t >> page_shift] * page_stride
    size_t page_stride;          //   + (t & page_mask) * hd elements (a paged cache)
    int page_shift, page_mask;
    const uint8_t *tail_k;       // position tail_t is read from these rows instead (the
    const uint8_t *tail_v;       //   step's own key and value); tail_t = -1: none
    int tail_t;
    uint8_t *stream;             // if set: shared memory for the streamed read of a chunk
    int stream_bytes;            //   in global memory (kAttnMaxSlots passes per warp at most)
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

// Eight consecutive elements of a cached key or value row (global or shared memory).
template <bool BF16>
__device__ __forceinline__ void load_row8(const uint8_t *row, int d0, float (&v)[8]) {
    if (BF16) {
        const uint4 u = *(const uint4 *)(row + d0 * 2);
        v[0] = bf16_lo(u.x); v[1] = bf16_hi(u.x); v[2] = bf16_lo(u.y); v[3] = bf16_hi(u.y);
        v[4] = bf16_lo(u.z); v[5] = bf16_hi(u.z); v[6] = bf16_lo(u.w); v[7] = bf16_hi(u.w);
    } else {
        const float4 a = *(const float4 *)(row + d0 * 4);
        const float4 b = *(const float4 *)(row + d0 * 4 + 16);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    }
}

// This warp's positions of one item: pass k takes positions t0 + (k * warps + warp) * PP
// ..., one per lane group of LPP lanes (each lane 8 of the head_dim elements).  Every
// pass scores the position against kMaxGroupPass query heads (heads past the group have
// q = 0 and are ignored by the caller) and folds it into each head's online softmax:
// the sums are rescaled only when the running max grows.
//
// SPLIT (LPP >= 4): the lane group's reduction of the four partial scores also hands
// out the heads: after two exchange rounds each quarter of the group holds one head's
// partial sums (head 2a + b for the lanes whose sub index has bits a = LPP/2, b = LPP/4),
// the remaining rounds finish that head's score, and each lane runs the softmax update
// of its one head; the weights (and, when a max grew, the rescale factors) are then
// broadcast to the group for the weighted sum of V, which every lane keeps for all heads
// on its 8 elements.  Otherwise every lane reduces and updates all four heads.
//
// Streamed (T.stream with room for at least two passes per warp): the warp's K and V
// rows of pass k are copied into slot k % S of its own shared-memory ring S - 1 passes
// ahead, so that each warp keeps S - 1 passes in flight (a long chunk read straight from
// the cache is bound by load latency).  Only cached rows [t0, tail) are copied; the new
// position is read from the tail rows.  Otherwise the rows are read where kbase / vbase
// point (the cache, or a whole-chunk copy in shared memory).
template <bool BF16, bool SPLIT>
__device__ __forceinline__ void attn_scan(const AttnTask &T, const float (&qv)[kMaxGroupPass][8],
                                          float (&mx)[kMaxGroupPass], float (&ls)[kMaxGroupPass],
                                          float (&o)[kMaxGroupPass][8], int warp, int lane, int LPP, int PP,
                                          int grp, bool lane_on, int d0) {
    static_assert(kMaxGroupPass == 4, "the head split hands out four heads");
    const int rowbytes = T.hd * (BF16 ? 2 : 4);
    const int t0 = T.t0, t1 = T.t1;
    const int stride = kComputeWarps * PP;     // positions of one pass of all warps
    const int slotb = 2 * PP * rowbytes;       // one warp's K and V rows of one pass
    const int per_warp = T.stream ? T.stream_bytes / kComputeWarps / 16 * 16 : 0;
    const int S = min(kAttnMaxSlots, per_warp / slotb);
    const bool streamed = S >= 2;
    uint8_t *ring = T.stream + (size_t)warp * per_warp;
    const int tc = T.tail_t >= 0 ? min(t1, T.tail_t) : t1;
    const int npass = (t1 - t0 + stride - 1) / stride;
    const int rows16 = rowbytes / 16;
    // head split: this lane's head, and the lane of its group that owns head h
    const int sub = lane & (LPP - 1), base = lane - sub;
    const bool bitA = SPLIT && (sub & (LPP >> 1)), bitB = SPLIT && (sub & (LPP >> 2));
    auto owner = [&](int h) { return base + (h >> 1) * (LPP >> 1) + (h & 1) * (LPP >> 2); };
    float m_own = -INFINITY, l_own = 0.f;
    int wr = 0, rd = 0;  // ring slots of the next copy and of the next pass
    // byte offset of position t's row (a pass's PP rows never cross a page: pages hold a
    // multiple of 16 rows and passes start at multiples of PP <= 16)
    auto row_off = [&](int t) -> size_t {
        return T.pages ? (size_t)__ldg(T.pages + (t >> T.page_shift)) * T.page_stride +
                             (size_t)(t & T.page_mask) * rowbytes
                       : (size_t)t * rowbytes;
    };
    auto issue = [&](int k) {
        if (k < npass) {
            const int p0 = t0 + k * stride + warp * PP;
            const int n = max(0, min(PP, tc - p0)) * rows16;  // 16-byte pieces
            uint8_t *dst = ring + (size_t)wr * slotb;
            const size_t src = n > 0 ? row_off(p0) : 0;
            for (int e = lane; e < n; e += 32) {
                cp_async16(dst + e * 16, T.kbase + src + e * 16);
                cp_async16(dst + PP * rowbytes + e * 16, T.vbase + src + e * 16);
            }
        }
        cp_async_commit();  // empty groups too: every lane counts the same groups
        wr = wr + 1 == S ? 0 : wr + 1;
    };
    if (streamed)
        for (int k = 0; k < S - 1; k++) issue(k);
    for (int k = 0; k < npass; k++) {
        const int p0 = t0 + k * stride + warp * PP;
        const uint8_t *kr, *vr;
        if (streamed) {
            issue(k + S - 1);
            cp_async_wait_upto(S - 1);  // this lane's copies of pass k have landed
            __syncwarp();               // ... and every lane's
            kr = ring + (size_t)rd * slotb;
            vr = kr + PP * rowbytes;
            rd = rd + 1 == S ? 0 : rd + 1;
        } else {
            const size_t off = p0 < t1 ? row_off(p0) : 0;
            kr = T.kbase + off;
            vr = T.vbase + off;
        }
        const int t = p0 + grp;
        const bool valid = t < t1;
        float kv8[8], vv8[8];
        if (valid && lane_on) {
            const bool tl = t == T.tail_t;
            load_row8<BF16>(tl ? T.tail_k : kr + grp * rowbytes, d0, kv8);
            load_row8<BF16>(tl ? T.tail_v : vr + grp * rowbytes, d0, vv8);
        } else {
#pragma unroll
            for (int d = 0; d < 8; d++) kv8[d] = vv8[d] = 0.f;
        }
        float s[kMaxGroupPass];
#pragma unroll
        for (int j = 0; j < kMaxGroupPass; j++) {
            float a = 0.f, b = 0.f;
#pragma unroll
            for (int d = 0; d < 8; d += 2) {
                a = fmaf(qv[j][d], kv8[d], a);
                b = fmaf(qv[j][d + 1], kv8[d + 1], b);
            }
            s[j] = a + b;
        }
        if (SPLIT) {
            float k0 = bitA ? s[2] : s[0], k1 = bitA ? s[3] : s[1];
            k0 += __shfl_xor_sync(0xffffffffu, bitA ? s[0] : s[2], LPP >> 1);
            k1 += __shfl_xor_sync(0xffffffffu, bitA ? s[1] : s[3], LPP >> 1);
            float sc = (bitB ? k1 : k0) + __shfl_xor_sync(0xffffffffu, bitB ? k0 : k1, LPP >> 2);
#pragma unroll
            for (int off = 1; off < 8; off <<= 1)
                if (off < (LPP >> 2)) sc += __shfl_xor_sync(0xffffffffu, sc, off);  // uniform
            float corr = 1.f, p = 0.f;
            if (valid) {
                if (sc > m_own) {  // a new running max (always at the first position)
                    corr = fast_exp2(m_own - sc);
                    l_own *= corr;
                    m_own = sc;
                }
                p = fast_exp2(sc - m_own);
                l_own += p;
            }
            if (__any_sync(0xffffffffu, corr != 1.f)) {
#pragma unroll
                for (int j = 0; j < kMaxGroupPass; j++) {
                    const float cj = __shfl_sync(0xffffffffu, corr, owner(j));
#pragma unroll
                    for (int d = 0; d < 8; d++) o[j][d] *= cj;
                }
            }
#pragma unroll
            for (int j = 0; j < kMaxGroupPass; j++) {
                const float pj = __shfl_sync(0xffffffffu, p, owner(j));
#pragma unroll
                for (int d = 0; d < 8; d++) o[j][d] = fmaf(pj, vv8[d], o[j][d]);
            }
        } else {
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                if (off < LPP) {  // uniform across the warp
#pragma unroll
                    for (int j = 0; j < kMaxGroupPass; j++) s[j] += __shfl_xor_sync(0xffffffffu, s[j], off);
                }
            }
            if (valid) {
#pragma unroll
                for (int j = 0; j < kMaxGroupPass; j++) {
                    if (s[j] > mx[j]) {  // a new running max (always at the first position)
                        const float corr = fast_exp2(mx[j] - s[j]);
                        ls[j] *= corr;
#pragma unroll
                        for (int d = 0; d < 8; d++) o[j][d] *= corr;
                        mx[j] = s[j];
                    }
                    const float p = fast_exp2(s[j] - mx[j]);
                    ls[j] += p;
#pragma unroll
                    for (int d = 0; d < 8; d++) o[j][d] = fmaf(p, vv8[d], o[j][d]);
                }
            }
        }
        if (streamed) __syncwarp();  // the slot just read is refilled by the next pass
    }
    if (streamed) cp_async_wait_upto(0);
    if (SPLIT) {  // every lane of the group takes each head's (max, sum) from its owner
#pragma unroll
        for (int j = 0; j < kMaxGroupPass; j++) {
            mx[j] = __shfl_sync(0xffffffffu, m_own, owner(j));
            ls[j] = __shfl_sync(0xffffffffu, l_own, owner(j));
        }
    }
}

// The scan of a long chunk on the tensor cores (bf16 cache, head_dim HD = 64, streamed).
// The chunk is a small dense contraction: the G query heads against the positions' keys,
// then the weights against the values; as CUDA-core code its per-position instructions
// (shuffles, the online update) bounded the phase, not HBM.  Here each warp takes
// passes of 8 positions: S = Q K^T (16 x 8, rows = heads, q as bf16 A fragments,
// mma.sync m16n8k16), the online softmax on the accumulator rows (quad shuffles), and
// O += P V (P as bf16 A fragments, mma.sync m16n8k8 over HD / 8 dim tiles) -- the
// prefill's precision (q and p enter as bf16, fp32 accumulation).  The rows of pass k
// reach its ring slot S - 1 passes ahead by cp.async, 16 bytes further apart than in
// the cache so that ldmatrix reads them without bank conflicts.  The warp's state
// (max, sum, weighted V) of each head j < Gp goes to ws like the CUDA-core scan's.
template <int HD>
__device__ __forceinline__ void attn_scan_mma(const AttnTask &T, const float *qs, int Gp, float *ws, int warp,
                                              int lane) {
    constexpr int RB = HD * 2, RS = RB + 16, NP = 8;  // row bytes, slot row stride, positions
    const int t0 = T.t0, t1 = T.t1;
    const int stride = kComputeWarps * NP;
    const int slotb = 2 * NP * RS;
    const int per_warp = T.stream_bytes / kComputeWarps / 16 * 16;
    const int S = min(kAttnMaxSlots, per_warp / slotb);  // >= 2: the caller checks
    uint8_t *ring = T.stream + (size_t)warp * per_warp;
    const int tc = T.tail_t >= 0 ? min(t1, T.tail_t) : t1;
    const int npass = (t1 - t0 + stride - 1) / stride;
    const int g4 = lane >> 2, t4 = lane & 3;
    auto row_off = [&](int t) -> size_t {
        return T.pages ? (size_t)__ldg(T.pages + (t >> T.page_shift)) * T.page_stride + (size_t)(t & T.page_mask) * RB
                       : (size_t)t * RB;
    };
    // q (already scaled to log2 units) as A fragments: rows = heads, zero past Gp
    uint32_t qa[HD / 16][4];
#pragma unroll
    for (int kk = 0; kk < HD / 16; kk++) {
        const int c = kk * 16 + 2 * t4;
        const bool on = g4 < Gp;
        qa[kk][0] = on ? pack_bf16x2(qs[g4 * HD + c], qs[g4 * HD + c + 1]) : 0u;
        qa[kk][1] = 0u;
        qa[kk][2] = on ? pack_bf16x2(qs[g4 * HD + c + 8], qs[g4 * HD + c + 9]) : 0u;
        qa[kk][3] = 0u;
    }
    float o[HD / 8][4];
#pragma unroll
    for (int n = 0; n < HD / 8; n++) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    float m_run = -INFINITY, l_run = 0.f;  // row g4 (this lane's two positions of each pass)
    int wr = 0, rd = 0;
    auto issue = [&](int k) {
        if (k < npass) {
            const int p0 = t0 + k * stride + warp * NP;
            const int n = max(0, min(NP, tc - p0)) * (RB / 16);  // 16-byte pieces of K (and of V)
            uint8_t *dst = ring + (size_t)wr * slotb;
            const size_t src = n > 0 ? row_off(p0) : 0;  // a pass never crosses a page
            for (int e = lane; e < n; e += 32) {
                const int r = e / (RB / 16), pc = e - r * (RB / 16);
                cp_async16(dst + r * RS + pc * 16, T.kbase + src + (size_t)r * RB + pc * 16);
                cp_async16(dst + (NP + r) * RS + pc * 16, T.vbase + src + (size_t)r * RB + pc * 16);
            }
        }
        cp_async_commit();
        wr = wr + 1 == S ? 0 : wr + 1;
    };
    for (int k = 0; k < S - 1; k++) issue(k);
    for (int k = 0; k < npass; k++) {
        const int p0 = t0 + k * stride + warp * NP;
        issue(k + S - 1);
        cp_async_wait_upto(S - 1);
        __syncwarp();
        uint8_t *ks = ring + (size_t)rd * slotb, *vs = ks + NP * RS;
        rd = rd + 1 == S ? 0 : rd + 1;
        if (p0 + NP > t1) {  // rows past the chunk: zero V (their weights are 0, and 0 * NaN is not)
            const int r0 = max(0, t1 - p0);
            for (int e = lane; e < (NP - r0) * (RB / 16); e += 32)
                *(uint4 *)(vs + (r0 + e / (RB / 16)) * RS + (e % (RB / 16)) * 16) = make_uint4(0, 0, 0, 0);
            __syncwarp();
        }
        if (T.tail_t >= p0 && T.tail_t < p0 + NP) {  // the new position's row from the exchange
            const int r = T.tail_t - p0;
            if (lane < RB / 16)
                *(uint4 *)(ks + r * RS + lane * 16) = *(const uint4 *)(T.tail_k + lane * 16);
            else if (lane < 2 * (RB / 16))
                *(uint4 *)(vs + r * RS + (lane - RB / 16) * 16) = *(const uint4 *)(T.tail_v + (lane - RB / 16) * 16);
            __syncwarp();
        }
        float sc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int kk = 0; kk < HD / 16; kk += 2) {  // two k steps per x4 load
            uint32_t b[4];
            ldsm_x4(b, ks + (lane & 7) * RS + (kk * 16 + (lane >> 3) * 8) * 2);
            mma_bf16_16816(sc, qa[kk], b[0], b[1]);
            mma_bf16_16816(sc, qa[kk + 1], b[2], b[3]);
        }
        const int pa = p0 + 2 * t4;
        const float s0 = pa < t1 ? sc[0] : -INFINITY, s1 = pa + 1 < t1 ? sc[1] : -INFINITY;
        float mx = fmaxf(s0, s1);
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        const float m_new = fmaxf(m_run, mx);
        if (m_new > m_run) {  // the running max grew (always at the first position)
            const float corr = fast_exp2(m_run - m_new);  // 0 when m_run = -inf
            l_run *= corr;
#pragma unroll
            for (int n = 0; n < HD / 8; n++) {
                o[n][0] *= corr;
                o[n][1] *= corr;
            }
            m_run = m_new;
        }
        const float p0v = m_run == -INFINITY ? 0.f : fast_exp2(s0 - m_run);
        const float p1v = m_run == -INFINITY ? 0.f : fast_exp2(s1 - m_run);
        l_run += p0v + p1v;
        const uint32_t pa0 = pack_bf16x2(p0v, p1v);
#pragma unroll
        for (int nb = 0; nb < HD / 32; nb++) {  // four dim tiles per x4 load
            uint32_t b[4];
            ldsm_x4_t(b, vs + (lane & 7) * RS + (nb * 32 + (lane >> 3) * 8) * 2);
#pragma unroll
            for (int i = 0; i < 4; i++) mma_bf16_1688(o[nb * 4 + i], pa0, 0u, b[i]);
        }
        __syncwarp();  // the slot just read is refilled by the next pass
    }
    cp_async_wait_upto(0);
    l_run += __shfl_xor_sync(0xffffffffu, l_run, 1);
    l_run += __shfl_xor_sync(0xffffffffu, l_run, 2);
    if (g4 < Gp) {
        float *w = ws + ((size_t)warp * kMaxGroupPass + g4) * (HD + 2);
#pragma unroll
        for (int n = 0; n < HD / 8; n++) {
            w[2 + n * 8 + 2 * t4] = o[n][0];
            w[3 + n * 8 + 2 * t4] = o[n][1];
        }
        if (t4 == 0) {
            w[0] = m_run;
            w[1] = l_run;
        }
    }
}

// All kComputeThreads threads of the CTA call this.  `scratch` holds
// kMaxGroupPass * hd + kComputeWarps * kMaxGroupPass * (hd + 2) floats; `flag` one int.
__device__ __forceinline__ void attn_core(const AttnTask &T, float *scratch, int *flag) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int hd = T.hd, G = T.G;
    const int nc = T.nc, c = T.c;
    const bool kvbf16 = T.kv_bf16;
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
        if (kvbf16 && hd == 64 && T.stream &&
            T.stream_bytes / kComputeWarps / 16 * 16 >= 2 * (2 * 8 * (64 * 2 + 16))) {
            attn_scan_mma<64>(T, qsrc, Gp, ws, warp, lane);  // long chunk: tensor cores
        } else {
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
        if (kvbf16 && LPP >= 4)
            attn_scan<true, true>(T, qv, mx, ls, o, warp, lane, LPP, PP, grp, lane_on, d0);
        else if (kvbf16)
            attn_scan<true, false>(T, qv, mx, ls, o, warp, lane, LPP, PP, grp, lane_on, d0);
        else
            attn_scan<false, false>(T, qv, mx, ls, o, warp, lane, LPP, PP, grp, lane_on, d0);
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
