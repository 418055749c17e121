// decode_kernel.cu -- the KV-cached greedy decode step as one persistent kernel.
//
// One cooperative launch computes a whole step for every batch row (kasahare 0.4.0 /
// simple-llm, "Architecture": RMSNorm, Wq/Wk/Wv without biases, RoPE, KV append, GQA
// softmax(q K^T / sqrt(d_head)) V, Wo + residual, RMSNorm, W2(silu(W1 x) * (W3 x)) +
// residual; then the final RMSNorm, the tied-embedding logits and the greedy argmax).
//
// Structure (one CTA per SM, 8 compute warps + 1 streaming warp):
//  * Weights do not depend on activations, so the streaming warp walks this CTA's
//    share of every matrix of the step (layer by layer, in consumption order) and
//    copies it HBM -> shared memory with cp.async.bulk into a ring of 16 KB slots,
//    signalled by mbarriers.  It runs ahead of the compute warps across phases.
//  * Each GEMV phase splits its output rows evenly over the CTAs.  A phase's input is
//    a vector produced by other CTAs; instead of grid barriers, producers publish every
//    element as a tagged 8-byte word (value + this launch's tag, one atomic store) and
//    consumers poll the words they need until the tags match: one L2 round trip per
//    hand-off, no fence, no counter.  Exchange buffers are per layer, so nothing is
//    rewritten within a launch.
//  * Each CTA keeps the residual rows it owns (the rows of Wo and W2 it computes) in
//    shared memory, so the residual adds read nothing from memory.
//  * GEMV: fp32 activations in shared memory, bf16 weights widened by shifts, fp32 FMA,
//    butterfly warp reduction.  Epilogues are fused: QKV publish, residual add (Wo,
//    W2), SwiGLU over interleaved W1/W3 rows, logits + argmax.
//  * Attention: work item = (row, kv head, chunk of positions), flash-decoding with an
//    online softmax per query head (attention.cuh); RoPE of q and k and the cache
//    append happen here.  Chunk states are either merged by the Wo consumers (small
//    batches) or by the last CTA to finish a (row, kv head).
//  * Every wait is bounded (1 s): on expiry the kernel records it in the status word,
//    raises an abort flag and finishes the step without waiting any further.
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "attention.cuh"
#include "device_common.cuh"
#include "slm_internal.h"

namespace slm {

// ------------------------------------------------------------------ shared memory

struct Shared {
    uint8_t *ring;      // [kRingSlots][kChunkBytes]
    uint64_t *full;     // [kRingSlots]
    uint64_t *empty;    // [kRingSlots]
    float *rs;          // [kMaxBatch] 1 / rms
    float *wbest_v;     // [kComputeWarps][kMaxBatch]
    int *wbest_i;       // [kComputeWarps][kMaxBatch]
    int *flags;         // [4]: 0 = last-arriver flag
    float *xown;        // [kMaxBatch][kMaxOwn] residual rows this CTA owns
    float *accs;        // [kMaxOwn][kMaxBatch] accumulators across K tiles
    float *xs;          // activation tile / attention scratch, kXsBudget bytes
};

constexpr int kRingBytes = kRingSlots * kChunkBytes;
constexpr int kMiscBytes = 2 * kRingSlots * 8 + kMaxBatch * 4 + 2 * kComputeWarps * kMaxBatch * 4 + 16;
constexpr int kOwnOffset = ((kRingBytes + kMiscBytes + 127) / 128) * 128;
constexpr int kAccOffset = kOwnOffset + kMaxBatch * kMaxOwn * 4;
constexpr int kXsOffset = kAccOffset + kMaxOwn * kMaxBatch * 4;
constexpr int kSmemBytes = kXsOffset + (int)kXsBudget;
static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");

__device__ __forceinline__ Shared carve(uint8_t *base) {
    Shared s;
    s.ring = base;
    uint8_t *p = base + kRingBytes;
    s.full = (uint64_t *)p;
    p += kRingSlots * 8;
    s.empty = (uint64_t *)p;
    p += kRingSlots * 8;
    s.rs = (float *)p;
    p += kMaxBatch * 4;
    s.wbest_v = (float *)p;
    p += kComputeWarps * kMaxBatch * 4;
    s.wbest_i = (int *)p;
    p += kComputeWarps * kMaxBatch * 4;
    s.flags = (int *)p;
    s.xown = (float *)(base + kOwnOffset);
    s.accs = (float *)(base + kAccOffset);
    s.xs = (float *)(base + kXsOffset);
    return s;
}

// ------------------------------------------------------------------ bounded waits

__device__ bool wait_slot(const StepParams &P, uint64_t *bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    if (ld_volatile_int(P.m.abort_flag)) return false;
    unsigned long long t0 = global_ns();
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if (ld_volatile_int(P.m.abort_flag)) return false;
        if (global_ns() - t0 > kWaitLimitNs) {
            atomicOr(P.m.status, kStRingTimeout);
            atomicExch(P.m.abort_flag, 1);
            return false;
        }
    }
}

// Poll rows x len tagged words (row stride src_ld) into shared memory (row stride
// dst_ld) until every tag equals `tag`.  Each thread keeps up to 8 loads in flight.
// All compute threads call it; it ends with a CTA barrier.
__device__ void ll_poll(const StepParams &P, const uint64_t *src, int src_ld, int rows, int len,
                        float *dst, int dst_ld, uint32_t tag) {
    constexpr int kBatch = 8;
    const int tid = threadIdx.x;
    const int n = rows * len;
    for (int base = 0; base < n; base += kComputeThreads * kBatch) {
        int so[kBatch], dof[kBatch];
        bool need[kBatch];
#pragma unroll
        for (int k = 0; k < kBatch; k++) {
            int i = base + k * kComputeThreads + tid;
            need[k] = i < n;
            int r = need[k] ? i / len : 0, j = need[k] ? i - r * len : 0;
            so[k] = r * src_ld + j;
            dof[k] = r * dst_ld + j;
        }
        unsigned long long t0 = 0;
        for (int it = 0;; it++) {
            uint64_t w[kBatch];
#pragma unroll
            for (int k = 0; k < kBatch; k++) w[k] = need[k] ? ll_load(src + so[k]) : 0;
            bool pending = false;
#pragma unroll
            for (int k = 0; k < kBatch; k++) {
                if (!need[k]) continue;
                if ((uint32_t)(w[k] >> 32) == tag) {
                    dst[dof[k]] = __uint_as_float((uint32_t)w[k]);
                    need[k] = false;
                } else {
                    pending = true;
                }
            }
            if (!pending) break;
            if (it == 0) t0 = global_ns();
            if ((it & 15) == 15) {  // the abort flag and the clock, every 16 rounds
                if (ld_volatile_int(P.m.abort_flag)) break;
                if (global_ns() - t0 > kWaitLimitNs) {
                    atomicOr(P.m.status, kStExchangeTimeout);
                    atomicExch(P.m.abort_flag, 1);
                    break;
                }
            }
        }
    }
    compute_sync();
}

// Timeline hook: thread 0 of each CTA stamps (phase, point) when tracing is on.
__device__ __forceinline__ void trace_mark(const StepParams &P, int slot, int point) {
    if (P.trace && threadIdx.x == 0)
        P.trace[((size_t)blockIdx.x * trace_slots(P.m.n_layers) + slot) * 3 + point] = global_ns();
}

// ------------------------------------------------------------------ chunk walk
// The streaming warp and the compute warps enumerate exactly the same chunks: this
// CTA's units [u0, u1) of the matrix, K tile by K tile.

struct Chunk {
    int kt;
    int unit0;       // first unit of the chunk, relative to the CTA's first unit
    int nunits;
    const uint8_t *src;
    uint32_t bytes;
};

template <typename F>
__device__ __forceinline__ void for_each_chunk(const Mat &M, int layer, int esz, int cta, int grid, F &&f) {
    const int units = M.rows / M.rows_per_unit;
    int u0, u1;
    unit_range(units, grid, cta, u0, u1);
    const int cu = M.rows_per_chunk / M.rows_per_unit;
    const uint8_t *lbase = M.base + (long long)layer * M.layer_stride;
    const long long rowbytes = (long long)M.KBp * esz;
    for (int kt = 0; kt < M.nkt; kt++) {
        for (int u = u0; u < u1; u += cu) {
            Chunk c;
            c.kt = kt;
            c.unit0 = u - u0;
            c.nunits = min(cu, u1 - u);
            c.src = lbase + ((long long)kt * M.rows + (long long)u * M.rows_per_unit) * rowbytes;
            c.bytes = (uint32_t)((long long)c.nunits * M.rows_per_unit * rowbytes);
            f(c);
        }
    }
}

// ------------------------------------------------------------------ streaming warp

__device__ void producer(const StepParams &P, Shared &S) {
    const Model &m = P.m;
    const int esz = m.weight_bf16 ? 2 : 4;
    const int cta = blockIdx.x, grid = P.grid;
    uint32_t issued = 0;
    bool dead = false;
    auto issue = [&](const Chunk &c) {
        if (dead) return;
        uint32_t slot = issued % kRingSlots;
        if (issued >= (uint32_t)kRingSlots) {
            uint32_t parity = ((issued / kRingSlots) - 1) & 1;
            if (!wait_slot(P, &S.empty[slot], parity)) {
                dead = true;
                return;
            }
        }
        mbar_expect_tx(&S.full[slot], c.bytes);
        bulk_g2s(S.ring + (size_t)slot * kChunkBytes, c.src, c.bytes, &S.full[slot]);
        issued++;
    };
    for (int l = 0; l < m.n_layers; l++) {
        for_each_chunk(m.qkv, l, esz, cta, grid, issue);
        for_each_chunk(m.wo, l, esz, cta, grid, issue);
        for_each_chunk(m.w13, l, esz, cta, grid, issue);
        for_each_chunk(m.w2, l, esz, cta, grid, issue);
    }
    if (P.do_logits) for_each_chunk(m.emb, 0, esz, cta, grid, issue);
    // Never leave with a copy in flight: wait (bounded, ignoring the abort flag) for the
    // completion of every slot that may still be filling.
    uint32_t first = issued > (uint32_t)kRingSlots ? issued - kRingSlots : 0;
    for (uint32_t i = first; i < issued; i++) {
        uint32_t slot = i % kRingSlots, parity = (i / kRingSlots) & 1;
        unsigned long long t0 = global_ns();
        while (!mbar_try_wait(&S.full[slot], parity)) {
            if (global_ns() - t0 > kWaitLimitNs) {
                atomicOr(P.m.status, kStRingTimeout);
                break;
            }
        }
    }
}

// ------------------------------------------------------------------ inputs of the GEMVs

enum Epi { EPI_QKV = 0, EPI_WO = 1, EPI_W13 = 2, EPI_W2 = 3, EPI_LOGITS = 4 };

__device__ __forceinline__ float emb_elem(const Model &m, int tok, int k) {
    const uint8_t *row = m.emb.base + (long long)tok * m.emb.KBp * (m.weight_bf16 ? 2 : 4);
    if (m.weight_bf16) {
        uint16_t b = ((const uint16_t *)row)[k];
        return __uint_as_float((uint32_t)b << 16);
    }
    return ((const float *)row)[k];
}

__device__ __forceinline__ int token_of(const StepParams &P, int b) {
    int t = __ldcg(P.tokens + b);
    if (t < 0 || t >= P.m.vocab) {
        if (threadIdx.x == 0 && blockIdx.x == 0) atomicOr(P.m.status, kStBadToken);
        t = 0;
    }
    return t;
}

// Offset of layer `layer`'s block in a per-layer exchange buffer of `per_row` words per row.
__device__ __forceinline__ size_t ll_layer(const StepParams &P, int layer, int per_row) {
    return ((size_t)layer * P.m.max_batch) * per_row;
}

// Residual rows this CTA owns (rows of Wo and W2 it computes) start as the embedding.
__device__ void init_residual(const StepParams &P, Shared &S) {
    const Model &m = P.m;
    int r0, r1;
    unit_range(m.dim, P.grid, blockIdx.x, r0, r1);
    for (int b = 0; b < P.batch; b++) {
        int tok = token_of(P, b);
        for (int i = threadIdx.x; i < r1 - r0; i += kComputeThreads)
            S.xown[b * kMaxOwn + i] = emb_elem(m, tok, r0 + i);
    }
}

// RMSNorm of the staged rows in place: xs[b][k] = xs[b][k] * rsqrt(mean + eps) * g[k].
__device__ void norm_in_place(const StepParams &P, float *xs, int ld, const float *g, Shared &S) {
    const Model &m = P.m;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    for (int b = warp; b < P.batch; b += kComputeWarps) {
        const float *r = xs + (size_t)b * ld;
        float ss = 0.f;
        for (int k = lane; k < m.dim; k += 32) ss = fmaf(r[k], r[k], ss);
        ss = warp_sum(ss);
        if (lane == 0) S.rs[b] = 1.0f / sqrtf(ss / (float)m.dim + m.norm_eps);
    }
    compute_sync();
    for (int b = 0; b < P.batch; b++) {
        float *r = xs + (size_t)b * ld;
        const float rs = S.rs[b];
        for (int k = tid; k < m.dim; k += kComputeThreads) r[k] = (r[k] * rs) * __ldg(g + k);
    }
    compute_sync();
}

__device__ void zero_pad(const StepParams &P, float *xs, int ld, int from) {
    for (int b = 0; b < P.batch; b++)
        for (int k = from + (int)threadIdx.x; k < ld; k += kComputeThreads) xs[(size_t)b * ld + k] = 0.f;
}

// Merge the chunk states of every (row, head) published by the attention items into
// the Wo input tile: o = sum_c 2^(m_c - M) O_c / sum_c 2^(m_c - M) l_c.
__device__ void merge_chunk_states(const StepParams &P, int layer, const Mat &M, Shared &S) {
    const Model &m = P.m;
    const int H = m.n_heads, hd = m.head_dim, st = hd + 2;
    int ncmax = 1;
    for (int b = 0; b < P.batch; b++) ncmax = max(ncmax, P.nchunk[b]);
    float *stage = S.xs + (size_t)P.batch * M.KBp;  // [batch][H][ncmax][hd + 2]
    const uint64_t *src = m.ll_part + ll_layer(P, layer, H * kMaxChunksA * st);
    for (int b = 0; b < P.batch; b++) {
        const int nc = P.nchunk[b];
        // rows (b, h) x (nc * st) words, source row stride kMaxChunksA * st
        ll_poll(P, src + (size_t)b * H * kMaxChunksA * st, kMaxChunksA * st, H, nc * st,
                stage + (size_t)b * H * ncmax * st, ncmax * st, P.tag);
    }
    for (int b = 0; b < P.batch; b++) {
        const int nc = P.nchunk[b];
        for (int e = threadIdx.x; e < H * hd; e += kComputeThreads) {
            const int h = e / hd, d = e - h * hd;
            const float *sp = stage + ((size_t)b * H + h) * ncmax * st;
            float Mx = -INFINITY;
            for (int c = 0; c < nc; c++) Mx = fmaxf(Mx, sp[(size_t)c * st]);
            float L = 0.f, O = 0.f;
            for (int c = 0; c < nc; c++) {
                const float mc = sp[(size_t)c * st];
                if (mc == -INFINITY) continue;
                const float sc = exp2f(mc - Mx);
                L = fmaf(sp[(size_t)c * st + 1], sc, L);
                O = fmaf(sp[(size_t)c * st + 2 + d], sc, O);
            }
            S.xs[(size_t)b * M.KBp + e] = O / L;
        }
    }
    zero_pad(P, S.xs, M.KBp, H * hd);
    compute_sync();
}

// Stage the input of phase `epi` (K tile kt) into S.xs as fp32 [batch][KBp].
__device__ void stage_input(const StepParams &P, int epi, int layer, const Mat &M, int kt, Shared &S) {
    const Model &m = P.m;
    const int tid = threadIdx.x;
    compute_sync();  // everyone is done with the previous tile
    if (epi == EPI_QKV || epi == EPI_W13 || epi == EPI_LOGITS) {
        if (epi == EPI_QKV && layer == 0) {
            for (int b = 0; b < P.batch; b++) {
                int tok = token_of(P, b);
                for (int k = tid; k < m.dim; k += kComputeThreads) S.xs[(size_t)b * M.KBp + k] = emb_elem(m, tok, k);
            }
            compute_sync();
        } else {
            const uint64_t *src = epi == EPI_W13 ? m.ll_xa + ll_layer(P, layer, m.dim)
                                                 : m.ll_x + ll_layer(P, epi == EPI_QKV ? layer : m.n_layers, m.dim);
            ll_poll(P, src, m.dim, P.batch, m.dim, S.xs, M.KBp, P.tag);
        }
        const float *g = epi == EPI_QKV   ? m.norms + (size_t)layer * 2 * m.dim
                         : epi == EPI_W13 ? m.norms + (size_t)layer * 2 * m.dim + m.dim
                                          : m.norms + (size_t)m.n_layers * 2 * m.dim;
        norm_in_place(P, S.xs, M.KBp, g, S);
        zero_pad(P, S.xs, M.KBp, m.dim);
        compute_sync();
    } else if (epi == EPI_WO) {
        if (P.attn_consumer_merge) {
            merge_chunk_states(P, layer, M, S);
        } else {
            const int qd = m.n_heads * m.head_dim;
            ll_poll(P, m.ll_o + ll_layer(P, layer, qd), qd, P.batch, qd, S.xs, M.KBp, P.tag);
            zero_pad(P, S.xs, M.KBp, qd);
            compute_sync();
        }
    } else {  // W2: tile kt of the SwiGLU output
        const int k0 = kt * M.KB, kn = min(M.K - k0, M.KB);
        ll_poll(P, m.ll_h + ll_layer(P, layer, m.hidden) + k0, m.hidden, P.batch, kn, S.xs, M.KBp, P.tag);
        zero_pad(P, S.xs, M.KBp, kn);
        compute_sync();
    }
}

// ------------------------------------------------------------------ GEMV arithmetic

// dot of one 16-byte weight piece with the matching activations of every row
template <int NB, bool WBF16>
__device__ __forceinline__ void piece_fma(const uint4 w, const float *xs, int KBp, int p, int batch,
                                          float (&acc)[NB]) {
    if constexpr (WBF16) {
        float wf[8] = {bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y),
                       bf16_lo(w.z), bf16_hi(w.z), bf16_lo(w.w), bf16_hi(w.w)};
#pragma unroll
        for (int b = 0; b < NB; b++) {
            if (NB > 1 && b >= batch) break;
            const float4 *xp = (const float4 *)(xs + (size_t)b * KBp + p * 8);
            float4 x0 = xp[0], x1 = xp[1];
            float a = acc[b];
            a = fmaf(wf[0], x0.x, a);
            a = fmaf(wf[1], x0.y, a);
            a = fmaf(wf[2], x0.z, a);
            a = fmaf(wf[3], x0.w, a);
            a = fmaf(wf[4], x1.x, a);
            a = fmaf(wf[5], x1.y, a);
            a = fmaf(wf[6], x1.z, a);
            a = fmaf(wf[7], x1.w, a);
            acc[b] = a;
        }
    } else {
        float wf[4] = {__uint_as_float(w.x), __uint_as_float(w.y), __uint_as_float(w.z),
                       __uint_as_float(w.w)};
#pragma unroll
        for (int b = 0; b < NB; b++) {
            if (NB > 1 && b >= batch) break;
            float4 x0 = *(const float4 *)(xs + (size_t)b * KBp + p * 4);
            float a = acc[b];
            a = fmaf(wf[0], x0.x, a);
            a = fmaf(wf[1], x0.y, a);
            a = fmaf(wf[2], x0.z, a);
            a = fmaf(wf[3], x0.w, a);
            acc[b] = a;
        }
    }
}

// One row of a ring slot against every batch row; returns the sums in every lane.
template <int NB, bool WBF16>
__device__ __forceinline__ void row_dot(const uint8_t *wrow, const float *xs, int KBp, int batch,
                                        float (&acc)[NB]) {
    const int lane = threadIdx.x & 31;
    constexpr int EPP = WBF16 ? 8 : 4;
    const int pieces = KBp / EPP;
#pragma unroll
    for (int b = 0; b < NB; b++) acc[b] = 0.f;
    const uint4 *w4 = (const uint4 *)wrow;
    int p = lane;
    for (; p + 32 < pieces; p += 64) {
        uint4 wa = w4[p], wb = w4[p + 32];
        piece_fma<NB, WBF16>(wa, xs, KBp, p, batch, acc);
        piece_fma<NB, WBF16>(wb, xs, KBp, p + 32, batch, acc);
    }
    if (p < pieces) piece_fma<NB, WBF16>(w4[p], xs, KBp, p, batch, acc);
#pragma unroll
    for (int b = 0; b < NB; b++) {
        if (NB > 1 && b >= batch) break;
        acc[b] = warp_sum(acc[b]);
    }
}

// ------------------------------------------------------------------ GEMV phases

template <int NB, bool WBF16>
__device__ void gemv_phase(const StepParams &P, int epi, int layer, const Mat &M, Shared &S,
                           uint32_t &chunk_i, float (&best_v)[NB], int (&best_i)[NB], int tslot) {
    const Model &m = P.m;
    const int esz = WBF16 ? 2 : 4;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int batch = P.batch;
    const uint32_t tag = P.tag;
    int u0, u1;
    unit_range(M.rows / M.rows_per_unit, P.grid, blockIdx.x, u0, u1);
    trace_mark(P, tslot, 0);
    if (u0 == u1) return;
    const bool split = M.nkt > 1;
    int cur_kt = -1;
    for_each_chunk(M, layer, esz, blockIdx.x, P.grid, [&](const Chunk &c) {
        if (c.kt != cur_kt) {
            stage_input(P, epi, layer, M, c.kt, S);
            if (cur_kt < 0) trace_mark(P, tslot, 1);
            cur_kt = c.kt;
        }
        const uint32_t slot = chunk_i % kRingSlots, parity = (chunk_i / kRingSlots) & 1;
        wait_slot(P, &S.full[slot], parity);
        const uint8_t *buf = S.ring + (size_t)slot * kChunkBytes;
        const size_t rowbytes = (size_t)M.KBp * esz;
        const bool last_tile = c.kt == M.nkt - 1;
        // unit i of the CTA's slice always belongs to warp i % 8 (accumulators stay put)
        const int first = (warp - c.unit0 % kComputeWarps + kComputeWarps) % kComputeWarps;
        for (int j = first; j < c.nunits; j += kComputeWarps) {
            const int i = c.unit0 + j;          // unit within the CTA's slice
            const int unit = u0 + i;            // global unit
            if (epi == EPI_W13) {
                float a[NB], g[NB];
                row_dot<NB, WBF16>(buf + (size_t)(2 * j) * rowbytes, S.xs, M.KBp, batch, a);
                row_dot<NB, WBF16>(buf + (size_t)(2 * j + 1) * rowbytes, S.xs, M.KBp, batch, g);
#pragma unroll
                for (int b = 0; b < NB; b++) {
                    if (b < batch && lane == b) {
                        float s = a[b] / (1.0f + __expf(-a[b]));
                        ll_store(m.ll_h + ll_layer(P, layer, m.hidden) + (size_t)b * m.hidden + unit, s * g[b], tag);
                    }
                }
                continue;
            }
            float acc[NB];
            row_dot<NB, WBF16>(buf + (size_t)j * rowbytes, S.xs, M.KBp, batch, acc);
#pragma unroll
            for (int b = 0; b < NB; b++) {
                if (b >= batch || lane != b) continue;
                float v = acc[b];
                if (split) {  // accumulate this K tile; finish after the last one
                    float *a = S.accs + (size_t)i * kMaxBatch + b;
                    v = (c.kt == 0 ? 0.f : *a) + v;
                    *a = v;
                    if (!last_tile) continue;
                }
                if (epi == EPI_QKV) {
                    ll_store(m.ll_qkv + ll_layer(P, layer, m.qkv.rows) + (size_t)b * m.qkv.rows + unit, v, tag);
                } else if (epi == EPI_WO || epi == EPI_W2) {
                    float *own = S.xown + b * kMaxOwn + i;
                    const float xn = *own + v;
                    *own = xn;
                    uint64_t *dst = epi == EPI_WO ? m.ll_xa + ll_layer(P, layer, m.dim)
                                                  : m.ll_x + ll_layer(P, layer + 1, m.dim);
                    ll_store(dst + (size_t)b * m.dim + unit, xn, tag);
                } else {  // logits
                    if (P.logits) P.logits[(size_t)b * m.vocab + unit] = v;
                    if (v != v)
                        atomicOr(m.status, kStNanLogits);
                    else if (v > best_v[b] || (v == best_v[b] && unit < best_i[b])) {
                        best_v[b] = v;
                        best_i[b] = unit;
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.empty[slot]);
        chunk_i++;
    });
    trace_mark(P, tslot, 2);
}

// Per-warp, then per-CTA argmax candidates; CTA 0 collects every CTA's candidate.
template <int NB>
__device__ void finish_argmax(const StepParams &P, Shared &S, float (&best_v)[NB], int (&best_i)[NB]) {
    const Model &m = P.m;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int batch = P.batch;
    compute_sync();  // the logits phase is done with S.xs
#pragma unroll
    for (int b = 0; b < NB; b++) {
        if (b < batch && lane == b) {
            S.wbest_v[warp * kMaxBatch + b] = best_v[b];
            S.wbest_i[warp * kMaxBatch + b] = best_i[b];
        }
    }
    compute_sync();
    if (tid < batch) {
        float bv = -INFINITY;
        int bi = 0x7fffffff;
        for (int w = 0; w < kComputeWarps; w++) {
            float v = S.wbest_v[w * kMaxBatch + tid];
            int i = S.wbest_i[w * kMaxBatch + tid];
            if (v > bv || (v == bv && i < bi)) {
                bv = v;
                bi = i;
            }
        }
        uint64_t *dst = m.ll_amax + ((size_t)tid * P.grid + blockIdx.x) * 2;
        ll_store(dst, bv, P.tag);
        ll_store(dst + 1, __int_as_float(bi), P.tag);
    }
    if (blockIdx.x != 0) return;
    // CTA 0: poll [batch][grid][2] words into shared memory, reduce per row
    ll_poll(P, m.ll_amax, P.grid * 2, batch, P.grid * 2, S.xs, P.grid * 2, P.tag);
    if (tid < batch) {
        float bv = -INFINITY;
        int bi = 0x7fffffff;
        const float *r = S.xs + (size_t)tid * P.grid * 2;
        for (int c = 0; c < P.grid; c++) {
            float v = r[2 * c];
            int i = __float_as_int(r[2 * c + 1]);
            if (v > bv || (v == bv && i < bi)) {
                bv = v;
                bi = i;
            }
        }
        if (bi == 0x7fffffff) bi = 0;  // all NaN: the status word already records it
        if (P.next_ids) P.next_ids[tid] = bi;
    }
}

// ------------------------------------------------------------------ attention phase

template <bool KVBF16>
__device__ void attn_item(const StepParams &P, int layer, int b, int g, int c, Shared &S) {
    const Model &m = P.m;
    const int tid = threadIdx.x;
    const int hd = m.head_dim, H = m.n_heads, KV = m.n_kv_heads, G = H / KV;
    const int half = hd / 2, qrows = m.qkv.rows;
    const int pos = P.pos[b], ctx = pos + 1, seq = P.seq[b];
    const int CH = P.attn_chunk, nc = P.nchunk[b];
    const int t0 = c * CH, t1 = min(ctx, t0 + CH);
    const size_t rowbytes = (size_t)hd * (KVBF16 ? 2 : 4);
    const size_t head_off = ((((size_t)layer * m.max_batch + seq) * KV + g) * m.max_seq) * rowbytes;
    uint8_t *kbase = m.kc + head_off;
    uint8_t *vbase = m.vc + head_off;
    const float *rope = m.rope + (size_t)pos * half * 2;
    const uint64_t *qkv = m.ll_qkv + ll_layer(P, layer, qrows) + (size_t)b * qrows;
    const bool appends = t1 == ctx;  // this chunk ends at the new position

    // Shared scratch after attn_core's: the group's raw [q heads; k; v] rows, then
    // (when it fits) a copy of the chunk's cached keys and values.  The cached rows do
    // not depend on this step, so their copy starts before waiting for q.
    float *raw = S.xs + kMaxGroupPass * hd + kComputeWarps * kMaxGroupPass * (hd + 2);
    uint8_t *kst = (uint8_t *)(raw + (size_t)(G + 2) * hd);
    const int tc = appends ? pos : t1;  // cached positions [t0, tc) of this chunk
    const bool stage = (size_t)(t1 - t0) * rowbytes * 2 <= kAttnStageBytes;
    uint8_t *vst = kst + (size_t)(t1 - t0) * rowbytes;
    compute_sync();  // the previous item is done with the scratch
    if (stage) {
        const int per_row = (int)(rowbytes / 16), n16 = (tc - t0) * per_row;
        for (int e = tid; e < n16; e += kComputeThreads) {
            const size_t off = (size_t)(e / per_row) * rowbytes + (size_t)(e % per_row) * 16;
            cp_async16(kst + off, kbase + (size_t)t0 * rowbytes + off);
            cp_async16(vst + off, vbase + (size_t)t0 * rowbytes + off);
        }
    }
    // one contiguous range: this group's q heads, then its k and v rows
    ll_poll(P, qkv + (size_t)g * (G + 2) * hd, hd, G + 2, hd, raw, hd, P.tag);
    if (appends) {
        uint8_t *kd = kbase + (size_t)pos * rowbytes;
        uint8_t *vd = vbase + (size_t)pos * rowbytes;
        uint8_t *ks = kst + (size_t)(pos - t0) * rowbytes;
        uint8_t *vs = vst + (size_t)(pos - t0) * rowbytes;
        const float *kr = raw + (size_t)G * hd, *vr = raw + (size_t)(G + 1) * hd;
        for (int i = tid; i < half; i += kComputeThreads) {
            float cs = __ldg(rope + 2 * i), sn = __ldg(rope + 2 * i + 1);
            float a = kr[i], bb = kr[i + half];
            float k0 = kv_round(a * cs - bb * sn, KVBF16), k1 = kv_round(a * sn + bb * cs, KVBF16);
            float v0 = kv_round(vr[i], KVBF16), v1 = kv_round(vr[i + half], KVBF16);
            if (KVBF16) {
                ((__nv_bfloat16 *)kd)[i] = __float2bfloat16_rn(k0);
                ((__nv_bfloat16 *)kd)[i + half] = __float2bfloat16_rn(k1);
                ((__nv_bfloat16 *)vd)[i] = __float2bfloat16_rn(v0);
                ((__nv_bfloat16 *)vd)[i + half] = __float2bfloat16_rn(v1);
                if (stage) {
                    ((__nv_bfloat16 *)ks)[i] = __float2bfloat16_rn(k0);
                    ((__nv_bfloat16 *)ks)[i + half] = __float2bfloat16_rn(k1);
                    ((__nv_bfloat16 *)vs)[i] = __float2bfloat16_rn(v0);
                    ((__nv_bfloat16 *)vs)[i + half] = __float2bfloat16_rn(v1);
                }
            } else {
                ((float *)kd)[i] = k0;
                ((float *)kd)[i + half] = k1;
                ((float *)vd)[i] = v0;
                ((float *)vd)[i + half] = v1;
                if (stage) {
                    ((float *)ks)[i] = k0;
                    ((float *)ks)[i + half] = k1;
                    ((float *)vs)[i] = v0;
                    ((float *)vs)[i + half] = v1;
                }
            }
        }
    }
    if (stage) cp_async_wait_all();  // attn_core's first barrier publishes the copies
    AttnTask T;
    T.q = raw;  // read by attn_core after its first barrier
    T.rope = rope;
    T.kbase = stage ? kst - (size_t)t0 * rowbytes : kbase;
    T.vbase = stage ? vst - (size_t)t0 * rowbytes : vbase;
    T.out = nullptr;
    const size_t pl = (size_t)layer * m.max_batch + b;
    T.part = m.part + (pl * H + (size_t)g * G) * kMaxChunksPerSeq * (hd + 2);
    T.counter = m.part_count + pl * KV + g;
    T.ll_part = P.attn_consumer_merge ? m.ll_part + (pl * H + (size_t)g * G) * kMaxChunksA * (hd + 2) : nullptr;
    T.ll_out = P.attn_consumer_merge ? nullptr : m.ll_o + pl * H * hd + (size_t)g * G * hd;
    T.tag = P.tag;
    T.ncap = kMaxChunksA;
    T.hd = hd;
    T.G = G;
    T.t0 = t0;
    T.t1 = t1;
    T.nc = nc;
    T.c = c;
    attn_core<KVBF16>(T, S.xs, &S.flags[0]);
}

template <bool KVBF16>
__device__ void attention_phase(const StepParams &P, int layer, Shared &S) {
    const int tslot = layer * kTracePerLayer + 1;
    trace_mark(P, tslot, 0);
    const int total = P.item_start[P.batch];
    const int KV = P.m.n_kv_heads;
    for (int item = blockIdx.x; item < total; item += P.grid) {
        int b = 0;
        while (item >= P.item_start[b + 1]) b++;
        const int local = item - P.item_start[b];
        const int nc = P.nchunk[b];
        const int g = local / nc, c = local - g * nc;
        if (g < KV) attn_item<KVBF16>(P, layer, b, g, c, S);
    }
    trace_mark(P, tslot, 2);
}

// ------------------------------------------------------------------ the kernel

template <int NB, bool WBF16>
__global__ void __launch_bounds__(kThreads, 1) decode_step_kernel(const __grid_constant__ StepParams P) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    Shared S = carve(smem_raw);
    const int tid = threadIdx.x;
    if (tid == 0) {
        for (int i = 0; i < kRingSlots; i++) {
            mbar_init(&S.full[i], 1);
            mbar_init(&S.empty[i], kComputeWarps);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (tid >= kComputeThreads) {
        if (tid == kComputeThreads) producer(P, S);
        return;
    }
    const Model &m = P.m;
    uint32_t chunk_i = 0;
    float best_v[NB];
    int best_i[NB];
#pragma unroll
    for (int b = 0; b < NB; b++) {
        best_v[b] = -INFINITY;
        best_i[b] = 0x7fffffff;
    }
    init_residual(P, S);
    for (int l = 0; l < m.n_layers; l++) {
        const int t = l * kTracePerLayer;
        gemv_phase<NB, WBF16>(P, EPI_QKV, l, m.qkv, S, chunk_i, best_v, best_i, t);
        if (m.kv_bf16)
            attention_phase<true>(P, l, S);
        else
            attention_phase<false>(P, l, S);
        gemv_phase<NB, WBF16>(P, EPI_WO, l, m.wo, S, chunk_i, best_v, best_i, t + 2);
        gemv_phase<NB, WBF16>(P, EPI_W13, l, m.w13, S, chunk_i, best_v, best_i, t + 3);
        gemv_phase<NB, WBF16>(P, EPI_W2, l, m.w2, S, chunk_i, best_v, best_i, t + 4);
    }
    if (P.do_logits) {
        const int t = m.n_layers * kTracePerLayer;
        gemv_phase<NB, WBF16>(P, EPI_LOGITS, 0, m.emb, S, chunk_i, best_v, best_i, t);
        trace_mark(P, t + 1, 0);
        finish_argmax<NB>(P, S, best_v, best_i);
        trace_mark(P, t + 1, 2);
    }
}

// ------------------------------------------------------------------ host-side launch

size_t decode_smem_bytes() { return (size_t)kSmemBytes; }

template <int NB, bool WBF16>
static cudaError_t launch_nb(const StepParams &P, cudaStream_t stream) {
    auto fn = decode_step_kernel<NB, WBF16>;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    void *args[] = {(void *)&P};
    return cudaLaunchCooperativeKernel((const void *)fn, dim3(P.grid), dim3(kThreads), args, kSmemBytes, stream);
}

template <bool WBF16>
static cudaError_t launch_w(const StepParams &P, cudaStream_t stream) {
    if (P.batch <= 1) return launch_nb<1, WBF16>(P, stream);
    if (P.batch <= 4) return launch_nb<4, WBF16>(P, stream);
    if (P.batch <= 8) return launch_nb<8, WBF16>(P, stream);
    return launch_nb<16, WBF16>(P, stream);
}

cudaError_t launch_decode_step(const StepParams &P, cudaStream_t stream) {
    return P.m.weight_bf16 ? launch_w<true>(P, stream) : launch_w<false>(P, stream);
}

cudaError_t decode_occupancy(int weight_bf16, int *blocks_per_sm) {
    auto fn = weight_bf16 ? decode_step_kernel<1, true> : decode_step_kernel<1, false>;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, fn, kThreads, kSmemBytes);
}

}  // namespace slm
