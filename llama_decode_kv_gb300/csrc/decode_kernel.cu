// decode_kernel.cu -- the KV-cached greedy decode step as one persistent kernel.
//
// One cooperative launch computes a whole step for every batch row (kasahare 0.4.0 /
// simple-llm, "Architecture": RMSNorm, Wq/Wk/Wv without biases, RoPE, KV append, GQA
// softmax(q K^T / sqrt(d_head)) V, Wo + residual, RMSNorm, W2(silu(W1 x) * (W3 x)) +
// residual; then the final RMSNorm, the tied-embedding logits and the greedy argmax).
//
// Structure (one CTA per SM, 8 compute warps + 1 streaming warp):
//  * Weights do not depend on activations: the streaming warp walks this CTA's share of
//    every matrix of the step in consumption order and copies it HBM -> shared memory
//    with cp.async.bulk into a ring of 8 KB slots signalled by mbarriers, running ahead
//    of the compute warps across phases.
//  * Each GEMV phase splits its output rows evenly over the CTAs.  Its input vector is
//    produced by other CTAs: producers publish every element as a tagged 8-byte word
//    (value + this launch's tag, one store) and consumers poll the words until the tags
//    match -- no fence, no counter, no grid barrier.  Exchange buffers are per layer, so
//    nothing is rewritten within a launch.
//  * RMSNorm is folded into that poll: the squares are summed as the elements arrive,
//    the gain is applied on arrival and 1/rms multiplies the finished dot products.
//  * QKV rows are stored in RoPE pairs (dims i and i + d/2 of a head side by side), so
//    the QKV epilogue rotates q and k, scales q for a base-2 softmax, rounds k and v to
//    the cache type and appends them to the cache.
//  * Each CTA keeps the residual rows it owns (the rows of Wo and W2 it computes) in
//    shared memory, so the residual adds read nothing from memory.
//  * Attention: work item = (row, kv head, chunk of positions), flash-decoding with an
//    online softmax per query head (attention.cuh); chunk states are merged by the Wo
//    consumers (small batches) or by the last CTA to finish a (row, kv head).
//  * The code is kept small: the four GEMV phases of a layer run through one body with a
//    run-time epilogue, so each helper is emitted once.  Every layer walks the whole
//    step's code again, and it has to stay in the SM's instruction caches.
//  * Every wait is bounded (1 s): on expiry the kernel records it in the status word,
//    raises an abort flag and finishes the step without waiting any further.
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "attention.cuh"
#include "device_common.cuh"
#include "gemv.cuh"
#include "slm_internal.h"

namespace slm {

// ------------------------------------------------------------------ shared memory

struct Shared {
    uint64_t *full;     // [kMaxRingSlots]
    uint64_t *empty;    // [kMaxRingSlots]
    float *ssp;         // [kComputeWarps][kMaxBatch] per-warp sums of squares of the
                        //   current RMSNorm input (every warp stores all its entries)
    float *wbest_v;     // [kComputeWarps][kMaxBatch]
    int *wbest_i;       // [kComputeWarps][kMaxBatch]
    int *flags;         // [4]: 0 = last-arriver flag
    float *xown;        // [max_batch][own_ld] residual rows this CTA owns
    float *accs;        // [own_ld][kMaxBatch] accumulators across K tiles (if any)
    float *xs;          // activation tile / attention scratch, P.xs_bytes
    uint8_t *ring;      // [P.ring_slots][kChunkBytes]
};

__device__ __forceinline__ Shared carve(uint8_t *base, const StepParams &P) {
    Shared s;
    uint8_t *p = base;
    s.full = (uint64_t *)p;
    p += kMaxRingSlots * 8;
    s.empty = (uint64_t *)p;
    p += kMaxRingSlots * 8;
    s.ssp = (float *)p;
    p += kComputeWarps * kMaxBatch * 4;
    s.wbest_v = (float *)p;
    p += kComputeWarps * kMaxBatch * 4;
    s.wbest_i = (int *)p;
    p += kComputeWarps * kMaxBatch * 4;
    s.flags = (int *)p;
    s.xs = (float *)(base + kSmallBytes);
    s.xown = (float *)(base + own_offset(P.xs_bytes));
    s.accs = (float *)(base + own_offset(P.xs_bytes) + own_bytes(P.m.max_batch, P.own_ld));
    s.ring = base + ring_offset(P.m.max_batch, P.own_ld, P.acc_bytes, P.xs_bytes);
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
        if (global_ns() - t0 > P.m.wait_ns) {
            atomicOr(P.m.status, kStRingTimeout);
            atomicExch(P.m.abort_flag, 1);
            return false;
        }
    }
}


// Batch-16 tensor-core phases keep their activations as two bf16 planes, hi and lo
// (x = hi + lo to about 16 mantissa bits), rows of `pld` elements, lo plane 16 rows
// after hi; element (r, j) of both at r * pld + j.
__device__ __forceinline__ void plane_store(uint16_t *hi, int pld, int r, int j, float x) {
    const __nv_bfloat16 h = __float2bfloat16_rn(x);
    const __nv_bfloat16 l = __float2bfloat16_rn(x - __bfloat162float(h));
    hi[r * pld + j] = *(const uint16_t *)&h;
    hi[kMaxBatch * pld + r * pld + j] = *(const uint16_t *)&l;
}

// Elements (r, j) and (r, j + 1), j even.
__device__ __forceinline__ void plane_store2(uint16_t *hi, int pld, int r, int j, float x0, float x1) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
    const float2 hf = __bfloat1622float2(h);
    const __nv_bfloat162 l = __floats2bfloat162_rn(x0 - hf.x, x1 - hf.y);
    *(__nv_bfloat162 *)(hi + r * pld + j) = h;
    *(__nv_bfloat162 *)(hi + kMaxBatch * pld + r * pld + j) = l;
}

__device__ __forceinline__ float plane_load(const uint16_t *hi, int pld, int r, int j) {
    return __uint_as_float((uint32_t)hi[r * pld + j] << 16) + __uint_as_float((uint32_t)hi[kMaxBatch * pld + r * pld + j] << 16);
}

// Timeline hook: thread 0 of each CTA stamps (phase, point) when tracing is on.
__device__ __forceinline__ void trace_mark(const StepParams &P, int slot, int point) {
    if (P.trace && threadIdx.x == 0)
        P.trace[((size_t)blockIdx.x * trace_slots(P.m.n_layers) + slot) * 3 + point] = global_ns();
}

// ------------------------------------------------------------------ polling

constexpr int kPollBatch = 8;   // loads each thread keeps in flight
constexpr int kPollBatchW = 8;   //   (rows of a batch)

// Poll rows x len tagged words src[r * src_ld + j] into shared memory dst[r * dst_ld +
// xpos(j)] (natural order when perm_ld is 0) until every tag equals the launch's tag.
// With `gain`: element j is stored as x_j * gain_j and each warp stores its part of row
// r's sum of x_j^2 in ssp[warp * kMaxBatch + r] (every r < rows; one row for WIDE = 1).
// All compute threads call it; it ends with their barrier.
template <int WIDE = 1>
__device__ __forceinline__ void poll_words(const StepParams &P, const uint64_t *src, int src_ld, int rows, int len,
                                        float *dst, int dst_ld, int perm_ld, const float *gain, float *ssp,
                                        bool planes = false) {
    const int tid = threadIdx.x;
    const uint32_t tag = P.tag;
    // WIDE = 2 (long vectors of batched rows): words are fetched two at a time (one
    // 16-byte load; each 8-byte word is still single-copy atomic and carries its own
    // tag) when rows and the source are aligned, which halves the load rounds.
    const int wpl = (((uintptr_t)src & 15) == 0 && (src_ld & 1) == 0 && (len & 1) == 0) ? 2 : 1;
    float ss = 0.f;
    if constexpr (WIDE == 1) {
        const int n = rows * len;
        for (int base = 0; base < n; base += kComputeThreads * kPollBatch) {
            int so[kPollBatch], dof[kPollBatch];
            float g[kPollBatch], xv[kPollBatch];  // xv: the words' values, squared in k order
            bool need[kPollBatch];
#pragma unroll
            for (int k = 0; k < kPollBatch; k++) {
                const int i = base + k * kComputeThreads + tid;
                need[k] = i < n;
                const int r = need[k] ? i / len : 0, j = need[k] ? i - r * len : 0;
                so[k] = r * src_ld + j;
                dof[k] = r * dst_ld + (perm_ld ? xpos(j, perm_ld, true) : j);
                g[k] = (gain && need[k]) ? __ldg(gain + j) : 1.f;
                xv[k] = 0.f;
            }
            unsigned long long t0 = 0;
            for (int it = 0;; it++) {
                uint64_t w[kPollBatch];
#pragma unroll
                for (int k = 0; k < kPollBatch; k++) w[k] = need[k] ? ll_load(src + so[k]) : 0;
                bool pending = false;
#pragma unroll
                for (int k = 0; k < kPollBatch; k++) {
                    if (!need[k]) continue;
                    if ((uint32_t)(w[k] >> 32) == tag) {
                        const float x = __uint_as_float((uint32_t)w[k]);
                        xv[k] = x;
                        dst[dof[k]] = x * g[k];
                        need[k] = false;
                    } else {
                        pending = true;
                    }
                }
                if (!pending) break;
                if (it == 0) t0 = global_ns();
                if ((it & 15) == 15) {  // the abort flag and the clock, every 16 rounds
                    if (ld_volatile_int(P.m.abort_flag)) break;
                    if (global_ns() - t0 > P.m.wait_ns) {
                        atomicOr(P.m.status, kStExchangeTimeout);
                        atomicExch(P.m.abort_flag, 1);
                        break;
                    }
                }
            }
            // the sum of squares in a fixed order, whatever order the words arrived in
#pragma unroll
            for (int k = 0; k < kPollBatch; k++) ss = fmaf(xv[k], xv[k], ss);
        }
        if (ssp) {
            ss = warp_sum(ss);
            if ((tid & 31) == 0) ssp[(tid >> 5) * kMaxBatch] = ss;
        }
    } else {
    // Row b is polled by threads [b * tpr, (b + 1) * tpr): a thread's words all belong to
    // one row, so its sum of squares is that row's.
    int rp = 1;
    while (rp < rows) rp <<= 1;
    const int tpr = kComputeThreads / rp;  // >= 16
    const int b = tid / tpr, t = tid - b * tpr;
    const int nl = len / wpl;  // loads per row
    // Every CTA reads the same block: each starts at its own column.
    const int rot = (int)(((long long)blockIdx.x * nl) / gridDim.x);
    if (b < rows) {
        const uint64_t *srow = src + (size_t)b * src_ld;
        for (int base = 0; base < nl; base += tpr * kPollBatchW) {
            int wj[kPollBatchW];  // first word (column) of load k
            float g0[kPollBatchW], g1[kPollBatchW];
            float xv[kPollBatchW][2];  // the words' values, squared in (k, h) order
            uint32_t pend = 0;   // bit 2k + h: word h of load k still missing
#pragma unroll
            for (int k = 0; k < kPollBatchW; k++) {
                const int l = base + k * tpr + t;
                int e = l + rot;
                if (e >= nl) e -= nl;
                wj[k] = l < nl ? e * wpl : 0;
                g0[k] = (gain && l < nl) ? __ldg(gain + wj[k]) : 1.f;
                g1[k] = (gain && l < nl && wpl == 2) ? __ldg(gain + wj[k] + 1) : 1.f;
                if (l < nl) pend |= (wpl == 2 ? 3u : 1u) << (2 * k);
                xv[k][0] = xv[k][1] = 0.f;
            }
            unsigned long long t0 = 0;
            for (int it = 0;; it++) {
                uint64_t w[kPollBatchW][2];
#pragma unroll
                for (int k = 0; k < kPollBatchW; k++) {
                    w[k][0] = w[k][1] = 0;
                    if (pend & (3u << (2 * k))) {
                        if (wpl == 2)
                            ll_load2(srow + wj[k], w[k][0], w[k][1]);
                        else
                            w[k][0] = ll_load(srow + wj[k]);
                    }
                }
#pragma unroll
                for (int k = 0; k < kPollBatchW; k++) {
                    if (planes && wpl == 2 && ((pend >> (2 * k)) & 3u) == 3u && (uint32_t)(w[k][0] >> 32) == tag &&
                        (uint32_t)(w[k][1] >> 32) == tag) {  // both words: one 32-bit store per plane
                        pend &= ~(3u << (2 * k));
                        const float x0 = __uint_as_float((uint32_t)w[k][0]), x1 = __uint_as_float((uint32_t)w[k][1]);
                        xv[k][0] = x0;
                        xv[k][1] = x1;
                        plane_store2((uint16_t *)dst, dst_ld, b, wj[k], x0 * g0[k], x1 * g1[k]);
                        continue;
                    }
#pragma unroll
                    for (int h = 0; h < 2; h++) {
                        const uint32_t bit = 1u << (2 * k + h);
                        if (!(pend & bit) || (uint32_t)(w[k][h] >> 32) != tag) continue;
                        pend &= ~bit;
                        const int j = wj[k] + h;
                        const float x = __uint_as_float((uint32_t)w[k][h]);
                        xv[k][h] = x;
                        const float y = x * (h ? g1[k] : g0[k]);
                        if (planes)  // dst_ld is the plane row length
                            plane_store((uint16_t *)dst, dst_ld, b, j, y);
                        else
                            dst[b * dst_ld + (perm_ld ? xpos(j, perm_ld, true) : j)] = y;
                    }
                }
                if (!pend) break;
                if (it == 0) t0 = global_ns();
                if ((it & 15) == 15) {  // the abort flag and the clock, every 16 rounds
                    if (ld_volatile_int(P.m.abort_flag)) break;
                    if (global_ns() - t0 > P.m.wait_ns) {
                        atomicOr(P.m.status, kStExchangeTimeout);
                        atomicExch(P.m.abort_flag, 1);
                        break;
                    }
                }
            }
#pragma unroll
            for (int k = 0; k < kPollBatchW; k++) ss = fmaf(xv[k][1], xv[k][1], fmaf(xv[k][0], xv[k][0], ss));
        }
    }
    if (ssp) {  // per warp and row: lanes of one row are min(tpr, 32) consecutive lanes
        const int wl = tpr < 32 ? tpr : 32;
        for (int off = wl >> 1; off >= 1; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
        const int warp = tid >> 5, lane = tid & 31;
        const float s0 = __shfl_sync(0xffffffffu, ss, 0), s16 = __shfl_sync(0xffffffffu, ss, 16);
        const int row_a = (warp * 32) / tpr, row_b = (warp * 32 + 16) / tpr;  // rows of lanes 0 and 16
        if (lane < rows) {
            float v = 0.f;
            if (lane == row_a) v += s0;
            if (row_b != row_a && lane == row_b) v += s16;
            ssp[warp * kMaxBatch + lane] = v;
        }
    }
    }
    compute_sync();
}

// ------------------------------------------------------------------ chunk walk
// The streaming warp and the compute warps enumerate exactly the same chunks: this
// CTA's units [u0, u1) of the matrix, K tile by K tile, rows_per_chunk rows at a time.

struct Chunk {
    const uint8_t *src;
    uint32_t bytes;
    uint32_t rowbytes;
};

// ------------------------------------------------------------------ streaming warp
// A cursor over the same chunk sequence as the compute warps walk: per layer QKV, Wo,
// W1/W3, W2, then the embedding (logits) when requested.

struct Cursor {
    int phase, layer, kt, u, u0, u1;
    bool done;
};

__device__ __forceinline__ const Mat &phase_mat(const Model &m, int phase) {
    return phase == 0 ? m.qkv : phase == 1 ? m.wo : phase == 2 ? m.w13 : phase == 3 ? m.w2 : m.emb;
}

__device__ void cursor_enter(const StepParams &P, Cursor &c) {
    const Mat &M = phase_mat(P.m, c.phase);
    phase_slice(P, c.phase, M.rows / M.rows_per_unit, blockIdx.x, c.u0, c.u1);
    c.kt = 0;
    c.u = c.u0;
}

// Next chunk of the sequence; false at the end.
__device__ bool cursor_next(const StepParams &P, Cursor &c, Chunk &out) {
    const Model &m = P.m;
    while (!c.done) {
        const Mat &M = phase_mat(m, c.phase);
        if (c.u < c.u1) {
            const int cu = M.rows_per_chunk / M.rows_per_unit;
            const long long rowbytes = tile_rowbytes(m.weight_type, M.KBp);
            const int nunits = min(cu, c.u1 - c.u);
            out.src = M.base + (long long)(c.phase == 4 ? 0 : c.layer) * M.layer_stride +
                      ((long long)c.kt * M.rows + (long long)c.u * M.rows_per_unit) * rowbytes;
            out.bytes = (uint32_t)((long long)nunits * M.rows_per_unit * rowbytes);
            out.rowbytes = (uint32_t)rowbytes;
            c.u += nunits;
            return true;
        }
        if (++c.kt < M.nkt) {
            c.u = c.u0;
            continue;
        }
        if (c.phase < 3) {
            c.phase++;
        } else if (c.phase == 3 && c.layer + 1 < m.n_layers) {
            c.layer++;
            c.phase = 0;
        } else if (c.phase == 3 && P.do_logits) {
            c.phase = 4;
        } else {
            c.done = true;
            break;
        }
        cursor_enter(P, c);
    }
    return false;
}

// Copies this CTA's chunks into the ring, in the order the compute warps use them; with
// PAD, row by row at a stride of rowbytes + kRowPad.
template <bool PAD>
__device__ __forceinline__ void producer(const StepParams &P, Shared &S) {
    const uint32_t slots = (uint32_t)P.ring_slots;
    Cursor ic;
    ic.phase = 0;
    ic.layer = 0;
    ic.done = false;
    cursor_enter(P, ic);
    uint32_t issued = 0;
    Chunk c;
    while (cursor_next(P, ic, c)) {
        const uint32_t slot = issued % slots;
        if (issued >= slots) {
            const uint32_t parity = ((issued / slots) - 1) & 1;
            if (!wait_slot(P, &S.empty[slot], parity)) break;
        }
        mbar_expect_tx(&S.full[slot], c.bytes);
        if (PAD) {
            for (uint32_t r = 0, n = c.bytes / c.rowbytes; r < n; r++)
                bulk_g2s(S.ring + (size_t)slot * kChunkBytes + r * (c.rowbytes + kRowPad), c.src + (size_t)r * c.rowbytes,
                         c.rowbytes, &S.full[slot]);
        } else {
            bulk_g2s(S.ring + (size_t)slot * kChunkBytes, c.src, c.bytes, &S.full[slot]);
        }
        issued++;
    }
    // Never leave with a copy in flight: wait (bounded, ignoring the abort flag) for the
    // completion of every slot that may still be filling.
    uint32_t first = issued > slots ? issued - slots : 0;
    for (uint32_t i = first; i < issued; i++) {
        uint32_t slot = i % slots, parity = (i / slots) & 1;
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
    const uint8_t *row = m.emb.base + (long long)tok * tile_rowbytes(m.weight_type, m.emb.KBp);
    if (m.weight_type == kWQ8)  // scale of k's block times its int8 value
        return ((const float *)(row + m.emb.KBp))[k / kQ8Block] * (float)((const int8_t *)row)[k];
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
__device__ __forceinline__ void init_residual(const StepParams &P, Shared &S) {
    const Model &m = P.m;
    int r0, r1;
    phase_slice(P, 1, m.dim, blockIdx.x, r0, r1);
    for (int b = 0; b < P.batch; b++) {
        int tok = token_of(P, b);
        for (int i = threadIdx.x; i < r1 - r0; i += kComputeThreads)
            S.xown[b * P.own_ld + i] = emb_elem(m, tok, r0 + i);
    }
}

// RMSNorm statistics of staged raw rows: each warp stores its part of sum_j x_j^2 of
// row b in ssp[warp * kMaxBatch + b] (0 for rows it does not hold) and every element is
// multiplied by its gain.  Rows are spread over power-of-two groups of threads.  Ends
// with a barrier.
__device__ __forceinline__ void norm_pass(const StepParams &P, float *xs, int ld, bool perm, const float *gain, float *ssp,
                                          int pld = 0) {
    const int batch = P.batch, dim = P.m.dim;
    int rp = 1;
    while (rp < batch) rp <<= 1;
    const int tpr = kComputeThreads / rp;  // threads per row, >= 16
    const int tid = threadIdx.x, b = tid / tpr, t = tid - b * tpr;
    float ss = 0.f;
    if (b < batch) {
        float *r = xs + (size_t)b * ld;
        constexpr int U = 4;  // gains fetched U at a time: no chain of dependent loads
        for (int j0 = t; j0 < dim; j0 += U * tpr) {
            float gv[U];
#pragma unroll
            for (int u = 0; u < U; u++) gv[u] = j0 + u * tpr < dim ? __ldg(gain + j0 + u * tpr) : 0.f;
#pragma unroll
            for (int u = 0; u < U; u++) {
                const int j = j0 + u * tpr;
                if (j >= dim) break;
                if (pld) {  // activation planes
                    const float x = plane_load((const uint16_t *)xs, pld, b, j);
                    ss = fmaf(x, x, ss);
                    plane_store((uint16_t *)xs, pld, b, j, x * gv[u]);
                    continue;
                }
                const int q = xpos(j, ld, perm);
                const float x = r[q];
                ss = fmaf(x, x, ss);
                r[q] = x * gv[u];
            }
        }
    }
    const int w = tpr < 32 ? tpr : 32;  // lanes of one row within a warp
    for (int off = w >> 1; off >= 1; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    const int warp = tid >> 5, lane = tid & 31;
    const float s0 = __shfl_sync(0xffffffffu, ss, 0), s16 = __shfl_sync(0xffffffffu, ss, 16);
    const int row_a = (warp * 32) / tpr, row_b = (warp * 32 + 16) / tpr;  // rows of lanes 0 and 16
    if (lane < batch) {
        float v = 0.f;
        if (lane == row_a) v += s0;
        if (row_b != row_a && lane == row_b) v += s16;
        ssp[warp * kMaxBatch + lane] = v;
    }
    compute_sync();
}

__device__ void zero_pad(const StepParams &P, float *xs, int ld, int from, bool perm, int pld = 0) {
    if (pld) {  // activation planes: columns [from, ld) of the live rows of both planes.
        // Rows past the batch may hold anything: an MMA output row depends only on its
        // own activation row, and those outputs are dropped.
        const int n = ld - from;
        if (n <= 0) return;
        uint16_t *h = (uint16_t *)xs;
        for (int e = threadIdx.x; e < 2 * P.batch * n; e += kComputeThreads) {
            const int q = e / n, k = from + (e - q * n);  // q: plane-row (plane q / batch)
            const int plane = q >= P.batch, r = q - plane * P.batch;
            h[(plane * kMaxBatch + r) * pld + k] = 0;
        }
        return;
    }
    for (int b = 0; b < P.batch; b++)
        for (int k = from + (int)threadIdx.x; k < ld; k += kComputeThreads) xs[(size_t)b * ld + xpos(k, ld, perm)] = 0.f;
}

// Merge the chunk states of every (row, head) published by the attention items into
// the Wo input tile: o = sum_c 2^(m_c - M) O_c / sum_c 2^(m_c - M) l_c.
__device__ __forceinline__ void merge_chunk_states(const StepParams &P, int layer, const Mat &M, Shared &S, int pld) {
    const Model &m = P.m;
    const bool perm = m.x_perm;
    const int H = m.n_heads, hd = m.head_dim, st = hd + 2;
    int ncmax = 1;
    for (int b = 0; b < P.batch; b++) ncmax = max(ncmax, P.nchunk[b]);
    float *stage = S.xs + (pld ? (size_t)kMaxBatch * pld : (size_t)P.batch * M.KBp);  // [batch][H][ncmax][hd + 2]
    const uint64_t *src = m.ll_part + ll_layer(P, layer, H * kMaxChunksA * st);
    zero_pad(P, S.xs, M.KBp, H * hd, perm, pld);
    for (int b = 0; b < P.batch; b++) {
        const int nc = P.nchunk[b];
        // rows (b, h) x (nc * st) words, source row stride kMaxChunksA * st
        poll_words(P, src + (size_t)b * H * kMaxChunksA * st, kMaxChunksA * st, H, nc * st,
                   stage + (size_t)b * H * ncmax * st, ncmax * st, 0, nullptr, nullptr);
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
            if (pld)
                plane_store((uint16_t *)S.xs, pld, b, e, O / L);
            else
                S.xs[(size_t)b * M.KBp + xpos(e, M.KBp, perm)] = O / L;
        }
    }
    compute_sync();
}

// Stage the input of phase `epi` (K tile kt) into S.xs as fp32 [batch][KBp] (element
// order given by xpos).  An RMSNorm input is left as x * gain, with the per-warp sums
// of x^2 in S.ssp.
template <int NB>
__device__ __forceinline__ void stage_input(const StepParams &P, int epi, int layer, const Mat &M, int kt, Shared &S) {
    const Model &m = P.m;
    const int tid = threadIdx.x;
    const bool perm = m.x_perm;
    const int pl = perm ? M.KBp : 0;
    const int pld = (NB == kMaxBatch && m.weight_bf16) ? M.KBp + 8 : 0;  // activation planes (tensor-core phases)
    float *dst = S.xs;
    const int dld = pld ? pld : M.KBp;
    compute_sync();  // everyone is done with the previous tile
    if (epi == EPI_QKV || epi == EPI_W13 || epi == EPI_LOGITS) {
        const float *g = epi == EPI_QKV   ? m.norms + (size_t)layer * 2 * m.dim
                         : epi == EPI_W13 ? m.norms + (size_t)layer * 2 * m.dim + m.dim
                                          : m.norms + (size_t)m.n_layers * 2 * m.dim;
        zero_pad(P, S.xs, M.KBp, m.dim, perm, pld);
        if (epi == EPI_QKV && tid < P.batch) {  // the QKV epilogue's RoPE rows, into L1 meanwhile
            const float *rr = m.rope + (size_t)P.pos[tid] * m.head_dim;
            for (int k = 0; k < m.head_dim; k += 32) prefetch_l1(rr + k);
        }
        if (epi == EPI_QKV && layer == 0) {
            for (int b = 0; b < P.batch; b++) {
                const int tok = token_of(P, b);
                for (int k = tid; k < m.dim; k += kComputeThreads) {
                    if (pld)
                        plane_store((uint16_t *)S.xs, pld, b, k, emb_elem(m, tok, k));
                    else
                        S.xs[(size_t)b * M.KBp + xpos(k, M.KBp, perm)] = emb_elem(m, tok, k);
                }
            }
            compute_sync();
            norm_pass(P, S.xs, M.KBp, perm, g, S.ssp, pld);
        } else {
            const uint64_t *src = epi == EPI_W13 ? m.ll_xa + ll_layer(P, layer, m.dim)
                                                 : m.ll_x + ll_layer(P, epi == EPI_QKV ? layer : m.n_layers, m.dim);
            poll_words<(NB > 1 ? 2 : 1)>(P, src, m.dim, P.batch, m.dim, dst, dld, pl, g, S.ssp, pld > 0);
        }
    } else if (epi == EPI_WO) {
        if (P.attn_consumer_merge) {
            merge_chunk_states(P, layer, M, S, pld);
        } else {
            const int qd = m.n_heads * m.head_dim;
            zero_pad(P, S.xs, M.KBp, qd, perm, pld);
            poll_words<(NB > 1 ? 2 : 1)>(P, m.ll_o + ll_layer(P, layer, qd), qd, P.batch, qd, dst, dld, pl, nullptr, nullptr,
                                         pld > 0);
        }
    } else {  // W2: tile kt of the SwiGLU output
        const int k0 = kt * M.KB, kn = min(M.K - k0, M.KB);
        zero_pad(P, S.xs, M.KBp, kn, perm, pld);
        poll_words<(NB > 1 ? 2 : 1)>(P, m.ll_h + ll_layer(P, layer, m.hidden) + k0, m.hidden, P.batch, kn, dst, dld, pl,
                                     nullptr, nullptr, pld > 0);
    }
}

// ------------------------------------------------------------------ GEMV arithmetic

// A warp works on RG rows at once: RG independent accumulator chains per batch row,
// one activation load per piece shared by all of them.
template <int NB> struct GemvShape {
    static constexpr int R = NB == 1 ? 4 : NB <= 4 ? 2 : 1;
};

// ------------------------------------------------------------------ epilogues

// 1 / rms of batch row b from the per-warp sums of squares.
__device__ __forceinline__ float inv_rms(const Model &m, const float *ssp, int b) {
    float ss = 0.f;
#pragma unroll
    for (int w = 0; w < kComputeWarps; w++) ss += ssp[w * kMaxBatch + b];
    return 1.0f / sqrtf(ss / (float)m.dim + m.norm_eps);
}

// What the lane that will hold a group's value does with it; everything that does not
// depend on the value is worked out before the input arrives.
enum { EK_Q = 0, EK_K = 1, EK_V = 2, EK_W13 = 3, EK_RES = 4, EK_LOGITS = 5 };
struct EpiCtx {
    uint64_t *dst;   // exchange word this lane publishes (RoPE pair: the first; second at + half)
    uint8_t *cache;  // key / value cache element of a RoPE pair's first dim
    float cs, sn;    // RoPE of a q / k pair
    int kind;        // EK_*
    int half;        // RoPE pair: dims between its two elements
    int own;         // Wo / W2: owned row within the CTA's slice; logits: vocabulary index
    int b;           // batch row of the value; -1: this lane publishes nothing
};

// Group of RG rows (RPU = 1) or one RoPE / SwiGLU pair unit (RG = RPU = 2) starting at
// unit j0 of a chunk whose first unit is unit0 of the CTA's slice [u0, ...); ng units.
template <int NB, int RG, int RPU>
__device__ __forceinline__ EpiCtx prepare_ctx(const StepParams &P, int epi, int layer, int u0, int unit0, int j0, int ng) {
    constexpr int V = RG * NB;
    constexpr int SHIFT = 5 - Log2<V>::value;
    const Model &m = P.m;
    const int lane = threadIdx.x & 31;
    const int idx = lane >> SHIFT;  // value this lane holds after the reduction
    const bool holder = (lane & ((1 << SHIFT) - 1)) == 0;
    const int r = idx / NB, b = idx - r * NB;
    EpiCtx c;
    c.b = -1;
    c.dst = nullptr;
    c.cache = nullptr;
    c.cs = 1.f;
    c.sn = 0.f;
    c.kind = EK_RES;
    c.half = 0;
    c.own = 0;
    if constexpr (RPU == 2) {  // the lane of the pair's first row publishes
        const int u = r >> 1;
        if (!holder || (r & 1) || u >= ng || b >= P.batch) return c;
        const int unit = u0 + unit0 + j0 + u;
        c.b = b;
        if (epi == EPI_W13) {
            c.kind = EK_W13;
            c.dst = m.ll_h + ll_layer(P, layer, m.hidden) + (size_t)b * m.hidden + unit;
            return c;
        }
        const int hd = m.head_dim, half = hd >> 1, G = m.n_heads / m.n_kv_heads;
        const int per_group = (G + 2) * half;
        const int g = unit / per_group, rem = unit - g * per_group;
        const int s = rem / half, i = rem - s * half;
        const int pos = P.pos[b];
        c.half = half;
        c.kind = s < G ? EK_Q : s == G ? EK_K : EK_V;
        if (s <= G) {
            const float *rp = m.rope + ((size_t)pos * half + i) * 2;
            c.cs = rp[0];
            c.sn = rp[1];
        }
        if (s >= G) {
            const int esz = m.kv_bf16 ? 2 : 4;
            c.cache = (s == G ? m.kc : m.vc) + (kv_row(m, layer, P.seq[b], g, pos) * hd + i) * esz;
        }
        c.dst = m.ll_qkv + ll_layer(P, layer, m.qkv.rows) + (size_t)b * m.qkv.rows + ((size_t)g * (G + 2) + s) * hd + i;
        return c;
    } else {
        if (!holder || r >= ng || b >= P.batch) return c;
        const int i = unit0 + j0 + r;  // unit within the CTA's slice
        c.b = b;
        c.own = i;
        if (epi == EPI_LOGITS) {
            c.kind = EK_LOGITS;
            c.own = u0 + i;
            return c;
        }
        c.dst = (epi == EPI_WO ? m.ll_xa + ll_layer(P, layer, m.dim) : m.ll_x + ll_layer(P, layer + 1, m.dim)) +
                (size_t)b * m.dim + u0 + i;
        return c;
    }
}

// A logits candidate this lane holds after a group (v = -inf: none).
struct Cand {
    float v;
    int i, b;
};

// The dots of a prepared group, the warp reduction and the epilogue.  rs1: 1/rms of the
// single batch row when NB = 1 (RMSNorm inputs).
template <int NB, int RG, int RPU, int WT>
__device__ __forceinline__ Cand group_compute(const StepParams &P, const Mat &M, Shared &S,
                                              const GroupW<NB, RG, WT> &G, const EpiCtx &c, const uint8_t *base,
                                              int nr, int kt, float rs1) {
    constexpr int V = RG * NB;
    constexpr int SHIFT = 5 - Log2<V>::value;
    const Model &m = P.m;
    const int lane = threadIdx.x & 31;
    const size_t rowbytes = (size_t)tile_rowbytes(WT, M.KBp);
    Cand cd{-INFINITY, 0, 0};
    float acc[V];
    rows_dot<NB, RG, WT>(G, base, rowbytes, nr, S.xs, M.KBp, P.batch, acc);
    const float val = reduce_scatter<V>(acc);
    float second = 0.f;
    if constexpr (RPU == 2) second = __shfl_sync(0xffffffffu, val, ((((lane >> SHIFT) + NB) << SHIFT) & 31));
    if (c.b < 0) return cd;
    const uint32_t tag = P.tag;
    const float rs = c.kind == EK_RES ? 1.f : NB == 1 ? rs1 : inv_rms(m, S.ssp, c.b);
    const float v = val * rs;
    if constexpr (RPU == 2) {
        const float x2 = second * rs;
        if (c.kind == EK_W13) {
            const float sg = v / (1.0f + __expf(-v));
            ll_store(c.dst, sg * x2, tag);
            return cd;
        }
        float o0 = v, o1 = x2;
        if (c.kind != EK_V) {
            o0 = v * c.cs - x2 * c.sn;
            o1 = v * c.sn + x2 * c.cs;
        }
        if (c.kind == EK_Q) {  // scores in base-2 units: q * log2(e) / sqrt(d)
            const float qscale = rsqrtf((float)m.head_dim) * 1.4426950408889634f;
            o0 *= qscale;
            o1 *= qscale;
        } else if (m.kv_bf16) {  // k, v: round to the cache type, append
            const __nv_bfloat16 h0 = __float2bfloat16_rn(o0), h1 = __float2bfloat16_rn(o1);
            ((__nv_bfloat16 *)c.cache)[0] = h0;
            ((__nv_bfloat16 *)c.cache)[c.half] = h1;
            o0 = __bfloat162float(h0);
            o1 = __bfloat162float(h1);
        } else {
            ((float *)c.cache)[0] = o0;
            ((float *)c.cache)[c.half] = o1;
        }
        ll_store(c.dst, o0, tag);
        ll_store(c.dst + c.half, o1, tag);
        return cd;
    } else {
        if (c.kind == EK_LOGITS) {
            if (P.logits) P.logits[(size_t)c.b * m.vocab + c.own] = v;
            if (v != v) {
                atomicOr(m.status, kStNanLogits);
            } else {
                cd.v = v;
                cd.i = c.own;
                cd.b = c.b;
            }
            return cd;
        }
        float t = v;
        if (M.nkt > 1) {  // accumulate this K tile; finish after the last one
            float *a = S.accs + (size_t)c.own * kMaxBatch + c.b;
            t = (kt == 0 ? 0.f : *a) + t;
            *a = t;
            if (kt != M.nkt - 1) return cd;
        }
        // Wo / W2: residual add on the owned row, publish the new residual
        float *own = S.xown + c.b * P.own_ld + c.own;
        const float xn = *own + t;
        *own = xn;
        if (m.fault && c.dst == m.ll_x + ll_layer(P, 1, m.dim)) return cd;  // test hook: a lost publish
        ll_store(c.dst, xn, tag);
        return cd;
    }
}

// ------------------------------------------------------------------ GEMV phases

template <int NB>
__device__ __forceinline__ void keep_best(const Cand &cd, float (&best_v)[NB], int (&best_i)[NB]) {
#pragma unroll
    for (int bb = 0; bb < NB; bb++)
        if (bb == cd.b && (cd.v > best_v[bb] || (cd.v == best_v[bb] && cd.i < best_i[bb]))) {
            best_v[bb] = cd.v;
            best_i[bb] = cd.i;
        }
}

__device__ __forceinline__ bool is_norm_input(int epi) { return epi == EPI_QKV || epi == EPI_W13 || epi == EPI_LOGITS; }

// The chunks of one of a layer's matrices for this CTA, K tile by K tile: chunk i of
// the step belongs to warp i % 8; with a multiple of 8 ring slots every use of a slot
// belongs to the same warp, which takes them in order.  At batch 1 a chunk of 4-8 rows
// is one row group; otherwise a group is a RoPE / SwiGLU pair or two rows (each
// activation load then serves two rows).  Each warp goes straight to its own chunks and, before the input is polled,
// waits for its first chunk's weights, loads its first group's pieces into registers
// and prepares that group's epilogue; after the poll only the arithmetic and the
// stores remain.  Returns the updated chunk counter.
template <int NB, int WT, int RG>
__device__ __forceinline__ uint32_t layer_walk(const StepParams &P, int epi, int layer, const Mat &M, Shared &S,
                                               uint32_t chunk_i, int tslot) {
    // RG: rows of a group (8 at batch 1 when chunks hold at least 4 rows, else 2)
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int u0, u1;
    phase_slice(P, epi, M.rows / M.rows_per_unit, blockIdx.x, u0, u1);
    trace_mark(P, tslot, 0);
    if (u0 == u1) return chunk_i;
    const int cu = M.rows_per_chunk / M.rows_per_unit;  // units per chunk
    const int cpk = (u1 - u0 + cu - 1) / cu;            // chunks per K tile
    const int nch = M.nkt * cpk;
    const uint32_t slots = (uint32_t)P.ring_slots;
    const size_t rowbytes = (size_t)tile_rowbytes(WT, M.KBp);
    const int pieces = M.KBp / Piece<WT>::elems;
    const bool pairs = M.rows_per_unit == 2;
    // the warp's chunks of the phase: j, j + 8, ...; the current group: units [g, g + ng)
    // of chunk j
    int j = (warp - (int)(chunk_i & 7)) & 7;
    int g = 0, ng = 0;
    GroupW<NB, RG, WT> wp;
    EpiCtx ctx;
    const uint8_t *buf = nullptr;
    // Prepare the group at unit g of chunk j: weights of its first pieces into registers,
    // epilogue.  j < 8 <= slots: the first chunk never waits for a chunk consumed after
    // the poll.
    auto prepare = [&]() {
        const uint32_t ci = chunk_i + (uint32_t)j;
        const int kt = j / cpk, unit0 = (j - kt * cpk) * cu, nunits = min(cu, u1 - u0 - unit0);
        ng = min(nunits - g, RG / M.rows_per_unit);  // batches: 2 rows share each activation load
        if (g == 0) wait_slot(P, &S.full[ci % slots], (ci / slots) & 1);
        buf = S.ring + (size_t)(ci % slots) * kChunkBytes + (size_t)g * M.rows_per_unit * rowbytes;
        load_pieces<NB, RG, WT>(wp, buf, rowbytes, ng * M.rows_per_unit, lane, pieces, M.KBp);
        ctx = pairs ? prepare_ctx<NB, RG, 2>(P, epi, layer, u0, unit0, g, ng)
                    : prepare_ctx<NB, RG, 1>(P, epi, layer, u0, unit0, g, ng);
    };
    if (j < nch) prepare();
#pragma unroll 1
    for (int kt = 0; kt < M.nkt; kt++) {
        stage_input<NB>(P, epi, layer, M, kt, S);
        if (kt == 0) trace_mark(P, tslot, 1);
        const float rs1 = (NB == 1 && is_norm_input(epi)) ? inv_rms(P.m, S.ssp, 0) : 1.f;
#pragma unroll 1
        while (j < nch && j < (kt + 1) * cpk) {
            const int unit0 = (j - kt * cpk) * cu, nunits = min(cu, u1 - u0 - unit0);
            if (pairs)
                group_compute<NB, RG, 2, WT>(P, M, S, wp, ctx, buf, ng * 2, kt, rs1);
            else
                group_compute<NB, RG, 1, WT>(P, M, S, wp, ctx, buf, ng, kt, rs1);
            g += ng;
            if (g >= nunits) {  // chunk done: release its slot, move to the warp's next one
                __syncwarp();
                if (lane == 0) mbar_arrive(&S.empty[(chunk_i + (uint32_t)j) % slots]);
                g = 0;
                j += kComputeWarps;
            }
            if (j < nch) prepare();
        }
    }
    if (P.trace) compute_sync();  // the timeline's "done" covers every warp
    trace_mark(P, tslot, 2);
    return chunk_i + (uint32_t)nch;
}

// The logits: chunks of up to R rows per group (8 at batch 1), each lane keeping the
// best (value, index) per batch row.
template <int NB, int WT, bool G8>
__device__ __forceinline__ uint32_t logits_walk(const StepParams &P, const Mat &M, Shared &S, uint32_t chunk_i, int tslot,
                                                float (&best_v)[NB], int (&best_i)[NB]) {
    constexpr int R = NB == 1 ? (G8 ? 8 : 2) : GemvShape<NB>::R;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int u0, u1;
    phase_slice(P, 4, M.rows, blockIdx.x, u0, u1);
    trace_mark(P, tslot, 0);
    if (u0 == u1) return chunk_i;
    const int cu = M.rows_per_chunk;
    const int nch = (u1 - u0 + cu - 1) / cu;
    const uint32_t slots = (uint32_t)P.ring_slots;
    const size_t rowbytes = (size_t)tile_rowbytes(WT, M.KBp);
    const int pieces = M.KBp / Piece<WT>::elems;
    int j = (warp - (int)(chunk_i & 7)) & 7;
    if (j < nch) wait_slot(P, &S.full[(chunk_i + (uint32_t)j) % slots], ((chunk_i + (uint32_t)j) / slots) & 1);
    stage_input<NB>(P, EPI_LOGITS, 0, M, 0, S);
    trace_mark(P, tslot, 1);
    const float rs1 = NB == 1 ? inv_rms(P.m, S.ssp, 0) : 1.f;
#pragma unroll 1
    for (; j < nch; j += kComputeWarps) {
        const uint32_t ci = chunk_i + (uint32_t)j, slot = ci % slots;
        wait_slot(P, &S.full[slot], (ci / slots) & 1);
        const int unit0 = j * cu, nunits = min(cu, u1 - u0 - unit0);
        const uint8_t *buf = S.ring + (size_t)slot * kChunkBytes;
#pragma unroll 1
        for (int g = 0; g < nunits; g += R) {
            const int ng = min(R, nunits - g);
            if (R > 1 && ng == 1) {
                GroupW<NB, 1, WT> w;
                load_pieces<NB, 1, WT>(w, buf + (size_t)g * rowbytes, rowbytes, 1, lane, pieces, M.KBp);
                const EpiCtx c = prepare_ctx<NB, 1, 1>(P, EPI_LOGITS, 0, u0, unit0, g, 1);
                keep_best<NB>(group_compute<NB, 1, 1, WT>(P, M, S, w, c, buf + (size_t)g * rowbytes, 1, 0, rs1),
                              best_v, best_i);
            } else {
                GroupW<NB, R, WT> w;
                load_pieces<NB, R, WT>(w, buf + (size_t)g * rowbytes, rowbytes, ng, lane, pieces, M.KBp);
                const EpiCtx c = prepare_ctx<NB, R, 1>(P, EPI_LOGITS, 0, u0, unit0, g, ng);
                keep_best<NB>(group_compute<NB, R, 1, WT>(P, M, S, w, c, buf + (size_t)g * rowbytes, ng, 0, rs1),
                              best_v, best_i);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.empty[slot]);
    }
    if (P.trace) compute_sync();
    trace_mark(P, tslot, 2);
    return chunk_i + (uint32_t)nch;
}

// ------------------------------------------------------------------ batch 16: tensor cores

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm4(uint32_t (&r)[4], const void *p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(smem_addr(p)));
}

__device__ __forceinline__ void ldsm2(uint32_t &r0, uint32_t &r1, const void *p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(smem_addr(p)));
}

// One value of a batch-16 tensor-core tile: row `unit` (pairs: its first row) of the
// CTA's slice for batch row b.  Same epilogues as the CUDA-core groups.
__device__ __forceinline__ Cand mma_epilogue(const StepParams &P, int epi, int layer, const Mat &M, Shared &S, int u0,
                                             int i, int b, float v, float v2, int kt) {
    const Model &m = P.m;
    Cand cd{-INFINITY, 0, 0};
    const uint32_t tag = P.tag;
    const int unit = u0 + i;
    if (epi == EPI_W13 || epi == EPI_QKV) {  // pair unit: v = first row, v2 = second
        const float rs = inv_rms(m, S.ssp, b);
        const float x1 = v * rs, x2 = v2 * rs;
        if (epi == EPI_W13) {
            const float sg = x1 / (1.0f + __expf(-x1));
            ll_store(m.ll_h + ll_layer(P, layer, m.hidden) + (size_t)b * m.hidden + unit, sg * x2, tag);
            return cd;
        }
        const int hd = m.head_dim, half = hd >> 1, G = m.n_heads / m.n_kv_heads;
        const int per_group = (G + 2) * half;
        const int g = unit / per_group, rem = unit - g * per_group;
        const int sub = rem / half, d = rem - sub * half;
        const int pos = P.pos[b];
        float o0 = x1, o1 = x2;
        if (sub <= G) {
            const float *rp = m.rope + ((size_t)pos * half + d) * 2;
            o0 = x1 * rp[0] - x2 * rp[1];
            o1 = x1 * rp[1] + x2 * rp[0];
        }
        if (sub < G) {
            const float qscale = rsqrtf((float)hd) * 1.4426950408889634f;
            o0 *= qscale;
            o1 *= qscale;
        } else {
            const bool bf = m.kv_bf16;
            uint8_t *row = (sub == G ? m.kc : m.vc) + kv_row(m, layer, P.seq[b], g, pos) * hd * (bf ? 2 : 4);
            if (bf) {
                const __nv_bfloat16 h0 = __float2bfloat16_rn(o0), h1 = __float2bfloat16_rn(o1);
                ((__nv_bfloat16 *)row)[d] = h0;
                ((__nv_bfloat16 *)row)[d + half] = h1;
                o0 = __bfloat162float(h0);
                o1 = __bfloat162float(h1);
            } else {
                ((float *)row)[d] = o0;
                ((float *)row)[d + half] = o1;
            }
        }
        uint64_t *dst = m.ll_qkv + ll_layer(P, layer, m.qkv.rows) + (size_t)b * m.qkv.rows + ((size_t)g * (G + 2) + sub) * hd + d;
        ll_store(dst, o0, tag);
        ll_store(dst + half, o1, tag);
        return cd;
    }
    if (epi == EPI_LOGITS) {
        v *= inv_rms(m, S.ssp, b);
        if (P.logits) P.logits[(size_t)b * m.vocab + unit] = v;
        if (v != v) {
            atomicOr(m.status, kStNanLogits);
        } else {
            cd.v = v;
            cd.i = unit;
            cd.b = b;
        }
        return cd;
    }
    float t = v;  // Wo / W2: K tiles accumulate, then the residual add
    if (M.nkt > 1) {
        float *a = S.accs + (size_t)i * kMaxBatch + b;
        t = (kt == 0 ? 0.f : *a) + t;
        *a = t;
        if (kt != M.nkt - 1) return cd;
    }
    float *own = S.xown + b * P.own_ld + i;
    const float xn = *own + t;
    *own = xn;
    uint64_t *dstw = epi == EPI_WO ? m.ll_xa + ll_layer(P, layer, m.dim) : m.ll_x + ll_layer(P, layer + 1, m.dim);
    ll_store(dstw + (size_t)b * m.dim + unit, xn, tag);
    return cd;
}

// A matrix's chunks for this CTA at batch 16, on the tensor cores: each chunk (at most 8
// rows) is one n8 tile of mma.sync m16n8k16 -- A = the 16 batch rows of activations
// (bf16 hi and lo planes: two MMAs per K step, fp32 accumulation), B = the chunk's
// weight rows read with ldmatrix straight from the ring slot.  Chunk ownership and
// ring protocol as in layer_walk.  For the logits, lanes keep their best candidates.
template <bool LOGITS>
__device__ __forceinline__ uint32_t mma_walk(const StepParams &P, int epi, int layer, const Mat &M, Shared &S,
                                             uint32_t chunk_i, int tslot, float (&best_v)[2], int (&best_i)[2]) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g4 = lane >> 2, t4 = lane & 3;
    int u0, u1;
    phase_slice(P, epi, M.rows / M.rows_per_unit, blockIdx.x, u0, u1);
    trace_mark(P, tslot, 0);
    if (u0 == u1) return chunk_i;
    const int rpu = M.rows_per_unit;
    const int cu = M.rows_per_chunk / rpu;
    const int cpk = (u1 - u0 + cu - 1) / cu;
    const int nch = M.nkt * cpk;
    const uint32_t slots = (uint32_t)P.ring_slots;
    const size_t rowbytes = (size_t)M.KBp * 2 + kRowPad;  // ring row stride (padded)
    const int pld = M.KBp + 8;
    const uint16_t *hi = (const uint16_t *)S.xs, *lo = hi + kMaxBatch * pld;
    int j = (warp - (int)(chunk_i & 7)) & 7;
    if (j < nch) wait_slot(P, &S.full[(chunk_i + (uint32_t)j) % slots], ((chunk_i + (uint32_t)j) / slots) & 1);
#pragma unroll 1
    for (int kt = 0; kt < M.nkt; kt++) {
        stage_input<kMaxBatch>(P, epi, layer, M, kt, S);
        if (kt == 0) trace_mark(P, tslot, 1);
#pragma unroll 1
        for (; j < nch && j < (kt + 1) * cpk; j += kComputeWarps) {
            const uint32_t ci = chunk_i + (uint32_t)j, slot = ci % slots;
            wait_slot(P, &S.full[slot], (ci / slots) & 1);
            const int unit0 = (j - kt * cpk) * cu, nunits = min(cu, u1 - u0 - unit0), nr = nunits * rpu;
            const uint8_t *buf = S.ring + (size_t)slot * kChunkBytes;
            // B rows: lanes 0-7 give the rows of k 0..7, lanes 8-15 of k 8..15 (rows past the
            // chunk read its last row; their outputs are dropped)
            const uint8_t *bp = buf + (size_t)min(lane & 7, nr - 1) * rowbytes + ((lane >> 3) & 1) * 16;
            const uint16_t *ah = hi + (lane & 15) * pld + (lane >> 4) * 8, *al = lo + (lane & 15) * pld + (lane >> 4) * 8;
            // four independent accumulators (hi / lo plane x even / odd K step) keep four
            // MMA chains in flight instead of one
            float d[4] = {0.f, 0.f, 0.f, 0.f}, e[4] = {0.f, 0.f, 0.f, 0.f};
            float f[4] = {0.f, 0.f, 0.f, 0.f}, g[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 2
            for (int k = 0; k < M.KBp; k += 32) {  // KBp is a multiple of 64
                uint32_t a[4], c[4], a2[4], c2[4], b0, b1, b2, b3;
                ldsm4(a, ah + k);
                ldsm4(c, al + k);
                ldsm2(b0, b1, bp + k * 2);
                ldsm4(a2, ah + k + 16);
                ldsm4(c2, al + k + 16);
                ldsm2(b2, b3, bp + (k + 16) * 2);
                mma16816(d, a, b0, b1);
                mma16816(e, c, b0, b1);
                mma16816(f, a2, b2, b3);
                mma16816(g, c2, b2, b3);
            }
#pragma unroll
            for (int q = 0; q < 4; q++) d[q] = (d[q] + f[q]) + (e[q] + g[q]);
            __syncwarp();
            if (lane == 0) mbar_arrive(&S.empty[slot]);
            // d0 = (batch g4, row 2 t4), d1 = (g4, 2 t4 + 1), d2 / d3 the same for batch g4 + 8
            const int n0 = 2 * t4;
#pragma unroll
            for (int h = 0; h < 2; h++) {
                const int b = g4 + 8 * h;
                if (b >= P.batch) continue;
                const float v0 = d[2 * h], v1 = d[2 * h + 1];
                if (rpu == 2) {
                    if (t4 < nunits) mma_epilogue(P, epi, layer, M, S, u0, unit0 + t4, b, v0, v1, kt);
                } else {
                    // a lane only ever holds batch rows g4 (h = 0) and g4 + 8 (h = 1): it keeps
                    // one candidate for each
                    if (n0 < nr) {
                        const Cand cd = mma_epilogue(P, epi, layer, M, S, u0, unit0 + n0, b, v0, 0.f, kt);
                        if constexpr (LOGITS)
                            if (cd.v > best_v[h] || (cd.v == best_v[h] && cd.i < best_i[h])) {
                                best_v[h] = cd.v;
                                best_i[h] = cd.i;
                            }
                    }
                    if (n0 + 1 < nr) {
                        const Cand cd = mma_epilogue(P, epi, layer, M, S, u0, unit0 + n0 + 1, b, v1, 0.f, kt);
                        if constexpr (LOGITS)
                            if (cd.v > best_v[h] || (cd.v == best_v[h] && cd.i < best_i[h])) {
                                best_v[h] = cd.v;
                                best_i[h] = cd.i;
                            }
                    }
                }
            }
        }
    }
    if (P.trace) compute_sync();
    trace_mark(P, tslot, 2);
    return chunk_i + (uint32_t)nch;
}

template <int NB, int WT, bool G8>
__device__ __forceinline__ uint32_t gemv_phase(const StepParams &P, int epi, int layer, const Mat &M, Shared &S,
                                            uint32_t chunk_i, int tslot) {
    if constexpr (NB == kMaxBatch && WT == kWBF16) {  // batch 16: tensor cores
        float bv[2];
        int bi[2];
        return mma_walk<false>(P, epi, layer, M, S, chunk_i, tslot, bv, bi);
    } else {
        return layer_walk<NB, WT, (NB == 1 && G8) ? 8 : 2>(P, epi, layer, M, S, chunk_i, tslot);
    }
}

// The logits and the greedy argmax: per lane, per warp, per CTA best candidates (lowest
// index on ties); CTA 0 collects every CTA's candidate.
template <int NB, int WT, bool G8>
__device__ __forceinline__ void logits_phase(const StepParams &P, Shared &S, uint32_t chunk_i, int tslot) {
    const Model &m = P.m;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int batch = P.batch;
    if constexpr (NB == kMaxBatch && WT == kWBF16) {
        // lane (g4, t4) holds candidates of batch rows g4 and g4 + 8: reduce over t4
        float bv[2] = {-INFINITY, -INFINITY};
        int bi[2] = {0x7fffffff, 0x7fffffff};
        mma_walk<true>(P, EPI_LOGITS, 0, m.emb, S, chunk_i, tslot, bv, bi);
        trace_mark(P, tslot + 1, 0);
        compute_sync();  // the logits phase is done with S.xs
#pragma unroll
        for (int h = 0; h < 2; h++) {
            float v = bv[h];
            int i = bi[h];
#pragma unroll
            for (int off = 1; off <= 2; off <<= 1) {
                const float v2 = __shfl_xor_sync(0xffffffffu, v, off);
                const int i2 = __shfl_xor_sync(0xffffffffu, i, off);
                if (v2 > v || (v2 == v && i2 < i)) {
                    v = v2;
                    i = i2;
                }
            }
            const int b = (lane >> 2) + 8 * h;
            if ((lane & 3) == 0 && b < batch) {
                S.wbest_v[warp * kMaxBatch + b] = v;
                S.wbest_i[warp * kMaxBatch + b] = i;
            }
        }
    } else {
    float best_v[NB];
    int best_i[NB];
#pragma unroll
    for (int b = 0; b < NB; b++) {
        best_v[b] = -INFINITY;
        best_i[b] = 0x7fffffff;
    }
    logits_walk<NB, WT, G8>(P, m.emb, S, chunk_i, tslot, best_v, best_i);
    trace_mark(P, tslot + 1, 0);
    compute_sync();  // the logits phase is done with S.xs
#pragma unroll
    for (int b = 0; b < NB; b++) {
        float v = best_v[b];
        int i = best_i[b];
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) {
            const float v2 = __shfl_xor_sync(0xffffffffu, v, off);
            const int i2 = __shfl_xor_sync(0xffffffffu, i, off);
            if (v2 > v || (v2 == v && i2 < i)) {
                v = v2;
                i = i2;
            }
        }
        if (b < batch && lane == 0) {
            S.wbest_v[warp * kMaxBatch + b] = v;
            S.wbest_i[warp * kMaxBatch + b] = i;
        }
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
    if (blockIdx.x == 0) {
        // CTA 0: poll [batch][grid][2] words into shared memory, reduce per row
        poll_words(P, m.ll_amax, P.grid * 2, batch, P.grid * 2, S.xs, P.grid * 2, 0, nullptr, nullptr);
        for (int b = warp; b < batch; b += kComputeWarps) {  // a warp per batch row
            float bv = -INFINITY;
            int bi = 0x7fffffff;
            const float *r = S.xs + (size_t)b * P.grid * 2;
            for (int c = lane; c < P.grid; c += 32) {
                const float v = r[2 * c];
                const int i = __float_as_int(r[2 * c + 1]);
                if (v > bv || (v == bv && i < bi)) {
                    bv = v;
                    bi = i;
                }
            }
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) {
                const float v2 = __shfl_xor_sync(0xffffffffu, bv, off);
                const int i2 = __shfl_xor_sync(0xffffffffu, bi, off);
                if (v2 > bv || (v2 == bv && i2 < bi)) {
                    bv = v2;
                    bi = i2;
                }
            }
            if (lane == 0) {
                if (bi == 0x7fffffff) bi = 0;  // all NaN: the status word already records it
                if (P.next_ids) P.next_ids[b] = bi;
            }
        }
        if (P.done_word) {  // host-memory ids: tell the host they are complete, with the status
            compute_sync();
            if (tid == 0) {
                ((volatile uint32_t *)P.done_word)[1] = (uint32_t)ld_volatile_int(m.status);
                __threadfence_system();
                *(volatile uint32_t *)P.done_word = P.tag;
            }
        }
    }
    trace_mark(P, tslot + 1, 2);
}

// ------------------------------------------------------------------ attention phase

// One work item: the query heads of kv group g of batch row b against positions
// [t0, t1) of chunk c.  q arrives rotated and scaled from the QKV epilogue; the chunk
// that ends at the new position also takes that position's key and value from the
// exchange words (the cache copy written by the QKV epilogue is for later steps).
__device__ __forceinline__ void attn_item(const StepParams &P, int layer, int b, int g, int c, Shared &S) {
    const Model &m = P.m;
    const int tid = threadIdx.x;
    const bool kvbf16 = m.kv_bf16;
    const int hd = m.head_dim, H = m.n_heads, KV = m.n_kv_heads, G = H / KV;
    const int qrows = m.qkv.rows;
    const int pos = P.pos[b], ctx = pos + 1, seq = P.seq[b];
    const int CH = P.attn_chunk, nc = P.nchunk[b];
    const int t0 = c * CH, t1 = min(ctx, t0 + CH);
    const size_t rowbytes = (size_t)hd * (kvbf16 ? 2 : 4);
    // rows of page 0 of this layer and kv head; the sequence's pages from its table row
    const size_t head_off = (((size_t)layer * m.kv_npages) * KV + g) * m.kv_rows * rowbytes;
    const size_t page_stride = (size_t)KV * m.kv_rows * rowbytes;
    const int *pages = m.kv_table + (size_t)seq * m.kv_pps;
    const uint8_t *kbase = m.kc + head_off;
    const uint8_t *vbase = m.vc + head_off;
    const uint64_t *qkv = m.ll_qkv + ll_layer(P, layer, qrows) + (size_t)b * qrows + (size_t)g * (G + 2) * hd;
    const bool appends = t1 == ctx;  // this chunk ends at the new position

    // Shared scratch after attn_core's: the group's [q heads; k; v] rows, then (when it
    // fits) a copy of the chunk's cached keys and values, else the new position's row.
    // The cached rows do not depend on this step, so their copy starts before the poll.
    float *raw = S.xs + kMaxGroupPass * hd + kComputeWarps * kMaxGroupPass * (hd + 2);
    uint8_t *kst = (uint8_t *)(raw + (size_t)(G + 2) * hd);
    const int tc = appends ? pos : t1;  // cached positions [t0, tc) of this chunk
    const bool stage = (size_t)(t1 - t0) * rowbytes * 2 <= (size_t)P.attn_stage_bytes;
    uint8_t *vst = kst + (size_t)(stage ? t1 - t0 : 1) * rowbytes;
    compute_sync();  // the previous item is done with the scratch
    if (stage) {
        const int per_row = (int)(rowbytes / 16), n16 = (tc - t0) * per_row;
        for (int e = tid; e < n16; e += kComputeThreads) {
            const int r = e / per_row, t = t0 + r;
            const size_t piece = (size_t)(e - r * per_row) * 16;
            const size_t src = (size_t)__ldg(pages + (t >> m.kv_shift)) * page_stride +
                               (size_t)(t & m.kv_mask) * rowbytes + piece;
            cp_async16(kst + (size_t)r * rowbytes + piece, kbase + src);
            cp_async16(vst + (size_t)r * rowbytes + piece, vbase + src);
        }
    }
    poll_words(P, qkv, hd, appends ? G + 2 : G, hd, raw, hd, 0, nullptr, nullptr);
    trace_mark(P, layer * kTracePerLayer + 1, 1);
    if (appends) {  // the new row, in the cache type (already rounded by the producer)
        uint8_t *kd = kst + (size_t)(stage ? pos - t0 : 0) * rowbytes;
        uint8_t *vd = vst + (size_t)(stage ? pos - t0 : 0) * rowbytes;
        const float *kr = raw + (size_t)G * hd, *vr = raw + (size_t)(G + 1) * hd;
        for (int i = tid; i < hd; i += kComputeThreads) {
            if (kvbf16) {
                ((__nv_bfloat16 *)kd)[i] = __float2bfloat16_rn(kr[i]);
                ((__nv_bfloat16 *)vd)[i] = __float2bfloat16_rn(vr[i]);
            } else {
                ((float *)kd)[i] = kr[i];
                ((float *)vd)[i] = vr[i];
            }
        }
    }
    if (stage) cp_async_wait_all();
    compute_sync();  // staged rows and the new row are visible to every warp
    AttnTask T;
    T.q = raw;
    T.q_ready = true;
    T.kv_bf16 = kvbf16;
    T.kbase = stage ? kst - (size_t)t0 * rowbytes : kbase;
    T.vbase = stage ? vst - (size_t)t0 * rowbytes : vbase;
    T.pages = stage ? nullptr : pages;
    T.page_stride = page_stride;
    T.page_shift = m.kv_shift;
    T.page_mask = m.kv_mask;
    T.tail_k = kst;
    T.tail_v = vst;
    T.tail_t = (appends && !stage) ? pos : -1;
    // a chunk too long to copy whole streams through the rest of the scratch region
    T.stream = stage ? nullptr : vst + rowbytes;
    T.stream_bytes = stage ? 0 : P.xs_bytes - (int)(T.stream - (uint8_t *)S.xs);
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
    attn_core(T, S.xs, &S.flags[0]);
}

// The cached keys and values an attention item of layer `layer` will read do not
// depend on this step: the CTAs that run items ask L2 for them when the layer starts,
// so that the item's copy into shared memory does not wait for HBM.  Only the first
// kPrefetchKvBytes of each: a long chunk streams through the per-warp rings anyway, and
// a layer's whole cache at long contexts is larger than L2 (measured: no change in the
// attention phase, 5 us less in the QKV phase that issues the prefetches).
constexpr size_t kPrefetchKvBytes = 128 * 1024;

__device__ __forceinline__ void prefetch_attention_kv(const StepParams &P, int layer) {
    const Model &m = P.m;
    const int total = P.item_start[P.batch];
    int a0, an;
    attention_ctas(P, a0, an);
    const int me = (int)blockIdx.x - a0;
    if (me < 0 || me >= an || me >= total || threadIdx.x >= 2) return;
    const size_t rowbytes = (size_t)m.head_dim * (m.kv_bf16 ? 2 : 4);
    for (int item = me; item < total; item += an) {
        int b = 0;
        while (item >= P.item_start[b + 1]) b++;
        const int local = item - P.item_start[b], nc = P.nchunk[b];
        const int g = local / nc, c = local - g * nc;
        const int t0 = c * P.attn_chunk, tc = min(P.pos[b], t0 + P.attn_chunk);  // cached rows
        if (g >= m.n_kv_heads || tc <= t0) continue;
        const int tend = t0 + (int)min((size_t)(tc - t0), kPrefetchKvBytes / rowbytes);
        for (int t = t0; t < tend;) {  // one bulk prefetch per page (each below 1 MB)
            const long long page_end = ((long long)(t >> m.kv_shift) + 1) << m.kv_shift;
            const int n = (int)min((long long)tend, min(page_end, (long long)t + (1 << 20) / (long long)rowbytes)) - t;
            bulk_prefetch_l2((threadIdx.x == 0 ? m.kc : m.vc) + kv_row(m, layer, P.seq[b], g, t) * rowbytes,
                             (uint32_t)(n * rowbytes));
            t += n;
        }
    }
}

__device__ __forceinline__ void attention_phase(const StepParams &P, int layer, Shared &S) {
    const int tslot = layer * kTracePerLayer + 1;
    trace_mark(P, tslot, 0);
    const int total = P.item_start[P.batch];
    const int KV = P.m.n_kv_heads;
    int a0, an;
    attention_ctas(P, a0, an);
    const int me = (int)blockIdx.x - a0;
    for (int item = me; me >= 0 && me < an && item < total; item += an) {
        int b = 0;
        while (item >= P.item_start[b + 1]) b++;
        const int local = item - P.item_start[b];
        const int nc = P.nchunk[b];
        const int g = local / nc, c = local - g * nc;
        if (g < KV) attn_item(P, layer, b, g, c, S);
    }
    if (P.trace) compute_sync();
    trace_mark(P, tslot, 2);
}

// ------------------------------------------------------------------ the kernel

// G8: batch-1 row groups of up to 8 rows (models whose chunks hold several rows);
// otherwise groups of 2 rows or one pair.
template <int NB, int WT, bool G8>
__global__ void __launch_bounds__(kThreads, 1) decode_step_kernel(const __grid_constant__ StepParams P) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    Shared S = carve(smem_raw, P);
    const int tid = threadIdx.x;
    if (tid == 0) {
        for (int i = 0; i < P.ring_slots; i++) {
            mbar_init(&S.full[i], 1);
            mbar_init(&S.empty[i], 1);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (tid >= kComputeThreads) {
        if (tid == kComputeThreads) producer<NB == kMaxBatch && WT == kWBF16>(P, S);
        return;
    }
    const Model &m = P.m;
    uint32_t chunk_i = 0;
    init_residual(P, S);
#pragma unroll 1
    for (int l = 0; l < m.n_layers; l++) {
        // phases: QKV, attention, Wo, W1/W3, W2; the four GEMV phases share one body
#pragma unroll 1
        for (int ph = 0; ph < kTracePerLayer; ph++) {
            const int t = l * kTracePerLayer + ph;
            if (ph == 0) prefetch_attention_kv(P, l);
            if (ph == 1) {
                attention_phase(P, l, S);
                continue;
            }
            const int epi = ph == 0 ? EPI_QKV : ph == 2 ? EPI_WO : ph == 3 ? EPI_W13 : EPI_W2;
            const Mat M = ph == 0 ? m.qkv : ph == 2 ? m.wo : ph == 3 ? m.w13 : m.w2;
            chunk_i = gemv_phase<NB, WT, G8>(P, epi, l, M, S, chunk_i, t);
        }
    }
    if (P.do_logits) logits_phase<NB, WT, G8>(P, S, chunk_i, m.n_layers * kTracePerLayer);
}

// ------------------------------------------------------------------ host-side launch

size_t decode_smem_bytes(int max_batch, int own_ld, int acc_bytes, int xs_bytes, int ring_slots) {
    return ring_offset(max_batch, own_ld, acc_bytes, xs_bytes) + (size_t)ring_slots * kChunkBytes;
}

template <int NB, int WT, bool G8>
static cudaError_t launch_nb(const StepParams &P, cudaStream_t stream) {
    auto fn = decode_step_kernel<NB, WT, G8>;
    const size_t smem = decode_smem_bytes(P.m.max_batch, P.own_ld, P.acc_bytes, P.xs_bytes, P.ring_slots);
    static size_t smem_set = 0;  // the attribute only grows; set it once per size (host latency per step)
    if (smem > smem_set) {
        cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        smem_set = smem;
    }
    void *args[] = {(void *)&P};
    return cudaLaunchCooperativeKernel((const void *)fn, dim3(P.grid), dim3(kThreads), args, smem, stream);
}

template <int WT>
static cudaError_t launch_w(const StepParams &P, cudaStream_t stream) {
    if (P.batch <= 1) return P.wide_groups ? launch_nb<1, WT, true>(P, stream) : launch_nb<1, WT, false>(P, stream);
    if (P.batch <= 4) return launch_nb<4, WT, false>(P, stream);
    if (P.batch <= 8) return launch_nb<8, WT, false>(P, stream);
    return launch_nb<16, WT, false>(P, stream);
}

cudaError_t launch_decode_step(const StepParams &P, cudaStream_t stream) {
    switch (P.m.weight_type) {
    case kWQ8: return launch_w<kWQ8>(P, stream);
    case kWBF16: return launch_w<kWBF16>(P, stream);
    default: return launch_w<kWF32>(P, stream);
    }
}

cudaError_t decode_occupancy(int weight_type, size_t smem, int *blocks_per_sm) {
    auto fn = weight_type == kWQ8     ? decode_step_kernel<1, kWQ8, true>
              : weight_type == kWBF16 ? decode_step_kernel<1, kWBF16, true>
                                      : decode_step_kernel<1, kWF32, true>;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, fn, kThreads, smem);
}

}  // namespace slm
