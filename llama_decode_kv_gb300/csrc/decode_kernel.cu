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
    uint64_t *full;     // [kMaxRingSlots]
    uint64_t *empty;    // [kMaxRingSlots]
    float *rs;          // [kMaxBatch] 1 / rms
    float *wbest_v;     // [kComputeWarps][kMaxBatch]
    int *wbest_i;       // [kComputeWarps][kMaxBatch]
    int *flags;         // [4]: 0 = last-arriver flag
    float *xown;        // [kMaxBatch][kMaxOwn] residual rows this CTA owns
    float *accs;        // [kMaxOwn][kMaxBatch] accumulators across K tiles
    float *xs;          // activation tile / attention scratch, P.xs_bytes
    uint8_t *ring;      // [P.ring_slots][kChunkBytes]
};

// Layout: barriers and small arrays, owned residual rows, K-tile accumulators, the
// activation tile, then the weight ring (sized at create time from what is left).
constexpr int kMiscBytes = 2 * kMaxRingSlots * 8 + kMaxBatch * 4 + 2 * kComputeWarps * kMaxBatch * 4 + 16;
constexpr int kOwnOffset = ((kMiscBytes + 127) / 128) * 128;
constexpr int kAccOffset = kOwnOffset + kMaxBatch * kMaxOwn * 4;
constexpr int kXsOffset = kAccOffset + kMaxOwn * kMaxBatch * 4;

__host__ __device__ inline size_t ring_offset(int xs_bytes) { return ((size_t)kXsOffset + xs_bytes + 1023) / 1024 * 1024; }

__device__ __forceinline__ Shared carve(uint8_t *base, const StepParams &P) {
    Shared s;
    uint8_t *p = base;
    s.full = (uint64_t *)p;
    p += kMaxRingSlots * 8;
    s.empty = (uint64_t *)p;
    p += kMaxRingSlots * 8;
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
    s.ring = base + ring_offset(P.xs_bytes);
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

// Shared-memory position of element k of a staged activation row.  With bf16 weights
// a lane multiplies the 8 elements 8p..8p+7 of piece p; storing elements 8p+e at plane
// e/4, offset 4p + e%4 makes every lane's two float4 reads contiguous across the warp
// (no bank conflicts).  fp32 weights keep the natural order.
__device__ __forceinline__ int xpos(int k, int KBp, bool perm) {
    return perm ? ((k & 4) ? (KBp >> 1) : 0) + ((k >> 3) << 2) + (k & 3) : k;
}

__device__ __forceinline__ int xinv(int q, int KBp, bool perm) {
    if (!perm) return q;
    const int h = q >= (KBp >> 1) ? 1 : 0, r = q - h * (KBp >> 1);
    return ((r >> 2) << 3) + (h << 2) + (r & 3);
}

// Poll rows x len tagged words (row stride src_ld) into shared memory (row stride
// dst_ld; element j of a row at xpos(j, perm_ld) when perm_ld > 0) until every tag
// equals `tag`.  Each thread keeps up to 8 loads in flight.  All compute threads call
// it; it ends with a CTA barrier.
__device__ void ll_poll(const StepParams &P, const uint64_t *src, int src_ld, int rows, int len,
                        float *dst, int dst_ld, uint32_t tag, int perm_ld = 0) {
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
            dof[k] = r * dst_ld + (perm_ld ? xpos(j, perm_ld, true) : j);
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
    unit_range(M.rows / M.rows_per_unit, P.grid, blockIdx.x, c.u0, c.u1);
    c.kt = 0;
    c.u = c.u0;
}

__device__ void cursor_init(const StepParams &P, Cursor &c) {
    c.phase = 0;
    c.layer = 0;
    c.done = false;
    cursor_enter(P, c);
}

// Next chunk of the sequence; false at the end.
__device__ bool cursor_next(const StepParams &P, Cursor &c, Chunk &out) {
    const Model &m = P.m;
    const int esz = m.weight_bf16 ? 2 : 4;
    while (!c.done) {
        const Mat &M = phase_mat(m, c.phase);
        if (c.u < c.u1) {
            const int cu = M.rows_per_chunk / M.rows_per_unit;
            const long long rowbytes = (long long)M.KBp * esz;
            out.kt = c.kt;
            out.unit0 = c.u - c.u0;
            out.nunits = min(cu, c.u1 - c.u);
            out.src = M.base + (long long)(c.phase == 4 ? 0 : c.layer) * M.layer_stride +
                      ((long long)c.kt * M.rows + (long long)c.u * M.rows_per_unit) * rowbytes;
            out.bytes = (uint32_t)((long long)out.nunits * M.rows_per_unit * rowbytes);
            c.u += out.nunits;
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

// Copies this CTA's chunks into the ring, in the order the compute warps use them.
__device__ void producer(const StepParams &P, Shared &S) {
    const uint32_t slots = (uint32_t)P.ring_slots;
    Cursor ic;
    cursor_init(P, ic);
    uint32_t issued = 0;
    Chunk c;
    while (cursor_next(P, ic, c)) {
        const uint32_t slot = issued % slots;
        if (issued >= slots) {
            const uint32_t parity = ((issued / slots) - 1) & 1;
            if (!wait_slot(P, &S.empty[slot], parity)) break;
        }
        mbar_expect_tx(&S.full[slot], c.bytes);
        bulk_g2s(S.ring + (size_t)slot * kChunkBytes, c.src, c.bytes, &S.full[slot]);
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

// RMSNorm of the staged rows in place: x[k] = x[k] * rsqrt(mean + eps) * g[k] for the
// dim logical elements; the padding past dim must already be zero.
__device__ void norm_in_place(const StepParams &P, float *xs, int ld, const float *g, bool perm, Shared &S) {
    const Model &m = P.m;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    for (int b = warp; b < P.batch; b += kComputeWarps) {
        const float *r = xs + (size_t)b * ld;
        float ss = 0.f;
        for (int q = lane; q < ld; q += 32) ss = fmaf(r[q], r[q], ss);
        ss = warp_sum(ss);
        if (lane == 0) S.rs[b] = 1.0f / sqrtf(ss / (float)m.dim + m.norm_eps);
    }
    compute_sync();
    for (int b = 0; b < P.batch; b++) {
        float *r = xs + (size_t)b * ld;
        const float rs = S.rs[b];
        for (int q = tid; q < ld; q += kComputeThreads) {
            const int k = xinv(q, ld, perm);
            if (k < m.dim) r[q] = (r[q] * rs) * g[k];
        }
    }
    compute_sync();
}

__device__ void zero_pad(const StepParams &P, float *xs, int ld, int from, bool perm) {
    for (int b = 0; b < P.batch; b++)
        for (int k = from + (int)threadIdx.x; k < ld; k += kComputeThreads) xs[(size_t)b * ld + xpos(k, ld, perm)] = 0.f;
}

// Merge the chunk states of every (row, head) published by the attention items into
// the Wo input tile: o = sum_c 2^(m_c - M) O_c / sum_c 2^(m_c - M) l_c.
__device__ void merge_chunk_states(const StepParams &P, int layer, const Mat &M, Shared &S) {
    const Model &m = P.m;
    const bool perm = m.weight_bf16;
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
            S.xs[(size_t)b * M.KBp + xpos(e, M.KBp, perm)] = O / L;
        }
    }
    zero_pad(P, S.xs, M.KBp, H * hd, perm);
    compute_sync();
}

// Stage the input of phase `epi` (K tile kt) into S.xs as fp32 [batch][KBp] (element
// order given by xpos).
__device__ void stage_input(const StepParams &P, int epi, int layer, const Mat &M, int kt, Shared &S) {
    const Model &m = P.m;
    const int tid = threadIdx.x;
    const bool perm = m.weight_bf16;
    const int pl = perm ? M.KBp : 0;
    compute_sync();  // everyone is done with the previous tile
    if (epi == EPI_QKV || epi == EPI_W13 || epi == EPI_LOGITS) {
        // the gains do not depend on this step: fetch them while waiting for x
        const float *g = epi == EPI_QKV   ? m.norms + (size_t)layer * 2 * m.dim
                         : epi == EPI_W13 ? m.norms + (size_t)layer * 2 * m.dim + m.dim
                                          : m.norms + (size_t)m.n_layers * 2 * m.dim;
        float *gs = S.xs + (size_t)P.batch * M.KBp;
        for (int k = tid * 4; k < m.dim; k += kComputeThreads * 4) cp_async16(gs + k, g + k);
        if (epi == EPI_QKV && layer == 0) {
            for (int b = 0; b < P.batch; b++) {
                int tok = token_of(P, b);
                for (int k = tid; k < m.dim; k += kComputeThreads)
                    S.xs[(size_t)b * M.KBp + xpos(k, M.KBp, perm)] = emb_elem(m, tok, k);
            }
        } else {
            const uint64_t *src = epi == EPI_W13 ? m.ll_xa + ll_layer(P, layer, m.dim)
                                                 : m.ll_x + ll_layer(P, epi == EPI_QKV ? layer : m.n_layers, m.dim);
            ll_poll(P, src, m.dim, P.batch, m.dim, S.xs, M.KBp, P.tag, pl);
        }
        zero_pad(P, S.xs, M.KBp, m.dim, perm);
        cp_async_wait_all();
        compute_sync();
        norm_in_place(P, S.xs, M.KBp, gs, perm, S);
    } else if (epi == EPI_WO) {
        if (P.attn_consumer_merge) {
            merge_chunk_states(P, layer, M, S);
        } else {
            const int qd = m.n_heads * m.head_dim;
            ll_poll(P, m.ll_o + ll_layer(P, layer, qd), qd, P.batch, qd, S.xs, M.KBp, P.tag, pl);
            zero_pad(P, S.xs, M.KBp, qd, perm);
            compute_sync();
        }
    } else {  // W2: tile kt of the SwiGLU output
        const int k0 = kt * M.KB, kn = min(M.K - k0, M.KB);
        ll_poll(P, m.ll_h + ll_layer(P, layer, m.hidden) + k0, m.hidden, P.batch, kn, S.xs, M.KBp, P.tag, pl);
        zero_pad(P, S.xs, M.KBp, kn, perm);
        compute_sync();
    }
}

// ------------------------------------------------------------------ GEMV arithmetic

// A warp works on RG rows at once: RG independent accumulator chains per batch row,
// one activation load per piece shared by all of them.
template <int NB> struct GemvShape {
    static constexpr int R = NB == 1 ? 4 : NB <= 4 ? 2 : 1;
};

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
    static constexpr int value = RG * NB >= 8 ? 1 : RG * NB >= 4 ? 2 : 4;
};

// Dots of RG weight rows with every staged batch row.  Group row r lives at
// base + (r / RPU) * unit_stride + (r % RPU) * rowbytes; rows r >= nr are skipped.
// Value index r * NB + b.  Pieces are taken U at a time into U separate accumulators.
template <int NB, int RG, int RPU, bool WBF16>
__device__ __forceinline__ void rows_dot(const uint8_t *base, size_t unit_stride, size_t rowbytes, int nr,
                                         const float *xs, int KBp, int batch, float (&out)[RG * NB]) {
    constexpr int U = Unroll<NB, RG>::value;
    constexpr int EPP = WBF16 ? 8 : 4;
    const int lane = threadIdx.x & 31;
    const int pieces = KBp / EPP;
    float acc[U][RG * NB];
#pragma unroll
    for (int u = 0; u < U; u++)
#pragma unroll
        for (int v = 0; v < RG * NB; v++) acc[u][v] = 0.f;
    const uint4 *rows[RG];
#pragma unroll
    for (int r = 0; r < RG; r++)
        rows[r] = (const uint4 *)(base + (size_t)((r < nr ? r : 0) / RPU) * unit_stride +
                                  (size_t)((r < nr ? r : 0) % RPU) * rowbytes);
    for (int p0 = lane; p0 < pieces; p0 += 32 * U) {
        uint4 w[U][RG];
#pragma unroll
        for (int u = 0; u < U; u++)
#pragma unroll
            for (int r = 0; r < RG; r++)
                w[u][r] = (p0 + 32 * u < pieces && r < nr) ? rows[r][p0 + 32 * u] : make_uint4(0, 0, 0, 0);
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
#pragma unroll
    for (int v = 0; v < RG * NB; v++) {
        float t = acc[0][v];
#pragma unroll
        for (int u = 1; u < U; u++) t += acc[u][v];
        out[v] = t;
    }
}

// ------------------------------------------------------------------ GEMV phases

// One group of a warp's units: finish the dots and run the phase's epilogue.
template <int NB, int RG, int RPU, bool WBF16>
__device__ __forceinline__ void gemv_group(const StepParams &P, int epi, int layer, const Mat &M, Shared &S,
                                           const uint8_t *buf, int j0, int ng, int c_unit0, int c_kt, int u0,
                                           float (&best_v)[NB], int (&best_i)[NB]) {
    constexpr int V = RG * NB;
    constexpr int SHIFT = 5 - Log2<V>::value;
    const Model &m = P.m;
    const int lane = threadIdx.x & 31;
    const int batch = P.batch;
    const size_t rowbytes = (size_t)M.KBp * (WBF16 ? 2 : 4);
    const size_t unit_stride = (size_t)RPU * rowbytes;  // the group's units are consecutive
    float acc[V];
    rows_dot<NB, RG, RPU, WBF16>(buf + (size_t)j0 * RPU * rowbytes, unit_stride, rowbytes, ng * RPU, S.xs, M.KBp,
                                 batch, acc);
    const float val = reduce_scatter<V>(acc);
    const int idx = lane >> SHIFT;              // value held by this lane
    const bool holder = (lane & ((1 << SHIFT) - 1)) == 0;
    const int r = idx / NB, b = idx - r * NB;   // group row, batch row
    const uint32_t tag = P.tag;
    if (epi == EPI_W13) {  // rows (2u, 2u + 1) = (gate, up) of group unit u
        const float up = __shfl_sync(0xffffffffu, val, ((idx + NB) << SHIFT) & 31);
        const int u = r >> 1;
        if (holder && (r & 1) == 0 && u < ng && b < batch) {
            const int unit = u0 + c_unit0 + j0 + u;
            const float s = val / (1.0f + __expf(-val));
            ll_store(m.ll_h + ll_layer(P, layer, m.hidden) + (size_t)b * m.hidden + unit, s * up, tag);
        }
        return;
    }
    if (!holder || r >= ng || b >= batch) return;
    const int i = c_unit0 + j0 + r;  // unit within the CTA's slice
    const int unit = u0 + i;
    float v = val;
    if (M.nkt > 1) {  // accumulate this K tile; finish after the last one
        float *a = S.accs + (size_t)i * kMaxBatch + b;
        v = (c_kt == 0 ? 0.f : *a) + v;
        *a = v;
        if (c_kt != M.nkt - 1) return;
    }
    if (epi == EPI_QKV) {
        ll_store(m.ll_qkv + ll_layer(P, layer, m.qkv.rows) + (size_t)b * m.qkv.rows + unit, v, tag);
    } else if (epi == EPI_WO || epi == EPI_W2) {
        float *own = S.xown + b * kMaxOwn + i;
        const float xn = *own + v;
        *own = xn;
        uint64_t *dst = epi == EPI_WO ? m.ll_xa + ll_layer(P, layer, m.dim) : m.ll_x + ll_layer(P, layer + 1, m.dim);
        ll_store(dst + (size_t)b * m.dim + unit, xn, tag);
    } else {  // logits: rows of one lane's value increase, so a strict > keeps the lowest index
        if (P.logits) P.logits[(size_t)b * m.vocab + unit] = v;
        if (v != v) {
            atomicOr(m.status, kStNanLogits);
        } else {
#pragma unroll
            for (int bb = 0; bb < NB; bb++)
                if (bb == b && (v > best_v[bb] || (v == best_v[bb] && unit < best_i[bb]))) {
                    best_v[bb] = v;
                    best_i[bb] = unit;
                }
        }
    }
}

template <int NB, bool WBF16>
__device__ void gemv_phase(const StepParams &P, int epi, int layer, const Mat &M, Shared &S,
                           uint32_t &chunk_i, float (&best_v)[NB], int (&best_i)[NB], int tslot) {
    constexpr int R = GemvShape<NB>::R;
    constexpr int RW = R < 2 ? 2 : R;  // W1/W3: whole (gate, up) pairs
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int u0, u1;
    unit_range(M.rows / M.rows_per_unit, P.grid, blockIdx.x, u0, u1);
    trace_mark(P, tslot, 0);
    if (u0 == u1) return;
    int cur_kt = -1;
    for_each_chunk(M, layer, WBF16 ? 2 : 4, blockIdx.x, P.grid, [&](const Chunk &c) {
        if (c.kt != cur_kt) {
            stage_input(P, epi, layer, M, c.kt, S);
            if (cur_kt < 0) trace_mark(P, tslot, 1);
            cur_kt = c.kt;
        }
        // chunk i belongs to warp i % 8; with a multiple of 8 slots every use of a slot
        // belongs to the same warp, which takes them in order
        if ((int)(chunk_i % kComputeWarps) == warp) {
            const uint32_t slot = chunk_i % (uint32_t)P.ring_slots, parity = (chunk_i / (uint32_t)P.ring_slots) & 1;
            wait_slot(P, &S.full[slot], parity);
            const uint8_t *buf = S.ring + (size_t)slot * kChunkBytes;
            if (epi == EPI_W13) {
                for (int j = 0; j < c.nunits; j += RW / 2)
                    gemv_group<NB, RW, 2, WBF16>(P, epi, layer, M, S, buf, j, min(RW / 2, c.nunits - j), c.unit0,
                                                 c.kt, u0, best_v, best_i);
            } else {  // groups of R rows, then of 2, then single rows: no idle accumulators
                int j = 0;
                for (; j + R <= c.nunits; j += R)
                    gemv_group<NB, R, 1, WBF16>(P, epi, layer, M, S, buf, j, R, c.unit0, c.kt, u0, best_v, best_i);
                if constexpr (R > 2) {
                    for (; j + 2 <= c.nunits; j += 2)
                        gemv_group<NB, 2, 1, WBF16>(P, epi, layer, M, S, buf, j, 2, c.unit0, c.kt, u0, best_v, best_i);
                }
                for (; j < c.nunits; j++)
                    gemv_group<NB, 1, 1, WBF16>(P, epi, layer, M, S, buf, j, 1, c.unit0, c.kt, u0, best_v, best_i);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&S.empty[slot]);
        }
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
    // each lane holds candidates for some rows: reduce over the warp (lowest index on ties)
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
    const bool stage = (size_t)(t1 - t0) * rowbytes * 2 <= (size_t)P.attn_stage_bytes;
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

size_t decode_smem_bytes(int xs_bytes, int ring_slots) {
    return ring_offset(xs_bytes) + (size_t)ring_slots * kChunkBytes;
}

template <int NB, bool WBF16>
static cudaError_t launch_nb(const StepParams &P, cudaStream_t stream) {
    auto fn = decode_step_kernel<NB, WBF16>;
    const size_t smem = decode_smem_bytes(P.xs_bytes, P.ring_slots);
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    void *args[] = {(void *)&P};
    return cudaLaunchCooperativeKernel((const void *)fn, dim3(P.grid), dim3(kThreads), args, smem, stream);
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

cudaError_t decode_occupancy(int weight_bf16, size_t smem, int *blocks_per_sm) {
    auto fn = weight_bf16 ? decode_step_kernel<1, true> : decode_step_kernel<1, false>;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, fn, kThreads, smem);
}

}  // namespace slm
