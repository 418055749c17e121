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
//    signalled by mbarriers.  It runs ahead of the compute warps across phase
//    boundaries, so the HBM stream does not stop while they wait at a grid barrier.
//  * The compute warps run the phases of the step; a phase's rows are split evenly
//    over the CTAs, and phases are separated by a grid-wide barrier (bounded spin).
//  * GEMV: the phase input (normalised residual, attention output or SwiGLU output)
//    sits in shared memory as fp32; each warp takes whole rows of a ring slot, each
//    lane reads 16-byte pieces (8 bf16) and accumulates in fp32, then a butterfly
//    reduction finishes the row.  Epilogues are fused: plain store (QKV), residual
//    add (Wo, W2), SwiGLU over interleaved W1/W3 rows, logits + argmax.
//  * Attention: work item = (row, kv head, chunk of positions); one item reads its
//    K/V chunk once for all query heads of the group (GQA), keeps an online softmax
//    per head, and split-K partials are merged by the last CTA to finish the
//    (row, kv head) -- flash-decoding.  RoPE of q and k and the cache append happen
//    in this phase, in the CTA whose chunk holds the new position.
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
    uint8_t *ring;           // [kRingSlots][kChunkBytes]
    uint64_t *full;          // [kRingSlots]
    uint64_t *empty;         // [kRingSlots]
    float *rs;               // [kMaxBatch] 1 / rms
    float *wbest_v;          // [kComputeWarps][kMaxBatch]
    int *wbest_i;            // [kComputeWarps][kMaxBatch]
    int *flags;              // [4]: 0 = last-arriver flag
    float *xs;               // activation tile / attention scratch
};

constexpr int kRingBytes = kRingSlots * kChunkBytes;
constexpr int kMiscBytes = 2 * kRingSlots * 8 + kMaxBatch * 4 + 2 * kComputeWarps * kMaxBatch * 4 + 16;
constexpr int kXsOffset = ((kRingBytes + kMiscBytes + 127) / 128) * 128;

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

// Grid-wide barrier number `idx` of this launch (all compute threads call it).
__device__ void grid_barrier(const StepParams &P, int idx) {
    compute_sync();
    if (threadIdx.x == 0) {
        __threadfence();
        atomicAdd(P.m.bar, 1ull);
        unsigned long long target = P.bar_base + (unsigned long long)(idx + 1) * (unsigned)P.grid;
        if (!ld_volatile_int(P.m.abort_flag)) {
            unsigned long long t0 = global_ns();
            while (ld_acquire_u64(P.m.bar) < target) {
                if (ld_volatile_int(P.m.abort_flag)) break;
                if (global_ns() - t0 > kWaitLimitNs) {
                    atomicOr(P.m.status, kStBarrierTimeout);
                    atomicExch(P.m.abort_flag, 1);
                    break;
                }
            }
        }
        __threadfence();
    }
    compute_sync();
}

// ------------------------------------------------------------------ chunk walk
// The streaming warp and the compute warps enumerate exactly the same chunks.

struct Chunk {
    int kt, row0, nrows;
    const uint8_t *src;
    uint32_t bytes;
};

template <typename F>
__device__ __forceinline__ void for_each_chunk(const Mat &M, int layer, int esz, int cta, int grid,
                                               F &&f) {
    const int upt = M.rows / M.rows_per_unit;
    int u0, u1;
    unit_range(M.nkt * upt, grid, cta, u0, u1);
    const int cu = M.rows_per_chunk / M.rows_per_unit;
    const uint8_t *lbase = M.base + (long long)layer * M.layer_stride;
    int u = u0;
    while (u < u1) {
        int kt = u / upt, ru = u - kt * upt;
        int n = min(min(u1 - u, upt - ru), cu);
        Chunk c;
        c.kt = kt;
        c.row0 = ru * M.rows_per_unit;
        c.nrows = n * M.rows_per_unit;
        c.src = lbase + ((long long)kt * M.rows + c.row0) * (long long)M.KBp * esz;
        c.bytes = (uint32_t)((long long)c.nrows * M.KBp * esz);
        f(c);
        u += n;
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
    // Never leave with a copy in flight: wait (bounded, ignoring the abort flag) for
    // the completion of every slot that may still be filling.
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

// ------------------------------------------------------------------ GEMV phases

enum Epi { EPI_QKV = 0, EPI_WO = 1, EPI_W13 = 2, EPI_W2 = 3, EPI_LOGITS = 4 };

// Residual source row for the first layer's norm: the token's embedding row.
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

// The residual stream starts as each row's embedding; every CTA writes its share of
// the columns.  Nobody reads x before the first Wo phase, two grid barriers later.
__device__ void init_residual(const StepParams &P) {
    const Model &m = P.m;
    int d0, d1;
    unit_range(m.dim, P.grid, blockIdx.x, d0, d1);
    for (int b = 0; b < P.batch; b++) {
        int tok = token_of(P, b);
        for (int k = d0 + (int)threadIdx.x; k < d1; k += kComputeThreads)
            m.x[(size_t)b * m.dim + k] = emb_elem(m, tok, k);
    }
}

// Stage the phase input tile kt into S.xs as fp32 [batch][KBp] (zero padded).
template <int NB>
__device__ void stage_input(const StepParams &P, int epi, int layer, const Mat &M, int kt, Shared &S) {
    const Model &m = P.m;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int batch = P.batch;
    compute_sync();  // everyone is done with the previous tile
    const bool from_emb = (epi == EPI_QKV && layer == 0);
    if (epi == EPI_QKV || epi == EPI_W13 || epi == EPI_LOGITS) {
        // 1 / rms of each row of the residual stream (recomputed by every CTA)
        for (int b = warp; b < batch; b += kComputeWarps) {
            float ss = 0.f;
            if (from_emb) {
                int tok = token_of(P, b);
                for (int k = lane; k < m.dim; k += 32) {
                    float v = emb_elem(m, tok, k);
                    ss += v * v;
                }
            } else {
                const float *xr = m.x + (size_t)b * m.dim;
                for (int k = lane; k < m.dim; k += 32) {
                    float v = __ldcg(xr + k);
                    ss += v * v;
                }
            }
            ss = warp_sum(ss);
            if (lane == 0) S.rs[b] = 1.0f / sqrtf(ss / (float)m.dim + m.norm_eps);
        }
        compute_sync();
        const float *g = epi == EPI_QKV   ? m.norms + (size_t)layer * 2 * m.dim
                         : epi == EPI_W13 ? m.norms + (size_t)layer * 2 * m.dim + m.dim
                                          : m.norms + (size_t)m.n_layers * 2 * m.dim;
        for (int b = 0; b < batch; b++) {
            float r = S.rs[b];
            float *dst = S.xs + (size_t)b * M.KBp;
            int tok = from_emb ? token_of(P, b) : 0;
            const float *xr = m.x + (size_t)b * m.dim;
            for (int k = tid; k < M.KBp; k += kComputeThreads) {
                float v = 0.f;
                if (k < m.dim) {
                    float xv = from_emb ? emb_elem(m, tok, k) : __ldcg(xr + k);
                    v = (xv * r) * __ldg(g + k);
                }
                dst[k] = v;
            }
        }
    } else {
        const float *src = epi == EPI_WO ? m.attn_out : m.hbuf;
        const int ld = epi == EPI_WO ? m.n_heads * m.head_dim : m.hidden;
        const int k0 = kt * M.KB;
        const int kend = min(M.K - k0, M.KB);
        for (int b = 0; b < batch; b++) {
            float *dst = S.xs + (size_t)b * M.KBp;
            const float *s = src + (size_t)b * ld + k0;
            for (int k = tid; k < M.KBp; k += kComputeThreads) dst[k] = k < kend ? __ldcg(s + k) : 0.f;
        }
    }
    compute_sync();
}

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

template <int NB, bool WBF16>
__device__ void gemv_phase(const StepParams &P, int epi, int layer, const Mat &M, Shared &S,
                           uint32_t &chunk_i, float (&best_v)[NB], int (&best_i)[NB]) {
    const Model &m = P.m;
    const int esz = WBF16 ? 2 : 4;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int batch = P.batch;
    int cur_kt = -1;
    for_each_chunk(M, layer, esz, blockIdx.x, P.grid, [&](const Chunk &c) {
        if (c.kt != cur_kt) {
            stage_input<NB>(P, epi, layer, M, c.kt, S);
            cur_kt = c.kt;
        }
        const uint32_t slot = chunk_i % kRingSlots, parity = (chunk_i / kRingSlots) & 1;
        wait_slot(P, &S.full[slot], parity);
        const uint8_t *buf = S.ring + (size_t)slot * kChunkBytes;
        const size_t rowbytes = (size_t)M.KBp * esz;
        const int nunits = c.nrows / M.rows_per_unit;
        for (int u = warp; u < nunits; u += kComputeWarps) {
            if (epi == EPI_W13) {
                float a[NB], g[NB];
                row_dot<NB, WBF16>(buf + (size_t)(2 * u) * rowbytes, S.xs, M.KBp, batch, a);
                row_dot<NB, WBF16>(buf + (size_t)(2 * u + 1) * rowbytes, S.xs, M.KBp, batch, g);
                const int j = (c.row0 >> 1) + u;
#pragma unroll
                for (int b = 0; b < NB; b++) {
                    if (b < batch && lane == b) {
                        float s = a[b] / (1.0f + __expf(-a[b]));
                        m.hbuf[(size_t)b * m.hidden + j] = s * g[b];
                    }
                }
            } else {
                float acc[NB];
                row_dot<NB, WBF16>(buf + (size_t)u * rowbytes, S.xs, M.KBp, batch, acc);
                const int row = c.row0 + u;
#pragma unroll
                for (int b = 0; b < NB; b++) {
                    if (b >= batch || lane != b) continue;
                    float v = acc[b];
                    if (epi == EPI_QKV) {
                        m.qkv_out[(size_t)b * m.qkv.rows + row] = v;
                    } else if (epi == EPI_WO || epi == EPI_W2) {
                        float *dst = m.x + (size_t)b * m.dim + row;
                        if (M.nkt == 1)
                            *dst = __ldcg(dst) + v;
                        else
                            atomicAdd(dst, v);
                    } else {  // logits
                        if (P.logits) P.logits[(size_t)b * m.vocab + row] = v;
                        if (v != v)
                            atomicOr(m.status, kStNanLogits);
                        else if (v > best_v[b]) {
                            best_v[b] = v;
                            best_i[b] = row;
                        }
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.empty[slot]);
        chunk_i++;
    });
}

// Merge the per-warp argmax candidates, then the per-CTA ones (last CTA to arrive).
template <int NB>
__device__ void finish_argmax(const StepParams &P, Shared &S, float (&best_v)[NB], int (&best_i)[NB]) {
    const Model &m = P.m;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int batch = P.batch;
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
        m.amax_val[(size_t)tid * P.grid + blockIdx.x] = bv;
        m.amax_idx[(size_t)tid * P.grid + blockIdx.x] = bi;
    }
    compute_sync();
    if (tid == 0) {
        __threadfence();
        int prev = atomicAdd(m.amax_count, 1);
        S.flags[0] = (prev == P.grid - 1);
    }
    compute_sync();
    if (S.flags[0]) {
        __threadfence();
        if (tid < batch) {
            float bv = -INFINITY;
            int bi = 0x7fffffff;
            for (int c = 0; c < P.grid; c++) {
                float v = __ldcg(m.amax_val + (size_t)tid * P.grid + c);
                int i = __ldcg(m.amax_idx + (size_t)tid * P.grid + c);
                if (v > bv || (v == bv && i < bi)) {
                    bv = v;
                    bi = i;
                }
            }
            if (bi == 0x7fffffff) bi = 0;  // all NaN: status already records it
            if (P.next_ids) P.next_ids[tid] = bi;
        }
        if (tid == 0) *(volatile int *)m.amax_count = 0;
    }
}

// ------------------------------------------------------------------ attention phase

template <bool KVBF16>
__device__ void attn_item(const StepParams &P, int layer, int b, int g, int c, Shared &S) {
    const Model &m = P.m;
    const int tid = threadIdx.x;
    const int hd = m.head_dim, H = m.n_heads, KV = m.n_kv_heads, G = H / KV;
    const int half = hd / 2;
    const int pos = P.pos[b], ctx = pos + 1, seq = P.seq[b];
    const int CH = P.attn_chunk, nc = P.nchunk[b];
    const int t0 = c * CH, t1 = min(ctx, t0 + CH);
    const int kvesz = KVBF16 ? 2 : 4;
    const size_t rowbytes = (size_t)hd * kvesz;
    const size_t head_off = ((((size_t)layer * m.max_batch + seq) * KV + g) * m.max_seq) * rowbytes;
    uint8_t *kbase = m.kc + head_off;
    uint8_t *vbase = m.vc + head_off;
    const float *qkv = m.qkv_out + (size_t)b * m.qkv.rows;
    const float *rope = m.rope + (size_t)pos * half * 2;

    // append k (rotated) and v at slot pos when this chunk ends at the new position
    if (t1 == ctx) {
        uint8_t *kd = kbase + (size_t)pos * rowbytes;
        uint8_t *vd = vbase + (size_t)pos * rowbytes;
        const float *kr = qkv + (size_t)(H + g) * hd;
        const float *vr = qkv + (size_t)(H + KV + g) * hd;
        for (int i = tid; i < half; i += kComputeThreads) {
            float cs = __ldg(rope + 2 * i), sn = __ldg(rope + 2 * i + 1);
            float a = __ldcg(kr + i), bb = __ldcg(kr + i + half);
            float k0 = kv_round(a * cs - bb * sn, KVBF16), k1 = kv_round(a * sn + bb * cs, KVBF16);
            float v0 = kv_round(__ldcg(vr + i), KVBF16), v1 = kv_round(__ldcg(vr + i + half), KVBF16);
            if (KVBF16) {
                ((__nv_bfloat16 *)kd)[i] = __float2bfloat16_rn(k0);
                ((__nv_bfloat16 *)kd)[i + half] = __float2bfloat16_rn(k1);
                ((__nv_bfloat16 *)vd)[i] = __float2bfloat16_rn(v0);
                ((__nv_bfloat16 *)vd)[i + half] = __float2bfloat16_rn(v1);
            } else {
                ((float *)kd)[i] = k0;
                ((float *)kd)[i + half] = k1;
                ((float *)vd)[i] = v0;
                ((float *)vd)[i + half] = v1;
            }
        }
    }

    AttnTask T;
    T.q = qkv + (size_t)g * G * hd;
    T.rope = rope;
    T.kbase = kbase;
    T.vbase = vbase;
    T.out = m.attn_out + ((size_t)b * H + (size_t)g * G) * hd;
    T.part = m.part + ((size_t)b * H + (size_t)g * G) * kMaxChunksPerSeq * (hd + 2);
    T.counter = m.part_count + (size_t)b * KV + g;
    T.hd = hd;
    T.G = G;
    T.t0 = t0;
    T.t1 = t1;
    T.nc = nc;
    T.c = c;
    // the appended row must be visible to every thread before the chunk is read
    attn_core<KVBF16>(T, S.xs, &S.flags[0]);
}

template <bool KVBF16>
__device__ void attention_phase(const StepParams &P, int layer, Shared &S) {
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
    int bar = 0;
    float best_v[NB];
    int best_i[NB];
#pragma unroll
    for (int b = 0; b < NB; b++) {
        best_v[b] = -INFINITY;
        best_i[b] = 0x7fffffff;
    }
    init_residual(P);
    for (int l = 0; l < m.n_layers; l++) {
        gemv_phase<NB, WBF16>(P, EPI_QKV, l, m.qkv, S, chunk_i, best_v, best_i);
        grid_barrier(P, bar++);
        if (m.kv_bf16)
            attention_phase<true>(P, l, S);
        else
            attention_phase<false>(P, l, S);
        grid_barrier(P, bar++);
        gemv_phase<NB, WBF16>(P, EPI_WO, l, m.wo, S, chunk_i, best_v, best_i);
        grid_barrier(P, bar++);
        gemv_phase<NB, WBF16>(P, EPI_W13, l, m.w13, S, chunk_i, best_v, best_i);
        grid_barrier(P, bar++);
        gemv_phase<NB, WBF16>(P, EPI_W2, l, m.w2, S, chunk_i, best_v, best_i);
        grid_barrier(P, bar++);
    }
    if (P.do_logits) {
        gemv_phase<NB, WBF16>(P, EPI_LOGITS, 0, m.emb, S, chunk_i, best_v, best_i);
        finish_argmax<NB>(P, S, best_v, best_i);
    }
}

// ------------------------------------------------------------------ host-side launch

size_t decode_smem_bytes(size_t xs_bytes) { return (size_t)kXsOffset + xs_bytes; }

template <int NB, bool WBF16>
static cudaError_t launch_nb(const StepParams &P, size_t smem, cudaStream_t stream) {
    auto fn = decode_step_kernel<NB, WBF16>;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    void *args[] = {(void *)&P};
    return cudaLaunchCooperativeKernel((const void *)fn, dim3(P.grid), dim3(kThreads), args, smem, stream);
}

template <bool WBF16>
static cudaError_t launch_w(const StepParams &P, size_t smem, cudaStream_t stream) {
    if (P.batch <= 1) return launch_nb<1, WBF16>(P, smem, stream);
    if (P.batch <= 4) return launch_nb<4, WBF16>(P, smem, stream);
    if (P.batch <= 8) return launch_nb<8, WBF16>(P, smem, stream);
    return launch_nb<16, WBF16>(P, smem, stream);
}

cudaError_t launch_decode_step(const StepParams &P, size_t smem, cudaStream_t stream) {
    return P.m.weight_bf16 ? launch_w<true>(P, smem, stream) : launch_w<false>(P, smem, stream);
}

cudaError_t decode_occupancy(int weight_bf16, size_t smem, int *blocks_per_sm) {
    auto fn = weight_bf16 ? decode_step_kernel<1, true> : decode_step_kernel<1, false>;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, fn, kThreads, smem);
}

}  // namespace slm
