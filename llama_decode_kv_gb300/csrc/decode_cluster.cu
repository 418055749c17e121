// decode_cluster.cu -- the single-row decode step of small models on thread-block clusters.
//
// The step computes the same block equations as decode_kernel.cu (kasahare 0.4.0 /
// simple-llm, "Architecture": RMSNorm, Wq/Wk/Wv, RoPE, KV append, GQA softmax(q K^T /
// sqrt(d_head)) V, Wo + residual, RMSNorm, W2(silu(W1 x) * (W3 x)) + residual; then the
// final RMSNorm, the tied-embedding logits and the greedy argmax), laid out so that a
// layer needs two grid-wide hand-offs instead of five:
//
//  * Attention cluster g (one per kv head, C CTAs): every CTA holds the whole residual
//    vector x.  CTA i computes its share of the group's QKV rows (RoPE pairs), rotates,
//    appends k and v to the cache and pushes q, k, v into every peer's shared memory;
//    then runs the online softmax over its share of the cached positions for the G query
//    heads and pushes its (max, sum, weighted V) states to every peer; every CTA merges
//    the states into o_g and computes its share of the rows of Wo[:, group g columns] o_g
//    (plus x, in cluster 0): a split-K partial of the attention block's output, published
//    as tagged words.
//  * FFN cluster c (C CTAs) owns hidden units [c hpc, (c + 1) hpc): each CTA polls the NA
//    attention partials (their sum is x after the attention block), normalises, computes
//    its W1/W3 row pairs and SwiGLU, pushes its h values to every peer, then its share of
//    the rows of W2[:, slice c] h (plus x, in cluster 0), published as tagged words.
//  * Attention CTA i polls column block i of the NF FFN partials, sums them in cluster
//    order and pushes the block to its peers: every CTA of the cluster then holds the
//    next layer's x.  After the last layer every CTA does the same and computes its share
//    of the vocabulary logits; CTA 0 reduces the per-CTA argmax candidates.
//
// Inside a cluster a push is st.async into the peer's shared memory, completing bytes on
// the peer's mbarrier, which the peer armed with the exact byte count of that exchange.
// Weights stream HBM -> shared memory through the same ring of cp.async.bulk chunks as
// in the persistent kernel (a dedicated warp running layers ahead).  Every wait is
// bounded (1 s): on expiry the kernel records it in the status word, raises the abort
// flag, stops arming barriers and skips to the final cluster barrier, which no CTA
// passes before its peers (none exits while a peer may still write into it).
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "device_common.cuh"
#include "gemv.cuh"
#include "slm_internal.h"

namespace slm {

// ------------------------------------------------------------------ cluster PTX helpers

__device__ __forceinline__ uint32_t cl_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Address of shared-memory location `a` (this CTA's shared::cta address) in CTA `rank`.
__device__ __forceinline__ uint32_t cl_map(uint32_t a, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
    return r;
}

// 4-byte store into a peer's shared memory that completes 4 bytes on the peer's mbarrier.
__device__ __forceinline__ void st_async(uint32_t raddr, float v, uint32_t rbar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(raddr),
                 "r"(__float_as_uint(v)), "r"(rbar)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_cl(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Barrier of the compute threads that also returns whether any of them passed `v`.
__device__ __forceinline__ bool compute_any(bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, 1, %2, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v), "n"(kComputeThreads)
        : "memory");
    return r != 0;
}

// ------------------------------------------------------------------ shared memory

enum { XB_X = 0, XB_QKV = 1, XB_ST = 2, XB_H = 3 };

struct CS {
    uint64_t *full, *empty;  // weight ring [kMaxRingSlots]
    uint64_t *xb;            // exchange barriers (XB_*)
    float *ssw;              // [kComputeWarps] per-warp sums of squares
    float *wbest_v;          // [kComputeWarps]
    int *wbest_i;            // [kComputeWarps]
    float *ml;               // [2 * kClusterMaxG] softmax max and sum per head
    float *rope;             // [hd] cos, sin pairs of this step's position
    int *utab;               // [2 * QKV units of this CTA] (head slot, dim) of each RoPE pair
    float *gain;             // [dim] RMSNorm gains of the current norm input
    float *yv;               // the phase's dot products (rows of this CTA's slice)
    float *xraw;             // [dim] residual input of the phase (x, or x after attention)
    float *xs;               // activation tile (xpos order)
    float *hb;               // [w2_kbp] the cluster's SwiGLU outputs (xpos order)
    float *qkv;              // [(G + 2) hd] the group's rotated q heads, k, v
    float *st;               // [C][G][hd + 2] attention states (max, sum, weighted V)
    float *pb;               // [G][positions per CTA] scores / probabilities
    float *hop;              // staging of polled words
    uint8_t *kst, *vst;      // staged cached keys / values, rows hd * esz + 16 bytes apart
    uint8_t *ring;
};

__device__ __forceinline__ CS carve_c(uint8_t *base, const ClusterParams &P) {
    CS s;
    s.full = (uint64_t *)base;
    s.empty = s.full + kMaxRingSlots;
    s.xb = s.empty + kMaxRingSlots;
    s.ssw = (float *)(s.xb + 4);
    s.wbest_v = s.ssw + kComputeWarps;
    s.wbest_i = (int *)(s.wbest_v + kComputeWarps);
    s.ml = (float *)(s.wbest_i + kComputeWarps);
    s.rope = (float *)(base + P.off_rope);
    s.utab = (int *)(base + P.off_utab);
    s.gain = (float *)(base + P.off_gain);
    s.yv = (float *)(base + P.off_yv);
    s.xraw = (float *)(base + P.off_xraw);
    s.xs = (float *)(base + P.off_xs);
    s.hb = (float *)(base + P.off_hb);
    s.qkv = (float *)(base + P.off_qkv);
    s.st = (float *)(base + P.off_st);
    s.pb = (float *)(base + P.off_p);
    s.kst = base + P.off_k;
    s.vst = base + P.off_v;
    s.hop = (float *)(base + P.off_hop);
    s.ring = base + P.off_ring;
    return s;
}

// ------------------------------------------------------------------ bounded waits

__device__ __forceinline__ void raise_abort(const Model &m, int bit) {
    atomicOr(m.status, bit);
    atomicExch(m.abort_flag, 1);
}

// Ring slot (CTA-scope mbarrier).
__device__ bool c_wait_slot(const Model &m, uint64_t *bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    if (ld_volatile_int(m.abort_flag)) return false;
    const unsigned long long t0 = global_ns();
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if (ld_volatile_int(m.abort_flag)) return false;
        if (global_ns() - t0 > m.wait_ns) {
            raise_abort(m, kStRingTimeout);
            return false;
        }
    }
}

// Exchange barrier: bytes pushed by the cluster's CTAs.
__device__ bool c_wait_xb(const Model &m, uint64_t *bar, uint32_t parity) {
    if (mbar_try_cl(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    for (int it = 0;; it++) {
        if (mbar_try_cl(bar, parity)) return true;
        if ((it & 15) == 15) {
            if (ld_volatile_int(m.abort_flag)) return false;
            if (global_ns() - t0 > m.wait_ns) {
                raise_abort(m, kStExchangeTimeout);
                return false;
            }
        }
    }
}

// Poll n tagged words (item e: src[(e / len) * src_ld + e % len]) into dst[e] until every
// tag equals the launch's; each thread keeps up to kPollBatch loads in flight.  Returns
// false if the wait ran out or another CTA aborted.  No barrier.
template <int K = 8>
__device__ bool poll_flat(const ClusterParams &P, const uint64_t *src, int n, int len, int src_ld, float *dst) {
    const int tid = threadIdx.x;
    const uint32_t tag = P.tag;
    bool ok = true;
    for (int base = 0; base < n && ok; base += kComputeThreads * K) {
        int off[K];
        bool need[K];
#pragma unroll
        for (int k = 0; k < K; k++) {
            const int e = base + k * kComputeThreads + tid;
            need[k] = e < n;
            const int s = need[k] ? e / len : 0;
            off[k] = need[k] ? s * src_ld + (e - s * len) : 0;
        }
        unsigned long long t0 = 0;
        for (int it = 0;; it++) {
            uint64_t w[K];
#pragma unroll
            for (int k = 0; k < K; k++) w[k] = need[k] ? ll_load(src + off[k]) : 0;
            bool pending = false;
#pragma unroll
            for (int k = 0; k < K; k++) {
                if (!need[k]) continue;
                if ((uint32_t)(w[k] >> 32) == tag) {
                    dst[base + k * kComputeThreads + tid] = __uint_as_float((uint32_t)w[k]);
                    need[k] = false;
                } else {
                    pending = true;
                }
            }
            if (!pending) break;
            if (it == 0) t0 = global_ns();
            if ((it & 15) == 15) {
                if (ld_volatile_int(P.m.abort_flag)) {
                    ok = false;
                    break;
                }
                if (global_ns() - t0 > P.m.wait_ns) {
                    raise_abort(P.m, kStExchangeTimeout);
                    ok = false;
                    break;
                }
            }
        }
    }
    return ok;
}

__device__ __forceinline__ void c_trace(const ClusterParams &P, int slot, int point) {
    if (P.trace && threadIdx.x == 0)
        P.trace[((size_t)blockIdx.x * trace_slots(P.m.n_layers) + slot) * 3 + point] = global_ns();
}

// ------------------------------------------------------------------ work split

enum { PH_QKV = 0, PH_WO = 1, PH_W13 = 2, PH_W2 = 3, PH_EMB = 4 };

// This CTA's slice of one phase's matrix: `units` units of `rpu` rows starting at `base`,
// cut into chunks of `upc` units (one ring slot each).
struct Phase {
    const uint8_t *base;
    uint32_t rowbytes;
    int u0;  // first unit within the phase's unit numbering
    int units, rpu, upc, nch;
};

struct Who {
    int cl, rank, g, c;  // cluster, rank in it, kv head (attention) or FFN cluster index
    bool attn;
};

__device__ __forceinline__ Who who(const ClusterParams &P) {
    Who w;
    w.cl = (int)blockIdx.x / P.C;
    w.rank = (int)cl_rank();
    w.attn = w.cl < P.NA;
    w.g = w.attn ? w.cl : -1;
    w.c = w.attn ? -1 : w.cl - P.NA;
    return w;
}

// Hidden units [h0, h0 + n) of FFN cluster c.
__device__ __forceinline__ void ffn_units(const ClusterParams &P, int c, int &h0, int &n) {
    h0 = c * P.hpc;
    n = max(0, min(P.m.hidden, h0 + P.hpc) - h0);
}

__device__ Phase cta_phase(const ClusterParams &P, int kind, int layer, const Who &w) {
    const Model &m = P.m;
    const int esz = m.weight_bf16 ? 2 : 4;
    Phase ph;
    int u0 = 0, u1 = 0;
    if (kind == PH_QKV) {
        const int hd = m.head_dim, G = m.n_heads / m.n_kv_heads;
        unit_range((G + 2) * hd / 2, P.C, w.rank, u0, u1);
        ph.rowbytes = (uint32_t)(m.qkv.KBp * esz);
        ph.base = m.qkv.base + (long long)layer * m.qkv.layer_stride +
                  ((long long)w.g * (G + 2) * hd + 2LL * u0) * ph.rowbytes;
        ph.rpu = 2;
        ph.upc = P.upc_qkv;
    } else if (kind == PH_WO || kind == PH_W2) {
        unit_range(m.dim, P.C, w.rank, u0, u1);
        const bool wo = kind == PH_WO;
        ph.rowbytes = (uint32_t)((wo ? P.wo_kbp : P.w2_kbp) * esz);
        ph.base = (wo ? P.wo_g + (long long)layer * P.wo_layer_stride : P.w2_c + (long long)layer * P.w2_layer_stride) +
                  ((long long)(wo ? w.g : w.c) * m.dim + u0) * ph.rowbytes;
        ph.rpu = 1;
        ph.upc = wo ? P.upc_wo : P.upc_w2;
    } else if (kind == PH_W13) {
        int h0, n;
        ffn_units(P, w.c, h0, n);
        unit_range(n, P.C, w.rank, u0, u1);
        ph.rowbytes = (uint32_t)(m.w13.KBp * esz);
        ph.base = m.w13.base + (long long)layer * m.w13.layer_stride + 2LL * (h0 + u0) * ph.rowbytes;
        ph.rpu = 2;
        ph.upc = P.upc_w13;
    } else {
        unit_range(m.vocab, P.grid, (int)blockIdx.x, u0, u1);
        ph.rowbytes = (uint32_t)(m.emb.KBp * esz);
        ph.base = m.emb.base + (long long)u0 * ph.rowbytes;
        ph.rpu = 1;
        ph.upc = P.upc_emb;
    }
    ph.u0 = u0;
    ph.units = u1 - u0;
    ph.nch = (ph.units + ph.upc - 1) / ph.upc;
    return ph;
}

// The phases of a CTA in consumption order: per layer QKV, Wo (attention) or W1/W3, W2
// (FFN); then the logits.
__device__ __forceinline__ int phase_kind(const Who &w, int k) { return w.attn ? (k == 0 ? PH_QKV : PH_WO) : (k == 0 ? PH_W13 : PH_W2); }

// ------------------------------------------------------------------ streaming warp

__device__ void c_producer(const ClusterParams &P, CS &S, const Who &w) {
    const uint32_t slots = (uint32_t)P.ring_slots;
    uint32_t issued = 0;
    const int L = P.m.n_layers;
    bool stop = false;
    for (int l = 0; l <= L && !stop; l++) {
        for (int k = 0; k < 2 && !stop; k++) {
            if (l == L && (k == 1 || !P.do_logits)) break;
            const Phase ph = cta_phase(P, l == L ? PH_EMB : phase_kind(w, k), l, w);
            for (int j = 0; j < ph.nch; j++) {
                const int u = j * ph.upc, nu = min(ph.upc, ph.units - u);
                const uint32_t bytes = (uint32_t)nu * ph.rpu * ph.rowbytes;
                const uint32_t slot = issued % slots;
                if (issued >= slots && !c_wait_slot(P.m, &S.empty[slot], ((issued / slots) - 1) & 1)) {
                    stop = true;
                    break;
                }
                mbar_expect_tx(&S.full[slot], bytes);
                bulk_g2s(S.ring + (size_t)slot * kChunkBytes, ph.base + (size_t)u * ph.rpu * ph.rowbytes, bytes, &S.full[slot]);
                issued++;
            }
        }
    }
    // never leave with a copy in flight
    const uint32_t first = issued > slots ? issued - slots : 0;
    for (uint32_t i = first; i < issued; i++) {
        const uint32_t slot = i % slots, parity = (i / slots) & 1;
        const unsigned long long t0 = global_ns();
        while (!mbar_try_wait(&S.full[slot], parity)) {
            if (global_ns() - t0 > kWaitLimitNs) {
                atomicOr(P.m.status, kStRingTimeout);
                break;
            }
        }
    }
}

// ------------------------------------------------------------------ per-CTA constants

// What a compute thread of this CTA works on; computed once per launch (registers).
struct Me {
    int b0, b1;        // column block of the residual this rank owns (Wo / W2 rows, hops)
    int t0, T, ns;     // attention: first position, positions, positions staged
    int sj[4], st[4];  // attention: this thread's (head, position) score items
    int nsc;           //   and their number
    int pj, pd;        // attention: the (head, dim) this thread weights and merges (pj < 0: none)
    uint32_t use[4];   // uses of each exchange barrier so far
};

__device__ __forceinline__ uint32_t xb_uses(const ClusterParams &P, const Who &w, int k) {
    const int L = P.m.n_layers;
    if (k == XB_X) return w.attn ? (uint32_t)(L - 1 + P.do_logits) : (uint32_t)P.do_logits;
    if (k == XB_H) return w.attn ? 0u : (uint32_t)L;
    return w.attn ? (uint32_t)L : 0u;
}

__device__ __forceinline__ uint32_t xb_bytes(const ClusterParams &P, const Who &w, int k) {
    const Model &m = P.m;
    const int G = m.n_heads / m.n_kv_heads, hd = m.head_dim;
    if (k == XB_X) return (uint32_t)m.dim * 4u;
    if (k == XB_QKV) return (uint32_t)((G + 2) * hd) * 4u;
    if (k == XB_ST) return (uint32_t)(P.C * G * (hd + 2)) * 4u;
    int h0 = 0, nh = 0;
    if (!w.attn) ffn_units(P, w.c, h0, nh);
    return (uint32_t)nh * 4u;
}

// Wait, on every compute thread, for the next use of exchange barrier k; thread 0 then
// re-arms it for the following use.  Uniform result.
__device__ __forceinline__ bool xwait(const ClusterParams &P, CS &S, const Who &w, Me &me, int k) {
    const bool ok = !compute_any(!c_wait_xb(P.m, &S.xb[k], me.use[k] & 1));
    if (!ok) return false;
    me.use[k]++;
    if (threadIdx.x == 0 && me.use[k] < xb_uses(P, w, k)) mbar_expect_tx(&S.xb[k], xb_bytes(P, w, k));
    return true;
}

// ------------------------------------------------------------------ phase inputs

// The RMSNorm gains of the next norm input into shared memory; issued while the phase
// waits for its input, so the global loads are off the critical path.
__device__ __forceinline__ void load_gain(const ClusterParams &P, CS &S, const float *gain) {
    for (int j = threadIdx.x; j < P.m.dim; j += kComputeThreads) S.gain[j] = __ldg(gain + j);
}

// RMSNorm of xraw into the activation tile: xs[xpos(j)] = x_j * gain_j, the padding
// [dim, kbp) zeroed.  Ends with a barrier; returns 1 / rms.
__device__ __forceinline__ float norm_stage(const ClusterParams &P, CS &S, int kbp) {
    const Model &m = P.m;
    const bool perm = m.weight_bf16;
    float ss = 0.f;
    for (int j = threadIdx.x; j < kbp; j += kComputeThreads) {
        float y = 0.f;
        if (j < m.dim) {
            const float x = S.xraw[j];
            ss = fmaf(x, x, ss);
            y = x * S.gain[j];
        }
        S.xs[xpos(j, kbp, perm)] = y;
    }
    ss = warp_sum(ss);
    if ((threadIdx.x & 31) == 0) S.ssw[threadIdx.x >> 5] = ss;
    compute_sync();
    float t = 0.f;
#pragma unroll
    for (int w = 0; w < kComputeWarps; w++) t += S.ssw[w];
    return 1.0f / sqrtf(t / (float)m.dim + m.norm_eps);
}

// The residual x = the sum of nsrc partial vectors (tagged words src[s * dim + j]), summed
// in source order into xraw.  Ends with a barrier; uniform result.
__device__ __forceinline__ bool hop_full(const ClusterParams &P, CS &S, const uint64_t *src, int nsrc) {
    const int dim = P.m.dim;
    if (compute_any(!poll_flat(P, src, nsrc * dim, dim, dim, S.hop))) return false;
    for (int j = threadIdx.x; j < dim; j += kComputeThreads) {
        float v = 0.f;
        for (int s = 0; s < nsrc; s++) v += S.hop[s * dim + j];  // source order: fixed
        S.xraw[j] = v;
    }
    compute_sync();
    return true;
}

// Column block [b0, b1) of the sum of nsrc partial vectors (tagged words src[s * dim + j])
// pushed to every CTA of the cluster (xraw, barrier XB_X).
template <int C>
__device__ __forceinline__ bool hop_block(const ClusterParams &P, CS &S, const Me &me, const uint64_t *src, int nsrc) {
    const int len = me.b1 - me.b0;
    bool ok = poll_flat(P, src + me.b0, nsrc * len, len, P.m.dim, S.hop);
    ok = !compute_any(!ok);
    if (!ok) return false;
    const uint32_t xa = smem_addr(S.xraw + me.b0), xbar = smem_addr(&S.xb[XB_X]);
    for (int e = threadIdx.x; e < len * C; e += kComputeThreads) {
        const int jj = e / C, peer = e % C;
        float v = 0.f;
        for (int s = 0; s < nsrc; s++) v += S.hop[s * len + jj];  // source order: fixed
        st_async(cl_map(xa + 4u * (uint32_t)jj, (uint32_t)peer), v, cl_map(xbar, (uint32_t)peer));
    }
    return true;
}

// ------------------------------------------------------------------ GEMV

constexpr int kRG = 8;  // rows per group (one warp reduction)

// A warp's walk over its chunks of a phase: chunk j of the phase (global index base + j)
// belongs to warp (base + j) % 8 and to ring slot (base + j) % slots.
template <bool WBF16>
struct Walk {
    int j, nr;
    const uint8_t *buf;
    GroupW<1, kRG, WBF16> gw;
};

// Wait for chunk j's weights and load the warp's first pieces of it into registers.
template <bool WBF16>
__device__ __forceinline__ void walk_load(const ClusterParams &P, CS &S, const Phase &ph, uint32_t base, int kbp, Walk<WBF16> &wk) {
    const uint32_t slots = (uint32_t)P.ring_slots, ci = base + (uint32_t)wk.j;
    c_wait_slot(P.m, &S.full[ci % slots], (ci / slots) & 1);
    wk.buf = S.ring + (size_t)(ci % slots) * kChunkBytes;
    wk.nr = min(ph.upc, ph.units - wk.j * ph.upc) * ph.rpu;
    load_pieces<1, kRG, WBF16>(wk.gw, wk.buf, ph.rowbytes, wk.nr, threadIdx.x & 31, kbp / (WBF16 ? 8 : 4), kbp);
}

template <bool WBF16>
__device__ __forceinline__ void walk_begin(const ClusterParams &P, CS &S, const Phase &ph, uint32_t base, int kbp, Walk<WBF16> &wk) {
    wk.j = ((int)(threadIdx.x >> 5) - (int)(base & 7)) & 7;
    if (wk.j < ph.nch) walk_load<WBF16>(P, S, ph, base, kbp, wk);
}

// The dot products of the warp's chunks into S.yv (row index within the CTA's slice).
template <bool WBF16>
__device__ __forceinline__ void walk_run(const ClusterParams &P, CS &S, const Phase &ph, uint32_t base, const float *xs,
                                         int kbp, Walk<WBF16> &wk) {
    constexpr int SHIFT = 5 - Log2<kRG>::value;
    const int lane = threadIdx.x & 31;
    const uint32_t slots = (uint32_t)P.ring_slots;
#pragma unroll 1
    while (wk.j < ph.nch) {
        float acc[kRG];
        rows_dot<1, kRG, WBF16>(wk.gw, wk.buf, ph.rowbytes, wk.nr, xs, kbp, 1, acc);
        const float val = reduce_scatter<kRG>(acc);
        const int r = lane >> SHIFT;  // row of the group this lane holds
        if ((lane & ((1 << SHIFT) - 1)) == 0 && r < wk.nr) S.yv[wk.j * ph.upc * ph.rpu + r] = val;
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.empty[(base + (uint32_t)wk.j) % slots]);
        wk.j += kComputeWarps;
        if (wk.j < ph.nch) walk_load<WBF16>(P, S, ph, base, kbp, wk);
    }
}

// ------------------------------------------------------------------ attention

// This CTA's cached positions [t0, t0 + ns) to shared memory (rows hd * esz + 16 bytes apart).
__device__ __forceinline__ void stage_kv(const ClusterParams &P, CS &S, const Me &me, int layer, int g) {
    const Model &m = P.m;
    const int esz = m.kv_bf16 ? 2 : 4;
    const int rb = m.head_dim * esz, srb = rb + 16, per = rb / 16;
    for (int e = threadIdx.x; e < me.ns * per; e += kComputeThreads) {
        const int t = e / per, q = e - t * per;
        const size_t src = kv_row(m, layer, P.seq, g, me.t0 + t) * rb + (size_t)q * 16;
        cp_async16(S.kst + (size_t)t * srb + q * 16, m.kc + src);
        cp_async16(S.vst + (size_t)t * srb + q * 16, m.vc + src);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
}

__device__ __forceinline__ float kv_elem(const uint8_t *row, int d, bool bf16) {
    return bf16 ? __uint_as_float((uint32_t)((const uint16_t *)row)[d] << 16) : ((const float *)row)[d];
}

// Online softmax of the G query heads over this CTA's positions; the states (max, sum,
// weighted V) are pushed to every CTA of the cluster (S.st[rank][j][0..hd + 2), XB_ST).
template <int C>
__device__ __forceinline__ void attention_cta(const ClusterParams &P, CS &S, const Me &me, int layer, const Who &w) {
    const Model &m = P.m;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int hd = m.head_dim, G = m.n_heads / m.n_kv_heads;
    const bool bf = m.kv_bf16;
    const int esz = bf ? 2 : 4, rb = hd * esz, srb = rb + 16;
    const int pos = P.pos, T = me.T, t0 = me.t0, ns = me.ns;
    const int tcap = (m.max_seq + C - 1) / C;
    // positions this CTA did not stage are read from the cache
    auto kg = [&](int t) { return m.kc + kv_row(m, layer, P.seq, w.g, t) * rb; };
    auto vg = [&](int t) { return m.vc + kv_row(m, layer, P.seq, w.g, t) * rb; };
    // scores s[j][t] = q_j . k_t (q carries log2(e) / sqrt(hd)); this thread's items
    for (int it = 0; it < me.nsc; it++) {
        const int j = me.sj[it], tt = me.st[it], t = t0 + tt;
        const float4 *q = (const float4 *)(S.qkv + j * hd);
        float s0 = 0.f, s1 = 0.f;
        if (t == pos) {
            const float4 *k = (const float4 *)(S.qkv + G * hd);
            for (int d = 0; d < hd / 4; d++) {
                const float4 a = q[d], b = k[d];
                s0 = fmaf(a.x, b.x, fmaf(a.y, b.y, s0));
                s1 = fmaf(a.z, b.z, fmaf(a.w, b.w, s1));
            }
        } else {
            const uint8_t *k = tt < ns ? S.kst + (size_t)tt * srb : kg(t);
            if (bf) {
                for (int d = 0; d < hd / 8; d++) {
                    const uint4 u = *(const uint4 *)(k + d * 16);
                    const float4 a = q[2 * d], b = q[2 * d + 1];
                    s0 = fmaf(a.x, bf16_lo(u.x), fmaf(a.y, bf16_hi(u.x), s0));
                    s1 = fmaf(a.z, bf16_lo(u.y), fmaf(a.w, bf16_hi(u.y), s1));
                    s0 = fmaf(b.x, bf16_lo(u.z), fmaf(b.y, bf16_hi(u.z), s0));
                    s1 = fmaf(b.z, bf16_lo(u.w), fmaf(b.w, bf16_hi(u.w), s1));
                }
            } else {
                for (int d = 0; d < hd / 4; d++) {
                    const float4 a = q[d], b = *(const float4 *)(k + d * 16);
                    s0 = fmaf(a.x, b.x, fmaf(a.y, b.y, s0));
                    s1 = fmaf(a.z, b.z, fmaf(a.w, b.w, s1));
                }
            }
        }
        S.pb[j * tcap + tt] = s0 + s1;
    }
    compute_sync();
    // per head (warp j): max, exponentials, sum
    if (warp < G) {
        float mx = -INFINITY;
        for (int tt = lane; tt < T; tt += 32) mx = fmaxf(mx, S.pb[warp * tcap + tt]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        float l = 0.f;
        for (int tt = lane; tt < T; tt += 32) {
            const float p = exp2f(S.pb[warp * tcap + tt] - mx);
            S.pb[warp * tcap + tt] = p;
            l += p;
        }
        l = warp_sum(l);
        if (lane == 0) {
            S.ml[2 * warp] = T > 0 ? mx : -INFINITY;
            S.ml[2 * warp + 1] = l;
        }
    }
    compute_sync();
    // weighted values of (head pj, dim pd), pushed with the head's max and sum
    if (me.pj >= 0) {
        const int j = me.pj, d = me.pd;
        float o0 = 0.f, o1 = 0.f;
        const float *p = S.pb + j * tcap;
        int tt = 0;
        for (; tt + 1 < T; tt += 2) {
            const int t = t0 + tt;
            const float v0 = t == pos ? S.qkv[(G + 1) * hd + d] : kv_elem(tt < ns ? S.vst + (size_t)tt * srb : vg(t), d, bf);
            const float v1 = t + 1 == pos ? S.qkv[(G + 1) * hd + d]
                                          : kv_elem(tt + 1 < ns ? S.vst + (size_t)(tt + 1) * srb : vg(t + 1), d, bf);
            o0 = fmaf(p[tt], v0, o0);
            o1 = fmaf(p[tt + 1], v1, o1);
        }
        if (tt < T) {
            const int t = t0 + tt;
            const float v0 = t == pos ? S.qkv[(G + 1) * hd + d] : kv_elem(tt < ns ? S.vst + (size_t)tt * srb : vg(t), d, bf);
            o0 = fmaf(p[tt], v0, o0);
        }
        const uint32_t sbar = smem_addr(&S.xb[XB_ST]);
        const uint32_t sa = smem_addr(S.st + (w.rank * G + j) * (hd + 2));
        const float o = o0 + o1, mx = S.ml[2 * j], l = S.ml[2 * j + 1];
#pragma unroll
        for (int peer = 0; peer < C; peer++) {
            const uint32_t rbar = cl_map(sbar, (uint32_t)peer), ra = cl_map(sa, (uint32_t)peer);
            st_async(ra + 8u + 4u * (uint32_t)d, o, rbar);
            if (d == 0) {
                st_async(ra, mx, rbar);
                st_async(ra + 4u, l, rbar);
            }
        }
    }
}

// Merge the cluster's attention states into o_g, the Wo activation tile.  Ends with a
// barrier.
template <int C>
__device__ __forceinline__ void merge_states(const ClusterParams &P, CS &S, const Me &me) {
    const Model &m = P.m;
    const int hd = m.head_dim, G = m.n_heads / m.n_kv_heads;
    const bool perm = m.weight_bf16;
    const int stride = G * (hd + 2);
    if (me.pj >= 0) {
        const int j = me.pj, d = me.pd;
        const float *s = S.st + j * (hd + 2);
        float M = -INFINITY;
#pragma unroll
        for (int i = 0; i < C; i++) M = fmaxf(M, s[i * stride]);
        float L = 0.f, O = 0.f;
#pragma unroll
        for (int i = 0; i < C; i++) {
            const float mi = s[i * stride];
            const float sc = mi == -INFINITY ? 0.f : exp2f(mi - M);
            L = fmaf(s[i * stride + 1], sc, L);
            O = fmaf(s[i * stride + 2 + d], sc, O);
        }
        S.xs[xpos(j * hd + d, P.wo_kbp, perm)] = O / L;
    }
    for (int e = G * hd + threadIdx.x; e < P.wo_kbp; e += kComputeThreads) S.xs[xpos(e, P.wo_kbp, perm)] = 0.f;
    compute_sync();
}

// ------------------------------------------------------------------ logits and argmax

__device__ __forceinline__ void better(float v, int i, float &bv, int &bi) {
    if (v > bv || (v == bv && i < bi)) {
        bv = v;
        bi = i;
    }
}

// The logits of this CTA's vocabulary rows (from S.yv) and the greedy argmax over the
// grid (lowest index on ties).
__device__ __forceinline__ void logits_tail(const ClusterParams &P, CS &S, const Phase &ph, float rs) {
    const Model &m = P.m;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    for (int t = tid; t < ph.units; t += kComputeThreads) {
        const int v = ph.u0 + t;
        const float lg = S.yv[t] * rs;
        if (P.logits) P.logits[v] = lg;
        if (lg != lg)
            atomicOr(m.status, kStNanLogits);
        else
            better(lg, v, bv, bi);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) better(__shfl_xor_sync(0xffffffffu, bv, o), __shfl_xor_sync(0xffffffffu, bi, o), bv, bi);
    if (lane == 0) {
        S.wbest_v[warp] = bv;
        S.wbest_i[warp] = bi;
    }
    compute_sync();
    if (tid != 0) return;
    float v = -INFINITY;
    int i = 0x7fffffff;
    for (int w = 0; w < kComputeWarps; w++) better(S.wbest_v[w], S.wbest_i[w], v, i);
    // The grid's best: one 64-bit atomicMax of (order-preserving bits of the value, ~index)
    // per CTA (larger value wins, then the lower index); the last CTA to arrive writes
    // the id and resets the two words for the next step.
    unsigned long long *best = (unsigned long long *)P.amax, *count = best + 1;
    if (i != 0x7fffffff) {
        const uint32_t b = __float_as_uint(v), ord = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
        atomicMax(best, ((unsigned long long)ord << 32) | (unsigned long long)(0xffffffffu - (uint32_t)i));
    }
    __threadfence();
    if (atomicAdd(count, 1ull) != (unsigned long long)(P.grid - 1)) return;
    __threadfence();
    const unsigned long long key = atomicAdd(best, 0ull);
    const int id = key ? (int)(0xffffffffu - (uint32_t)(key & 0xffffffffu)) : 0;  // none: all NaN (status records it)
    *(volatile unsigned long long *)best = 0ull;
    *(volatile unsigned long long *)count = 0ull;
    if (P.next_ids) P.next_ids[0] = id;
    if (P.done_word) {  // host-memory ids: tell the host they are complete, with the status
        ((volatile uint32_t *)P.done_word)[1] = (uint32_t)ld_volatile_int(m.status);
        __threadfence_system();
        *(volatile uint32_t *)P.done_word = P.tag;
    }
}

// ------------------------------------------------------------------ the kernel

// Every phase: before its input is waited for, each warp waits for its first chunk and
// loads its first pieces into registers, so that afterwards only arithmetic and stores
// remain; the dot products go to S.yv, a barrier, then one thread per output item runs the
// epilogue.
template <bool WBF16, int C>
__device__ __forceinline__ void compute_cta(const ClusterParams &P, CS &S, const Who &w, Me &me) {
    const Model &m = P.m;
    const int tid = threadIdx.x, L = m.n_layers, dim = m.dim;
    const int hd = m.head_dim, half = hd / 2, G = m.n_heads / m.n_kv_heads;
    const bool perm = m.weight_bf16;
    const uint32_t tag = P.tag;
    unit_range(dim, C, w.rank, me.b0, me.b1);
    for (int k = 0; k < 4; k++) me.use[k] = 0;
    me.pj = -1;
    me.pd = 0;
    me.nsc = 0;
    me.t0 = me.T = me.ns = 0;
    int h0 = 0, nh = 0;
    if (w.attn) {
        int t1;
        unit_range(P.pos + 1, C, w.rank, me.t0, t1);
        me.T = t1 - me.t0;
        me.ns = max(0, min(min(t1, P.pos) - me.t0, P.stage_rows));
        for (int e = tid; e < G * me.T && me.nsc < 4; e += kComputeThreads) {
            me.sj[me.nsc] = e / me.T;
            me.st[me.nsc] = e - (e / me.T) * me.T;
            me.nsc++;
        }
        if (tid < G * hd) {
            me.pj = tid / hd;
            me.pd = tid - me.pj * hd;
        }
        // the RoPE row of this position (the same in every layer) and the QKV units' heads
        for (int i = tid; i < half; i += kComputeThreads) {
            S.rope[2 * i] = m.rope[((size_t)P.pos * half + i) * 2];
            S.rope[2 * i + 1] = m.rope[((size_t)P.pos * half + i) * 2 + 1];
        }
        const Phase pq = cta_phase(P, PH_QKV, 0, w);
        for (int t = tid; t < pq.units; t += kComputeThreads) {
            const int unit = pq.u0 + t, sub = unit / half;
            S.utab[2 * t] = sub;
            S.utab[2 * t + 1] = unit - sub * half;
        }
    } else {
        ffn_units(P, w.c, h0, nh);
    }
    compute_sync();
    uint32_t chunk = 0;
    float rs = 1.f;
    for (int l = 0; l < L; l++) {
        if (w.attn) {
            // ---------------- QKV: RoPE pairs of the group's [G q heads; k; v] rows
            stage_kv(P, S, me, l, w.g);  // cached rows: independent of this step
            const Phase pq = cta_phase(P, PH_QKV, l, w);
            c_trace(P, l * kTracePerLayer + 0, 0);
            Walk<WBF16> wk;
            walk_begin<WBF16>(P, S, pq, chunk, m.qkv.KBp, wk);
            load_gain(P, S, m.norms + (size_t)l * 2 * dim);
            if (l == 0) {
                int tok = __ldcg(P.tokens);
                if (tok < 0 || tok >= m.vocab) {
                    if (tid == 0 && blockIdx.x == 0) atomicOr(m.status, kStBadToken);
                    tok = 0;
                }
                const uint8_t *row = m.emb.base + (size_t)tok * m.emb.KBp * (WBF16 ? 2 : 4);
                for (int j = tid; j < dim; j += kComputeThreads)
                    S.xraw[j] = WBF16 ? __uint_as_float((uint32_t)((const uint16_t *)row)[j] << 16) : ((const float *)row)[j];
                compute_sync();
            } else {
                if (!hop_block<C>(P, S, me, P.p_ffn + (size_t)(l - 1) * P.NF * dim, P.NF)) return;
                if (!xwait(P, S, w, me, XB_X)) return;
            }
            rs = norm_stage(P, S, m.qkv.KBp);
            c_trace(P, l * kTracePerLayer + 0, 1);
            walk_run<WBF16>(P, S, pq, chunk, S.xs, m.qkv.KBp, wk);
            chunk += (uint32_t)pq.nch;
            compute_sync();
            {  // one item per (pair, peer): rotate, scale q / round k, v (peer 0 appends), push
                const uint32_t qa = smem_addr(S.qkv), qbar = smem_addr(&S.xb[XB_QKV]);
                const float qscale = rsqrtf((float)hd) * 1.4426950408889634f;  // scores in log2 units
                for (int e = tid; e < pq.units * C; e += kComputeThreads) {
                    const int t = e / C, peer = e % C;
                    const int sub = S.utab[2 * t], i = S.utab[2 * t + 1];
                    float o0 = S.yv[2 * t] * rs, o1 = S.yv[2 * t + 1] * rs;
                    if (sub <= G) {
                        const float c = S.rope[2 * i], sn = S.rope[2 * i + 1];
                        const float r0 = o0 * c - o1 * sn, r1 = o0 * sn + o1 * c;
                        o0 = r0;
                        o1 = r1;
                    }
                    if (sub < G) {
                        o0 *= qscale;
                        o1 *= qscale;
                    } else if (m.kv_bf16) {
                        const __nv_bfloat16 h0v = __float2bfloat16_rn(o0), h1v = __float2bfloat16_rn(o1);
                        o0 = __bfloat162float(h0v);
                        o1 = __bfloat162float(h1v);
                        if (peer == 0) {
                            __nv_bfloat16 *row = (__nv_bfloat16 *)(sub == G ? m.kc : m.vc) +
                                                 kv_row(m, l, P.seq, w.g, P.pos) * hd;
                            row[i] = h0v;
                            row[i + half] = h1v;
                        }
                    } else if (peer == 0) {
                        float *row = (float *)(sub == G ? m.kc : m.vc) + kv_row(m, l, P.seq, w.g, P.pos) * hd;
                        row[i] = o0;
                        row[i + half] = o1;
                    }
                    const uint32_t e0 = cl_map(qa + 4u * (uint32_t)(sub * hd + i), (uint32_t)peer), rbar = cl_map(qbar, (uint32_t)peer);
                    st_async(e0, o0, rbar);
                    st_async(e0 + 4u * (uint32_t)half, o1, rbar);
                }
            }
            c_trace(P, l * kTracePerLayer + 0, 2);
            // ---------------- attention over this CTA's positions
            c_trace(P, l * kTracePerLayer + 1, 0);
            asm volatile("cp.async.wait_group 0;" ::: "memory");
            if (!xwait(P, S, w, me, XB_QKV)) return;
            c_trace(P, l * kTracePerLayer + 1, 1);
            attention_cta<C>(P, S, me, l, w);
            c_trace(P, l * kTracePerLayer + 1, 2);
            // ---------------- Wo: split-K partial over the group's columns (+ x in cluster 0)
            const Phase po = cta_phase(P, PH_WO, l, w);
            c_trace(P, l * kTracePerLayer + 2, 0);
            walk_begin<WBF16>(P, S, po, chunk, P.wo_kbp, wk);
            if (!xwait(P, S, w, me, XB_ST)) return;
            merge_states<C>(P, S, me);
            c_trace(P, l * kTracePerLayer + 2, 1);
            walk_run<WBF16>(P, S, po, chunk, S.xs, P.wo_kbp, wk);
            chunk += (uint32_t)po.nch;
            compute_sync();
            {
                uint64_t *dst = P.p_att + ((size_t)l * P.NA + w.g) * dim;
                const bool res = w.g == 0;
                for (int t = tid; t < po.units; t += kComputeThreads) {
                    const int row = po.u0 + t;
                    ll_store(dst + row, res ? S.xraw[row] + S.yv[t] : S.yv[t], tag);
                }
            }
            c_trace(P, l * kTracePerLayer + 2, 2);
        } else {
            // ---------------- W1/W3 + SwiGLU over the cluster's hidden slice
            const Phase p13 = cta_phase(P, PH_W13, l, w);
            c_trace(P, l * kTracePerLayer + 3, 0);
            Walk<WBF16> wk;
            walk_begin<WBF16>(P, S, p13, chunk, m.w13.KBp, wk);
            load_gain(P, S, m.norms + (size_t)l * 2 * dim + dim);
            // x after the attention block: the sum of the NA partials, in cluster order
            if (!hop_full(P, S, P.p_att + (size_t)l * P.NA * dim, P.NA)) return;
            rs = norm_stage(P, S, m.w13.KBp);
            c_trace(P, l * kTracePerLayer + 3, 1);
            walk_run<WBF16>(P, S, p13, chunk, S.xs, m.w13.KBp, wk);
            chunk += (uint32_t)p13.nch;
            compute_sync();
            {  // one item per (unit, peer): SwiGLU into the peer's W2 activation tile
                const uint32_t ha = smem_addr(S.hb), hbar = smem_addr(&S.xb[XB_H]);
                for (int e = tid; e < p13.units * C; e += kComputeThreads) {
                    const int t = e / C, peer = e % C;
                    const float x1 = S.yv[2 * t] * rs, x2 = S.yv[2 * t + 1] * rs;
                    const float h = x1 / (1.0f + __expf(-x1)) * x2;
                    st_async(cl_map(ha + 4u * (uint32_t)xpos(p13.u0 + t, P.w2_kbp, perm), (uint32_t)peer), h,
                             cl_map(hbar, (uint32_t)peer));
                }
            }
            c_trace(P, l * kTracePerLayer + 3, 2);
            // ---------------- W2: split-K partial over the hidden slice (+ x in cluster 0)
            const Phase p2 = cta_phase(P, PH_W2, l, w);
            c_trace(P, l * kTracePerLayer + 4, 0);
            walk_begin<WBF16>(P, S, p2, chunk, P.w2_kbp, wk);
            if (!xwait(P, S, w, me, XB_H)) return;
            c_trace(P, l * kTracePerLayer + 4, 1);
            walk_run<WBF16>(P, S, p2, chunk, S.hb, P.w2_kbp, wk);
            chunk += (uint32_t)p2.nch;
            compute_sync();
            {
                uint64_t *dst = P.p_ffn + ((size_t)l * P.NF + w.c) * dim;
                const bool res = w.c == 0;
                const bool lost = m.fault && l == 0 && w.c == 0 && w.rank == 0;  // test hook: a lost publish
                for (int t = tid; t < p2.units && !lost; t += kComputeThreads) {
                    const int row = p2.u0 + t;
                    ll_store(dst + row, res ? S.xraw[row] + S.yv[t] : S.yv[t], tag);
                }
            }
            c_trace(P, l * kTracePerLayer + 4, 2);
        }
    }
    if (!P.do_logits) return;
    // ---------------- the logits: every CTA, its share of the vocabulary
    const int tslot = L * kTracePerLayer;
    const Phase pe = cta_phase(P, PH_EMB, L, w);
    c_trace(P, tslot, 0);
    Walk<WBF16> wk;
    walk_begin<WBF16>(P, S, pe, chunk, m.emb.KBp, wk);
    load_gain(P, S, m.norms + (size_t)L * 2 * dim);
    if (!hop_block<C>(P, S, me, P.p_ffn + (size_t)(L - 1) * P.NF * dim, P.NF)) return;
    if (!xwait(P, S, w, me, XB_X)) return;
    rs = norm_stage(P, S, m.emb.KBp);
    c_trace(P, tslot, 1);
    walk_run<WBF16>(P, S, pe, chunk, S.xs, m.emb.KBp, wk);
    compute_sync();
    c_trace(P, tslot, 2);
    c_trace(P, tslot + 1, 0);
    logits_tail(P, S, pe, rs);
    c_trace(P, tslot + 1, 2);
}

template <bool WBF16, int C>
__global__ void __launch_bounds__(kThreads, 1) decode_cluster_kernel(const __grid_constant__ ClusterParams P) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    CS S = carve_c(smem_raw, P);
    const int tid = threadIdx.x;
    const Who w = who(P);
    const Model &m = P.m;
    if (tid == 0) {
        for (int i = 0; i < P.ring_slots; i++) {
            mbar_init(&S.full[i], 1);
            mbar_init(&S.empty[i], 1);
        }
        for (int k = 0; k < 4; k++) mbar_init(&S.xb[k], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        // first use of each exchange barrier this CTA waits on
        for (int k = 0; k < 4; k++)
            if (xb_uses(P, w, k) > 0) mbar_expect_tx(&S.xb[k], xb_bytes(P, w, k));
    }
    // the cluster's SwiGLU tile padding is never pushed: zero it once
    if (!w.attn) {
        int h0, nh;
        ffn_units(P, w.c, h0, nh);
        for (int k = tid; k < P.w2_kbp; k += kThreads)
            if (k >= nh) S.hb[xpos(k, P.w2_kbp, m.weight_bf16)] = 0.f;
    }
    __syncthreads();
    cluster_sync_all();  // every peer's barriers are initialised before the first push
    if (tid >= kComputeThreads) {
        if (tid == kComputeThreads) c_producer(P, S, w);
    } else {
        Me me;
        compute_cta<WBF16, C>(P, S, w, me);
        // An aborted step may leave this thread's cached-row copies in flight: they land
        // in this CTA's shared memory, so it may not exit before they complete.
        asm volatile("cp.async.wait_all;" ::: "memory");
        if (tid == 0)
            for (int k = 0; k < 4; k++) S.wbest_i[k] = (int)me.use[k];
    }
    // No CTA leaves while a peer may still push into its shared memory: first every CTA
    // of the cluster has issued its last push; then, in a step that stopped early, each
    // waits (briefly, bounded) for the pushes of exchanges it armed but did not await;
    // then all leave together.
    __syncwarp();
    cluster_sync_all();
    if (tid == 0) {
        for (int k = 0; k < 4; k++) {
            const uint32_t u = (uint32_t)S.wbest_i[k];
            if (u >= xb_uses(P, w, k)) continue;  // every armed use of this barrier was awaited
            const unsigned long long t0 = global_ns();
            while (!mbar_try_cl(&S.xb[k], u & 1))
                if (global_ns() - t0 > 100000ull) break;  // bytes that were never sent
        }
    }
    __syncthreads();
    cluster_sync_all();
}

// ------------------------------------------------------------------ host side

static const void *cluster_fn(int weight_bf16, int C) {
    if (C == 16) return weight_bf16 ? (const void *)decode_cluster_kernel<true, 16> : (const void *)decode_cluster_kernel<false, 16>;
    return weight_bf16 ? (const void *)decode_cluster_kernel<true, 8> : (const void *)decode_cluster_kernel<false, 8>;
}

cudaError_t cluster_kernel_attrs(int weight_bf16, size_t smem, int C) {
    if (C != 8 && C != 16) return cudaErrorInvalidValue;
    const void *fn = cluster_fn(weight_bf16, C);
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    if (C > 8) e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    return e;
}

// Clusters of C CTAs that can be resident at once with `smem` bytes per CTA.
cudaError_t cluster_capacity(int weight_bf16, size_t smem, int C, int *clusters) {
    cudaError_t e = cluster_kernel_attrs(weight_bf16, smem, C);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = (unsigned)C;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3((unsigned)C);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaOccupancyMaxActiveClusters(clusters, cluster_fn(weight_bf16, C), &cfg);
}

// The CTAs wait on each other, so all of them must be resident at once: the grid is the
// number of clusters the occupancy API reports resident together (one CTA per SM), on a
// GPU this process has to itself.  Should some cluster not be scheduled, its peers'
// bounded waits end the step with a timeout status instead of a hang.  (A cooperative
// launch would state the guarantee, but Nsight Compute fails to launch cooperative
// cluster kernels; the plain cluster launch profiles normally.)
cudaError_t launch_decode_cluster(const ClusterParams &P, size_t smem, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = (unsigned)P.C;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3((unsigned)P.grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    void *args[] = {(void *)&P};
    return cudaLaunchKernelExC(&cfg, cluster_fn(P.m.weight_bf16, P.C), args);
}

}  // namespace slm
