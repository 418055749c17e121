// prefill.cu -- tensor-core prefill of the prompts of one or several sequences.
//
// The prompt positions are processed in blocks of up to `rows` positions (a block may
// hold the prompts of several sequences: a segment table maps rows to sequences).  Per
// block and layer:
//   xn  = rmsnorm(x), as two bf16 planes hi + lo (x ~ hi + lo to ~16 mantissa bits)
//   qkv = xn . Wqkv^T                               (tcgen05 GEMM: bf16 weights x the hi
//                                                    and the lo plane, fp32 accumulation)
//   RoPE of q and k; k, v appended to the cache     (positions p0 .. p0 + T - 1)
//   o   = causal GQA attention                      (flash-style on the tensor cores:
//                                                    mma.sync bf16 QK^T and PV, fp32
//                                                    online softmax), as hi + lo planes
//   x  += o . Wo^T                                  (GEMM, residual epilogue)
//   xn  = rmsnorm(x) as hi + lo planes
//   h   = silu(xn . W1^T) * (xn . W3^T)             (GEMM, SwiGLU epilogue on interleaved
//                                                    rows), as hi + lo planes
//   x  += h . W2^T                                  (GEMM, residual epilogue)
// and finally the logits of each sequence's last position (GEMM with the tied
// embedding) and its argmax.  The block equations are those of the decode step
// (kasahare 0.4.0 / simple-llm, "Architecture"); weights enter as stored (bf16), the
// residual stream and every accumulation are fp32.  Every kernel of this chain is
// launched with programmatic dependent launch (launch_pdl) and waits for its predecessor
// (pdl_wait) before it reads anything, so launches overlap the previous kernel's tail.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "device_common.cuh"
#include "gemm_tc.cuh"
#include "prefill.cuh"
#include "slm_internal.h"

namespace slm {

__device__ __forceinline__ float bf16_bits_to_f32(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

__device__ __forceinline__ uint16_t f32_to_bf16_bits(float v) {
    __nv_bfloat16 h = __float2bfloat16_rn(v);
    return *(uint16_t *)&h;
}

// x[t][:] = E[tok[t]] (widened); one CTA per row.
__global__ void embed_rows_kernel(const Model m, const int *tokens, float *x, int *status) {
    pdl_wait();
    pdl_trigger();
    const int t = blockIdx.x;
    int tok = __ldg(tokens + t);
    if (tok < 0 || tok >= m.vocab) {
        if (threadIdx.x == 0) atomicOr(status, kStBadToken);
        tok = 0;
    }
    const uint16_t *row = (const uint16_t *)m.emb.base + (size_t)tok * m.emb.KBp;
    for (int k = threadIdx.x; k < m.dim; k += blockDim.x) x[(size_t)t * m.dim + k] = bf16_bits_to_f32(row[k]);
}

// Split v into bf16 hi + lo parts.
__device__ __forceinline__ void split_store(uint16_t *hi, uint16_t *lo, size_t i, float v) {
    const __nv_bfloat16 h = __float2bfloat16_rn(v);
    const __nv_bfloat16 l = __float2bfloat16_rn(v - __bfloat162float(h));
    hi[i] = *(const uint16_t *)&h;
    lo[i] = *(const uint16_t *)&l;
}

// out = (x[t][:] * rsqrt(mean(x^2) + eps)) * g as bf16 hi (out) + lo (out + lo_off);
// one CTA per row (a few hundred rows: every thread of the row's CTA takes a few
// elements, the shortest chain).
__global__ void rmsnorm_bf16_kernel(const float *x, const float *g, uint16_t *out, size_t lo_off, int dim, float eps) {
    pdl_wait();
    pdl_trigger();
    __shared__ float red[32];
    const int t = blockIdx.x;
    const float *r = x + (size_t)t * dim;
    float ss = 0.f;
    for (int k = threadIdx.x; k < dim; k += blockDim.x) ss = fmaf(r[k], r[k], ss);
    ss = warp_sum(ss);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) red[warp] = ss;
    __syncthreads();
    ss = 0.f;
    for (int w = 0; w < (int)(blockDim.x >> 5); w++) ss += red[w];
    const float rs = 1.0f / sqrtf(ss / (float)dim + eps);
    for (int k = threadIdx.x; k < dim; k += blockDim.x)
        split_store(out, out + lo_off, (size_t)t * dim + k, (r[k] * rs) * g[k]);
}

// The same for many rows (thousands): one warp per row, 8 rows per CTA (fewer, fuller
// CTAs: measured 16.6 -> ~8 us per launch at 8,192 rows of 576).
__global__ void rmsnorm_bf16_rows_kernel(const float *x, const float *g, uint16_t *out, size_t lo_off, int dim,
                                         float eps, int rows) {
    pdl_wait();
    pdl_trigger();
    const int t = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (t >= rows) return;
    const float *r = x + (size_t)t * dim;
    float ss = 0.f;
    for (int k = lane; k < dim; k += 32) ss = fmaf(r[k], r[k], ss);
    ss = warp_sum(ss);
    const float rs = 1.0f / sqrtf(ss / (float)dim + eps);
    for (int k = lane; k < dim; k += 32) split_store(out, out + lo_off, (size_t)t * dim + k, (r[k] * rs) * g[k]);
}

static cudaError_t rmsnorm_launch(const float *x, const float *g, uint16_t *out, size_t lo_off, int dim, float eps,
                                  int rows, cudaStream_t s) {
    if (rows >= 2048)
        return launch_pdl(rmsnorm_bf16_rows_kernel, dim3((rows + 7) / 8), dim3(256), 0, s, x, g, out, lo_off, dim, eps, rows);
    else
        return launch_pdl(rmsnorm_bf16_kernel, dim3(rows), dim3(256), 0, s, x, g, out, lo_off, dim, eps);
}

// RoPE of q (in place) and k; k and v of positions p0 + t appended to the bf16 cache.
// qkv rows are grouped per kv head, [q heads g*G .. g*G+G-1; k; v], each head's columns
// in RoPE pairs (column 2i = dim i, column 2i + 1 = dim i + hd/2, the weights' stored
// order); q leaves in natural order.  One warp per row: lane l takes the pairs l, l + 32,
// ... of every head (hd/2 is a multiple of 32), as 8-byte loads of up to 8 heads at a
// time, all in flight, before any of those heads is written back.
static inline int rope_rpc(int rows) { return rows >= 4096 ? 8 : 2; }  // rows (warps) per CTA

template <int HD>
__global__ void __launch_bounds__(256) rope_append_kernel(const Model m, float *qkv, int layer, const PfSegs sg,
                                                          int rows) {
    pdl_wait();
    pdl_trigger();
    constexpr int HALF = HD / 2, PPL = HALF / 32, CH = 8;  // pairs per lane and head, heads per round
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);  // row of the block
    if (t >= rows) return;  // (no block-wide barrier below: each warp keeps to its row)
    int k = 0;
    while (k + 1 < sg.n && t >= sg.row[k + 1]) k++;
    const int seq = sg.seq[k], pos = sg.pos0[k] + (t - sg.row[k]);
    const int KV = m.n_kv_heads, G = m.n_heads / KV, S = G + 2, heads = KV * S;
    float *row = qkv + (size_t)t * m.qkv.rows;
    float2 cs[PPL];  // (cos, sin) of this lane's pairs at this position
#pragma unroll
    for (int p = 0; p < PPL; p++) cs[p] = *(const float2 *)(m.rope + ((size_t)pos * HALF + lane + 32 * p) * 2);
    for (int j0 = 0; j0 < heads; j0 += CH) {
        float2 v[CH][PPL];
#pragma unroll
        for (int c = 0; c < CH; c++)
#pragma unroll
            for (int p = 0; p < PPL; p++)
                v[c][p] = j0 + c < heads ? *(const float2 *)(row + (size_t)(j0 + c) * HD + 2 * (lane + 32 * p))
                                         : make_float2(0.f, 0.f);
        __syncwarp();  // every lane has read these heads before any lane overwrites them
#pragma unroll
        for (int c = 0; c < CH; c++) {
            const int jh = j0 + c;
            if (jh >= heads) break;
            const int g = jh / S, j = jh - g * S;  // kv group, slot: q (< G), k (= G), v (= G + 1)
            if (j < G) {
                float *h = row + (size_t)jh * HD;
#pragma unroll
                for (int p = 0; p < PPL; p++) {
                    const int i = lane + 32 * p;
                    const float a = v[c][p].x, b = v[c][p].y, cn = cs[p].x, sn = cs[p].y;
                    h[i] = a * cn - b * sn;
                    h[i + HALF] = a * sn + b * cn;
                }
            } else {
                uint16_t *d = (uint16_t *)((j == G ? m.kc : m.vc) + kv_row(m, layer, seq, g, pos) * (size_t)(HD * 2));
#pragma unroll
                for (int p = 0; p < PPL; p++) {
                    const int i = lane + 32 * p;
                    const float a = v[c][p].x, b = v[c][p].y, cn = cs[p].x, sn = cs[p].y;
                    d[i] = f32_to_bf16_bits(j == G ? a * cn - b * sn : a);
                    d[i + HALF] = f32_to_bf16_bits(j == G ? a * sn + b * cn : b);
                }
            }
        }
    }
}

static cudaError_t rope_launch(const Model &m, float *qkv, int layer, const PfSegs &sg, int rows, cudaStream_t s) {
    const int rpc = rope_rpc(rows);
    if (m.head_dim == 64)
        return launch_pdl(rope_append_kernel<64>, dim3((rows + rpc - 1) / rpc), dim3(32 * rpc), 0, s, m, qkv, layer, sg, rows);
    else
        return launch_pdl(rope_append_kernel<128>, dim3((rows + rpc - 1) / rpc), dim3(32 * rpc), 0, s, m, qkv, layer, sg, rows);
}

// ---- tensor-core causal attention (flash-attention style, mma.sync bf16 -> fp32)

// Causal attention of query rows p0 .. p0 + T - 1 of one query head on the tensor cores:
// a CTA takes 64 rows (4 warps x 16), walks the cached keys / values 64 positions at a
// time (bf16, copied to padded shared memory with cp.async through a ring of kAttnStages
// buffers), S = Q K^T and O += P V by mma.sync m16n8k16 with fp32 accumulation, online
// softmax in the log2 domain (q is pre-multiplied by log2(e) / sqrt(HD)), causal mask on
// the blocks that reach the rows' own positions.  Q and P enter the MMAs as bf16.  The
// CTAs of one (head, sequence) start with the last query block, the one with the most
// key blocks, so the short ones fill the tail of the launch.
template <int HD> struct AttnStages {
    static constexpr int value = HD == 64 ? 3 : 2;  // HD 128: two stages keep 2 CTAs per SM
};
template <int HD>
__global__ void __launch_bounds__(128) attn_prefill_tc_kernel(const Model m, const float *qkv_blk, uint16_t *out_blk,
                                                              size_t lo_off, int layer, const PfSegs sg) {
    pdl_wait();
    pdl_trigger();
    constexpr int QB = 64, KB = 64, LD = HD + 8;  // rows per CTA, keys per block, padded row (elements)
    constexpr int NST = AttnStages<HD>::value;
    // segment blockIdx.z of the block: its rows, sequence and first position
    const int sgi = blockIdx.z, seq = sg.seq[sgi], p0 = sg.pos0[sgi], T = sg.count[sgi];
    const int qb = (int)(gridDim.x - 1 - blockIdx.x);  // query block, longest first
    if (qb * QB >= T) return;
    const float *qkv = qkv_blk + (size_t)sg.row[sgi] * m.qkv.rows;
    uint16_t *out = out_blk + (size_t)sg.row[sgi] * m.n_heads * HD;
    extern __shared__ __align__(16) uint16_t sm[];
    uint16_t *qs = sm;                  // [QB][LD]
    // key / value ring: buffer b = [KB][LD] keys, then [KB][LD] values
    auto kbuf = [&](int b) { return qs + QB * LD + b * 2 * KB * LD; };
    auto vbuf = [&](int b) { return qs + QB * LD + b * 2 * KB * LD + KB * LD; };
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g4 = lane >> 2, t4 = lane & 3;
    const int h = blockIdx.y, KV = m.n_kv_heads, G = m.n_heads / KV, g = h / G;
    const int q0 = qb * QB;                               // first row of the CTA
    const int last = p0 + min(T, q0 + QB) - 1;            // last position any row reads
    const size_t rowbytes = (size_t)HD * 2;

    // key / value block k0 into buffer b as one cp.async group (zeros past `last`); past
    // the end an empty group, so that every iteration waits for the same group count.
    // A thread copies the same 16-byte column of rows j0, j0 + RPP, ...; with pages of 64
    // positions or more (or no paging) the block lies in one page, so one table lookup
    // gives every row.
    auto load = [&](int k0, int b) {
        if (k0 <= last) {
            constexpr int PPR = HD / 8, RPP = 128 / PPR;  // 16-byte pieces per row, rows per pass
            const int j0 = tid / PPR, c = (tid % PPR) * 8;
            const bool one_page = m.kv_shift >= 6;
            const size_t row0 = one_page ? kv_row(m, layer, seq, g, k0) : 0;
#pragma unroll
            for (int i = 0; i < KB / RPP; i++) {
                const int j = j0 + i * RPP, kp = k0 + j;
                uint16_t *kd = kbuf(b) + j * LD + c, *vd = vbuf(b) + j * LD + c;
                if (kp <= last) {
                    const size_t row = one_page ? row0 + j : kv_row(m, layer, seq, g, kp);
                    const size_t src = row * rowbytes + c * 2;
                    cp_async16(kd, m.kc + src);
                    cp_async16(vd, m.vc + src);
                } else {
                    *(uint4 *)kd = make_uint4(0, 0, 0, 0);
                    *(uint4 *)vd = make_uint4(0, 0, 0, 0);
                }
            }
        }
        cp_async_commit();
    };
    // the first NST - 1 key / value blocks load while the Q tile is read
#pragma unroll
    for (int b = 0; b < NST - 1; b++) load(b * KB, b);

    // Q tile: fp32 -> scaled bf16; every thread's 16-byte loads are issued before use
    const float qscale = rsqrtf((float)HD) * 1.4426950408889634f;
    const size_t qcol = ((size_t)g * (G + 2) + (h - g * G)) * HD;
    constexpr int QV = QB * HD / 4 / 128;  // float4 per thread
    float4 qv[QV];
#pragma unroll
    for (int i = 0; i < QV; i++) {
        const int e = (tid + i * 128) * 4, r = e / HD, d = e - r * HD, t = q0 + r;
        qv[i] = t < T ? *(const float4 *)(qkv + (size_t)t * m.qkv.rows + qcol + d) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int i = 0; i < QV; i++) {
        const int e = (tid + i * 128) * 4, r = e / HD, d = e - r * HD;
        *(uint2 *)(qs + r * LD + d) = make_uint2(pack_bf16x2(qv[i].x * qscale, qv[i].y * qscale),
                                                 pack_bf16x2(qv[i].z * qscale, qv[i].w * qscale));
    }
    __syncthreads();
    uint32_t qa[HD / 16][4];  // A fragments of this warp's 16 rows
#pragma unroll
    for (int kk = 0; kk < HD / 16; kk++) {
        const int r = warp * 16 + (lane & 7) + ((lane >> 3) & 1) * 8, c = kk * 16 + (lane >> 4) * 8;
        ldsm_x4(qa[kk], qs + r * LD + c);
    }
    float o[HD / 8][4];
#pragma unroll
    for (int n = 0; n < HD / 8; n++) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    float mrow[2] = {-INFINITY, -INFINITY}, lrow[2] = {0.f, 0.f};  // rows g4, g4 + 8
    const int pos0 = p0 + q0 + warp * 16 + g4, pos1 = pos0 + 8;    // this lane's two rows

    for (int k0 = 0, kb = 0; k0 <= last; k0 += KB, kb++) {
        // block kb + NST - 1 loads while this one is computed
        load(k0 + (NST - 1) * KB, (kb + NST - 1) % NST);
        cp_async_wait_upto(NST - 1);
        __syncthreads();  // block kb (and its zero fill) is visible to every warp
        const uint16_t *ks = kbuf(kb % NST), *vs = vbuf(kb % NST);
        // S = Q K^T for 64 keys: 8 tiles of 8 keys
        float sc[KB / 8][4];
#pragma unroll
        for (int n = 0; n < KB / 8; n++) {
            sc[n][0] = sc[n][1] = sc[n][2] = sc[n][3] = 0.f;
#pragma unroll
            for (int kk = 0; kk < HD / 16; kk += 2) {  // two k-steps per x4 load
                uint32_t b[4];
                const int r = n * 8 + (lane & 7), c = kk * 16 + (lane >> 3) * 8;
                ldsm_x4(b, ks + r * LD + c);
                mma_bf16_16816(sc[n], qa[kk], b[0], b[1]);
                mma_bf16_16816(sc[n], qa[kk + 1], b[2], b[3]);
            }
        }
        // causal mask, row maxima
        const bool diag = k0 + KB - 1 > pos0;
        float mx0 = mrow[0], mx1 = mrow[1];
#pragma unroll
        for (int n = 0; n < KB / 8; n++) {
            const int kp = k0 + n * 8 + 2 * t4;
            if (diag) {
                if (kp > pos0) sc[n][0] = -INFINITY;
                if (kp + 1 > pos0) sc[n][1] = -INFINITY;
                if (kp > pos1) sc[n][2] = -INFINITY;
                if (kp + 1 > pos1) sc[n][3] = -INFINITY;
            }
            mx0 = fmaxf(mx0, fmaxf(sc[n][0], sc[n][1]));
            mx1 = fmaxf(mx1, fmaxf(sc[n][2], sc[n][3]));
        }
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
        const float c0 = fast_exp2(mrow[0] - mx0), c1 = fast_exp2(mrow[1] - mx1);  // exp2(-inf) = 0
        mrow[0] = mx0;
        mrow[1] = mx1;
        lrow[0] *= c0;
        lrow[1] *= c1;
#pragma unroll
        for (int n = 0; n < HD / 8; n++) {
            o[n][0] *= c0;
            o[n][1] *= c0;
            o[n][2] *= c1;
            o[n][3] *= c1;
        }
        // P = 2^(S - m) as bf16 A fragments; O += P V
#pragma unroll
        for (int kk = 0; kk < KB / 16; kk++) {
            float p[8];
            p[0] = fast_exp2(sc[2 * kk][0] - mx0);
            p[1] = fast_exp2(sc[2 * kk][1] - mx0);
            p[2] = fast_exp2(sc[2 * kk][2] - mx1);
            p[3] = fast_exp2(sc[2 * kk][3] - mx1);
            p[4] = fast_exp2(sc[2 * kk + 1][0] - mx0);
            p[5] = fast_exp2(sc[2 * kk + 1][1] - mx0);
            p[6] = fast_exp2(sc[2 * kk + 1][2] - mx1);
            p[7] = fast_exp2(sc[2 * kk + 1][3] - mx1);
            lrow[0] += p[0] + p[1] + p[4] + p[5];
            lrow[1] += p[2] + p[3] + p[6] + p[7];
            uint32_t pa[4];
            pa[0] = pack_bf16x2(p[0], p[1]);
            pa[1] = pack_bf16x2(p[2], p[3]);
            pa[2] = pack_bf16x2(p[4], p[5]);
            pa[3] = pack_bf16x2(p[6], p[7]);
#pragma unroll
            for (int n = 0; n < HD / 8; n += 2) {  // two dim tiles per x4 load
                uint32_t b[4];
                const int r = kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8, c = n * 8 + (lane >> 4) * 8;
                ldsm_x4_t(b, vs + r * LD + c);
                mma_bf16_16816(o[n], pa, b[0], b[1]);
                mma_bf16_16816(o[n + 1], pa, b[2], b[3]);
            }
        }
        __syncthreads();  // every warp is done with this buffer before the next prefetch fills it
    }
    // row sums over the quad, normalise, store (bf16 hi + lo planes)
    float l0 = lrow[0], l1 = lrow[1];
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    const int t0 = q0 + warp * 16 + g4, t1 = t0 + 8;
    const float i0 = 1.0f / l0, i1 = 1.0f / l1;
#pragma unroll
    for (int n = 0; n < HD / 8; n++) {
        const int d = n * 8 + 2 * t4;
        if (t0 < T) {
            const size_t row = (size_t)t0 * m.n_heads * HD + (size_t)h * HD + d;
            split_store(out, out + lo_off, row, o[n][0] * i0);
            split_store(out, out + lo_off, row + 1, o[n][1] * i0);
        }
        if (t1 < T) {
            const size_t row = (size_t)t1 * m.n_heads * HD + (size_t)h * HD + d;
            split_store(out, out + lo_off, row, o[n][2] * i1);
            split_store(out, out + lo_off, row + 1, o[n][3] * i1);
        }
    }
}

template <int HD>
static size_t attn_tc_smem() { return (size_t)(1 + 2 * AttnStages<HD>::value) * 64 * (HD + 8) * 2; }  // Q + K / V ring

// argmax of one row (lowest index on ties); a NaN sets the status word.
// Row blockIdx.x of v [rows][n]: its argmax (lowest index on ties) into out[blockIdx.x].
__global__ void argmax_kernel(const float *v, int n, int *out, int *status) {
    pdl_wait();
    pdl_trigger();
    v += (size_t)blockIdx.x * n;
    out += blockIdx.x;
    __shared__ float bv[32];
    __shared__ int bi[32];
    float best = -INFINITY;
    int idx = 0x7fffffff;
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
        const float x = v[i];
        if (x != x) {
            atomicOr(status, kStNanLogits);
            continue;
        }
        if (x > best || (x == best && i < idx)) {
            best = x;
            idx = i;
        }
    }
    for (int off = 16; off; off >>= 1) {
        const float b2 = __shfl_xor_sync(0xffffffffu, best, off);
        const int i2 = __shfl_xor_sync(0xffffffffu, idx, off);
        if (b2 > best || (b2 == best && i2 < idx)) {
            best = b2;
            idx = i2;
        }
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) {
        bv[warp] = best;
        bi[warp] = idx;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < (int)(blockDim.x >> 5); w++)
            if (bv[w] > best || (bv[w] == best && bi[w] < idx)) {
                best = bv[w];
                idx = bi[w];
            }
        *out = idx == 0x7fffffff ? 0 : idx;
    }
}

// ------------------------------------------------------------------ host side

bool prefill_supported(const Model &m) {
    return m.weight_bf16 && m.kv_bf16 && m.dim % 64 == 0 && (m.n_heads * m.head_dim) % 64 == 0 &&
           m.hidden % 8 == 0 && (m.head_dim == 64 || m.head_dim == 128);
}

// Two maps per weight matrix: boxes of 64 rows (64-column tiles) and of 128 rows.
static cudaError_t weight_map(CUtensorMap *map, const Mat &M, int layer) {
    cudaError_t e = make_bf16_tiled_map(map, M.base + (long long)layer * M.layer_stride, M.nkt, M.rows, M.KBp, 64);
    if (e != cudaSuccess) return e;
    return make_bf16_tiled_map(map + 1, M.base + (long long)layer * M.layer_stride, M.nkt, M.rows, M.KBp, 128);
}

cudaError_t prefill_prepare(const Model &m, PrefillPlan &p, int rows) {
    p.rows = rows;
    {
        cudaError_t e = cudaFuncSetAttribute(attn_prefill_tc_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)attn_tc_smem<64>());
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(attn_prefill_tc_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)attn_tc_smem<128>());
        if (e != cudaSuccess) return e;
    }
    p.maps.resize(2 * ((size_t)4 * m.n_layers + 1));
    for (int l = 0; l < m.n_layers; l++) {
        cudaError_t e;
        if ((e = weight_map(&p.maps[2 * (4 * l + 0)], m.qkv, l)) != cudaSuccess) return e;
        if ((e = weight_map(&p.maps[2 * (4 * l + 1)], m.wo, l)) != cudaSuccess) return e;
        if ((e = weight_map(&p.maps[2 * (4 * l + 2)], m.w13, l)) != cudaSuccess) return e;
        if ((e = weight_map(&p.maps[2 * (4 * l + 3)], m.w2, l)) != cudaSuccess) return e;
    }
    cudaError_t e = weight_map(&p.maps[2 * (4 * m.n_layers)], m.emb, 0);
    if (e != cudaSuccess) return e;
    const int qd = m.n_heads * m.head_dim;
    if ((e = make_bf16_map(&p.xn_map, p.xn, rows, m.dim, m.dim)) != cudaSuccess) return e;
    if ((e = make_bf16_map(&p.o_map, p.o, rows, qd, qd)) != cudaSuccess) return e;
    if ((e = make_bf16_map(&p.h_map, p.h, rows, m.hidden, m.hidden)) != cudaSuccess) return e;
    if ((e = make_bf16_map(&p.xn_lo_map, p.xn + (size_t)rows * m.dim, rows, m.dim, m.dim)) != cudaSuccess) return e;
    if ((e = make_bf16_map(&p.o_lo_map, p.o + (size_t)rows * qd, rows, qd, qd)) != cudaSuccess) return e;
    if ((e = make_bf16_map(&p.h_lo_map, p.h + (size_t)rows * m.hidden, rows, m.hidden, m.hidden)) != cudaSuccess)
        return e;
    return cudaSuccess;
}

static cudaError_t gemm(const CUtensorMap &a, const CUtensorMap &a_lo, const CUtensorMap *b, const Mat &M, int rows,
                        int epi, float *of, uint16_t *ob, uint16_t *ob_lo, int ldo, int *status, cudaStream_t s) {
    GemmArgs g{};
    g.a_map = a;
    g.a_lo_map = a_lo;
    g.a_split = 1;
    g.b_map = b[0];
    g.b_map_wide = b[1];
    g.out_bf16_lo = ob_lo;
    g.b_tile_k = M.KBp;
    g.M = rows;
    g.N = M.rows;
    g.K = M.nkt * M.KBp;
    g.epi = epi;
    g.out_f32 = of;
    g.out_bf16 = ob;
    g.ldo = ldo;
    g.status = status;
    return gemm_bf16_tn(g, s);
}

cudaError_t prefill_run(const Model &m, const PrefillPlan &p, int seq, const int *tokens, int n, float *last_logits,
                        int *next_id, cudaStream_t s) {
    const int qd = m.n_heads * m.head_dim;
    cudaError_t e = cudaSuccess;
#define PF_CK(x)                                   \
    do {                                           \
        if ((e = (x)) != cudaSuccess) return e;    \
    } while (0)
    for (int p0 = 0; p0 < n; p0 += p.rows) {
        const int T = n - p0 < p.rows ? n - p0 : p.rows;
        PF_CK(launch_pdl(embed_rows_kernel, dim3(T), dim3(256), 0, s, m, tokens + p0, p.x, m.status));
        const size_t xlo = (size_t)p.rows * m.dim, olo = (size_t)p.rows * qd, hlo = (size_t)p.rows * m.hidden;
        for (int l = 0; l < m.n_layers; l++) {
            const float *gn = m.norms + (size_t)l * 2 * m.dim;
            PF_CK(rmsnorm_launch(p.x, gn, p.xn, xlo, m.dim, m.norm_eps, T, s));
            PF_CK(gemm(p.xn_map, p.xn_lo_map, &p.maps[2 * (4 * l + 0)], m.qkv, T, GEMM_STORE_F32, p.qkv, nullptr, nullptr,
                       m.qkv.rows, m.status, s));
            PfSegs one{};
            one.n = 1;
            one.seq[0] = seq;
            one.pos0[0] = p0;
            one.count[0] = T;
            one.row[0] = 0;
            PF_CK(rope_launch(m, p.qkv, l, one, T, s));
            dim3 ag((T + 63) / 64, m.n_heads, 1);
            if (m.head_dim == 64)
                PF_CK(launch_pdl(attn_prefill_tc_kernel<64>, ag, dim3(128), attn_tc_smem<64>(), s, m, (const float *)p.qkv, p.o,
                                 olo, l, one));
            else
                PF_CK(launch_pdl(attn_prefill_tc_kernel<128>, ag, dim3(128), attn_tc_smem<128>(), s, m, (const float *)p.qkv,
                                 p.o, olo, l, one));
            PF_CK(gemm(p.o_map, p.o_lo_map, &p.maps[2 * (4 * l + 1)], m.wo, T, GEMM_ADD_F32, p.x, nullptr, nullptr, m.dim,
                       m.status, s));
            PF_CK(rmsnorm_launch(p.x, gn + m.dim, p.xn, xlo, m.dim, m.norm_eps, T, s));
            PF_CK(gemm(p.xn_map, p.xn_lo_map, &p.maps[2 * (4 * l + 2)], m.w13, T, GEMM_SWIGLU, nullptr, p.h, p.h + hlo,
                       m.hidden, m.status, s));
            PF_CK(gemm(p.h_map, p.h_lo_map, &p.maps[2 * (4 * l + 3)], m.w2, T, GEMM_ADD_F32, p.x, nullptr, nullptr, m.dim,
                       m.status, s));
        }
        if (p0 + T == n) {  // logits of the last position (its normalised row goes to xn row 0)
            PF_CK(launch_pdl(rmsnorm_bf16_kernel, dim3(1), dim3(256), 0, s, (const float *)(p.x + (size_t)(T - 1) * m.dim),
                             (const float *)(m.norms + (size_t)m.n_layers * 2 * m.dim), p.xn, xlo, m.dim, m.norm_eps));
            float *lg = last_logits ? last_logits : p.logits;
            PF_CK(gemm(p.xn_map, p.xn_lo_map, &p.maps[2 * (4 * m.n_layers)], m.emb, 1, GEMM_STORE_F32, lg, nullptr, nullptr,
                       m.vocab, m.status, s));
            PF_CK(launch_pdl(argmax_kernel, dim3(1), dim3(1024), 0, s, (const float *)lg, m.vocab, next_id, m.status));
        }
    }
#undef PF_CK
    return cudaSuccess;
}

// Several empty sequences at once: their prompts, concatenated in order, are cut into
// blocks of up to p.rows rows; every GEMM and norm of a block runs over all its rows
// (rows are independent there), RoPE / append and the causal attention run per segment
// (one sequence's consecutive positions inside the block).  The logits of every sequence
// whose last position falls in the block are computed together.
cudaError_t prefill_run_batch(const Model &m, const PrefillPlan &p, int nseq, const int *seqs, const int *lens,
                              const int *tokens, float *last_logits, int *next_ids, cudaStream_t s) {
    const int qd = m.n_heads * m.head_dim;
    cudaError_t e = cudaSuccess;
#define PF_CK(x)                                   \
    do {                                           \
        if ((e = (x)) != cudaSuccess) return e;    \
    } while (0)
    long long total = 0;
    for (int i = 0; i < nseq; i++) total += lens[i];
    const size_t xlo = (size_t)p.rows * m.dim, olo = (size_t)p.rows * qd, hlo = (size_t)p.rows * m.hidden;
    int si = 0, spos = 0;  // the next row to place: sequence si, its position spos
    for (long long r0 = 0; r0 < total;) {
        struct Seg { int seq, idx, pos0, count, row; };
        Seg segs[kMaxBatch + 1];
        int nsegs = 0, T = 0;
        while (T < p.rows && si < nseq) {
            const int take = std::min(lens[si] - spos, p.rows - T);
            segs[nsegs++] = {seqs[si], si, spos, take, T};
            T += take;
            spos += take;
            if (spos == lens[si]) {
                si++;
                spos = 0;
            }
        }
        PfSegs tab{};
        int maxcount = 0;
        tab.n = nsegs;
        for (int k = 0; k < nsegs; k++) {
            tab.seq[k] = segs[k].seq;
            tab.pos0[k] = segs[k].pos0;
            tab.count[k] = segs[k].count;
            tab.row[k] = segs[k].row;
            maxcount = std::max(maxcount, segs[k].count);
        }
        PF_CK(launch_pdl(embed_rows_kernel, dim3(T), dim3(256), 0, s, m, tokens + r0, p.x, m.status));
        for (int l = 0; l < m.n_layers; l++) {
            const float *gn = m.norms + (size_t)l * 2 * m.dim;
            PF_CK(rmsnorm_launch(p.x, gn, p.xn, xlo, m.dim, m.norm_eps, T, s));
            PF_CK(gemm(p.xn_map, p.xn_lo_map, &p.maps[2 * (4 * l + 0)], m.qkv, T, GEMM_STORE_F32, p.qkv, nullptr, nullptr,
                       m.qkv.rows, m.status, s));
            PF_CK(rope_launch(m, p.qkv, l, tab, T, s));
            dim3 ag((maxcount + 63) / 64, m.n_heads, nsegs);  // every segment in one launch
            if (m.head_dim == 64)
                PF_CK(launch_pdl(attn_prefill_tc_kernel<64>, ag, dim3(128), attn_tc_smem<64>(), s, m, (const float *)p.qkv, p.o,
                                 olo, l, tab));
            else
                PF_CK(launch_pdl(attn_prefill_tc_kernel<128>, ag, dim3(128), attn_tc_smem<128>(), s, m, (const float *)p.qkv,
                                 p.o, olo, l, tab));
            PF_CK(gemm(p.o_map, p.o_lo_map, &p.maps[2 * (4 * l + 1)], m.wo, T, GEMM_ADD_F32, p.x, nullptr, nullptr, m.dim,
                       m.status, s));
            PF_CK(rmsnorm_launch(p.x, gn + m.dim, p.xn, xlo, m.dim, m.norm_eps, T, s));
            PF_CK(gemm(p.xn_map, p.xn_lo_map, &p.maps[2 * (4 * l + 2)], m.w13, T, GEMM_SWIGLU, nullptr, p.h, p.h + hlo,
                       m.hidden, m.status, s));
            PF_CK(gemm(p.h_map, p.h_lo_map, &p.maps[2 * (4 * l + 3)], m.w2, T, GEMM_ADD_F32, p.x, nullptr, nullptr, m.dim,
                       m.status, s));
        }
        // sequences that end in this block: their last rows' final norms into xn rows
        // 0..k-1, one logits GEMM, one argmax each
        int first = -1, k = 0;
        for (int j = 0; j < nsegs; j++) {
            const Seg &g = segs[j];
            if (g.pos0 + g.count != lens[g.idx]) continue;
            if (first < 0) first = g.idx;
            PF_CK(launch_pdl(rmsnorm_bf16_kernel, dim3(1), dim3(256), 0, s,
                             (const float *)(p.x + (size_t)(g.row + g.count - 1) * m.dim),
                             (const float *)(m.norms + (size_t)m.n_layers * 2 * m.dim), p.xn + (size_t)k * m.dim, xlo,
                             m.dim, m.norm_eps));
            k++;
        }
        if (k > 0) {
            float *lg = (last_logits ? last_logits : p.logits) + (last_logits ? (size_t)first * m.vocab : 0);
            PF_CK(gemm(p.xn_map, p.xn_lo_map, &p.maps[2 * (4 * m.n_layers)], m.emb, k, GEMM_STORE_F32, lg, nullptr,
                       nullptr, m.vocab, m.status, s));
            PF_CK(launch_pdl(argmax_kernel, dim3(k), dim3(1024), 0, s, (const float *)lg, m.vocab, next_ids + first,
                             m.status));  // one CTA per row
        }
        r0 += T;
    }
#undef PF_CK
    return cudaSuccess;
}

}  // namespace slm
