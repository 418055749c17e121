// prefill.cu -- tensor-core prefill of one sequence's prompt.
//
// The prompt is processed in blocks of up to `rows` positions.  Per block and layer:
//   xn  = rmsnorm(x) as bf16                       (one CTA per row)
//   qkv = xn . Wqkv^T                              (tcgen05 GEMM, fp32 out)
//   RoPE of q and k; k, v appended to the cache    (positions p0 .. p0 + T - 1)
//   o   = causal GQA attention, as bf16            (flash-style, CUDA cores, fp32 math)
//   x  += o . Wo^T                                 (GEMM, residual epilogue)
//   xn  = rmsnorm(x) as bf16
//   h   = silu(xn . W1^T) * (xn . W3^T) as bf16    (GEMM, SwiGLU epilogue on interleaved rows)
//   x  += h . W2^T                                 (GEMM, residual epilogue)
// and finally the logits of the last position (GEMM with the tied embedding) and its
// argmax.  The block equations are those of the decode step (kasahare 0.4.0 /
// simple-llm, "Architecture"); the GEMM operands are bf16 (weights as stored,
// activations rounded), accumulation fp32, the residual stream fp32.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

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

__device__ __forceinline__ float block_sum(float v, float *red) {
    v = warp_sum(v);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float t = 0.f;
    for (int w = 0; w < (int)(blockDim.x >> 5); w++) t += red[w];
    __syncthreads();
    return t;
}

// x[t][:] = E[tok[t]] (widened); one CTA per row.
__global__ void embed_rows_kernel(const Model m, const int *tokens, float *x, int *status) {
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
// one CTA per row.
__global__ void rmsnorm_bf16_kernel(const float *x, const float *g, uint16_t *out, size_t lo_off, int dim, float eps) {
    __shared__ float red[32];
    const int t = blockIdx.x;
    const float *r = x + (size_t)t * dim;
    float ss = 0.f;
    for (int k = threadIdx.x; k < dim; k += blockDim.x) ss = fmaf(r[k], r[k], ss);
    ss = block_sum(ss, red);
    const float rs = 1.0f / sqrtf(ss / (float)dim + eps);
    for (int k = threadIdx.x; k < dim; k += blockDim.x)
        split_store(out, out + lo_off, (size_t)t * dim + k, (r[k] * rs) * g[k]);
}

// RoPE of q (in place) and k; k and v of positions p0 + t appended to the cache.
// qkv rows are grouped per kv head, [q heads g*G .. g*G+G-1; k; v], each head's columns
// in RoPE pairs (column 2i = dim i, column 2i + 1 = dim i + hd/2, the weights' stored
// order).  The row is read into shared memory first and written back in natural order.
template <bool KVBF16>
__global__ void rope_append_kernel(const Model m, float *qkv, int layer, int seq, int p0) {
    extern __shared__ float rowbuf[];  // [qkv.rows]
    const int t = blockIdx.x, pos = p0 + t;
    const int hd = m.head_dim, half = hd / 2, KV = m.n_kv_heads, G = m.n_heads / KV;
    const float *rope = m.rope + (size_t)pos * half * 2;
    float *row = qkv + (size_t)t * m.qkv.rows;
    const size_t rowbytes = (size_t)hd * (KVBF16 ? 2 : 4);
    for (int e = threadIdx.x; e < m.qkv.rows; e += blockDim.x) rowbuf[e] = row[e];
    __syncthreads();
    for (int e = threadIdx.x; e < KV * (G + 2) * half; e += blockDim.x) {
        const int g = e / ((G + 2) * half), r = e - g * (G + 2) * half;
        const int j = r / half, i = r - j * half;  // head slot j in the group: q (< G), k (= G), v (= G + 1)
        const size_t h0 = ((size_t)g * (G + 2) + j) * hd;
        float *h = row + h0;
        const float cs = rope[2 * i], sn = rope[2 * i + 1];
        const float a = rowbuf[h0 + 2 * i], b = rowbuf[h0 + 2 * i + 1];
        if (j <= G) {
            const float a2 = a * cs - b * sn, b2 = a * sn + b * cs;
            if (j < G) {
                h[i] = a2;
                h[i + half] = b2;
                continue;
            }
            uint8_t *kd = m.kc + ((((size_t)layer * m.max_batch + seq) * KV + g) * m.max_seq + pos) * rowbytes;
            if (KVBF16) {
                ((uint16_t *)kd)[i] = f32_to_bf16_bits(a2);
                ((uint16_t *)kd)[i + half] = f32_to_bf16_bits(b2);
            } else {
                ((float *)kd)[i] = a2;
                ((float *)kd)[i + half] = b2;
            }
        } else {
            uint8_t *vd = m.vc + ((((size_t)layer * m.max_batch + seq) * KV + g) * m.max_seq + pos) * rowbytes;
            if (KVBF16) {
                ((uint16_t *)vd)[i] = f32_to_bf16_bits(a);
                ((uint16_t *)vd)[i + half] = f32_to_bf16_bits(b);
            } else {
                ((float *)vd)[i] = a;
                ((float *)vd)[i + half] = b;
            }
        }
    }
}

// Causal attention of query rows p0 .. p0 + T - 1 (one CTA: 64 rows of one query head).
// Four threads per row each hold HD/4 dimensions of q and of the output; keys and values
// are staged 64 positions at a time in shared memory; online softmax in the log2 domain.
template <int HD, bool KVBF16>
__global__ void __launch_bounds__(256) attn_prefill_kernel(const Model m, const float *qkv, uint16_t *out, size_t lo_off,
                                                           int layer, int seq, int p0, int T) {
    constexpr int DPT = HD / 4, QB = 64, KB = 4096 / HD;  // query rows per CTA, keys per stage
    __shared__ float ks[KB][HD + 1];
    __shared__ float vs[KB][HD];
    const int h = blockIdx.y, KV = m.n_kv_heads, G = m.n_heads / KV, g = h / G;
    const int r = threadIdx.x >> 2, sub = threadIdx.x & 3;
    const int t = blockIdx.x * QB + r;           // row within the block
    const int pos = p0 + t;                      // this row's position
    const bool live = t < T;
    const int last = p0 + min(T, (int)(blockIdx.x + 1) * QB) - 1;  // last position of the CTA
    const float qscale = rsqrtf((float)HD) * 1.4426950408889634f;
    float q[DPT], o[DPT];
    const float *qr = qkv + (size_t)(live ? t : 0) * m.qkv.rows + ((size_t)g * (G + 2) + (h - g * G)) * HD + sub * DPT;
#pragma unroll
    for (int d = 0; d < DPT; d++) {
        q[d] = live ? qr[d] * qscale : 0.f;
        o[d] = 0.f;
    }
    float mx = -INFINITY, l = 0.f;
    const size_t rowbytes = (size_t)HD * (KVBF16 ? 2 : 4);
    const uint8_t *kbase = m.kc + ((((size_t)layer * m.max_batch + seq) * KV + g) * m.max_seq) * rowbytes;
    const uint8_t *vbase = m.vc + ((((size_t)layer * m.max_batch + seq) * KV + g) * m.max_seq) * rowbytes;
    for (int k0 = 0; k0 <= last; k0 += KB) {
        __syncthreads();
        for (int e = threadIdx.x; e < KB * HD; e += blockDim.x) {
            const int j = e / HD, d = e - j * HD, kp = k0 + j;
            float kv = 0.f, vv = 0.f;
            if (kp <= last) {
                if (KVBF16) {
                    kv = bf16_bits_to_f32(((const uint16_t *)(kbase + (size_t)kp * rowbytes))[d]);
                    vv = bf16_bits_to_f32(((const uint16_t *)(vbase + (size_t)kp * rowbytes))[d]);
                } else {
                    kv = ((const float *)(kbase + (size_t)kp * rowbytes))[d];
                    vv = ((const float *)(vbase + (size_t)kp * rowbytes))[d];
                }
            }
            ks[j][d] = kv;
            vs[j][d] = vv;
        }
        __syncthreads();
        const int jmax = min(KB, last - k0 + 1);
        for (int j = 0; j < jmax; j++) {
            float s = 0.f;
#pragma unroll
            for (int d = 0; d < DPT; d++) s = fmaf(q[d], ks[j][sub * DPT + d], s);
            s += __shfl_xor_sync(0xffffffffu, s, 1);
            s += __shfl_xor_sync(0xffffffffu, s, 2);
            if (k0 + j > pos) continue;  // causal mask (uniform within a row's 4 threads)
            const float mn = fmaxf(mx, s);
            const float corr = exp2f(mx - mn), p = exp2f(s - mn);
            l = l * corr + p;
#pragma unroll
            for (int d = 0; d < DPT; d++) o[d] = fmaf(p, vs[j][sub * DPT + d], o[d] * corr);
            mx = mn;
        }
    }
    if (!live) return;
    const size_t orow = (size_t)t * m.n_heads * HD + (size_t)h * HD + sub * DPT;
    const float inv = 1.0f / l;
#pragma unroll
    for (int d = 0; d < DPT; d++) split_store(out, out + lo_off, orow + d, o[d] * inv);
}

// argmax of one row (lowest index on ties); a NaN sets the status word.
__global__ void argmax_kernel(const float *v, int n, int *out, int *status) {
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
           m.hidden % 8 == 0 && (m.head_dim == 64 || m.head_dim == 128) && (size_t)m.qkv.rows * 4 <= 48 * 1024;
}

static cudaError_t weight_map(CUtensorMap *map, const Mat &M, int layer) {
    return make_bf16_tiled_map(map, M.base + (long long)layer * M.layer_stride, M.nkt, M.rows, M.KBp);
}

cudaError_t prefill_prepare(const Model &m, PrefillPlan &p, int rows) {
    p.rows = rows;
    p.maps.resize((size_t)4 * m.n_layers + 1);
    for (int l = 0; l < m.n_layers; l++) {
        cudaError_t e;
        if ((e = weight_map(&p.maps[4 * l + 0], m.qkv, l)) != cudaSuccess) return e;
        if ((e = weight_map(&p.maps[4 * l + 1], m.wo, l)) != cudaSuccess) return e;
        if ((e = weight_map(&p.maps[4 * l + 2], m.w13, l)) != cudaSuccess) return e;
        if ((e = weight_map(&p.maps[4 * l + 3], m.w2, l)) != cudaSuccess) return e;
    }
    cudaError_t e = weight_map(&p.maps[4 * m.n_layers], m.emb, 0);
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

static cudaError_t gemm(const CUtensorMap &a, const CUtensorMap &a_lo, const CUtensorMap &b, const Mat &M, int rows,
                        int epi, float *of, uint16_t *ob, uint16_t *ob_lo, int ldo, int *status, cudaStream_t s) {
    GemmArgs g{};
    g.a_map = a;
    g.a_lo_map = a_lo;
    g.a_split = 1;
    g.b_map = b;
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
        embed_rows_kernel<<<T, 256, 0, s>>>(m, tokens + p0, p.x, m.status);
        PF_CK(cudaGetLastError());
        const size_t xlo = (size_t)p.rows * m.dim, olo = (size_t)p.rows * qd, hlo = (size_t)p.rows * m.hidden;
        for (int l = 0; l < m.n_layers; l++) {
            const float *gn = m.norms + (size_t)l * 2 * m.dim;
            rmsnorm_bf16_kernel<<<T, 256, 0, s>>>(p.x, gn, p.xn, xlo, m.dim, m.norm_eps);
            PF_CK(gemm(p.xn_map, p.xn_lo_map, p.maps[4 * l + 0], m.qkv, T, GEMM_STORE_F32, p.qkv, nullptr, nullptr,
                       m.qkv.rows, m.status, s));
            rope_append_kernel<true><<<T, 256, (size_t)m.qkv.rows * 4, s>>>(m, p.qkv, l, seq, p0);
            dim3 ag((T + 63) / 64, m.n_heads);
            if (m.head_dim == 64)
                attn_prefill_kernel<64, true><<<ag, 256, 0, s>>>(m, p.qkv, p.o, olo, l, seq, p0, T);
            else
                attn_prefill_kernel<128, true><<<ag, 256, 0, s>>>(m, p.qkv, p.o, olo, l, seq, p0, T);
            PF_CK(cudaGetLastError());
            PF_CK(gemm(p.o_map, p.o_lo_map, p.maps[4 * l + 1], m.wo, T, GEMM_ADD_F32, p.x, nullptr, nullptr, m.dim,
                       m.status, s));
            rmsnorm_bf16_kernel<<<T, 256, 0, s>>>(p.x, gn + m.dim, p.xn, xlo, m.dim, m.norm_eps);
            PF_CK(gemm(p.xn_map, p.xn_lo_map, p.maps[4 * l + 2], m.w13, T, GEMM_SWIGLU, nullptr, p.h, p.h + hlo,
                       m.hidden, m.status, s));
            PF_CK(gemm(p.h_map, p.h_lo_map, p.maps[4 * l + 3], m.w2, T, GEMM_ADD_F32, p.x, nullptr, nullptr, m.dim,
                       m.status, s));
        }
        if (p0 + T == n) {  // logits of the last position (its normalised row goes to xn row 0)
            rmsnorm_bf16_kernel<<<1, 256, 0, s>>>(p.x + (size_t)(T - 1) * m.dim, m.norms + (size_t)m.n_layers * 2 * m.dim,
                                                  p.xn, xlo, m.dim, m.norm_eps);
            float *lg = last_logits ? last_logits : p.logits;
            PF_CK(gemm(p.xn_map, p.xn_lo_map, p.maps[4 * m.n_layers], m.emb, 1, GEMM_STORE_F32, lg, nullptr, nullptr,
                       m.vocab, m.status, s));
            argmax_kernel<<<1, 1024, 0, s>>>(lg, m.vocab, next_id, m.status);
            PF_CK(cudaGetLastError());
        }
    }
#undef PF_CK
    return cudaSuccess;
}

}  // namespace slm
