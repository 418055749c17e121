// sampling.cu -- the next token drawn on the device from rows of logits.
//
// "Inside nanochat Part 4: Understanding Inference" (The Sampling Function, Greedy
// Decoding, Temperature Sampling, Top-K Filtering), with top-p as nucleus filtering after
// top-k (kasahare 0.4.0, "CLI flags" names it beside top-k).  The uniform variate of the
// draw is an input, one per row; the draw is the inverse cumulative distribution over
// the candidates (top-k: largest logit first, ties by lower index; no top-k: index
// order).  One CTA of 1024 threads per row:
//   greedy       block argmax (lowest index on ties);
//   top-k        radix select of the k-th largest order-preserving key (4 passes of 8
//                bits, shared histogram), a deterministic gather (ties filled by the
//                lowest indices), a bitonic sort of the candidates, softmax weights,
//                block scan, top-p cut, the draw; for large vocabularies split over
//                several CTAs per row (each slice's top k, then one merge per row);
//   whole vocab  per-thread index-ordered ranges, block scan of the range sums, the
//                draw inside the range that holds it.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "slm_internal.h"

namespace slm {

constexpr int kSampleThreads = 1024;

// Monotone map of a float to an unsigned key: a < b  <=>  key(a) < key(b).
__device__ __forceinline__ uint32_t order_key(float f) {
    const uint32_t b = __float_as_uint(f);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// Inclusive scan over the block's 1024 threads (warp shuffles, then the 32 warp totals).
template <typename T>
__device__ __forceinline__ T block_scan(T v, T *wsum) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const T n = __shfl_up_sync(0xffffffffu, v, off);
        if (lane >= off) v += n;
    }
    if (lane == 31) wsum[warp] = v;
    __syncthreads();
    if (warp == 0) {
        T s = wsum[lane];
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const T n = __shfl_up_sync(0xffffffffu, s, off);
            if (lane >= off) s += n;
        }
        wsum[lane] = s;
    }
    __syncthreads();
    if (warp > 0) v += wsum[warp - 1];
    __syncthreads();  // wsum is reused by the next scan
    return v;
}

// Bitonic sort of c[0, n) (n a power of two, n / 1024 entries per thread), largest first.
__device__ void bitonic_desc(unsigned long long *c, int n) {
    for (int size = 2; size <= n; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int i = threadIdx.x; i < n; i += kSampleThreads) {
                const int j = i ^ stride;
                if (j > i) {
                    const unsigned long long ci = c[i], cj = c[j];
                    const bool desc = (i & size) == 0;
                    if (desc ? (ci < cj) : (ci > cj)) {
                        c[i] = cj;
                        c[j] = ci;
                    }
                }
            }
            __syncthreads();
        }
    }
}

// The value and token of a composite key.
__device__ __forceinline__ float key_value(unsigned long long c) {
    const uint32_t k = (uint32_t)(c >> 32);
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}
__device__ __forceinline__ int key_token(unsigned long long c) { return (int)(0xffffffffu - (uint32_t)(c & 0xffffffffu)); }

// The draw from candidates sorted largest first in cand[0, k): softmax(value / T) weights,
// running sums, the top-p cut, the inverse CDF at u.  Returns the token (thread 0).
__device__ int draw_sorted(const unsigned long long *cand, int k, float temperature, float top_p, float u, float *cum,
                           float *wsum_f, int *sel) {
    const int tid = threadIdx.x;
    const float v0 = key_value(cand[0]) / temperature;
    const float w = tid < k ? expf(key_value(cand[tid]) / temperature - v0) : 0.0f;
    const float c = block_scan<float>(w, wsum_f);
    cum[tid] = c;
    if (tid == 0) sel[2] = k - 1;
    __syncthreads();
    const float Z = cum[k - 1];
    if (top_p < 1.0f && tid < k) {
        const float lim = top_p * Z;
        if (c >= lim && (tid == 0 || cum[tid - 1] < lim)) sel[2] = tid;
    }
    __syncthreads();
    const int m = sel[2];
    const float target = u * cum[m];
    if (tid == 0) sel[0] = m;
    __syncthreads();
    if (tid <= m && c > target && (tid == 0 || cum[tid - 1] <= target)) sel[0] = tid;
    __syncthreads();
    return key_token(cand[sel[0]]);
}

// The k largest entries of x[0, n) (k <= n, k <= kMaxTopK) as composite keys
// (order_key(value) << 32) | ~(base + i), sorted largest first into cand[0, k); cand[k,
// kMaxTopK) is zero.  Ties at the k-th value take the lowest indices.  All 1024 threads.
__device__ void select_topk(const float *x, int n, int base, int k, unsigned long long *cand, int *hist, int *sel,
                            int *wsum_i) {
    const int tid = threadIdx.x;
    const int per = (n + kSampleThreads - 1) / kSampleThreads;  // contiguous index range per thread
    const int lo = min(n, tid * per), hi = min(n, lo + per);
    // the k-th largest key, 8 bits at a time from the top
    uint32_t prefix = 0, mask = 0;
    int remaining = k;  // how many keys equal to the final prefix to take
    for (int d = 3; d >= 0; d--) {
        if (tid < 256) hist[tid] = 0;
        __syncthreads();
#pragma unroll 4
        for (int i = tid; i < n; i += kSampleThreads) {
            const uint32_t key = order_key(__ldg(x + i));
            if ((key & mask) == prefix) atomicAdd(&hist[(key >> (8 * d)) & 255u], 1);
        }
        __syncthreads();
        if (tid < 32) {  // the bin where the count from the top reaches `remaining`: lane l
                         // holds bins 255 - 8l .. 248 - 8l, a warp scan gives each lane the
                         // count above its bins
            const int lane = tid;
            int cnt[8], t = 0;
#pragma unroll
            for (int j = 0; j < 8; j++) {
                cnt[j] = hist[255 - 8 * lane - j];
                t += cnt[j];
            }
            int incl = t;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int nb = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += nb;
            }
            int above = incl - t;
            if (above < remaining && remaining <= incl) {
#pragma unroll
                for (int j = 0; j < 8; j++) {
                    if (above + cnt[j] >= remaining) {
                        sel[0] = 255 - 8 * lane - j;
                        sel[1] = remaining - above;
                        break;
                    }
                    above += cnt[j];
                }
            }
        }
        __syncthreads();
        prefix |= (uint32_t)sel[0] << (8 * d);
        mask |= 0xffu << (8 * d);
        remaining = sel[1];
        __syncthreads();
    }
    const uint32_t T = prefix;
    const int n_gt = k - remaining;
    // gather: keys above T, then the `remaining` lowest indices whose key is T
    int ngt = 0, neq = 0;
    for (int i = lo; i < hi; i++) {
        const uint32_t key = order_key(__ldg(x + i));
        ngt += key > T;
        neq += key == T;
    }
    int gt_off = block_scan<int>(ngt, wsum_i) - ngt;
    int eq_off = block_scan<int>(neq, wsum_i) - neq;
    for (int i = tid; i < kMaxTopK; i += kSampleThreads) cand[i] = 0ull;  // below every real entry
    __syncthreads();
    for (int i = lo; i < hi; i++) {
        const uint32_t key = order_key(__ldg(x + i));
        const unsigned long long c = ((unsigned long long)key << 32) | (0xffffffffu - (uint32_t)(base + i));
        if (key > T) {
            cand[gt_off++] = c;
        } else if (key == T) {
            if (eq_off < remaining) cand[n_gt + eq_off] = c;
            eq_off++;
        }
    }
    __syncthreads();
    int npow = 2;  // the sort only needs the k real entries (zeros pad to a power of two)
    while (npow < k) npow <<= 1;
    bitonic_desc(cand, npow);
}

__global__ void __launch_bounds__(kSampleThreads) sample_kernel(const SampleArgs a) {
    __shared__ unsigned long long cand[kMaxTopK];  // (key << 32) | (~index): sorted largest first
    __shared__ float cum[kMaxTopK];
    __shared__ int hist[256];
    __shared__ float wsum_f[32];
    __shared__ int wsum_i[32];
    __shared__ int sel[3];
    __shared__ float bestv[32];
    __shared__ int besti[32];
    const int row = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const float *x = a.logits + (size_t)row * a.ld;
    const int V = a.vocab;

    if (a.temperature == 0.0f) {  // greedy
        float bv = -INFINITY;
        int bi = 0x7fffffff;
        for (int i = tid; i < V; i += kSampleThreads) {
            const float v = __ldg(x + i);
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
            bestv[warp] = bv;
            besti[warp] = bi;
        }
        __syncthreads();
        if (tid == 0) {
            for (int w = 1; w < 32; w++)
                if (bestv[w] > bv || (bestv[w] == bv && besti[w] < bi)) {
                    bv = bestv[w];
                    bi = besti[w];
                }
            a.next_ids[row] = bi == 0x7fffffff ? 0 : bi;
        }
        return;
    }

    const float u = a.uniforms[row];
    const int per = (V + kSampleThreads - 1) / kSampleThreads;  // contiguous index range per thread
    const int lo = min(V, tid * per), hi = min(V, lo + per);

    if (a.top_k >= 1) {
        const int k = min(a.top_k, V);
        select_topk(x, V, 0, k, cand, hist, sel, wsum_i);
        const int tok = draw_sorted(cand, k, a.temperature, a.top_p, u, cum, wsum_f, sel);
        if (tid == 0) a.next_ids[row] = tok;
        return;
    }

    // the whole vocabulary in index order
    float mx = -INFINITY;
    for (int i = tid; i < V; i += kSampleThreads) mx = fmaxf(mx, __ldg(x + i));
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    if (lane == 0) bestv[warp] = mx;
    __syncthreads();
    mx = bestv[0];
    for (int w = 1; w < 32; w++) mx = fmaxf(mx, bestv[w]);
    const float vmax = mx / a.temperature;
    float s = 0.0f;
    for (int i = lo; i < hi; i++) s += expf(__ldg(x + i) / a.temperature - vmax);
    const float incl = block_scan<float>(s, wsum_f);
    cum[tid] = incl;  // range t covers [cum[t - 1], cum[t]): the ranges partition [0, Z)
    if (tid == 0) sel[0] = V - 1;
    __syncthreads();
    const float pre = tid ? cum[tid - 1] : 0.0f;
    const float target = u * cum[kSampleThreads - 1];
    if (s > 0.0f && pre <= target && target < incl) {
        float run = pre;
        int pick = hi - 1;
        for (int i = lo; i < hi; i++) {
            run += expf(__ldg(x + i) / a.temperature - vmax);
            if (run > target) {
                pick = i;
                break;
            }
        }
        sel[0] = pick;
    }
    __syncthreads();
    if (tid == 0) a.next_ids[row] = sel[0];
}

// Top-k over several CTAs per row.  Stage 1: slice s of a row (V / C logits) keeps its
// k largest entries, sorted, as composite keys; every entry of the row's top k is among
// its slice's top k.  Stage 2: one CTA per row sorts the C lists together and draws
// from the first k (the same keys, so the same order and ties as one CTA over the row).
__global__ void __launch_bounds__(kSampleThreads) topk_slice_kernel(const SampleArgs a, int C, int kq,
                                                                    unsigned long long *out) {
    __shared__ unsigned long long cand[kMaxTopK];
    __shared__ int hist[256];
    __shared__ int wsum_i[32];
    __shared__ int sel[3];
    const int sl = blockIdx.x, row = blockIdx.y, V = a.vocab;
    const int i0 = (int)((long long)V * sl / C), i1 = (int)((long long)V * (sl + 1) / C);
    select_topk(a.logits + (size_t)row * a.ld + i0, i1 - i0, i0, min(kq, i1 - i0), cand, hist, sel, wsum_i);
    for (int j = threadIdx.x; j < kq; j += kSampleThreads) out[((size_t)row * C + sl) * kq + j] = cand[j];
}

__global__ void __launch_bounds__(kSampleThreads) sample_merge_kernel(const SampleArgs a, int C, int kq, int npow,
                                                                      const unsigned long long *in) {
    extern __shared__ unsigned long long all[];  // [npow]
    __shared__ float cum[kMaxTopK];
    __shared__ float wsum_f[32];
    __shared__ int sel[3];
    const int row = blockIdx.x, total = C * kq;
    for (int j = threadIdx.x; j < npow; j += kSampleThreads) all[j] = j < total ? in[(size_t)row * total + j] : 0ull;
    __syncthreads();
    bitonic_desc(all, npow);
    const int tok = draw_sorted(all, min(a.top_k, a.vocab), a.temperature, a.top_p, a.uniforms[row], cum, wsum_f, sel);
    if (threadIdx.x == 0) a.next_ids[row] = tok;
}

cudaError_t sample_launch(const SampleArgs &a, int batch, cudaStream_t stream) {
    if (a.temperature > 0.0f && a.top_k >= 1) {
        // slices of at least max(2k, 4096) logits, at most 16, with C * k <= 4096 keys to merge
        const int k = min(a.top_k, a.vocab);
        int C = a.vocab / max(2 * k, 4096);
        C = min(C, 16);
        C = min(C, 4096 / k);
        if (C >= 2) {
            int npow = 2;
            while (npow < C * k) npow <<= 1;
            unsigned long long *buf = nullptr;
            if (cudaMallocAsync((void **)&buf, (size_t)batch * C * k * 8, stream) == cudaSuccess) {
                topk_slice_kernel<<<dim3(C, batch), kSampleThreads, 0, stream>>>(a, C, k, buf);
                sample_merge_kernel<<<batch, kSampleThreads, (size_t)npow * 8, stream>>>(a, C, k, npow, buf);
                const cudaError_t e = cudaGetLastError();
                cudaFreeAsync(buf, stream);
                return e;
            }
            cudaGetLastError();  // no scratch: one CTA per row
        }
    }
    sample_kernel<<<batch, kSampleThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace slm
