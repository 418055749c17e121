// attention_op.cu -- the decode-attention step on its own, behind the C ABI:
// slm_attention_workspace_bytes and slm_attention_decode (include/slm.h).
//
// Same split-K GQA kernel body as the decode step (attention.cuh), launched with one
// CTA per work item (row, kv head, chunk of positions) over caller-owned buffers.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <mutex>

#include "attention.cuh"
#include "slm_internal.h"

namespace slm {

struct AttnOpParams {
    int batch, H, KV, hd, cap, chunk;
    int ctx[kMaxBatch];
    int nchunk[kMaxBatch];
    int item_start[kMaxBatch + 1];
    const float *q;
    const uint8_t *k, *v;
    float *out;
    float *part;
    int *counters;
};

template <bool KVBF16>
__global__ void __launch_bounds__(kComputeThreads) attention_decode_kernel(const __grid_constant__ AttnOpParams P) {
    extern __shared__ __align__(16) float scratch[];
    __shared__ int flag;
    const int item = blockIdx.x;
    int b = 0;
    while (item >= P.item_start[b + 1]) b++;
    const int local = item - P.item_start[b];
    const int nc = P.nchunk[b];
    const int g = local / nc, c = local - g * nc;
    const int G = P.H / P.KV, hd = P.hd;
    const size_t rowbytes = (size_t)hd * (KVBF16 ? 2 : 4);
    AttnTask T;
    T.q = P.q + ((size_t)b * P.H + (size_t)g * G) * hd;
    T.q_ready = false;
    T.kv_bf16 = KVBF16;
    T.tail_k = T.tail_v = nullptr;
    T.tail_t = -1;
    T.pages = nullptr;
    T.page_stride = 0;
    T.page_shift = 0;
    T.page_mask = 0;
    T.stream = nullptr;
    T.stream_bytes = 0;
    T.kbase = P.k + ((size_t)b * P.KV + g) * P.cap * rowbytes;
    T.vbase = P.v + ((size_t)b * P.KV + g) * P.cap * rowbytes;
    T.out = P.out + ((size_t)b * P.H + (size_t)g * G) * hd;
    T.part = P.part + ((size_t)b * P.H + (size_t)g * G) * kMaxChunksPerSeq * (hd + 2);
    T.counter = P.counters + (size_t)b * P.KV + g;
    T.ll_part = nullptr;
    T.ll_out = nullptr;
    T.tag = 0;
    T.ncap = 0;
    T.hd = hd;
    T.G = G;
    T.t0 = c * P.chunk;
    T.t1 = min(P.ctx[b], T.t0 + P.chunk);
    T.nc = nc;
    T.c = c;
    attn_core(T, scratch, &flag);
}

// ------------------------------------------------------------------ host side

int attn_fail(int code, const char *fmt, ...) {
    char buf[256];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    set_detached_error(buf);
    return code;
}

static size_t align256(size_t v) { return (v + 255) / 256 * 256; }

size_t attn_partials_bytes(int batch, int H, int hd) {
    return align256((size_t)batch * H * kMaxChunksPerSeq * (hd + 2) * sizeof(float));
}

size_t attn_counters_bytes(int batch, int KV) { return align256((size_t)batch * KV * sizeof(int)); }

// Validate the shape and plan the split-K chunks; fills everything but the pointers.
int attn_plan(int batch, int H, int KV, int hd, int cap, int kv_dtype, const int *ctx, AttnOpParams &P) {
    if (batch < 1 || batch > kMaxBatch) return attn_fail(SLM_EINVAL, "batch %d outside [1, %d]", batch, kMaxBatch);
    if (H < 1 || KV < 1 || H % KV) return attn_fail(SLM_EINVAL, "n_heads %d must be a positive multiple of n_kv_heads %d", H, KV);
    if (hd < 8 || hd % 8 || hd > 256) return attn_fail(SLM_EINVAL, "head_dim %d must be a multiple of 8 in [8, 256]", hd);
    if (cap < 1) return attn_fail(SLM_EINVAL, "capacity %d < 1", cap);
    if (kv_dtype != SLM_F32 && kv_dtype != SLM_BF16) return attn_fail(SLM_EINVAL, "kv_dtype %d", kv_dtype);
    if (!ctx) return attn_fail(SLM_EINVAL, "ctx_len is NULL");
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return attn_fail(SLM_ECUDA, "no CUDA device");
    long long work = 0;
    int max_ctx = 1;
    for (int b = 0; b < batch; b++) {
        if (ctx[b] < 1 || ctx[b] > cap) return attn_fail(SLM_EINVAL, "ctx_len[%d] = %d outside [1, %d]", b, ctx[b], cap);
        work += (long long)ctx[b] * KV;
        max_ctx = std::max(max_ctx, ctx[b]);
    }
    long long ch = (work + 2LL * sms - 1) / (2LL * sms);
    ch = std::max<long long>(ch, kMinAttnChunk);
    ch = std::max<long long>(ch, (max_ctx + kMaxChunksPerSeq - 1) / kMaxChunksPerSeq);
    ch = (ch + 31) / 32 * 32;
    P.batch = batch;
    P.H = H;
    P.KV = KV;
    P.hd = hd;
    P.cap = cap;
    P.chunk = (int)ch;
    P.item_start[0] = 0;
    for (int b = 0; b < batch; b++) {
        P.ctx[b] = ctx[b];
        P.nchunk[b] = (int)((ctx[b] + ch - 1) / ch);
        P.item_start[b + 1] = P.item_start[b] + KV * P.nchunk[b];
    }
    return SLM_OK;
}

// Clear the arrival counters, then run one CTA per work item.
int attn_launch(const AttnOpParams &P, int kv_dtype, cudaStream_t s) {
    cudaError_t e = cudaMemsetAsync(P.counters, 0, (size_t)P.batch * P.KV * sizeof(int), s);
    if (e != cudaSuccess) return attn_fail(SLM_ECUDA, "cudaMemsetAsync: %s", cudaGetErrorString(e));
    size_t smem = (size_t)(kMaxGroupPass * P.hd + kComputeWarps * kMaxGroupPass * (P.hd + 2)) * sizeof(float);
    if (kv_dtype == SLM_BF16)
        attention_decode_kernel<true><<<P.item_start[P.batch], kComputeThreads, smem, s>>>(P);
    else
        attention_decode_kernel<false><<<P.item_start[P.batch], kComputeThreads, smem, s>>>(P);
    e = cudaGetLastError();
    if (e != cudaSuccess) return attn_fail(SLM_ECUDA, "attention launch: %s", cudaGetErrorString(e));
    return SLM_OK;
}

}  // namespace slm

using namespace slm;

extern "C" size_t slm_attention_workspace_bytes(int32_t batch, int32_t n_heads, int32_t n_kv_heads,
                                                int32_t head_dim) {
    if (batch < 1 || n_heads < 1 || n_kv_heads < 1 || head_dim < 1) return 0;
    return attn_partials_bytes(batch, n_heads, head_dim) + attn_counters_bytes(batch, n_kv_heads);
}

extern "C" int slm_attention_decode(int32_t batch, int32_t n_heads, int32_t n_kv_heads, int32_t head_dim,
                                    int32_t capacity, int32_t kv_dtype, const float *q, const void *k_cache,
                                    const void *v_cache, const int32_t *ctx_len, float *out, void *workspace,
                                    size_t workspace_bytes, void *stream) {
    AttnOpParams P{};
    int rc = attn_plan(batch, n_heads, n_kv_heads, head_dim, capacity, kv_dtype, ctx_len, P);
    if (rc) return rc;
    if (!q || !k_cache || !v_cache || !out || !workspace)
        return attn_fail(SLM_EINVAL, "q, k_cache, v_cache, out and workspace must be non-NULL");
    size_t need = slm_attention_workspace_bytes(batch, n_heads, n_kv_heads, head_dim);
    if (workspace_bytes < need)
        return attn_fail(SLM_EINVAL, "workspace of %zu bytes, %zu needed", workspace_bytes, need);
    if ((uintptr_t)workspace % 256)
        return attn_fail(SLM_EINVAL, "workspace must be 256-byte aligned");
    if (((uintptr_t)k_cache | (uintptr_t)v_cache) & 15)
        return attn_fail(SLM_EINVAL, "k_cache and v_cache must be 16-byte aligned (rows are read 16 bytes at a time)");
    P.q = q;
    P.k = (const uint8_t *)k_cache;
    P.v = (const uint8_t *)v_cache;
    P.out = out;
    P.part = (float *)workspace;
    P.counters = (int *)((uint8_t *)workspace + attn_partials_bytes(batch, n_heads, head_dim));
    return attn_launch(P, kv_dtype, (cudaStream_t)stream);
}

// ------------------------------------------------------------------ allocation-free variant
//
// For callers that cannot allocate device memory: the split-K partial states and the
// arrival counters live in one fixed array compiled into the library instead of a
// caller-provided workspace.  Every GPU that loads the library holds this array until
// the process exits.

static constexpr size_t kNoAllocScratchBytes = 4u << 20;  // 4 MiB
static __device__ __align__(256) unsigned char g_attn_scratch[kNoAllocScratchBytes];

static std::mutex g_scratch_mu;
static void *g_scratch_ptr[64];  // device address of g_attn_scratch, per device ordinal ...
static void *g_scratch_ctx[64];  // ... valid for the context it was looked up in

// The context current on this thread (the driver's cuCtxGetCurrent, reached through the
// runtime), or null.
static void *current_context() {
    using GetCurrent = int (*)(void **);
    static GetCurrent fn = [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess) {
            cudaGetLastError();
            f = nullptr;
        }
        return (GetCurrent)f;
    }();
    void *ctx = nullptr;
    if (!fn || fn(&ctx) != 0) return nullptr;
    return ctx;
}

// The host cannot use g_attn_scratch's name as a device address; look the address up
// once per device, with that device current, and again whenever the device's context
// changed since (a reset context reloads the module, and the array may move).
static int scratch_address(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return attn_fail(SLM_ECUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= 64) return attn_fail(SLM_EUNSUPPORTED, "device ordinal %d above 63", dev);
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    void *ctx = current_context();
    if (!g_scratch_ptr[dev] || !ctx || ctx != g_scratch_ctx[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_attn_scratch);
        if (e != cudaSuccess || !p)
            return attn_fail(SLM_ECUDA, "cudaGetSymbolAddress(scratch): %s", cudaGetErrorString(e));
        g_scratch_ptr[dev] = p;
        g_scratch_ctx[dev] = current_context();  // the lookup made the primary context current
    }
    *out = g_scratch_ptr[dev];
    return SLM_OK;
}

extern "C" size_t slm_attention_noalloc_max_bytes(void) { return kNoAllocScratchBytes; }

extern "C" int slm_attention_decode_noalloc(int32_t batch, int32_t n_heads, int32_t n_kv_heads, int32_t head_dim,
                                            int32_t capacity, int32_t kv_dtype, const float *q, const void *k_cache,
                                            const void *v_cache, const int32_t *ctx_len, float *out, void *stream) {
    AttnOpParams P{};
    int rc = attn_plan(batch, n_heads, n_kv_heads, head_dim, capacity, kv_dtype, ctx_len, P);
    if (rc) return rc;
    if (!q || !k_cache || !v_cache || !out)
        return attn_fail(SLM_EINVAL, "q, k_cache, v_cache and out must be non-NULL");
    if (((uintptr_t)k_cache | (uintptr_t)v_cache) & 15)
        return attn_fail(SLM_EINVAL, "k_cache and v_cache must be 16-byte aligned (rows are read 16 bytes at a time)");
    size_t need = slm_attention_workspace_bytes(batch, n_heads, n_kv_heads, head_dim);
    if (need > kNoAllocScratchBytes)
        return attn_fail(SLM_EINVAL,
                         "this shape needs %zu bytes of scratch; the fixed scratch array holds %zu "
                         "(use slm_attention_decode with a workspace)",
                         need, kNoAllocScratchBytes);
    void *scratch = nullptr;
    if ((rc = scratch_address(&scratch))) return rc;
    P.q = q;
    P.k = (const uint8_t *)k_cache;
    P.v = (const uint8_t *)v_cache;
    P.out = out;
    P.part = (float *)scratch;
    P.counters = (int *)((uint8_t *)scratch + attn_partials_bytes(batch, n_heads, head_dim));
    // attn_launch clears the arrival counters before the kernel runs; the partial
    // states need no clearing (each is written before it is read)
    return attn_launch(P, kv_dtype, (cudaStream_t)stream);
}
