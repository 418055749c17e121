// slm_api.cu -- host runtime behind the C ABI declared in include/slm.h.
//
// Owns the device copy of the weights (repacked into the K-tiled layout the decode
// kernel streams), the preallocated KV cache (kasahare 0.4.0 / simple-llm,
// "Optimisations": a pre-allocated KvSlot per head per layer), the per-step scratch,
// and the host-side sequence lengths that validate every position before launch.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <chrono>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>
#include <string>
#include <vector>

#include "kv_pages.h"
#include "prefill.cuh"
#include "slm_internal.h"

namespace slm {
cudaError_t launch_decode_step(const StepParams &P, cudaStream_t stream);
cudaError_t decode_occupancy(int weight_type, size_t smem, int *blocks_per_sm);
size_t decode_smem_bytes(int max_batch, int own_ld, int acc_bytes, int xs_bytes, int ring_slots);
cudaError_t cluster_capacity(int weight_bf16, size_t smem, int C, int *clusters);
cudaError_t cluster_kernel_attrs(int weight_bf16, size_t smem, int C);
cudaError_t launch_decode_cluster(const ClusterParams &P, size_t smem, cudaStream_t stream);
}  // namespace slm

using namespace slm;

struct slm_ctx {
    slm_config cfg{};
    int device = 0;
    int grid = 0;
    size_t smem = 0;
    int ring_slots = 0, xs_bytes = 0, xs_plan = 0, attn_stage = 0;
    int attn_chunk_min = 0;      // SLM_ATTN_CHUNK: lower bound on the split-K chunk (tests)
    int own_ld = 0, acc_bytes = 0;  // decode kernel shared-memory layout (see ring_offset)
    Model m{};
    std::vector<void *> allocs;
    std::vector<int> len;
    KvPages pages;               // the KV cache's page table (host copy) and pool
    int *d_table = nullptr;      //   device copy of the table
    uint32_t launch_seq = 0;     // exchange tag of the last launch
    unsigned long long *d_trace = nullptr;  // phase timeline, when tracing is on
    bool prefill_tc = false;     // long prompts go through the tensor-core prefill
    bool roles = false;          // CTA roles for steps of at most kRolesMaxBatch rows
    int role0[5] = {0, 0, 0, 0, 0};
    PrefillPlan plan;
    bool trace_on = false;
    int *d_tokens = nullptr;     // staging for host-provided tokens [max(max_seq, max_batch)]
    float *d_logits = nullptr;   // staging for host-requested logits [max_batch][vocab]
    int *d_ids = nullptr;        // staging for host-requested ids [max_batch]
    int *h_ids = nullptr;        // pinned
    int *h_step = nullptr;       // mapped pinned [2][kMaxBatch] + 1: host tokens, ids, the done word
    int *d_step = nullptr;       //   its device address (the kernel reads / writes it directly)
    // Single-row steps on thread-block clusters (decode_cluster.cu), when the plan allows.
    bool cl_on = false;
    ClusterParams cp{};          // the engine part (model, geometry, buffers, layout)
    size_t cl_smem = 0;
    std::string err;
};

static thread_local std::string g_create_err;

void slm::set_detached_error(const char *msg) { g_create_err = msg; }

static int fail(slm_ctx *c, int code, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    if (c)
        c->err = buf;
    else
        g_create_err = buf;
    return code;
}

#define CK(ctx, call)                                                                          \
    do {                                                                                       \
        cudaError_t e_ = (call);                                                               \
        if (e_ != cudaSuccess)                                                                 \
            return fail((ctx), SLM_ECUDA, "%s failed: %s", #call, cudaGetErrorString(e_));     \
    } while (0)

// Allocation failures can be injected for tests: SLM_FAULT_ALLOC_AFTER=n makes the
// (n+1)-th device allocation of the process fail.
static int g_alloc_calls = 0;

static int dev_alloc(slm_ctx *c, void **p, size_t bytes) {
    const char *inj = getenv("SLM_FAULT_ALLOC_AFTER");
    if (inj && g_alloc_calls++ >= atoi(inj)) return fail(c, SLM_ENOMEM, "injected allocation failure");
    cudaError_t e = cudaMalloc(p, bytes ? bytes : 16);
    if (e != cudaSuccess) {
        cudaGetLastError();
        *p = nullptr;
        return fail(c, e == cudaErrorMemoryAllocation ? SLM_ENOMEM : SLM_ECUDA,
                    "cudaMalloc(%zu) failed: %s", bytes, cudaGetErrorString(e));
    }
    c->allocs.push_back(*p);
    return SLM_OK;
}

static bool is_device_ptr(const void *p) {
    if (!p) return false;
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged;
}

// ------------------------------------------------------------------ layout planning

static size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Choose the K tiling of a [rows][K] matrix: one tile when the fp32 activation tile of
// every batch row fits in shared memory and a unit of rows fits in one ring slot;
// otherwise split K (only for residual-add epilogues, where the tiles' partial sums are
// accumulated).  A chunk (one warp's piece of work) holds whole units: enough that a
// CTA's share (of `ctas` CTAs) splits into about one chunk per warp or more, at most one
// slot and at most 8 rows (one row group of the batch-1 kernel).
static bool plan_mat(Mat &M, int rows, int K, int rows_per_unit, int wt, int max_batch,
                     bool allow_split, int ctas, size_t budget) {
    // int8 rows (KB bytes + KB / 8 bytes of scales) are whole 16-byte units, as the bulk
    // copies into the ring need, when KB is a multiple of 128
    const size_t pad = wt == kWQ8 ? 128 : kPadElems;
    for (int nkt = 1; nkt <= 64; nkt++) {
        int KB = (int)round_up((size_t)((K + nkt - 1) / nkt), pad);
        int real_nkt = (K + KB - 1) / KB;
        // batches of more than 8 rows run the tensor-core kernel: 16 rows of bf16 hi + lo
        // planes, padded by 8 elements
        size_t xs = max_batch > 8 ? (size_t)kMaxBatch * (KB + 8) * 4 : (size_t)max_batch * KB * 4;
        size_t unit_bytes = (size_t)tile_rowbytes(wt, KB) * rows_per_unit;
        // (the batch-16 tensor-core kernel pads every bf16 row in the ring by kRowPad)
        const size_t slot_unit = unit_bytes + (max_batch > 8 && wt == kWBF16 ? (size_t)kRowPad * rows_per_unit : 0);
        if (xs <= budget && slot_unit <= (size_t)kChunkBytes) {
            if (real_nkt > 1 && !allow_split) return false;
            M.rows = rows;
            M.K = K;
            M.KB = KB;
            M.KBp = KB;
            M.nkt = real_nkt;
            M.rows_per_unit = rows_per_unit;
            M.units = real_nkt * (rows / rows_per_unit);
            const int units = rows / rows_per_unit;
            const int per_cta = (units + ctas - 1) / ctas;
            const int fit = std::min((int)(kChunkBytes / slot_unit), 8 / rows_per_unit);
            // batches: at least two single rows per chunk, so that a row group reuses
            // each activation load for two rows
            const int want = (per_cta + kComputeWarps - 1) / kComputeWarps;
            const int upc = std::max(1, std::min(fit, max_batch > 1 && rows_per_unit == 1 ? std::max(2, want) : want));
            M.rows_per_chunk = upc * rows_per_unit;
            M.layer_stride = (long long)real_nkt * rows * tile_rowbytes(wt, KB);
            return true;
        }
        if (!allow_split) return false;
    }
    return false;
}

// Copy rows [r0, r0 + n) of a row-major [*, K] source into the tiled layout at row
// offset dst_row0 of a matrix with `rows` rows.
// Block-quantised int8: for each block of kQ8Block consecutive weights of a row (the
// last block of a row may be shorter), d = max|w| / 127 and q = w / d rounded to the
// nearest integer, halves away from zero (an all-zero block: d = 0, q = 0).
extern "C" int slm_quantize_q8(const float *w, int32_t rows, int32_t cols, int8_t *q, float *d) {
    if (!w || !q || !d || rows < 0 || cols < 1) return SLM_EINVAL;
    const int nb = (cols + kQ8Block - 1) / kQ8Block;
    for (int32_t r = 0; r < rows; r++) {
        const float *wr = w + (size_t)r * cols;
        for (int b = 0; b < nb; b++) {
            const int j0 = b * kQ8Block, j1 = std::min(cols, j0 + kQ8Block);
            float amax = 0.0f;
            for (int j = j0; j < j1; j++) amax = std::max(amax, std::fabs(wr[j]));
            const float scale = amax / 127.0f;
            d[(size_t)r * nb + b] = scale;
            for (int j = j0; j < j1; j++) {
                float v = scale > 0.0f ? std::round(wr[j] / scale) : 0.0f;
                v = std::min(127.0f, std::max(-127.0f, v));
                q[(size_t)r * cols + j] = (int8_t)v;
            }
        }
    }
    return SLM_OK;
}

// Copy rows [r0, r0 + n) of a row-major [*, K] source (elements of `src_esz` bytes) into
// the tiled layout of weight type wt at row offset dst_row0 of a matrix with `rows`
// rows.  int8 rows (fp32 source) are quantised here, blocks counted from column 0.
static void pack_rows(uint8_t *dst, const Mat &M, int dst_row0, const uint8_t *src, int n, int src_esz, int wt = -1) {
    if (wt < 0) wt = src_esz == 2 ? kWBF16 : kWF32;
    const size_t rb = (size_t)tile_rowbytes(wt, M.KBp);
    std::vector<int8_t> q;
    std::vector<float> d;
    if (wt == kWQ8) {
        q.resize(M.K);
        d.resize((M.K + kQ8Block - 1) / kQ8Block);
    }
    for (int r = 0; r < n; r++) {
        const uint8_t *s = src + (size_t)r * M.K * src_esz;
        if (wt == kWQ8) slm_quantize_q8((const float *)s, 1, M.K, q.data(), d.data());
        for (int kt = 0; kt < M.nkt; kt++) {
            const int k0 = kt * M.KB, kn = std::min(M.KB, M.K - k0);
            uint8_t *o = dst + ((size_t)kt * M.rows + dst_row0 + r) * rb;
            memset(o, 0, rb);
            if (wt == kWQ8) {  // KB is a multiple of kQ8Block: tiles hold whole blocks
                memcpy(o, q.data() + k0, (size_t)kn);
                const int b0 = k0 / kQ8Block, nb = (kn + kQ8Block - 1) / kQ8Block;
                memcpy(o + M.KBp, d.data() + b0, (size_t)nb * 4);
            } else {
                memcpy(o, s + (size_t)k0 * src_esz, (size_t)kn * src_esz);
            }
        }
    }
}

static float widen(const uint8_t *p, int esz, size_t i) {
    if (esz == 4) {
        float f;
        memcpy(&f, p + i * 4, 4);
        return f;
    }
    uint16_t b;
    memcpy(&b, p + i * 2, 2);
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

static bool config_ok(const slm_config *c, std::string &why) {
    char buf[256];
    if (c->dim <= 0 || c->n_layers <= 0 || c->n_heads <= 0 || c->n_kv_heads <= 0 || c->head_dim <= 0 ||
        c->hidden <= 0 || c->vocab <= 0 || c->max_seq <= 0 || c->max_batch <= 0) {
        why = "every size in the config must be positive";
        return false;
    }
    if (c->n_heads % c->n_kv_heads) {
        why = "n_heads must be a multiple of n_kv_heads";
        return false;
    }
    if (c->dim % 4) {
        snprintf(buf, sizeof buf, "dim %d must be a multiple of 4", c->dim);
        why = buf;
        return false;
    }
    if (c->head_dim % 8 || c->head_dim > 256) {
        snprintf(buf, sizeof buf, "head_dim %d must be a multiple of 8 and at most 256", c->head_dim);
        why = buf;
        return false;
    }
    if (c->kv_page_size != 0 &&
        (c->kv_page_size < 16 || c->kv_page_size > (1 << 20) || (c->kv_page_size & (c->kv_page_size - 1)))) {
        snprintf(buf, sizeof buf, "kv_page_size %d must be 0 or a power of two in [16, 2^20]", c->kv_page_size);
        why = buf;
        return false;
    }
    if (c->kv_pages < 0 || (c->kv_pages > 0 && c->kv_page_size == 0)) {
        why = "kv_pages must be >= 0, and 0 without paging";
        return false;
    }
    if (c->kv_page_size != 0 && c->kv_pages != 0 && c->kv_pages < (c->max_seq + c->kv_page_size - 1) / c->kv_page_size) {
        snprintf(buf, sizeof buf, "kv_pages %d cannot hold one sequence of max_seq %d", c->kv_pages, c->max_seq);
        why = buf;
        return false;
    }
    if (c->max_batch > kMaxBatch) {
        snprintf(buf, sizeof buf, "max_batch %d above %d", c->max_batch, kMaxBatch);
        why = buf;
        return false;
    }
    if (c->weight_dtype != SLM_F32 && c->weight_dtype != SLM_BF16 && c->weight_dtype != SLM_Q8) {
        why = "weight_dtype must be SLM_F32, SLM_BF16 or SLM_Q8";
        return false;
    }
    if (c->kv_dtype != SLM_F32 && c->kv_dtype != SLM_BF16) {
        why = "kv_dtype must be SLM_F32 or SLM_BF16";
        return false;
    }
    if (!(c->norm_eps >= 0.f) || !(c->rope_theta > 0.f) || !std::isfinite(c->rope_theta)) {
        why = "norm_eps must be >= 0 and rope_theta > 0";
        return false;
    }
    return true;
}

static size_t weight_count(const slm_config *c) {
    size_t dim = c->dim, qd = (size_t)c->n_heads * c->head_dim, kvd = (size_t)c->n_kv_heads * c->head_dim,
           hid = c->hidden;
    size_t per_layer = 2 * dim + qd * dim + 2 * kvd * dim + dim * qd + 3 * hid * dim;
    return (size_t)c->vocab * dim + (size_t)c->n_layers * per_layer + dim;
}

// ------------------------------------------------------------------ ABI

extern "C" const char *slm_status_string(int s) {
    switch (s) {
    case SLM_OK: return "ok";
    case SLM_EINVAL: return "invalid argument";
    case SLM_ENOMEM: return "out of memory";
    case SLM_ECAPACITY: return "sequence capacity (max_seq) reached";
    case SLM_EPOS: return "position does not match the sequence length";
    case SLM_ESTATE: return "sequence in the wrong state";
    case SLM_ECUDA: return "CUDA runtime error";
    case SLM_ETIMEOUT: return "a bounded device-side wait ran out";
    case SLM_EDEVICE: return "device reported a numeric fault";
    case SLM_EUNSUPPORTED: return "configuration not supported by this build";
    default: return "unknown status";
    }
}

extern "C" const char *slm_last_error(const slm_ctx *ctx) {
    return ctx ? ctx->err.c_str() : g_create_err.c_str();
}

extern "C" void slm_destroy(slm_ctx *ctx) {
    if (!ctx) return;
    cudaDeviceSynchronize();
    for (void *p : ctx->allocs) cudaFree(p);
    if (ctx->h_ids) cudaFreeHost(ctx->h_ids);
    if (ctx->h_step) cudaFreeHost(ctx->h_step);
    delete ctx;
}

// The engine's work split and shared-memory layout for `sms` CTAs (one per SM): pure
// arithmetic on the config, no device calls (slm_debug_plan runs it on the host).
static int plan_engine(slm_ctx *c, const slm_config *cfg, int sms) {
    const int wt = cfg->weight_dtype == SLM_Q8 ? kWQ8 : cfg->weight_dtype == SLM_BF16 ? kWBF16 : kWF32;
    const double esz = wt == kWQ8 ? 1.125 : wt == kWBF16 ? 2.0 : 4.0;  // stored bytes per weight
    const int dim = cfg->dim, H = cfg->n_heads, KV = cfg->n_kv_heads, hd = cfg->head_dim;
    const int hid = cfg->hidden, V = cfg->vocab, L = cfg->n_layers, B = cfg->max_batch;
    const int qd = H * hd, kvd = KV * hd, qkv_rows = qd + 2 * kvd;
    Model &m = c->m;
    m.dim = dim;
    m.n_layers = L;
    m.n_heads = H;
    m.n_kv_heads = KV;
    m.head_dim = hd;
    m.hidden = hid;
    m.vocab = V;
    m.max_seq = cfg->max_seq;
    m.max_batch = B;
    m.norm_eps = cfg->norm_eps;
    m.weight_bf16 = wt == kWBF16;
    m.weight_type = wt;
    m.x_perm = wt != kWF32;
    m.kv_bf16 = cfg->kv_dtype == SLM_BF16;
    m.wait_ns = kWaitLimitNs;
    m.fault = 0;

    // Shared memory of the decode kernel: the activation tile / attention scratch region
    // takes what this shape needs, the weight ring (8 KB slots, a multiple of 8, at
    // least 16) takes the rest.  The grid is one CTA per SM.
    c->grid = sms;
    const int grid = c->grid;
    // Roles (see StepParams): engines of small models at small batches.  CTAs
    // [role0[r], role0[r + 1]) take role r; the sizes follow each role's weight bytes.
    {
        bool ok = true;
        if (const char *e = getenv("SLM_NO_ROLES")) ok = atoi(e) == 0;
        const double b_qkv = (double)qkv_rows * dim, b_w13 = 2.0 * hid * dim, b_res = (double)dim * qd + (double)dim * hid;
        const double total = b_qkv + b_w13 + b_res;
        const int R = grid - kRoleAttnCtas;
        ok = ok && B <= kRolesMaxBatch && total * esz <= kRolesMaxLayerBytes && R >= 3;
        if (ok) {
            const int n_qkv = std::max(1, (int)std::lround(R * b_qkv / total));
            const int n_w13 = std::max(1, (int)std::lround(R * b_w13 / total));
            const int n_res = R - n_qkv - n_w13;
            ok = n_res >= 1 && (dim + n_res - 1) / n_res <= kMaxOwn;
            c->role0[0] = 0;
            c->role0[1] = n_qkv;
            c->role0[2] = n_qkv + kRoleAttnCtas;
            c->role0[3] = n_qkv + kRoleAttnCtas + n_res;
            c->role0[4] = grid;
        }
        c->roles = ok;
    }
    const int ctas_qkv = c->roles ? c->role0[1] - c->role0[0] : grid;
    const int ctas_res = c->roles ? c->role0[3] - c->role0[2] : grid;
    const int ctas_w13 = c->roles ? c->role0[4] - c->role0[3] : grid;
    // Residual rows a CTA may own: with roles the residual CTAs' share; otherwise the
    // share when up to a quarter of the CTAs are left to attention (res_cta0).
    c->own_ld = c->roles ? (dim + ctas_res - 1) / ctas_res : (dim + (grid - grid / 4) - 1) / (grid - grid / 4);
    if (c->own_ld > kMaxOwn) return fail(c, SLM_EUNSUPPORTED, "dim %d too large for %d CTAs", dim, grid);
    // The activation tile takes what a 16-slot ring leaves; the norm inputs also keep a
    // dim-long row beside it.  The residual matrices are planned first without K-tile
    // accumulators, and again with them if either has to be split.
    auto budget = [&](size_t acc) {
        return kSmemLimit - (size_t)kMinRingSlots * kChunkBytes - layout_overhead(B, c->own_ld, (int)acc);
    };
    c->acc_bytes = 0;
    bool planned = plan_mat(m.wo, dim, qd, 1, wt, B, true, ctas_res, budget(0)) &&
                   plan_mat(m.w2, dim, hid, 1, wt, B, true, ctas_res, budget(0));
    if (planned && (m.wo.nkt > 1 || m.w2.nkt > 1)) {
        c->acc_bytes = (int)acc_bytes_for(c->own_ld);
        planned = plan_mat(m.wo, dim, qd, 1, wt, B, true, ctas_res, budget(c->acc_bytes)) &&
                  plan_mat(m.w2, dim, hid, 1, wt, B, true, ctas_res, budget(c->acc_bytes));
    }
    const size_t bn = budget(c->acc_bytes) - (size_t)dim * 4;
    planned = planned && plan_mat(m.emb, V, dim, 1, wt, B, false, grid, bn) &&
              plan_mat(m.qkv, qkv_rows, dim, 2, wt, B, false, ctas_qkv, bn) &&
              plan_mat(m.w13, 2 * hid, dim, 2, wt, B, false, ctas_w13, bn);
    if (!planned)
        return fail(c, SLM_EUNSUPPORTED,
                    "activation tile of max_batch=%d rows does not fit in shared memory for this shape", B);
    m.emb.layer_stride = 0;
    {
        const int G = H / KV;
        size_t need = 0;
        // activation tile (the tensor-core kernel of batches > 8 keeps 16 padded rows)
        auto tile = [&](const Mat *M) { return B > 8 ? (size_t)kMaxBatch * (M->KBp + 8) * 4 : (size_t)B * M->KBp * 4; };
        for (const Mat *M : {&m.emb, &m.qkv, &m.w13}) need = std::max(need, tile(M) + (size_t)dim * 4);
        for (const Mat *M : {&m.wo, &m.w2}) need = std::max(need, tile(M));
        c->attn_stage = B <= 2 ? 16 * 1024 : 32 * 1024;
        if (const char *e = getenv("SLM_ATTN_STAGE"))  // tests: a smaller whole-chunk copy budget
            c->attn_stage = std::max(0, std::min(c->attn_stage, atoi(e)));
        need = std::max(need, (size_t)(kMaxGroupPass * hd + kComputeWarps * kMaxGroupPass * (hd + 2) + (G + 2) * hd) * 4 +
                                  std::max(c->attn_stage, 2 * hd * 4));  // at least the new row
        need = std::max(need, (size_t)B * grid * 2 * 4);  // argmax candidates
        c->xs_bytes = (int)round_up(need, 128);
        const size_t base = decode_smem_bytes(B, c->own_ld, c->acc_bytes, c->xs_bytes, 0);
        int slots = base < kSmemLimit ? (int)((kSmemLimit - base) / kChunkBytes) : 0;
        slots = std::min(kMaxRingSlots, slots / 8 * 8);
        if (slots < kMinRingSlots)
            return fail(c, SLM_EUNSUPPORTED, "shared memory too small: %zu B of scratch leaves %d ring slots", need, slots);
        c->ring_slots = slots;
        c->smem = decode_smem_bytes(B, c->own_ld, c->acc_bytes, c->xs_bytes, slots);
        if (const char *e = getenv("SLM_ATTN_CHUNK")) c->attn_chunk_min = std::max(0, atoi(e));
        // What the ring slots leave goes to the scratch region too: attention chunks too
        // long to copy whole stream through it (deeper per-warp rings).  The step plans
        // keep using the size the shape needs.
        c->xs_plan = c->xs_bytes;
        const size_t spare = kSmemLimit > c->smem ? (kSmemLimit - c->smem) / 128 * 128 : 0;
        c->xs_bytes += (int)spare;
        c->smem = decode_smem_bytes(B, c->own_ld, c->acc_bytes, c->xs_bytes, slots);
    }
    return SLM_OK;
}

// The cluster plan of an engine (see ClusterParams): clusters of C CTAs, `clusters` of
// them resident at once.  Pure arithmetic on the config and the engine plan; leaves
// cl_on false (with the reason in `why`) when the shape does not suit the cluster kernel.
static void plan_cluster(slm_ctx *c, int clusters, int C, std::string &why) {
    const slm_config *cfg = &c->cfg;
    const Model &m = c->m;
    c->cl_on = false;
    if (const char *e = getenv("SLM_NO_CLUSTER"))
        if (atoi(e) != 0) {
            why = "disabled by SLM_NO_CLUSTER";
            return;
        }
    if (m.weight_type == kWQ8) {
        why = "int8 weights run on the persistent kernel";
        return;
    }
    const int esz = cfg->weight_dtype == SLM_BF16 ? 2 : 4, kvesz = cfg->kv_dtype == SLM_BF16 ? 2 : 4;
    const int dim = cfg->dim, H = cfg->n_heads, KV = cfg->n_kv_heads, hd = cfg->head_dim, hid = cfg->hidden;
    const int G = H / KV, qd = H * hd, kvd = KV * hd;
    const double layer_bytes = ((double)(qd + 2 * kvd) * dim + (double)dim * qd + 3.0 * hid * dim) * esz;
    if (layer_bytes > kRolesMaxLayerBytes) {
        why = "layers too large: each phase needs every SM's bandwidth";
        return;
    }
    if (dim > 8 * kComputeThreads) {
        why = "dim above the kernel's per-thread gain registers";
        return;
    }
    if ((C != 8 && C != 16) || G > kClusterMaxG || hd > kClusterMaxHd || G * hd > kComputeThreads ||
        (size_t)G * ((cfg->max_seq + C - 1) / C) > 4 * (size_t)kComputeThreads) {
        why = "cluster size or head geometry outside the kernel's limits";
        return;
    }
    if (clusters < KV + 1) {
        why = "not enough resident clusters for one attention cluster per kv head plus an FFN cluster";
        return;
    }
    ClusterParams &P = c->cp;
    P.C = C;
    P.NA = KV;
    int NF = std::min(clusters - KV, hid);
    P.hpc = (hid + NF - 1) / NF;
    P.NF = (hid + P.hpc - 1) / P.hpc;
    P.grid = (P.NA + P.NF) * C;
    P.wo_kbp = (int)round_up((size_t)G * hd, kPadElems);
    P.w2_kbp = (int)round_up((size_t)P.hpc, kPadElems);
    // units per chunk: at most 8 rows (one row group), at most one ring slot, about one
    // chunk per warp
    auto upc = [&](int units_per_cta, int rpu, size_t rowbytes) {
        const int fit = std::min(8 / rpu, (int)(kChunkBytes / (rowbytes * rpu)));
        const int want = (units_per_cta + kComputeWarps - 1) / kComputeWarps;
        return std::max(1, std::min(fit, want));
    };
    const size_t rb_qkv = (size_t)m.qkv.KBp * esz, rb_w13 = (size_t)m.w13.KBp * esz, rb_emb = (size_t)m.emb.KBp * esz;
    const size_t rb_wo = (size_t)P.wo_kbp * esz, rb_w2 = (size_t)P.w2_kbp * esz;
    for (size_t rb : {rb_qkv * 2, rb_w13 * 2, rb_emb, rb_wo, rb_w2})
        if (rb > (size_t)kChunkBytes) {
            why = "a unit of rows exceeds one ring slot";
            return;
        }
    P.upc_qkv = upc(((G + 2) * hd / 2 + C - 1) / C, 2, rb_qkv);
    P.upc_wo = upc((dim + C - 1) / C, 1, rb_wo);
    P.upc_w13 = upc((P.hpc + C - 1) / C, 2, rb_w13);
    P.upc_w2 = upc((dim + C - 1) / C, 1, rb_w2);
    P.upc_emb = upc((cfg->vocab + P.grid - 1) / P.grid, 1, rb_emb);
    // shared memory
    const int tcap = (cfg->max_seq + C - 1) / C;
    P.stage_rows = std::min(tcap, kClusterStageMax);
    P.xs_floats = std::max({m.qkv.KBp, m.w13.KBp, m.emb.KBp, P.wo_kbp});
    size_t off = 1024;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off = round_up(off + bytes, 128);
        return (int)o;
    };
    P.off_xraw = take((size_t)dim * 4);
    P.off_xs = take((size_t)P.xs_floats * 4);
    P.off_hb = take((size_t)P.w2_kbp * 4);
    P.off_qkv = take((size_t)(G + 2) * hd * 4);
    P.off_st = take((size_t)C * G * (hd + 2) * 4);
    P.off_p = take((size_t)G * tcap * 4);
    P.off_k = take((size_t)P.stage_rows * (hd * kvesz + 16));
    P.off_v = take((size_t)P.stage_rows * (hd * kvesz + 16));
    const size_t blk = (size_t)(dim + C - 1) / C;  // Wo / W2 rows per CTA
    P.off_hop = take(std::max((size_t)P.NF * blk, (size_t)P.NA * dim) * 4);  // polled partials
    P.off_gain = take((size_t)dim * 4);
    // dot products of the largest slice (or the attention's weighted values)
    const size_t yv = std::max({(size_t)2 * (((G + 2) * hd / 2 + C - 1) / C), blk, (size_t)2 * ((P.hpc + C - 1) / C),
                                (size_t)(cfg->vocab + P.grid - 1) / P.grid, (size_t)G * hd});
    P.off_yv = take(yv * 4);
    P.off_rope = take((size_t)hd * 4);
    P.off_utab = take((size_t)2 * (((G + 2) * hd / 2 + C - 1) / C) * 4);
    P.off_ring = (int)round_up(off, 1024);
    int slots = P.off_ring < (int)kSmemLimit ? (int)((kSmemLimit - P.off_ring) / kChunkBytes) : 0;
    slots = std::min(kMaxRingSlots, slots / 8 * 8);
    if (slots < 8) {
        why = "shared memory leaves fewer than 8 ring slots";
        return;
    }
    P.ring_slots = slots;
    c->cl_smem = (size_t)P.off_ring + (size_t)slots * kChunkBytes;
    c->cl_on = true;
}

static int create_impl(slm_ctx *c, const slm_config *cfg, const void *weights, size_t nbytes) {
    std::string why;
    if (!config_ok(cfg, why)) return fail(c, SLM_EINVAL, "bad config: %s", why.c_str());
    const int esz = cfg->weight_dtype == SLM_BF16 ? 2 : 4;  // of the caller's weights (int8: fp32 in)
    const size_t n_w = weight_count(cfg);
    if (nbytes != n_w * esz)
        return fail(c, SLM_EINVAL, "weights are %zu bytes, the config needs %zu", nbytes, n_w * esz);
    c->cfg = *cfg;
    CK(c, cudaGetDevice(&c->device));
    int sms = 0;
    CK(c, cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, c->device));
    int coop = 0;
    CK(c, cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, c->device));
    if (!coop) return fail(c, SLM_EUNSUPPORTED, "device lacks cooperative launch");
    int rc = plan_engine(c, cfg, sms);
    if (rc) return rc;
    const int dim = cfg->dim, H = cfg->n_heads, KV = cfg->n_kv_heads, hd = cfg->head_dim;
    const int hid = cfg->hidden, V = cfg->vocab, L = cfg->n_layers, B = cfg->max_batch;
    const int qd = H * hd, kvd = KV * hd, qkv_rows = qd + 2 * kvd;
    Model &m = c->m;
    const int grid = c->grid;
    (void)qkv_rows;
    (void)grid;
    int per_sm = 0;
    CK(c, decode_occupancy(m.weight_type, c->smem, &per_sm));
    if (per_sm < 1) return fail(c, SLM_EUNSUPPORTED, "decode kernel does not fit on an SM (%zu B smem)", c->smem);
    {
        // clusters of 16 CTAs (measured faster at the SmolLM2 shape: less work per CTA
        // in each phase), else 8; SLM_CLUSTER_SIZE picks one
        int sizes[2] = {16, 8}, n = 2;
        if (const char *e = getenv("SLM_CLUSTER_SIZE")) {
            sizes[0] = atoi(e);
            n = 1;
        }
        std::string why;
        c->cl_on = false;
        for (int i = 0; i < n && !c->cl_on; i++) {
            int clusters = 0;
            if (cluster_capacity(m.weight_bf16, kSmemLimit, sizes[i], &clusters) == cudaSuccess)
                plan_cluster(c, clusters, sizes[i], why);
            else
                cudaGetLastError();
        }
        if (c->cl_on) CK(c, cluster_kernel_attrs(m.weight_bf16, c->cl_smem, c->cp.C));
    }

    // ---- weights: repack on the host, then one copy to the device
    std::vector<uint8_t> src;
    const uint8_t *w = (const uint8_t *)weights;
    if (is_device_ptr(weights)) {
        try {
            src.resize(nbytes);
        } catch (const std::bad_alloc &) {
            return fail(c, SLM_ENOMEM, "host staging of %zu bytes failed", nbytes);
        }
        CK(c, cudaMemcpy(src.data(), weights, nbytes, cudaMemcpyDeviceToHost));
        w = src.data();
    }
    const size_t al = 256;
    size_t off_emb = 0;
    const int wt = m.weight_type;
    size_t off_qkv = round_up(off_emb + (size_t)m.emb.nkt * V * tile_rowbytes(wt, m.emb.KBp), al);
    size_t off_wo = round_up(off_qkv + (size_t)L * m.qkv.layer_stride, al);
    size_t off_w13 = round_up(off_wo + (size_t)L * m.wo.layer_stride, al);
    size_t off_w2 = round_up(off_w13 + (size_t)L * m.w13.layer_stride, al);
    // cluster kernel copies: Wo by head group, W2 by hidden slice
    const int Gq = H / KV;
    ClusterParams &cp = c->cp;
    const long long wo_g_stride = c->cl_on ? (long long)KV * dim * cp.wo_kbp * esz : 0;
    const long long w2_c_stride = c->cl_on ? (long long)cp.NF * dim * cp.w2_kbp * esz : 0;
    size_t off_wog = round_up(off_w2 + (size_t)L * m.w2.layer_stride, al);
    size_t off_w2c = round_up(off_wog + (size_t)L * wo_g_stride, al);
    size_t off_norm = round_up(off_w2c + (size_t)L * w2_c_stride, al);
    size_t off_rope = round_up(off_norm + ((size_t)L * 2 + 1) * dim * 4, al);
    size_t total = round_up(off_rope + (size_t)cfg->max_seq * (hd / 2) * 2 * 4, al);
    std::vector<uint8_t> h;
    try {
        h.assign(total, 0);
    } catch (const std::bad_alloc &) {
        return fail(c, SLM_ENOMEM, "host staging of %zu bytes failed", total);
    }
    // walk the canonical order
    size_t cur = 0;
    auto take = [&](size_t count) {
        const uint8_t *p = w + cur * esz;
        cur += count;
        return p;
    };
    pack_rows(h.data() + off_emb, m.emb, 0, take((size_t)V * dim), V, esz, wt);
    float *norms = (float *)(h.data() + off_norm);
    for (int l = 0; l < L; l++) {
        const uint8_t *an = take(dim);
        for (int i = 0; i < dim; i++) norms[(size_t)l * 2 * dim + i] = widen(an, esz, i);
        // QKV rows grouped by kv head: [q heads g*G .. g*G+G-1; k head g; v head g], and
        // within each head in RoPE pairs: stored rows 2i, 2i + 1 = dims i, i + hd/2
        uint8_t *qkv = h.data() + off_qkv + (size_t)l * m.qkv.layer_stride;
        const uint8_t *wq = take((size_t)qd * dim), *wk = take((size_t)kvd * dim), *wv = take((size_t)kvd * dim);
        const int G = H / KV, half = hd / 2;
        auto pack_head = [&](int dst0, const uint8_t *src) {
            for (int i = 0; i < half; i++) {
                pack_rows(qkv, m.qkv, dst0 + 2 * i, src + (size_t)i * dim * esz, 1, esz, wt);
                pack_rows(qkv, m.qkv, dst0 + 2 * i + 1, src + (size_t)(i + half) * dim * esz, 1, esz, wt);
            }
        };
        for (int g = 0; g < KV; g++) {
            const int r0 = g * (G + 2) * hd;
            for (int j = 0; j < G; j++) pack_head(r0 + j * hd, wq + (size_t)(g * G + j) * hd * dim * esz);
            pack_head(r0 + G * hd, wk + (size_t)g * hd * dim * esz);
            pack_head(r0 + (G + 1) * hd, wv + (size_t)g * hd * dim * esz);
        }
        const uint8_t *wo_src = take((size_t)dim * qd);
        pack_rows(h.data() + off_wo + (size_t)l * m.wo.layer_stride, m.wo, 0, wo_src, dim, esz, wt);
        if (c->cl_on) {  // [kv head g][dim][wo_kbp]: columns g G hd .. (g + 1) G hd - 1 of Wo
            uint8_t *dst = h.data() + off_wog + (size_t)l * wo_g_stride;
            const size_t gw = (size_t)Gq * hd;
            for (int g = 0; g < KV; g++)
                for (int r = 0; r < dim; r++)
                    memcpy(dst + (((size_t)g * dim + r) * cp.wo_kbp) * esz, wo_src + ((size_t)r * qd + g * gw) * esz, gw * esz);
        }
        const uint8_t *fn = take(dim);
        for (int i = 0; i < dim; i++) norms[(size_t)l * 2 * dim + dim + i] = widen(fn, esz, i);
        const uint8_t *w1 = take((size_t)hid * dim);
        const uint8_t *w3 = take((size_t)hid * dim);
        uint8_t *w13 = h.data() + off_w13 + (size_t)l * m.w13.layer_stride;
        for (int j = 0; j < hid; j++) {  // interleave gate and up rows
            pack_rows(w13, m.w13, 2 * j, w1 + (size_t)j * dim * esz, 1, esz, wt);
            pack_rows(w13, m.w13, 2 * j + 1, w3 + (size_t)j * dim * esz, 1, esz, wt);
        }
        const uint8_t *w2_src = take((size_t)dim * hid);
        pack_rows(h.data() + off_w2 + (size_t)l * m.w2.layer_stride, m.w2, 0, w2_src, dim, esz, wt);
        if (c->cl_on) {  // [FFN cluster f][dim][w2_kbp]: columns f hpc .. (f + 1) hpc - 1 of W2
            uint8_t *dst = h.data() + off_w2c + (size_t)l * w2_c_stride;
            for (int f = 0; f < cp.NF; f++) {
                const int h0 = f * cp.hpc, n = std::min(hid, h0 + cp.hpc) - h0;
                for (int r = 0; r < dim; r++)
                    memcpy(dst + (((size_t)f * dim + r) * cp.w2_kbp) * esz, w2_src + ((size_t)r * hid + h0) * esz,
                           (size_t)n * esz);
            }
        }
    }
    const uint8_t *on = take(dim);
    for (int i = 0; i < dim; i++) norms[(size_t)L * 2 * dim + i] = widen(on, esz, i);
    if (cur != n_w) return fail(c, SLM_EINVAL, "internal: weight walk consumed %zu of %zu", cur, n_w);
    // RoPE table: angle pos * theta^(-2i/hd) in double, cos/sin rounded to fp32
    float *rope = (float *)(h.data() + off_rope);
    for (int p = 0; p < cfg->max_seq; p++)
        for (int i = 0; i < hd / 2; i++) {
            double a = (double)p * std::pow((double)cfg->rope_theta, -2.0 * i / hd);
            rope[((size_t)p * (hd / 2) + i) * 2] = (float)std::cos(a);
            rope[((size_t)p * (hd / 2) + i) * 2 + 1] = (float)std::sin(a);
        }
    void *dblock = nullptr;
    rc = dev_alloc(c, &dblock, total);
    if (rc) return rc;
    CK(c, cudaMemcpy(dblock, h.data(), total, cudaMemcpyHostToDevice));
    uint8_t *d = (uint8_t *)dblock;
    m.emb.base = d + off_emb;
    m.qkv.base = d + off_qkv;
    m.wo.base = d + off_wo;
    m.w13.base = d + off_w13;
    m.w2.base = d + off_w2;
    m.norms = (const float *)(d + off_norm);
    m.rope = (const float *)(d + off_rope);
    if (c->cl_on) {
        cp.wo_g = d + off_wog;
        cp.wo_layer_stride = wo_g_stride;
        cp.w2_c = d + off_w2c;
        cp.w2_layer_stride = w2_c_stride;
    }

    // ---- KV cache and scratch
    const size_t kvesz = m.kv_bf16 ? 2 : 4;
    KvPages &kp = c->pages;
    if (cfg->kv_page_size == 0) {
        kp.init_contiguous(B, cfg->max_seq);
    } else {
        const int pps = (cfg->max_seq + cfg->kv_page_size - 1) / cfg->kv_page_size;
        kp.init_paged(B, cfg->max_seq, cfg->kv_page_size, cfg->kv_pages ? cfg->kv_pages : B * pps);
    }
    const size_t kv_bytes = (size_t)L * kp.npages * KV * kp.rows * hd * kvesz;
    void *p;
    if ((rc = dev_alloc(c, &p, kv_bytes))) return rc;
    m.kc = (uint8_t *)p;
    if ((rc = dev_alloc(c, &p, kv_bytes))) return rc;
    m.vc = (uint8_t *)p;
    CK(c, cudaMemset(m.kc, 0, kv_bytes));
    CK(c, cudaMemset(m.vc, 0, kv_bytes));
    if ((rc = dev_alloc(c, &p, kp.table.size() * 4))) return rc;
    c->d_table = (int *)p;
    CK(c, cudaMemcpy(c->d_table, kp.table.data(), kp.table.size() * 4, cudaMemcpyHostToDevice));
    kp.clear_queue();
    m.kv_table = c->d_table;
    m.kv_pps = kp.pps;
    m.kv_shift = kp.shift;
    m.kv_mask = kp.contiguous ? 0x7fffffff : kp.rows - 1;
    m.kv_rows = kp.rows;
    m.kv_npages = kp.npages;
    const size_t Lz = L;
    struct {
        void **dst;
        size_t bytes;
    } bufs[] = {
        {(void **)&m.ll_x, (Lz + 1) * B * dim * 8},
        {(void **)&m.ll_qkv, Lz * B * qkv_rows * 8},
        {(void **)&m.ll_part, Lz * B * H * kMaxChunksA * (hd + 2) * 8},
        {(void **)&m.ll_o, Lz * B * qd * 8},
        {(void **)&m.ll_xa, Lz * B * dim * 8},
        {(void **)&m.ll_h, Lz * B * hid * 8},
        {(void **)&m.ll_amax, (size_t)B * c->grid * 2 * 8},
        {(void **)&m.part, Lz * B * H * kMaxChunksPerSeq * (hd + 2) * 4},
        {(void **)&m.part_count, Lz * B * KV * 4},
        {(void **)&m.status, 4},
        {(void **)&m.abort_flag, 4},
        {(void **)&c->d_tokens, (size_t)std::max(cfg->max_seq, B) * 4},
        {(void **)&c->d_logits, (size_t)B * V * 4},
        {(void **)&c->d_ids, (size_t)B * 4},
    };
    for (auto &b : bufs) {
        if ((rc = dev_alloc(c, b.dst, b.bytes))) return rc;
        CK(c, cudaMemset(*b.dst, 0, b.bytes));
    }
    if (c->cl_on) {
        struct {
            void **dst;
            size_t bytes;
        } cb[] = {
            {(void **)&cp.p_att, Lz * cp.NA * dim * 8},
            {(void **)&cp.p_ffn, Lz * cp.NF * dim * 8},
            {(void **)&cp.amax, 2 * 8},  // argmax: best (value, index) word, arrival count
        };
        for (auto &b : cb) {
            if ((rc = dev_alloc(c, b.dst, b.bytes))) return rc;
            CK(c, cudaMemset(*b.dst, 0, b.bytes));
        }
    }
    CK(c, cudaMallocHost((void **)&c->h_ids, (size_t)B * 4));
    // mapped [host tokens; ids; done word; the device status at the done word]
    CK(c, cudaHostAlloc((void **)&c->h_step, (size_t)(2 * kMaxBatch + 2) * 4, cudaHostAllocMapped));
    c->h_step[2 * kMaxBatch] = 0;
    c->h_step[2 * kMaxBatch + 1] = 0;
    CK(c, cudaHostGetDevicePointer((void **)&c->d_step, c->h_step, 0));
    // tensor-core prefill buffers (blocks of up to 2048 prompt positions)
    if (prefill_supported(m)) {
        PrefillPlan &pp = c->plan;
        // blocks of up to 8,192 prompt positions: one block holds the 16 x 512 batched
        // prefill (measured 24.3 -> 11.4 ms against 1,024-position blocks: every launch
        // of a block is latency-bound, so fewer, larger launches win)
        const int rows = (int)std::min<long long>(8192, (long long)cfg->max_seq * cfg->max_batch);
        struct {
            void **dst;
            size_t bytes;
        } pb[] = {
            {(void **)&pp.x, (size_t)rows * dim * 4},        {(void **)&pp.xn, (size_t)rows * dim * 2 * 2},
            {(void **)&pp.qkv, (size_t)rows * qkv_rows * 4}, {(void **)&pp.o, (size_t)rows * qd * 2 * 2},
            {(void **)&pp.h, (size_t)rows * hid * 2 * 2},    {(void **)&pp.logits, (size_t)B * V * 4},
        };
        for (auto &b : pb) {
            if ((rc = dev_alloc(c, b.dst, b.bytes))) return rc;
            CK(c, cudaMemset(*b.dst, 0, b.bytes));
        }
        CK(c, prefill_prepare(m, pp, rows));
        c->prefill_tc = true;
    }
    c->len.assign(B, 0);
    CK(c, cudaDeviceSynchronize());
    return SLM_OK;
}

extern "C" int slm_debug_plan(const slm_config *config, int32_t sms, int32_t *out, int32_t out_len) {
    if (!config || !out || sms < 1 || out_len < 47) {
        set_detached_error("slm_debug_plan: config, out (47 entries) and sms >= 1 are required");
        return SLM_EINVAL;
    }
    slm_ctx *c = new (std::nothrow) slm_ctx();
    if (!c) return SLM_ENOMEM;
    std::string why;
    int rc;
    if (!config_ok(config, why)) {
        rc = fail(c, SLM_EINVAL, "bad config: %s", why.c_str());
    } else {
        c->cfg = *config;
        rc = plan_engine(c, config, sms);
    }
    if (rc == SLM_OK) {
        int k = 0;
        out[k++] = c->grid;
        out[k++] = c->roles;
        for (int r = 0; r < 5; r++) out[k++] = c->role0[r];
        out[k++] = c->own_ld;
        out[k++] = c->acc_bytes;
        out[k++] = c->xs_bytes;
        out[k++] = c->ring_slots;
        out[k++] = (int32_t)c->smem;
        for (const Mat *M : {&c->m.emb, &c->m.qkv, &c->m.wo, &c->m.w13, &c->m.w2}) {
            out[k++] = M->rows;
            out[k++] = M->K;
            out[k++] = M->KB;
            out[k++] = M->KBp;
            out[k++] = M->nkt;
            out[k++] = M->rows_per_unit;
            out[k++] = M->rows_per_chunk;
        }
    } else {
        set_detached_error(c->err.c_str());
    }
    slm_destroy(c);
    return rc;
}

extern "C" int slm_create(const slm_config *config, const void *weights, size_t nbytes, slm_ctx **out) {
    if (!out) return fail(nullptr, SLM_EINVAL, "out is NULL");
    *out = nullptr;
    if (!config || !weights) return fail(nullptr, SLM_EINVAL, "config or weights is NULL");
    slm_ctx *c = new (std::nothrow) slm_ctx();
    if (!c) return fail(nullptr, SLM_ENOMEM, "context allocation failed");
    int rc = create_impl(c, config, weights, nbytes);
    if (rc != SLM_OK) {
        g_create_err = c->err;
        slm_destroy(c);
        return rc;
    }
    *out = c;
    return SLM_OK;
}

// Work split of this step: the engine's roles when it has them and the batch is small
// (the step is then bound by the hand-offs between phases, and a CTA that loops over
// one small piece of code keeps it in the SM's instruction cache).
static void plan_roles(const slm_ctx *c, StepParams &P) {
    P.roles = c->roles && P.batch <= kRolesMaxBatch;
    for (int r = 0; r < 5; r++) P.role0[r] = c->role0[r];
}

// Split-K geometry of the attention phase for this step: about two items per CTA (at
// most kRoleAttnCtas items when the CTAs have roles), at least kMinAttnChunk positions
// per chunk, at most kMaxChunksPerSeq chunks per row.  When every row's chunk states
// fit the Wo consumers' shared-memory tile (and at most kMaxChunksA chunks per row),
// the consumers merge them; otherwise the last CTA to finish a (row, kv head) merges
// and publishes the output.
static void plan_attention(const slm_ctx *c, StepParams &P) {
    const Model &m = c->m;
    const int KV = m.n_kv_heads, H = m.n_heads, hd = m.head_dim;
    long long work = 0;
    int max_ctx = 1;
    for (int b = 0; b < P.batch; b++) {
        work += (long long)(P.pos[b] + 1) * KV;
        max_ctx = std::max(max_ctx, P.pos[b] + 1);
    }
    plan_roles(c, P);
    long long ch;
    if (P.roles) {  // chunks so that the items fit kRoleAttnCtas CTAs
        const long long per_row = std::max(1, kRoleAttnCtas / (P.batch * KV));
        ch = (max_ctx + per_row - 1) / per_row;
    } else {
        ch = (work + 2LL * c->grid - 1) / (2LL * c->grid);
    }
    ch = std::max<long long>(ch, std::max(kMinAttnChunk, c->attn_chunk_min));
    ch = std::max<long long>(ch, (max_ctx + kMaxChunksPerSeq - 1) / kMaxChunksPerSeq);
    ch = (ch + 31) / 32 * 32;
    if (!P.roles) {
        // Item i runs on CTA i mod grid, so the phase lasts ceil(items / grid) chunks: of
        // the chunk lengths up to twice this one, take the one whose busiest CTA reads
        // the fewest positions (rounding each row up to whole chunks can leave a few CTAs
        // with one item more than the rest), and of equal ones the longest (fewer items:
        // each has its own poll, setup and partial state to merge).
        long long best = ch, best_load = -1;
        for (long long cand = ch; cand <= 2 * ch; cand += 32) {
            long long items = 0;
            for (int b = 0; b < P.batch; b++) items += (long long)KV * ((P.pos[b] + cand) / cand);
            const long long load = (items + c->grid - 1) / c->grid * cand;
            if (best_load < 0 || load <= best_load) {
                best = cand;
                best_load = load;
            }
        }
        ch = best;
    }
    // consumer merge: batch * (KBp(Wo) + H * nc * (hd + 2)) floats must fit the tile
    const long long tile = (long long)(c->xs_plan / 4) / P.batch - m.wo.KBp;
    long long nc_fit = tile > 0 ? tile / ((long long)H * (hd + 2)) : 0;
    nc_fit = std::min<long long>(nc_fit, kMaxChunksA);
    // consumers poll batch * H * nc * (hd + 2) words: beyond ~8K words the polling rounds
    // cost more than letting the last CTA of each (row, kv head) merge
    nc_fit = std::min<long long>(nc_fit, 8192 / ((long long)P.batch * H * (hd + 2)));
    P.attn_consumer_merge = 0;
    if (nc_fit >= 1 && P.batch <= 8) {  // larger batches: producer merge (the Wo tile is planes there)
        long long ch_a = std::max<long long>(ch, (max_ctx + nc_fit - 1) / nc_fit);
        ch_a = (ch_a + 31) / 32 * 32;
        if (ch_a <= 4 * std::max<long long>(ch, 128)) {
            ch = ch_a;
            P.attn_consumer_merge = 1;
        }
    }
    P.attn_chunk = (int)ch;
    P.item_start[0] = 0;
    for (int b = 0; b < P.batch; b++) {
        P.nchunk[b] = (int)((P.pos[b] + 1 + ch - 1) / ch);
        P.item_start[b + 1] = P.item_start[b] + KV * P.nchunk[b];
    }
    const int items = P.item_start[P.batch];
    if (!P.roles) {
        // The CTAs that run attention items (CTA i takes item i) finish that phase last;
        // when they are few, the Wo / W2 rows go to the others so that nobody waits for
        // them twice.
        const int rest = c->grid - items;
        P.res_cta0 = (items <= c->grid / 4 && rest > 0 && (m.dim + rest - 1) / rest <= c->own_ld) ? items : 0;
    }
}

static int launch(slm_ctx *c, StepParams &P, cudaStream_t s) {
    if (++c->launch_seq == 0) c->launch_seq = 1;  // tag 0 marks never-written words
    if (c->cl_on && P.batch == 1) {
        ClusterParams Q = c->cp;
        Q.m = c->m;
        Q.seq = P.seq[0];
        Q.pos = P.pos[0];
        Q.tokens = P.tokens;
        Q.logits = P.logits;
        Q.next_ids = P.next_ids;
        Q.done_word = P.done_word;
        Q.do_logits = P.do_logits;
        Q.tag = c->launch_seq;
        Q.trace = c->trace_on ? c->d_trace : nullptr;
        cudaError_t e = launch_decode_cluster(Q, c->cl_smem, s);
        if (e != cudaSuccess) {
            cudaGetLastError();
            return fail(c, SLM_ECUDA, "cluster decode launch failed: %s", cudaGetErrorString(e));
        }
        P.tag = Q.tag;
        return SLM_OK;
    }
    P.m = c->m;
    P.grid = c->grid;
    P.wide_groups = c->m.w13.rows_per_chunk >= 4;  // the largest layer matrix sets the group width
    P.tag = c->launch_seq;
    P.trace = c->trace_on ? c->d_trace : nullptr;
    P.ring_slots = c->ring_slots;
    P.own_ld = c->own_ld;
    P.acc_bytes = c->acc_bytes;
    P.xs_bytes = c->xs_bytes;
    P.attn_stage_bytes = c->attn_stage;
    plan_attention(c, P);
    cudaError_t e = launch_decode_step(P, s);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(c, SLM_ECUDA, "decode launch failed: %s", cudaGetErrorString(e));
    }
    return SLM_OK;
}

// After a call with host buffers has waited for its step: a nonzero device status means
// every result of the step is invalid (a bounded wait ran out, NaN logits or a bad token);
// the status stays set until slm_sync reads and clears it.
static int host_status(slm_ctx *c, uint32_t st) {
    if (st == 0) return SLM_OK;
    if (st & (kStExchangeTimeout | kStRingTimeout))
        return fail(c, SLM_ETIMEOUT, "device wait timed out (status 0x%x); results invalid until slm_sync", st);
    return fail(c, SLM_EDEVICE, "device status 0x%x (NaN logits or token out of range); results invalid until slm_sync", st);
}

static int read_status(slm_ctx *c, uint32_t *st) {
    CK(c, cudaMemcpy(st, c->m.status, 4, cudaMemcpyDeviceToHost));
    return SLM_OK;
}

// Launch the page-table writes and page copies queued on the host, in stream order
// before the kernels that read the cache.
static int flush_pages(slm_ctx *c, cudaStream_t s) {
    KvPages &kp = c->pages;
    for (size_t i = 0; i < kp.copies.size(); i += kMaxBatch) {
        PageCopies a{};
        for (size_t j = i; j < kp.copies.size() && a.n < kMaxBatch; j++, a.n++) {
            a.src[a.n] = kp.copies[j].src;
            a.dst[a.n] = kp.copies[j].dst;
            a.rows[a.n] = kp.copies[j].rows;
        }
        CK(c, copy_kv_pages(c->m, a, s));
    }
    for (size_t i = 0; i < kp.upd_idx.size(); i += kTableWritesMax) {
        TableWrites w{};
        for (size_t j = i; j < kp.upd_idx.size() && w.n < kTableWritesMax; j++, w.n++) {
            w.idx[w.n] = kp.upd_idx[j];
            w.val[w.n] = kp.upd_val[j];
        }
        CK(c, write_kv_table(c->d_table, w, s));
    }
    kp.clear_queue();
    return SLM_OK;
}

// Pages for `n` sequences to grow from lens[i] to tos[i] positions: all of them, or
// SLM_ECAPACITY and nothing taken.  Then the table and copies reach the device.
static int reserve_pages(slm_ctx *c, int n, const int *seqs, const int *lens, const int *tos, cudaStream_t s) {
    KvPages &kp = c->pages;
    if (!kp.contiguous) {
        int need = 0;
        for (int i = 0; i < n; i++) need += kp.pages_needed(seqs[i], lens[i], tos[i]);
        if (need > kp.pages_free())
            return fail(c, SLM_ECAPACITY, "KV page pool exhausted: %d pages needed, %d free of %d", need,
                        kp.pages_free(), kp.npages);
        for (int i = 0; i < n; i++) kp.prepare(seqs[i], lens[i], tos[i]);
    }
    return flush_pages(c, s);
}

extern "C" int slm_decode_step(slm_ctx *c, int32_t batch, const int32_t *seq_ids, const int32_t *tokens,
                               const int32_t *positions, float *logits, int32_t *next_ids, void *stream) {
    if (!c) return SLM_EINVAL;
    if (!seq_ids || !tokens || !positions || !next_ids)
        return fail(c, SLM_EINVAL, "seq_ids, tokens, positions and next_ids must be non-NULL");
    if (batch < 1 || batch > c->cfg.max_batch)
        return fail(c, SLM_EINVAL, "batch %d outside [1, %d]", batch, c->cfg.max_batch);
    StepParams P{};
    P.batch = batch;
    for (int i = 0; i < batch; i++) {
        int s = seq_ids[i];
        if (s < 0 || s >= c->cfg.max_batch) return fail(c, SLM_EINVAL, "seq id %d out of range", s);
        for (int j = 0; j < i; j++)
            if (seq_ids[j] == s) return fail(c, SLM_EINVAL, "seq id %d repeated in one step", s);
        if (positions[i] != c->len[s])
            return fail(c, SLM_EPOS, "row %d: position %d but sequence %d holds %d positions", i,
                        positions[i], s, c->len[s]);
        if (positions[i] >= c->cfg.max_seq)
            return fail(c, SLM_ECAPACITY, "row %d: position %d reaches max_seq %d", i, positions[i],
                        c->cfg.max_seq);
        P.seq[i] = s;
        P.pos[i] = positions[i];
    }
    cudaStream_t s = (cudaStream_t)stream;
    const bool tok_dev = is_device_ptr(tokens);
    const bool log_dev = !logits || is_device_ptr(logits);
    const bool ids_dev = is_device_ptr(next_ids);
    if (!tok_dev) {
        for (int i = 0; i < batch; i++)
            if (tokens[i] < 0 || tokens[i] >= c->cfg.vocab)
                return fail(c, SLM_EINVAL, "token %d out of range at row %d", tokens[i], i);
        // host tokens: the kernel reads them from mapped pinned memory (no copy launch);
        // every call with host buffers ends with a synchronisation, so no earlier step
        // still reads this buffer
        memcpy(c->h_step, tokens, (size_t)batch * 4);
        P.tokens = c->d_step;
    } else {
        P.tokens = tokens;
    }
    P.logits = logits ? (log_dev ? logits : c->d_logits) : nullptr;
    P.next_ids = ids_dev ? next_ids : c->d_step + kMaxBatch;  // host ids: written straight to mapped memory
    // host ids with device (or no) logits: the last CTA stamps a done word after the ids,
    // and the host waits for it instead of for the whole launch to retire
    const bool spin = !ids_dev && log_dev;
    P.done_word = spin ? (uint32_t *)(c->d_step + 2 * kMaxBatch) : nullptr;
    P.do_logits = 1;
    {
        int tos[kMaxBatch];
        for (int i = 0; i < batch; i++) tos[i] = P.pos[i] + 1;
        if (int rp = reserve_pages(c, batch, P.seq, P.pos, tos, s)) return rp;
    }
    int rc = launch(c, P, s);
    if (rc) return rc;
    for (int i = 0; i < batch; i++) c->len[P.seq[i]] = P.pos[i] + 1;
    if (!log_dev) CK(c, cudaMemcpyAsync(logits, c->d_logits, (size_t)batch * c->cfg.vocab * 4, cudaMemcpyDeviceToHost, s));
    if (spin) {
        const volatile uint32_t *done = (const volatile uint32_t *)(c->h_step + 2 * kMaxBatch);
        const auto t0 = std::chrono::steady_clock::now();
        bool seen = false;
        while (!(seen = (*done == P.tag))) {  // bounded: an aborted step falls back to the stream
            if (std::chrono::steady_clock::now() - t0 > std::chrono::seconds(3)) break;
        }
        std::atomic_thread_fence(std::memory_order_acquire);
        uint32_t st = (uint32_t)c->h_step[2 * kMaxBatch + 1];
        if (!seen) {
            CK(c, cudaStreamSynchronize(s));
            if ((rc = read_status(c, &st))) return rc;
        }
        memcpy(next_ids, c->h_step + kMaxBatch, (size_t)batch * 4);
        return host_status(c, st);
    } else if (!tok_dev || !log_dev || !ids_dev) {
        CK(c, cudaStreamSynchronize(s));
        if (!ids_dev) memcpy(next_ids, c->h_step + kMaxBatch, (size_t)batch * 4);
        uint32_t st = 0;
        if ((rc = read_status(c, &st))) return rc;
        return host_status(c, st);
    }
    return SLM_OK;
}

extern "C" int slm_prefill_batch(slm_ctx *c, int32_t nseq, const int32_t *seqs, const int32_t *lens,
                                 const int32_t *tokens, float *last_logits, int32_t *next_ids, void *stream) {
    if (!c) return SLM_EINVAL;
    if (!seqs || !lens || !tokens || !next_ids) return fail(c, SLM_EINVAL, "seqs, lens, tokens and next_ids must be non-NULL");
    if (nseq < 1 || nseq > c->cfg.max_batch) return fail(c, SLM_EINVAL, "nseq %d outside [1, %d]", nseq, c->cfg.max_batch);
    if (!is_device_ptr(tokens) || !is_device_ptr(next_ids) || (last_logits && !is_device_ptr(last_logits)))
        return fail(c, SLM_EINVAL, "tokens, last_logits and next_ids must be device memory");
    bool tc = c->prefill_tc;
    for (int i = 0; i < nseq; i++) {
        const int q = seqs[i];
        if (q < 0 || q >= c->cfg.max_batch) return fail(c, SLM_EINVAL, "seq %d out of range", q);
        for (int j = 0; j < i; j++)
            if (seqs[j] == q) return fail(c, SLM_EINVAL, "seq %d repeated", q);
        if (c->len[q] != 0) return fail(c, SLM_ESTATE, "sequence %d is not empty (%d positions)", q, c->len[q]);
        if (lens[i] < 1) return fail(c, SLM_EINVAL, "prompt length %d < 1", lens[i]);
        if (lens[i] > c->cfg.max_seq)
            return fail(c, SLM_ECAPACITY, "prompt of %d tokens exceeds max_seq %d", lens[i], c->cfg.max_seq);
        if (lens[i] < kTensorPrefillMin) tc = false;
    }
    cudaStream_t s = (cudaStream_t)stream;
    {
        int zeros[kMaxBatch] = {0};
        if (int rp = reserve_pages(c, nseq, seqs, zeros, lens, s)) return rp;
    }
    if (tc) {
        cudaError_t e = prefill_run_batch(c->m, c->plan, nseq, seqs, lens, tokens, last_logits, next_ids, s);
        if (e != cudaSuccess) {
            cudaGetLastError();
            return fail(c, SLM_ECUDA, "batched tensor-core prefill failed: %s", cudaGetErrorString(e));
        }
        for (int i = 0; i < nseq; i++) c->len[seqs[i]] = lens[i];
        return SLM_OK;
    }
    size_t off = 0;  // short prompts or no tensor-core path: one sequence at a time
    for (int i = 0; i < nseq; i++) {
        const int rc = slm_prefill(c, seqs[i], tokens + off, lens[i],
                                   last_logits ? last_logits + (size_t)i * c->cfg.vocab : nullptr, next_ids + i, stream);
        if (rc) return rc;
        off += (size_t)lens[i];
    }
    return SLM_OK;
}

extern "C" int slm_prefill(slm_ctx *c, int32_t seq, const int32_t *tokens, int32_t n, float *last_logits,
                           int32_t *next_id, void *stream) {
    if (!c) return SLM_EINVAL;
    if (!tokens || !next_id) return fail(c, SLM_EINVAL, "tokens and next_id must be non-NULL");
    if (seq < 0 || seq >= c->cfg.max_batch) return fail(c, SLM_EINVAL, "seq %d out of range", seq);
    if (n < 1) return fail(c, SLM_EINVAL, "prompt length %d < 1", n);
    if (c->len[seq] != 0) return fail(c, SLM_ESTATE, "sequence %d is not empty (%d positions)", seq, c->len[seq]);
    if (n > c->cfg.max_seq) return fail(c, SLM_ECAPACITY, "prompt of %d tokens exceeds max_seq %d", n, c->cfg.max_seq);
    cudaStream_t s = (cudaStream_t)stream;
    const bool tok_dev = is_device_ptr(tokens);
    const bool log_dev = !last_logits || is_device_ptr(last_logits);
    const bool ids_dev = is_device_ptr(next_id);
    const int32_t *dtok = tokens;
    {
        const int zero = 0;
        if (int rp = reserve_pages(c, 1, &seq, &zero, &n, s)) return rp;
    }
    if (!tok_dev) {
        for (int i = 0; i < n; i++)
            if (tokens[i] < 0 || tokens[i] >= c->cfg.vocab)
                return fail(c, SLM_EINVAL, "token %d out of range at %d", tokens[i], i);
        CK(c, cudaMemcpyAsync(c->d_tokens, tokens, (size_t)n * 4, cudaMemcpyHostToDevice, s));
        dtok = c->d_tokens;
    }
    if (c->prefill_tc && n >= kTensorPrefillMin) {
        const bool ids_dev2 = ids_dev;
        cudaError_t e = prefill_run(c->m, c->plan, seq, dtok, n, last_logits ? (log_dev ? last_logits : c->d_logits) : nullptr,
                                    ids_dev2 ? next_id : c->d_ids, s);
        if (e != cudaSuccess) {
            cudaGetLastError();
            return fail(c, SLM_ECUDA, "tensor-core prefill failed: %s", cudaGetErrorString(e));
        }
        c->len[seq] = n;
        if (!log_dev) CK(c, cudaMemcpyAsync(last_logits, c->d_logits, (size_t)c->cfg.vocab * 4, cudaMemcpyDeviceToHost, s));
        if (!ids_dev) CK(c, cudaMemcpyAsync(c->h_ids, c->d_ids, 4, cudaMemcpyDeviceToHost, s));
        if (!tok_dev || !log_dev || !ids_dev) {
            CK(c, cudaStreamSynchronize(s));
            if (!ids_dev) *next_id = c->h_ids[0];
            uint32_t st = 0;
            if (int rs = read_status(c, &st)) return rs;
            return host_status(c, st);
        }
        return SLM_OK;
    }
    for (int p = 0; p < n; p++) {
        StepParams P{};
        P.batch = 1;
        P.seq[0] = seq;
        P.pos[0] = p;
        P.tokens = dtok + p;
        const bool last = p == n - 1;
        P.do_logits = last;
        P.logits = last && last_logits ? (log_dev ? last_logits : c->d_logits) : nullptr;
        P.next_ids = last ? (ids_dev ? next_id : c->d_ids) : nullptr;
        int rc = launch(c, P, s);
        if (rc) {
            c->len[seq] = p;
            return rc;
        }
    }
    c->len[seq] = n;
    if (!log_dev) CK(c, cudaMemcpyAsync(last_logits, c->d_logits, (size_t)c->cfg.vocab * 4, cudaMemcpyDeviceToHost, s));
    if (!ids_dev) CK(c, cudaMemcpyAsync(c->h_ids, c->d_ids, 4, cudaMemcpyDeviceToHost, s));
    if (!tok_dev || !log_dev || !ids_dev) {
        CK(c, cudaStreamSynchronize(s));
        if (!ids_dev) *next_id = c->h_ids[0];
        uint32_t st = 0;
        int rc = read_status(c, &st);
        if (rc) return rc;
        return host_status(c, st);
    }
    return SLM_OK;
}

extern "C" int slm_reset(slm_ctx *c, int32_t seq) {
    if (!c) return SLM_EINVAL;
    if (seq == -1) {
        std::fill(c->len.begin(), c->len.end(), 0);
        for (int q = 0; q < c->cfg.max_batch; q++) c->pages.release(q);
        return SLM_OK;
    }
    if (seq < 0 || seq >= c->cfg.max_batch) return fail(c, SLM_EINVAL, "seq %d out of range", seq);
    c->len[seq] = 0;
    c->pages.release(seq);
    return SLM_OK;
}

static int sample_fail(int code, const char *msg) {
    set_detached_error(msg);
    return code;
}

extern "C" int slm_sample(int32_t batch, int32_t vocab, const float *logits, int32_t ld, float temperature,
                          int32_t top_k, float top_p, const float *uniforms, int32_t *next_ids, void *stream) {
    if (batch < 1 || vocab < 1 || ld < vocab) return sample_fail(SLM_EINVAL, "slm_sample: bad batch, vocab or ld");
    if (!logits || !uniforms || !next_ids) return sample_fail(SLM_EINVAL, "slm_sample: NULL pointer");
    if (!is_device_ptr(logits) || !is_device_ptr(uniforms) || !is_device_ptr(next_ids))
        return sample_fail(SLM_EINVAL, "slm_sample: logits, uniforms and next_ids must be device memory");
    if (!(temperature >= 0.0f) || !std::isfinite(temperature))
        return sample_fail(SLM_EINVAL, "slm_sample: temperature must be finite and >= 0");
    if (top_k < 0 || top_k > kMaxTopK) return sample_fail(SLM_EINVAL, "slm_sample: top_k must be in [0, 1024]");
    if (!(top_p > 0.0f && top_p <= 1.0f)) return sample_fail(SLM_EINVAL, "slm_sample: top_p must be in (0, 1]");
    if (top_p < 1.0f && top_k < 1 && temperature > 0.0f)
        return sample_fail(SLM_EINVAL, "slm_sample: top_p < 1 needs top_k >= 1");
    SampleArgs a;
    a.logits = logits;
    a.uniforms = uniforms;
    a.next_ids = next_ids;
    a.ld = ld;
    a.vocab = vocab;
    a.top_k = top_k;
    a.temperature = temperature;
    a.top_p = top_p;
    cudaError_t e = sample_launch(a, batch, (cudaStream_t)stream);
    if (e != cudaSuccess) return sample_fail(SLM_ECUDA, cudaGetErrorString(e));
    return SLM_OK;
}

extern "C" int slm_fork(slm_ctx *c, int32_t src, int32_t n_dst, const int32_t *dst_seqs, void *stream) {
    if (!c) return SLM_EINVAL;
    if (!dst_seqs) return fail(c, SLM_EINVAL, "dst_seqs is NULL");
    const int B = c->cfg.max_batch;
    if (src < 0 || src >= B) return fail(c, SLM_EINVAL, "source sequence %d out of range", src);
    if (n_dst < 1 || n_dst > B - 1 || n_dst > kMaxBatch)
        return fail(c, SLM_EINVAL, "n_dst %d out of range [1, %d]", n_dst, B - 1);
    if (c->len[src] < 1) return fail(c, SLM_ESTATE, "source sequence %d is empty", src);
    for (int i = 0; i < n_dst; i++) {
        const int d = dst_seqs[i];
        if (d < 0 || d >= B) return fail(c, SLM_EINVAL, "destination sequence %d out of range", d);
        if (d == src) return fail(c, SLM_EINVAL, "destination %d is the source", d);
        for (int j = 0; j < i; j++)
            if (dst_seqs[j] == d) return fail(c, SLM_EINVAL, "destination %d repeated", d);
        if (c->len[d] != 0)
            return fail(c, SLM_ESTATE, "destination sequence %d is not empty (%d positions)", d, c->len[d]);
    }
    // paged: the clones share the source's pages (copied on their first write);
    // otherwise the rows are copied into each clone's own page
    for (int i = 0; i < n_dst; i++) c->pages.fork(src, dst_seqs[i], c->len[src]);
    if (int rc = flush_pages(c, (cudaStream_t)stream)) return rc;
    for (int i = 0; i < n_dst; i++) c->len[dst_seqs[i]] = c->len[src];
    return SLM_OK;
}

extern "C" int32_t slm_kv_pages_free(const slm_ctx *c) {
    if (!c) return SLM_EINVAL;
    return c->pages.contiguous ? 0 : c->pages.pages_free();
}

extern "C" int32_t slm_debug_page_table(const slm_ctx *c, int32_t seq, int32_t *out, int32_t out_len) {
    if (!c || seq < 0 || seq >= c->cfg.max_batch || (!out && out_len > 0) || out_len < 0) return SLM_EINVAL;
    const KvPages &kp = c->pages;
    const int n = std::min(out_len, kp.pps);
    for (int i = 0; i < n; i++) out[i] = kp.table[(size_t)seq * kp.pps + i];
    return kp.pps;
}

extern "C" int32_t slm_seq_len(const slm_ctx *c, int32_t seq) {
    if (!c || seq < 0 || seq >= c->cfg.max_batch) return SLM_EINVAL;
    return c->len[seq];
}

extern "C" int slm_sync(slm_ctx *c, void *stream) {
    if (!c) return SLM_EINVAL;
    CK(c, cudaStreamSynchronize((cudaStream_t)stream));
    int st = 0;
    CK(c, cudaMemcpy(&st, c->m.status, 4, cudaMemcpyDeviceToHost));
    if (st == 0) return SLM_OK;
    // clear the sticky state so that the next step starts clean
    CK(c, cudaMemset(c->m.status, 0, 4));
    CK(c, cudaMemset(c->m.abort_flag, 0, 4));
    CK(c, cudaMemset(c->m.part_count, 0, (size_t)c->cfg.n_layers * c->cfg.max_batch * c->cfg.n_kv_heads * 4));
    if (c->cl_on) CK(c, cudaMemset(c->cp.amax, 0, 2 * 8));  // an aborted step's argmax words
    CK(c, cudaDeviceSynchronize());
    if (st & (kStExchangeTimeout | kStRingTimeout))
        return fail(c, SLM_ETIMEOUT, "device wait timed out (status 0x%x)", st);
    return fail(c, SLM_EDEVICE, "device status 0x%x (NaN logits or token out of range)", st);
}

// ------------------------------------------------------------------ test hooks

__global__ void fill_kv_kernel(uint8_t *p, size_t n, float v, int bf16) {
    size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x;
    size_t stride = (size_t)gridDim.x * blockDim.x;
    if (bf16) {
        __nv_bfloat16 b = __float2bfloat16_rn(v);
        for (; i < n; i += stride) ((__nv_bfloat16 *)p)[i] = b;
    } else {
        for (; i < n; i += stride) ((float *)p)[i] = v;
    }
}

extern "C" int slm_debug_trace(slm_ctx *c, int32_t enable, unsigned long long *out_host, size_t out_len) {
    if (!c) return SLM_EINVAL;
    const size_t n = (size_t)c->grid * trace_slots(c->cfg.n_layers) * 3;
    if (enable && !c->d_trace) {
        void *p;
        int rc = dev_alloc(c, &p, n * 8);
        if (rc) return rc;
        c->d_trace = (unsigned long long *)p;
    }
    if (enable && !c->trace_on) CK(c, cudaMemset(c->d_trace, 0, n * 8));
    c->trace_on = enable != 0;
    if (out_host) {
        if (!c->d_trace) return fail(c, SLM_ESTATE, "tracing was never enabled");
        if (out_len < n) return fail(c, SLM_EINVAL, "trace needs %zu entries", n);
        CK(c, cudaDeviceSynchronize());
        CK(c, cudaMemcpy(out_host, c->d_trace, n * 8, cudaMemcpyDeviceToHost));
    }
    return (int)c->grid;
}

extern "C" int slm_debug_faults(slm_ctx *c, unsigned long long wait_ns, int32_t lost_publish) {
    if (!c) return SLM_EINVAL;
    if (lost_publish != 0 && lost_publish != 1) return fail(c, SLM_EINVAL, "lost_publish must be 0 or 1");
    c->m.wait_ns = wait_ns ? wait_ns : kWaitLimitNs;
    c->m.fault = lost_publish;
    return SLM_OK;
}

extern "C" int slm_debug_cluster(const slm_ctx *c, int32_t *out, int32_t out_len) {
    if (!c) return SLM_EINVAL;
    if (out && out_len < 12) return SLM_EINVAL;
    if (out) {
        const ClusterParams &p = c->cp;
        const int32_t v[12] = {p.C, p.NA, p.NF, p.grid, p.hpc, p.ring_slots, (int32_t)c->cl_smem,
                               p.upc_qkv, p.upc_wo, p.upc_w13, p.upc_w2, p.upc_emb};
        for (int i = 0; i < 12; i++) out[i] = c->cl_on ? v[i] : 0;
    }
    return c->cl_on ? 1 : 0;
}

extern "C" int slm_debug_fill_kv(slm_ctx *c, float value) {
    if (!c) return SLM_EINVAL;
    const slm_config &g = c->cfg;
    size_t n = (size_t)g.n_layers * c->pages.npages * g.n_kv_heads * c->pages.rows * g.head_dim;
    fill_kv_kernel<<<1024, 256>>>(c->m.kc, n, value, c->m.kv_bf16);
    fill_kv_kernel<<<1024, 256>>>(c->m.vc, n, value, c->m.kv_bf16);
    CK(c, cudaGetLastError());
    CK(c, cudaDeviceSynchronize());
    return SLM_OK;
}

extern "C" int slm_debug_copy_kv(slm_ctx *c, int32_t layer, int32_t seq, int32_t n_pos, float *k_host,
                                 float *v_host) {
    if (!c) return SLM_EINVAL;
    const slm_config &g = c->cfg;
    if (layer < 0 || layer >= g.n_layers || seq < 0 || seq >= g.max_batch)
        return fail(c, SLM_EINVAL, "layer %d / seq %d out of range", layer, seq);
    if (n_pos < -1 || n_pos > g.max_seq) return fail(c, SLM_EINVAL, "n_pos %d outside [-1, max_seq]", n_pos);
    CK(c, cudaDeviceSynchronize());
    const int n = n_pos < 0 ? c->len[seq] : n_pos, hd = g.head_dim;
    const size_t esz = c->m.kv_bf16 ? 2 : 4;
    std::vector<uint8_t> tmp((size_t)n * hd * esz + 1);
    for (int which = 0; which < 2; which++) {
        float *dst = which ? v_host : k_host;
        if (!dst) continue;
        const uint8_t *base = which ? c->m.vc : c->m.kc;
        const KvPages &kp = c->pages;
        for (int kvh = 0; kvh < g.n_kv_heads; kvh++) {
            for (int t = 0; t < n;) {  // one run per page
                const int pg = kp.table[(size_t)seq * kp.pps + (t >> kp.shift)];
                const int r0 = kp.contiguous ? t : (t & (kp.rows - 1));
                const int cnt = std::min(n - t, kp.rows - r0);
                if (pg < 0) return fail(c, SLM_ESTATE, "position %d of sequence %d has no page", t, seq);
                const size_t off = ((((size_t)layer * kp.npages + pg) * g.n_kv_heads + kvh) * kp.rows + r0) * hd * esz;
                CK(c, cudaMemcpy(tmp.data() + (size_t)t * hd * esz, base + off, (size_t)cnt * hd * esz,
                                 cudaMemcpyDeviceToHost));
                t += cnt;
            }
            float *o = dst + (size_t)kvh * n * hd;
            for (size_t i = 0; i < (size_t)n * hd; i++) o[i] = widen(tmp.data(), (int)esz, i);
        }
    }
    return n;
}
