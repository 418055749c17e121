// slm_internal.h -- device layout and launch parameters shared by the host runtime
// (slm_api.cu) and the decode kernel (decode_kernel.cu).  Not part of the public ABI.
#pragma once

#include <cstddef>
#include <cstdint>

#include "../../include/slm.h"

namespace slm {

// ---------------------------------------------------------------- launch geometry
constexpr int kComputeWarps = 8;                      // warps that do the arithmetic
constexpr int kThreads = (kComputeWarps + 1) * 32;     // + one weight-streaming warp
constexpr int kComputeThreads = kComputeWarps * 32;
constexpr int kMaxRingSlots = 32;                     // weight ring depth per CTA (a multiple
constexpr int kMinRingSlots = 16;                     //   of 8: slot s is always warp s % 8's)
constexpr int kChunkBytes = 8192;                     // one ring slot = one warp's chunk
constexpr int kMaxBatch = 16;
constexpr int kMaxGroupPass = 4;                      // query heads per attention pass
constexpr int kAttnMaxSlots = 8;                      // streamed attention: passes per warp ring
constexpr int kMaxChunksPerSeq = 64;                  // split-K chunks per (row, kv head)
constexpr int kMaxChunksA = 16;                       // chunks when consumers merge them
constexpr int kMinAttnChunk = 32;                     // positions
constexpr int kRoleAttnCtas = 16;                     // attention CTAs when CTAs have roles
constexpr int kRolesMaxBatch = 4;                     // roles only up to this batch ...
constexpr double kRolesMaxLayerBytes = 16e6;          //   ... and these weight bytes per layer
constexpr int kTensorPrefillMin = 16;                 // prompts this long use the GEMM prefill
constexpr size_t kSmemLimit = 227 * 1024;             // dynamic shared memory per CTA
constexpr int kMaxOwn = 32;                           // residual rows one CTA may own
constexpr int kPadElems = 64;                         // K tiles are padded to 64 elements
                                                      //   (one tensor-core K block)
// The batch-16 tensor-core kernel reads a chunk's rows with ldmatrix, eight rows at one
// K offset: its ring keeps rows kRowPad bytes further apart than memory does, so that
// those eight 16-byte reads fall in different bank groups (row bytes are multiples of 128).
constexpr int kRowPad = 16;

// status word bits (device side)
constexpr int kStExchangeTimeout = 1;
constexpr int kStRingTimeout = 2;
constexpr int kStNanLogits = 4;
constexpr int kStBadToken = 8;
constexpr unsigned long long kWaitLimitNs = 1000000000ull;  // 1 s per wait

// A repacked weight matrix.  Logical [rows][K] row-major; stored as nkt K-tiles,
// tile t = [rows][KBp] elements (columns t*KB .. t*KB+KB-1, zero padded to KBp),
// tiles back to back; one copy per layer, layer_stride bytes apart.
struct Mat {
    const uint8_t *base;
    long long layer_stride;  // bytes
    int rows;
    int K;
    int KB;       // logical columns per tile
    int KBp;      // stored columns per tile (multiple of kPadElems)
    int nkt;      // number of tiles
    int units;    // work units split across CTAs (rows, or row pairs for W1/W3)
    int rows_per_unit;
    int rows_per_chunk;  // multiple of rows_per_unit
};

// Weight storage types: fp32, bf16, block-quantised int8 (a stored row of a K tile is
// its KBp int8 values, then one fp32 scale per block of kQ8Block elements).
constexpr int kWF32 = 0, kWBF16 = 1, kWQ8 = 2;
constexpr int kQ8Block = 32;
__host__ __device__ inline long long tile_rowbytes(int wt, int KBp) {
    return wt == kWQ8 ? (long long)KBp + (long long)(KBp / kQ8Block) * 4 : (long long)KBp * (wt == kWBF16 ? 2 : 4);
}

struct Model {
    int dim, n_layers, n_heads, n_kv_heads, head_dim, hidden, vocab, max_seq, max_batch;
    float norm_eps;
    int weight_bf16;   // 1 = bf16 weights, 0 = fp32 or int8
    int weight_type;   // kWF32, kWBF16 or kWQ8
    int x_perm;        // activation tiles in the xpos() order (8-element weight pieces)
    int kv_bf16;       // 1 = bf16 cache, 0 = fp32
    Mat emb;           // [vocab][dim], also the tied output projection
    Mat qkv;           // [(H + 2 KV) hd][dim]: per kv group g, its G q heads, k, v rows
    Mat wo;            // [dim][H hd]
    Mat w13;           // [2 hidden][dim], rows 2j / 2j+1 = W1 row j / W3 row j
    Mat w2;            // [dim][hidden]
    const float *norms;      // [n_layers][2][dim] (attn, ffn) then [dim] output norm
    const float *rope;       // [max_seq][head_dim/2][2] = (cos, sin)
    // KV cache in pages: position p of sequence s is row (p & kv_mask) of page
    // kv_table[s * kv_pps + (p >> kv_shift)]; a page holds kv_rows rows per (layer, kv
    // head): kc / vc [n_layers][kv_npages][KV][kv_rows][hd].  Without paging every
    // sequence owns one page of max_seq rows (page s, kv_shift 31), which is the plain
    // [n_layers][max_batch][KV][max_seq][hd] layout.
    uint8_t *kc, *vc;
    const int *kv_table;     // device [max_batch][kv_pps]
    int kv_pps, kv_shift, kv_mask, kv_rows, kv_npages;
    // Exchange buffers.  Every element is a tagged 8-byte word (value in the low half,
    // the launch's tag in the high half) so that consumers poll the data itself.  They
    // are per layer: nothing is rewritten within one launch.
    uint64_t *ll_x;     // [n_layers + 1][max_batch][dim]: residual entering layer l
    uint64_t *ll_qkv;   // [n_layers][max_batch][(H + 2 KV) hd]
    uint64_t *ll_part;  // [n_layers][max_batch][H][kMaxChunksA][hd + 2] chunk states
    uint64_t *ll_o;     // [n_layers][max_batch][H hd] merged attention output
    uint64_t *ll_xa;    // [n_layers][max_batch][dim]: residual after the attention block
    uint64_t *ll_h;     // [n_layers][max_batch][hidden] SwiGLU output
    uint64_t *ll_amax;  // [max_batch][grid][2] per-CTA argmax (value, index)
    float *part;        // [n_layers][max_batch][H][kMaxChunksPerSeq][hd + 2] (producer merge)
    int *part_count;    // [n_layers][max_batch][KV] arrival counters (producer merge)
    int *status;        // device status word
    int *abort_flag;
    unsigned long long wait_ns;  // limit of one bounded wait (kWaitLimitNs unless a test shortens it)
    int fault;                   // test hook: 1 = one producer skips one publish (slm_debug_faults)
};

struct StepParams {
    Model m;
    int batch;
    int seq[kMaxBatch];
    int pos[kMaxBatch];
    int item_start[kMaxBatch + 1];  // attention work items per row: KV * nchunks
    int nchunk[kMaxBatch];
    int attn_chunk;                 // positions per split-K chunk
    int attn_consumer_merge;        // 1: Wo consumers merge chunk states; 0: last CTA merges
    // How the CTAs share the work.  roles = 0: every CTA takes a slice of every matrix,
    // attention item i runs on CTA i, and Wo / W2 rows (the residual) go to CTAs
    // [res_cta0, grid) (the attention CTAs finish that phase last).  roles = 1: each CTA
    // keeps one role for the whole step, so that it loops over one small piece of code:
    // CTAs [role0[r], role0[r + 1]) take role r = 0 QKV rows, 1 attention items, 2 the
    // residual rows (Wo and W2), 3 W1/W3 pairs; all CTAs share the logits.
    int res_cta0;
    int roles;
    int role0[5];
    int wide_groups;                // batch 1: row groups of up to 8 rows (else 2)
    const int *tokens;              // device [batch]
    float *logits;                  // device [batch][vocab] or null
    int *next_ids;                  // device [batch] or null
    uint32_t *done_word;            // null, or mapped host word set to `tag` once next_ids are written
    int do_logits;                  // 0: skip the vocabulary projection (prefill)
    uint32_t tag;                   // this launch's exchange tag (never 0)
    int grid;
    int ring_slots;                 // weight ring depth (multiple of 8)
    int own_ld;                     // residual rows a CTA may own (xown row length)
    int acc_bytes;                  // K-tile accumulators (0: no residual matrix is K-split)
    int xs_bytes;                   // activation tile / scratch region
    int attn_stage_bytes;           // K + V chunk copy budget within it
    unsigned long long *trace;      // null, or [grid][trace_slots][3] phase timestamps
};

// Phase timeline of one step (slm_debug_trace): per CTA and phase, three %globaltimer
// readings (ns): phase entered, inputs ready, phase done.  Phases: 5 per layer (QKV,
// attention, Wo, W1/W3, W2), then logits and argmax.
constexpr int kTracePerLayer = 5;
__host__ __device__ inline int trace_slots(int n_layers) { return kTracePerLayer * n_layers + 2; }

// Dynamic shared memory of the decode kernel, in order: barriers and small arrays
// (kSmallBytes), the activation tile / scratch (xs_bytes; at a constant offset, so that
// its addresses need no register), the residual rows the CTA owns ([max_batch][own_ld]
// floats), the K-tile accumulators (acc_bytes), the weight ring.
constexpr int kSmallBytes = ((2 * kMaxRingSlots * 8 + 3 * kComputeWarps * kMaxBatch * 4 + 16 + 127) / 128) * 128;
__host__ __device__ inline size_t own_bytes(int max_batch, int own_ld) {
    return ((size_t)max_batch * own_ld * 4 + 127) / 128 * 128;
}
__host__ __device__ inline size_t acc_bytes_for(int own_ld) { return ((size_t)own_ld * kMaxBatch * 4 + 127) / 128 * 128; }
__host__ __device__ inline size_t own_offset(int xs_bytes) { return kSmallBytes + ((size_t)xs_bytes + 127) / 128 * 128; }
// Bytes before the activation tile plus what follows it up to the ring.
__host__ __device__ inline size_t layout_overhead(int max_batch, int own_ld, int acc_bytes) {
    return kSmallBytes + own_bytes(max_batch, own_ld) + (size_t)acc_bytes;
}
__host__ __device__ inline size_t ring_offset(int max_batch, int own_ld, int acc_bytes, int xs_bytes) {
    return (own_offset(xs_bytes) + own_bytes(max_batch, own_ld) + (size_t)acc_bytes + 1023) / 1024 * 1024;
}

// ------------------------------------------------------------------ cluster decode kernel
// Single-row steps of small models run on thread-block clusters (decode_cluster.cu):
// clusters [0, NA) are attention clusters, one per kv head (its query heads' QKV rows,
// RoPE, append, attention over the cached positions split across the cluster, Wo as a
// split-K partial over the head group's columns); clusters [NA, NA + NF) are FFN
// clusters, each owning a slice of the hidden units (W1/W3 rows, SwiGLU, W2 as a split-K
// partial over the slice).  Inside a cluster, vectors move through distributed shared
// memory (st.async + mbarrier); between the two kinds of cluster, through tagged words in
// global memory.
constexpr int kClusterMax = 16;           // cluster size limit (non-portable above 8)
constexpr int kClusterMaxG = 8;           // query heads per kv head
constexpr int kClusterMaxHd = 128;        // head_dim
constexpr int kClusterStageMax = 64;      // cached positions per CTA staged in shared memory

struct ClusterParams {
    Model m;
    int C, NA, NF, grid;
    int hpc;                     // hidden units per FFN cluster: cluster c owns [c hpc, (c + 1) hpc) ∩ [0, hidden)
    // Wo by head group: [layer][kv head g][dim rows][wo_kbp] (columns g G hd .. (g + 1) G hd - 1)
    const uint8_t *wo_g;
    long long wo_layer_stride;
    int wo_kbp;
    // W2 by hidden slice: [layer][cluster c][dim rows][w2_kbp] (columns c hpc .. (c + 1) hpc - 1)
    const uint8_t *w2_c;
    long long w2_layer_stride;
    int w2_kbp;
    int upc_qkv, upc_wo, upc_w13, upc_w2, upc_emb;  // work units per ring chunk, per phase
    uint64_t *p_att;             // [n_layers][NA][dim] tagged words: attention cluster partials
    uint64_t *p_ffn;             // [n_layers][NF][dim] tagged words: FFN cluster partials
    uint64_t *amax;              // [2]: the grid's best (value, index) key and the CTAs' arrival count
    int ring_slots;
    int stage_rows;              // cached positions per CTA copied to shared memory
    int xs_floats;               // activation tile length
    // shared-memory offsets (bytes)
    int off_xraw, off_xs, off_hb, off_qkv, off_st, off_p, off_k, off_v, off_hop, off_gain, off_yv, off_rope, off_utab, off_ring;
    // the step (one row)
    int seq, pos;
    const int *tokens;
    float *logits;
    int *next_ids;
    uint32_t *done_word;
    int do_logits;
    uint32_t tag;
    unsigned long long *trace;
};

// Cache replication (cache_ops.cu): positions [0, len) of sequence src into dst[0..n).
// KV cache pages (cache_ops.cu): rows [0, rows[i]) of page src[i] copied into page dst[i],
// every layer and kv head, keys and values (a fork without paging, or a copy on write).
struct PageCopies {
    int n;
    int src[kMaxBatch], dst[kMaxBatch], rows[kMaxBatch];
};
cudaError_t copy_kv_pages(const Model &m, const PageCopies &a, cudaStream_t stream);
// Page-table entries written on the device: table[idx[i]] = val[i].
constexpr int kTableWritesMax = 256;
struct TableWrites {
    int n;
    int idx[kTableWritesMax], val[kTableWritesMax];
};
cudaError_t write_kv_table(int *table, const TableWrites &w, cudaStream_t stream);

// Next-token sampling (sampling.cu), one CTA per row.
constexpr int kMaxTopK = 1024;
struct SampleArgs {
    const float *logits;  // [batch][ld]
    const float *uniforms;  // [batch], in [0, 1)
    int *next_ids;        // [batch]
    int ld, vocab, top_k;
    float temperature, top_p;
};
cudaError_t sample_launch(const SampleArgs &a, int batch, cudaStream_t stream);

// Record the error text of a failed call that has no context (slm_last_error(NULL)).
void set_detached_error(const char *msg);

// Per-CTA slice of a matrix: units [u0, u1) in tile-major order.
__host__ __device__ inline void unit_range(int units_total, int grid, int cta, int &u0, int &u1) {
    long long t = units_total;
    u0 = (int)(t * cta / grid);
    u1 = (int)(t * (cta + 1) / grid);
}

// The slice of phase `phase` (0 QKV, 1 Wo, 2 W1/W3, 3 W2, 4 logits) for CTA cta.
__host__ __device__ inline void phase_slice(const StepParams &P, int phase, int units_total, int cta, int &u0,
                                            int &u1) {
    if (phase == 4) {
        unit_range(units_total, P.grid, cta, u0, u1);
        return;
    }
    int lo = 0, hi = P.grid;
    if (P.roles) {
        const int r = phase == 0 ? 0 : (phase == 1 || phase == 3) ? 2 : 3;
        lo = P.role0[r];
        hi = P.role0[r + 1];
    } else if (phase == 1 || phase == 3) {
        lo = P.res_cta0;
    }
    if (cta < lo || cta >= hi) {
        u0 = u1 = 0;
        return;
    }
    unit_range(units_total, hi - lo, cta - lo, u0, u1);
}

// The CTAs that run attention items: item i on CTA first + i (mod count).
__host__ __device__ inline void attention_ctas(const StepParams &P, int &first, int &count) {
    first = P.roles ? P.role0[1] : 0;
    count = P.roles ? P.role0[2] - P.role0[1] : P.grid;
}

}  // namespace slm
