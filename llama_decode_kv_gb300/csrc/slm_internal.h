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
constexpr int kRingSlots = 6;                         // weight ring depth per CTA
constexpr int kChunkBytes = 16384;                    // one ring slot
constexpr int kMaxBatch = 16;
constexpr int kMaxGroupPass = 4;                      // query heads per attention pass
constexpr int kMaxChunksPerSeq = 64;                  // split-K chunks per (row, kv head)
constexpr int kMinAttnChunk = 32;                     // positions
constexpr size_t kXsBudget = 120 * 1024;              // activation tile in shared memory
constexpr int kPadElems = 8;                          // K tiles are padded to 8 elements

// status word bits (device side)
constexpr int kStBarrierTimeout = 1;
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

struct Model {
    int dim, n_layers, n_heads, n_kv_heads, head_dim, hidden, vocab, max_seq, max_batch;
    float norm_eps;
    int weight_bf16;   // 1 = bf16 weights, 0 = fp32
    int kv_bf16;       // 1 = bf16 cache, 0 = fp32
    Mat emb;           // [vocab][dim], also the tied output projection
    Mat qkv;           // [(H + 2 KV) hd][dim]
    Mat wo;            // [dim][H hd]
    Mat w13;           // [2 hidden][dim], rows 2j / 2j+1 = W1 row j / W3 row j
    Mat w2;            // [dim][hidden]
    const float *norms;      // [n_layers][2][dim] (attn, ffn) then [dim] output norm
    const float *rope;       // [max_seq][head_dim/2][2] = (cos, sin)
    uint8_t *kc, *vc;        // [n_layers][max_batch][KV][max_seq][hd]
    // scratch
    float *x;          // [max_batch][dim] residual stream
    float *qkv_out;    // [max_batch][(H + 2 KV) hd]
    float *attn_out;   // [max_batch][H hd]
    float *hbuf;       // [max_batch][hidden]
    float *part;       // [max_batch][H][kMaxChunksPerSeq][hd + 2] split-K partials
    int *part_count;   // [max_batch][KV] arrival counters
    float *amax_val;   // [max_batch][grid] per-CTA argmax partials
    int *amax_idx;
    int *amax_count;   // [1]
    unsigned long long *bar;  // grid barrier counter
    int *status;       // device status word
    int *abort_flag;
};

struct StepParams {
    Model m;
    int batch;
    int seq[kMaxBatch];
    int pos[kMaxBatch];
    int item_start[kMaxBatch + 1];  // attention work items per row: KV * nchunks
    int nchunk[kMaxBatch];
    int attn_chunk;                 // positions per split-K chunk
    const int *tokens;              // device [batch]
    float *logits;                  // device [batch][vocab] or null
    int *next_ids;                  // device [batch] or null
    int do_logits;                  // 0: skip the vocabulary projection (prefill)
    unsigned long long bar_base;    // barrier counter value at launch
    int grid;
    int n_barriers;
};

// Record the error text of a failed call that has no context (slm_last_error(NULL)).
void set_detached_error(const char *msg);

// Per-CTA slice of a matrix: units [u0, u1) in tile-major order.
__host__ __device__ inline void unit_range(int units_total, int grid, int cta, int &u0, int &u1) {
    long long t = units_total;
    u0 = (int)(t * cta / grid);
    u1 = (int)(t * (cta + 1) / grid);
}

}  // namespace slm
