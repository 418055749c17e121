// prefill.cuh -- tensor-core prefill (prefill.cu), used by slm_prefill for long prompts.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <vector>

#include "slm_internal.h"

namespace slm {

// Device buffers for one block of `rows` prompt positions, plus the tensor maps of the
// weights and of the GEMM activation operands.
struct PrefillPlan {
    int rows = 0;
    // GEMM activation operands are split in two bf16 parts, v = hi + lo, so that the
    // tensor cores see them to ~16 mantissa bits
    float *x = nullptr;        // [rows][dim] residual stream
    uint16_t *xn = nullptr;    // [2][rows][dim] normalised (hi, lo)
    float *qkv = nullptr;      // [rows][(H + 2 KV) hd]
    uint16_t *o = nullptr;     // [2][rows][H hd] attention output (hi, lo)
    uint16_t *h = nullptr;     // [2][rows][hidden] SwiGLU output (hi, lo)
    float *logits = nullptr;   // [max_batch][vocab] when the caller wants no logits
    std::vector<CUtensorMap> maps;  // per layer: qkv, wo, w13, w2; then the embedding (each: 64-, 128-row boxes)
    CUtensorMap xn_map, o_map, h_map, xn_lo_map, o_lo_map, h_lo_map;
};

// Shapes the tensor-core prefill handles: bf16 weights and cache, dim and H * hd
// multiples of 64, head_dim 64 or 128.
bool prefill_supported(const Model &m);

// Encode the tensor maps (buffers already allocated).
cudaError_t prefill_prepare(const Model &m, PrefillPlan &p, int rows);

// Enqueue the prefill of positions 0 .. n-1 of sequence `seq` (tokens on the device).
// Segments of one prefill block: segment k is `count` consecutive positions from pos0 of
// sequence seq, at block rows [row, row + count).
struct PfSegs {
    int n;
    int seq[kMaxBatch + 1], pos0[kMaxBatch + 1], count[kMaxBatch + 1], row[kMaxBatch + 1];
};

// Prompts of nseq empty sequences, concatenated in `tokens` (device); last_logits null or
// [nseq][vocab]; next_ids [nseq] (device).
cudaError_t prefill_run_batch(const Model &m, const PrefillPlan &p, int nseq, const int *seqs, const int *lens,
                              const int *tokens, float *last_logits, int *next_ids, cudaStream_t s);

cudaError_t prefill_run(const Model &m, const PrefillPlan &p, int seq, const int *tokens, int n, float *last_logits,
                        int *next_id, cudaStream_t s);

}  // namespace slm
