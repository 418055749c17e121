// gemm_tc.cuh -- bf16 tensor-core GEMM tile for sm_103a: TMA (cp.async.bulk.tensor)
// loads into 128-byte-swizzled shared memory, tcgen05.mma with the fp32 accumulator in
// tensor memory, tcgen05.ld epilogue.  C[m][n] = sum_k A[m][k] B[n][k] (both K-major).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace slm {

// Epilogue applied to each fp32 accumulator element (row m, column n).
enum GemmEpi {
    GEMM_STORE_F32 = 0,  // out_f32[m * ldo + n] = acc
    GEMM_ADD_F32 = 1,    // out_f32[m * ldo + n] += acc          (residual add)
    GEMM_SWIGLU = 2,     // columns (2j, 2j+1) = (gate, up): h = silu(g) * u stored as bf16
                         //   hi (out_bf16) + lo (out_bf16_lo) parts at [m * ldo + j]
};

struct GemmArgs {
    CUtensorMap a_map;   // A [M][K] bf16, box 128 x 64 (the high part when a_split)
    CUtensorMap a_lo_map;  // with a_split: the low part, A = hi + lo to ~16 mantissa bits
    int a_split;
    CUtensorMap b_map;   // B [N][K] bf16, box 64 rows x 64; 3-D [tiles][N][b_tile_k] when b_tile_k > 0
    CUtensorMap b_map_wide;  // the same with boxes of 128 rows (128-column tiles load once)
    int b_tile_k;        // 0, or the K extent of each K tile of a K-tiled B (a multiple of 64)
    int M, N, K;
    int epi;
    float *out_f32;
    uint16_t *out_bf16;
    uint16_t *out_bf16_lo;
    int ldo;
    int *status;         // set to 1 if a bounded wait runs out
};

// Tensor map of a row-major [rows][cols] bf16 matrix (row stride ld elements, ld * 2 a
// multiple of 16 bytes, base 16-byte aligned), boxes of box_rows rows x 64 columns (128
// for activations, 64 for weights), 128-byte swizzle.
cudaError_t make_bf16_map(CUtensorMap *map, const void *base, int rows, int cols, int ld, int box_rows = 128);

// Tensor map of a K-tiled bf16 matrix [tiles][rows][tile_k] (tile_k a multiple of 64),
// boxes of 64 columns x box_rows rows x 1, 128-byte swizzle.
cudaError_t make_bf16_tiled_map(CUtensorMap *map, const void *base, int tiles, int rows, int tile_k, int box_rows);

// Enqueue C = A . B^T with the given epilogue.  K must be a multiple of 64.
cudaError_t gemm_bf16_tn(const GemmArgs &args, cudaStream_t stream);

}  // namespace slm
