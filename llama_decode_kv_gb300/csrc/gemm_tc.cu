// gemm_tc.cu -- bf16 x bf16 -> fp32 GEMM tile on the 5th-generation tensor cores.
//
// Output tiles of 128 x BN (BN = 128, or 64 when 128-wide tiles would not fill the GPU
// once), the N index fastest; a persistent grid of at most one CTA per SM walks them
// (tile blockIdx.x, then + gridDim.x, ...).  The activation operand may come as two bf16
// parts (hi + lo, ~16 mantissa bits together): each K step then issues two MMAs into the
// same accumulator against the one weight tile.
//   warp 4 (one lane)  : TMA producer, cp.async.bulk.tensor of the A and B K-blocks
//                        (rows x 64 bf16 = one 128-byte swizzle atom wide) into a
//                        4-stage ring that runs on across tiles, completion on mbarriers;
//   warp 5 (one lane)  : tcgen05.mma.cta_group::1.kind::f16 (M 128, N BN, K 16) issuer,
//                        accumulating in one of two tensor-memory buffers (tile i in
//                        buffer i % 2); tcgen05.commit frees each stage and signals the
//                        epilogue when a tile's accumulator is complete;
//   warps 0-3          : allocate 2 BN TMEM columns, then per tile read the accumulator
//                        back with tcgen05.ld (warp w owns TMEM lanes 32w..32w+31 = tile
//                        rows), apply the fused epilogue and hand the buffer back -- so
//                        the epilogue of tile i overlaps the loads and MMAs of tile i + 1.
// Every wait is bounded (the first one to run out stops every role); TMEM is always
// freed.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <algorithm>

#include "device_common.cuh"
#include "gemm_tc.cuh"
#include "slm_internal.h"

namespace slm {

constexpr int kBM = 128, kBK = 64, kStages = 4;
constexpr int kBRows = 64;  // rows of the narrow weight (B) box, for 64-column tiles
constexpr int kTileBytes = kBM * kBK * 2;            // 16 KB per operand per stage
constexpr int kGemmThreads = 192;
constexpr int kEpiBytes = 4 * 32 * 33 * 4;             // per-warp [32][33] fp32 transpose tiles
constexpr int kGemmSmem = 1024 + kStages * 3 * kTileBytes + kEpiBytes + 256;

// ------------------------------------------------------------------ PTX wrappers

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            smem_addr(dst)),
        "l"(map), "r"(x), "r"(y), "r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, int x, int y, int z, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(
            smem_addr(dst)),
        "l"(map), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, rows 128 bytes
// apart, 8-row groups 1024 bytes apart (stride byte offset), descriptor version 1.
__device__ __forceinline__ uint64_t sdesc_sw128(const void *p) {
    const uint32_t a = smem_addr(p);
    uint64_t d = (uint64_t)((a & 0x3FFFF) >> 4);
    d |= (uint64_t)(16 >> 4) << 16;     // leading byte offset (unused with this swizzle)
    d |= (uint64_t)(1024 >> 4) << 32;   // stride byte offset
    d |= (uint64_t)1 << 46;             // version
    d |= (uint64_t)2 << 61;             // 128-byte swizzle
    return d;
}

// Instruction descriptor, kind::f16: fp32 accumulator, bf16 A and B, both K-major.
__host__ __device__ constexpr uint32_t idesc_bf16(int m, int n) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}

__device__ __forceinline__ void umma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
                 : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Bounded wait; the first wait of the CTA to run out raises *stop, and every later wait
// gives up at once, so that no role waits for work another role abandoned.
__device__ bool gemm_wait(uint64_t *bar, uint32_t parity, int *status, volatile int *stop) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (*stop) return false;
        if (global_ns() - t0 > kWaitLimitNs) {
            atomicOr(status, 1);
            *stop = 1;
            return false;
        }
    }
    return true;
}

// ------------------------------------------------------------------ the kernel

template <int BN>  // output columns per tile: 128, or 64 when 128-wide tiles would not fill the GPU
__global__ void __launch_bounds__(kGemmThreads, 1) gemm_bf16_tn_kernel(const __grid_constant__ GemmArgs g) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);  // 1024-B aligned stages
    uint8_t *sa = base;                                 // [kStages][128 rows][128 B]
    uint8_t *sl = base + kStages * kTileBytes;          // low parts of A (split operand)
    uint8_t *sb = base + 2 * kStages * kTileBytes;      // [kStages][128 rows][128 B]
    float *epi_tiles = (float *)(sb + kStages * kTileBytes);  // [4 warps][32][33]
    uint64_t *full = (uint64_t *)((uint8_t *)epi_tiles + kEpiBytes);
    uint64_t *empty = full + kStages;
    uint64_t *acc_full = empty + kStages;   // [2]: a tile's accumulator is complete
    uint64_t *acc_empty = acc_full + 2;     // [2]: the epilogue is done with a buffer
    uint32_t *tmem_slot = (uint32_t *)(acc_empty + 2);
    volatile int *stop = (volatile int *)(tmem_slot + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nk = g.K / kBK;
    const int ntn = (g.N + BN - 1) / BN, ntiles = ntn * ((g.M + kBM - 1) / kBM);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; s++) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; b++) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], 4);  // one arrival per epilogue warp
        }
        *stop = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {  // two accumulators of BN fp32 columns
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tmem_slot)),
                     "r"(2 * BN)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_wait();  // A, B and the residual come from earlier kernels (launched with launch_pdl)
    pdl_trigger();

    if (warp == 4 && lane == 0) {
        // producer: for each of this CTA's tiles, A rows m0.., B rows n0.., K block kb;
        // the stage ring runs on from one tile into the next
        uint32_t q = 0;  // K blocks issued so far
        for (int t = blockIdx.x; t < ntiles; t += gridDim.x) {
            const int m0 = (t / ntn) * kBM, n0 = (t % ntn) * BN;
            bool ok = true;
            for (int kb = 0; kb < nk; kb++, q++) {
                const int s = (int)(q % kStages);
                const uint32_t u = q / kStages;
                if (q >= (uint32_t)kStages && !gemm_wait(&empty[s], (u - 1) & 1, g.status, stop)) {
                    ok = false;
                    break;
                }
                mbar_expect_tx(&full[s], (g.a_split ? 2 : 1) * kTileBytes + BN * kBK * 2);
                tma_load_2d(sa + s * kTileBytes, &g.a_map, kb * kBK, m0, &full[s]);
                if (g.a_split) tma_load_2d(sl + s * kTileBytes, &g.a_lo_map, kb * kBK, m0, &full[s]);
                // B: one box of BN rows (the wide map for 128-column tiles)
                const CUtensorMap *bm = BN == 128 ? &g.b_map_wide : &g.b_map;
                if (g.b_tile_k > 0) {
                    const int k = kb * kBK, z = k / g.b_tile_k;
                    tma_load_3d(sb + s * kTileBytes, bm, k - z * g.b_tile_k, n0, z, &full[s]);
                } else {
                    tma_load_2d(sb + s * kTileBytes, bm, kb * kBK, n0, &full[s]);
                }
            }
            if (!ok) break;
        }
    } else if (warp == 5 && lane == 0) {
        // MMA issuer: 4 K-steps of 16 per stage; the descriptor advances 32 bytes per step
        const uint32_t idesc = idesc_bf16(kBM, BN);
        uint32_t q = 0;
        int it = 0;  // this CTA's tile count
        for (int t = blockIdx.x; t < ntiles && !*stop; t += gridDim.x, it++) {
            const int b = it & 1;
            if (it >= 2 && !gemm_wait(&acc_empty[b], ((it >> 1) - 1) & 1, g.status, stop)) break;
            tc_fence_after();
            const uint32_t acc = tmem + (uint32_t)(b * BN);
            bool ok = true;
            for (int kb = 0; kb < nk; kb++, q++) {
                const int s = (int)(q % kStages);
                const uint32_t u = q / kStages;
                if (!gemm_wait(&full[s], u & 1, g.status, stop)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint64_t ad = sdesc_sw128(sa + s * kTileBytes), bd = sdesc_sw128(sb + s * kTileBytes);
                const uint64_t ld = sdesc_sw128(sl + s * kTileBytes);
#pragma unroll
                for (int k = 0; k < kBK / 16; k++) {
                    umma_bf16(acc, ad + (uint64_t)(2 * k), bd + (uint64_t)(2 * k), idesc, (kb | k) != 0);
                    if (g.a_split) umma_bf16(acc, ld + (uint64_t)(2 * k), bd + (uint64_t)(2 * k), idesc, 1);
                }
                umma_commit(&empty[s]);
            }
            if (!ok) break;
            umma_commit(&acc_full[b]);
        }
    } else if (warp < 4) {
        // epilogue: per tile, wait for its accumulator, then 32 columns at a time; fp32
        // results go through the warp's [32][33] shared tile so that each row leaves as
        // one 128-byte run; the buffer goes back to the MMA issuer when read
        float *T = epi_tiles + warp * 32 * 33;
        const bool vec = (g.ldo & 7) == 0;
        int it = 0;
        for (int t = blockIdx.x; t < ntiles; t += gridDim.x, it++) {
            const int m0 = (t / ntn) * kBM, n0 = (t % ntn) * BN;
            const int b = it & 1;
            if (!gemm_wait(&acc_full[b], (it >> 1) & 1, g.status, stop)) break;
            __syncwarp();  // tcgen05.ld is warp-collective
            tc_fence_after();
            const int row0 = m0 + warp * 32;
            const uint32_t acc = tmem + (uint32_t)(b * BN);
            for (int c = 0; c < BN; c += 32) {
                uint32_t r[32];
                tmem_ld16(acc + ((uint32_t)(warp * 32) << 16) + (uint32_t)c, *(uint32_t(*)[16])r);
                tmem_ld16(acc + ((uint32_t)(warp * 32) << 16) + (uint32_t)(c + 16), *(uint32_t(*)[16])(r + 16));
                if (g.epi == GEMM_SWIGLU) {
                    // this lane's row: 16 outputs (gate / up pairs), bf16 hi and lo parts
                    const int row = row0 + lane;
                    if (row >= g.M) continue;
                    uint32_t hw[8], lw[8];
#pragma unroll
                    for (int j = 0; j < 16; j++) {
                        const float gt = __uint_as_float(r[2 * j]), up = __uint_as_float(r[2 * j + 1]);
                        const float h = gt / (1.0f + __expf(-gt)) * up;
                        const __nv_bfloat16 hb = __float2bfloat16_rn(h);
                        const __nv_bfloat16 lb = __float2bfloat16_rn(h - __bfloat162float(hb));
                        const uint32_t hu = *(const uint16_t *)&hb, lu = *(const uint16_t *)&lb;
                        hw[j >> 1] = (j & 1) ? (hw[j >> 1] | (hu << 16)) : hu;
                        lw[j >> 1] = (j & 1) ? (lw[j >> 1] | (lu << 16)) : lu;
                    }
                    const int o0 = (n0 + c) >> 1;  // first output column
                    uint16_t *dh = g.out_bf16 + (size_t)row * g.ldo + o0;
                    uint16_t *dl = g.out_bf16_lo ? g.out_bf16_lo + (size_t)row * g.ldo + o0 : nullptr;
                    if (vec && n0 + c + 32 <= g.N) {
                        ((uint4 *)dh)[0] = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                        ((uint4 *)dh)[1] = make_uint4(hw[4], hw[5], hw[6], hw[7]);
                        if (dl) {
                            ((uint4 *)dl)[0] = make_uint4(lw[0], lw[1], lw[2], lw[3]);
                            ((uint4 *)dl)[1] = make_uint4(lw[4], lw[5], lw[6], lw[7]);
                        }
                    } else {
                        for (int j = 0; j < 16 && n0 + c + 2 * j + 1 < g.N; j++) {
                            dh[j] = (uint16_t)(hw[j >> 1] >> (16 * (j & 1)));
                            if (dl) dl[j] = (uint16_t)(lw[j >> 1] >> (16 * (j & 1)));
                        }
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 32; j++) T[lane * 33 + j] = __uint_as_float(r[j]);
                    __syncwarp();
                    const int n = n0 + c + lane;
                    const int nrows = min(32, g.M - row0);
                    float *o = g.out_f32 + (size_t)row0 * g.ldo + n;
                    float old[32];  // the residual rows, all loads in flight before the first add
#pragma unroll
                    for (int rr = 0; rr < 32; rr++)
                        old[rr] = (g.epi == GEMM_ADD_F32 && rr < nrows && n < g.N) ? o[(size_t)rr * g.ldo] : 0.0f;
#pragma unroll
                    for (int rr = 0; rr < 32; rr++)
                        if (rr < nrows && n < g.N) o[(size_t)rr * g.ldo] = old[rr] + T[rr * 33 + lane];
                    __syncwarp();
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[b]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(2 * BN) : "memory");
    }
}

// ------------------------------------------------------------------ host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (EncodeTiledFn)p;
    }
    return fn;
}

cudaError_t make_bf16_map(CUtensorMap *map, const void *base, int rows, int cols, int ld, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return cudaErrorNotSupported;
    if (((uintptr_t)base & 15) || ((size_t)ld * 2) % 16) return cudaErrorInvalidValue;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
    cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t make_bf16_tiled_map(CUtensorMap *map, const void *base, int tiles, int rows, int tile_k, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return cudaErrorNotSupported;
    if (((uintptr_t)base & 15) || tile_k % kBK) return cudaErrorInvalidValue;
    cuuint64_t dims[3] = {(cuuint64_t)tile_k, (cuuint64_t)rows, (cuuint64_t)tiles};
    cuuint64_t strides[2] = {(cuuint64_t)tile_k * 2, (cuuint64_t)rows * tile_k * 2};
    cuuint32_t box[3] = {(cuuint32_t)kBK, (cuuint32_t)box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t gemm_bf16_tn(const GemmArgs &args, cudaStream_t stream) {
    if (args.K <= 0 || args.K % kBK || args.M <= 0 || args.N <= 0) return cudaErrorInvalidValue;
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(gemm_bf16_tn_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, kGemmSmem);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(gemm_bf16_tn_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, kGemmSmem);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    // 128-column tiles when they fill the GPU at least once, else 64-column tiles (twice
    // the CTAs, each with half the MMA and B traffic)
    static int sms = 0;
    if (!sms && cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0) != cudaSuccess) return cudaErrorUnknown;
    const long long mt = (args.M + kBM - 1) / kBM;
    const long long t128 = mt * ((args.N + 127) / 128), t64 = mt * ((args.N + 63) / 64);
    if (t128 >= 148)
        return launch_pdl(gemm_bf16_tn_kernel<128>, dim3((unsigned)std::min<long long>(t128, sms)), dim3(kGemmThreads),
                          (size_t)kGemmSmem, stream, args);
    return launch_pdl(gemm_bf16_tn_kernel<64>, dim3((unsigned)std::min<long long>(t64, sms)), dim3(kGemmThreads),
                      (size_t)kGemmSmem, stream, args);
}

}  // namespace slm

// ------------------------------------------------------------------ test hook

using namespace slm;

extern "C" int slm_debug_gemm_bf16(int32_t M, int32_t N, int32_t K, const void *A, const void *B, float *C,
                                   void *stream) {
    if (M <= 0 || N <= 0 || K <= 0 || K % kBK || !A || !B || !C) {
        set_detached_error("slm_debug_gemm_bf16: M, N > 0, K a positive multiple of 64, non-NULL pointers");
        return SLM_EINVAL;
    }
    static int *status = nullptr;
    if (!status && cudaMalloc(&status, sizeof(int)) != cudaSuccess) return SLM_ENOMEM;
    GemmArgs g{};
    g.b_tile_k = 0;
    g.a_split = 0;
    if (make_bf16_map(&g.a_map, A, M, K, K, kBM) != cudaSuccess ||
        make_bf16_map(&g.b_map, B, N, K, K, kBRows) != cudaSuccess ||
        make_bf16_map(&g.b_map_wide, B, N, K, K, kBM) != cudaSuccess) {
        set_detached_error("slm_debug_gemm_bf16: tensor map encoding failed (alignment?)");
        return SLM_EINVAL;
    }
    g.M = M;
    g.N = N;
    g.K = K;
    g.epi = GEMM_STORE_F32;
    g.out_f32 = C;
    g.ldo = N;
    g.status = status;
    cudaStream_t s = (cudaStream_t)stream;
    if (cudaMemsetAsync(status, 0, sizeof(int), s) != cudaSuccess || gemm_bf16_tn(g, s) != cudaSuccess) {
        set_detached_error("slm_debug_gemm_bf16: launch failed");
        return SLM_ECUDA;
    }
    int st = 0;
    if (cudaMemcpyAsync(&st, status, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return SLM_ECUDA;
    return st ? SLM_ETIMEOUT : SLM_OK;
}
