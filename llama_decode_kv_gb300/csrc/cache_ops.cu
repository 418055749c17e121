// cache_ops.cu -- operations on cached pages.
//
// Cache replication ("Inside nanochat Part 4: Understanding Inference", Batch
// Prefilling via Cache Replication) and copy on write of a shared page both copy the
// first rows of one page into another: every layer and kv head, keys and values.  A
// page's rows of one (layer, kv head) are one contiguous run of rows * head_dim
// elements (layout [layer][page][kv head][page rows][head_dim]; without paging a page
// is a whole sequence), so a copy is 2 * layers * kv heads runs, moved as 4-byte words
// (head_dim is even).
#include <cuda_runtime.h>
#include <stdint.h>

#include "slm_internal.h"

namespace slm {

__global__ void copy_kv_pages_kernel(const Model m, const PageCopies a) {
    const size_t esz = m.kv_bf16 ? 2 : 4;
    const int i = blockIdx.y;
    const size_t words = (size_t)a.rows[i] * m.head_dim * esz / 4;  // per run
    const size_t runs = (size_t)m.n_layers * m.n_kv_heads * 2;      // (layer, kv head, K or V)
    const size_t head_bytes = (size_t)m.kv_rows * m.head_dim * esz;  // one (page, kv head)
    for (size_t e = (size_t)blockIdx.x * blockDim.x + threadIdx.x; e < runs * words;
         e += (size_t)gridDim.x * blockDim.x) {
        const size_t run = e / words, w = e - run * words;
        const int is_v = (int)(run & 1);
        const size_t lg = run >> 1;
        const size_t l = lg / m.n_kv_heads, g = lg - l * m.n_kv_heads;
        uint8_t *base = is_v ? m.vc : m.kc;
        const uint32_t *s =
            (const uint32_t *)(base + (((l * m.kv_npages + a.src[i]) * m.n_kv_heads + g) * head_bytes));
        uint32_t *d = (uint32_t *)(base + (((l * m.kv_npages + a.dst[i]) * m.n_kv_heads + g) * head_bytes));
        d[w] = s[w];
    }
}

cudaError_t copy_kv_pages(const Model &m, const PageCopies &a, cudaStream_t stream) {
    if (a.n < 1) return cudaSuccess;
    const size_t esz = m.kv_bf16 ? 2 : 4;
    int most = 1;
    for (int i = 0; i < a.n; i++) most = a.rows[i] > most ? a.rows[i] : most;
    const size_t total = (size_t)most * m.head_dim * esz / 4 * m.n_layers * m.n_kv_heads * 2;
    const int threads = 256;
    size_t blocks = (total + threads - 1) / threads;
    if (blocks > 1024) blocks = 1024;
    if (blocks < 1) blocks = 1;
    copy_kv_pages_kernel<<<dim3((unsigned)blocks, (unsigned)a.n), threads, 0, stream>>>(m, a);
    return cudaGetLastError();
}

__global__ void write_kv_table_kernel(int *table, const TableWrites w) {
    for (int i = threadIdx.x; i < w.n; i += blockDim.x) table[w.idx[i]] = w.val[i];
}

cudaError_t write_kv_table(int *table, const TableWrites &w, cudaStream_t stream) {
    if (w.n < 1) return cudaSuccess;
    write_kv_table_kernel<<<1, 256, 0, stream>>>(table, w);
    return cudaGetLastError();
}

}  // namespace slm
