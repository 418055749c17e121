// cache_ops.cu -- operations on whole cached sequences.
//
// Cache replication ("Inside nanochat Part 4: Understanding Inference", Batch
// Prefilling via Cache Replication): positions [0, len) of one sequence's keys and
// values, every layer and kv head, copied into other (empty) sequences.  In the cache
// layout [layer][seq][kv head][max_seq][head_dim] each (layer, kv head) of a sequence
// is one contiguous run of len * head_dim elements, so the copy is 2 * layers * kv heads
// runs per destination, moved as 4-byte words (head_dim is even).
#include <cuda_runtime.h>
#include <stdint.h>

#include "slm_internal.h"

namespace slm {

__global__ void fork_kv_kernel(const Model m, const ForkArgs a) {
    const size_t esz = m.kv_bf16 ? 2 : 4;
    const size_t words = (size_t)a.len * m.head_dim * esz / 4;  // per run
    const size_t runs = (size_t)m.n_layers * m.n_kv_heads * 2;  // (layer, kv head, K or V)
    const int dst = a.dst[blockIdx.y];
    const size_t seq_stride = (size_t)m.n_kv_heads * m.max_seq * m.head_dim * esz;  // bytes
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < runs * words;
         i += (size_t)gridDim.x * blockDim.x) {
        const size_t run = i / words, w = i - run * words;
        const int is_v = (int)(run & 1);
        const size_t lg = run >> 1;
        const size_t l = lg / m.n_kv_heads, g = lg - l * m.n_kv_heads;
        uint8_t *base = is_v ? m.vc : m.kc;
        const size_t head = (g * m.max_seq) * m.head_dim * esz;
        const uint32_t *s = (const uint32_t *)(base + (l * m.max_batch + a.src) * seq_stride + head);
        uint32_t *d = (uint32_t *)(base + (l * m.max_batch + dst) * seq_stride + head);
        d[w] = s[w];
    }
}

cudaError_t fork_kv(const Model &m, const ForkArgs &a, int n_dst, cudaStream_t stream) {
    const size_t esz = m.kv_bf16 ? 2 : 4;
    const size_t total = (size_t)a.len * m.head_dim * esz / 4 * m.n_layers * m.n_kv_heads * 2;
    const int threads = 256;
    size_t blocks = (total + threads - 1) / threads;
    if (blocks > 1024) blocks = 1024;
    if (blocks < 1) blocks = 1;
    fork_kv_kernel<<<dim3((unsigned)blocks, (unsigned)n_dst), threads, 0, stream>>>(m, a);
    return cudaGetLastError();
}

}  // namespace slm
