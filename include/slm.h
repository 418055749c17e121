/*
 * slm.h -- C ABI of the GB300 (sm_103a) KV-cached greedy decode library for
 * LLaMA-style decoders.
 *
 * What one decode step computes (kasahare 0.4.0 / simple-llm, "Architecture"), for
 * every batch row, at the row's position pos:
 *     x = E[token]                                   (tied embedding, bf16 widened)
 *     per block:  xn = rmsnorm(x, attn_norm)
 *                 q, k, v = Wq xn, Wk xn, Wv xn       (no biases)
 *                 q, k = RoPE(q, k, pos)              (pairs (i, i + head_dim/2))
 *                 append k, v to the cache at slot pos
 *                 o = softmax(q K^T / sqrt(head_dim)) V over slots 0..pos (GQA)
 *                 x = x + Wo o
 *                 xn = rmsnorm(x, ffn_norm)
 *                 x = x + W2( silu(W1 xn) * (W3 xn) )
 *     logits = E rmsnorm(x, output_norm);  next id = argmax (lowest index on ties)
 * The KV cache keeps each position's key and value rows and reuses them for every
 * later token (GOTOken: An Inference Engine in QBasic, "About one token per second").
 *
 * Conventions for every entry point:
 *   - Return 0 (SLM_OK) or a negative SLM_E* code; nothing aborts, nothing throws.
 *     After a failure, slm_last_error() returns a one-line description.
 *   - "device" pointers are CUDA device (or managed) memory of the current device;
 *     "host" pointers are ordinary host memory.  Where a parameter says "host or
 *     device", the library checks the pointer's kind itself.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream).
 *     Work is enqueued asynchronously on it unless the call says otherwise.  Stream
 *     order holds as usual: the prefill's kernels are launched with programmatic
 *     dependent launch among themselves, and each waits for the work before it on the
 *     stream to complete before it reads or writes any memory.
 *   - A context is not thread-safe: calls on one context must not overlap.
 *   - Every device-side wait in the library's kernels is bounded in time; a wait that
 *     runs out sets the context's device status word, which slm_sync() reports as
 *     SLM_ETIMEOUT.  No kernel traps.
 */
#ifndef SLM_H
#define SLM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* element types */
enum { SLM_F32 = 0, SLM_BF16 = 1, SLM_Q8 = 2 };

/* status codes */
enum {
    SLM_OK = 0,
    SLM_EINVAL = -1,      /* bad argument or config                                  */
    SLM_ENOMEM = -2,      /* a device or pinned-host allocation failed                */
    SLM_ECAPACITY = -3,   /* a position would reach max_seq                           */
    SLM_EPOS = -4,        /* a position is not the sequence's current length          */
    SLM_ESTATE = -5,      /* the sequence is in the wrong state (prefill of non-empty) */
    SLM_ECUDA = -6,       /* a CUDA runtime call failed                               */
    SLM_ETIMEOUT = -7,    /* a bounded device-side wait ran out                       */
    SLM_EDEVICE = -8,     /* the device reported a numeric fault (NaN logits)         */
    SLM_EUNSUPPORTED = -9 /* valid config outside what this build implements          */
};

/*
 * Model shape and storage.  Field meanings follow the kasahare config blob and the
 * nanochat model config: dim, n_layers, n_heads, n_kv_heads (< n_heads for GQA, = for
 * MHA, 1 for MQA: kasahare "Architecture"), head_dim, hidden (SwiGLU width), vocab.
 * max_seq is the per-sequence cache capacity (GOTOken keeps a fixed context constant;
 * kasahare preallocates its KvSlots), max_batch the number of sequence slots.
 * Embeddings are always tied (kasahare "Optimisations").  weight_dtype: SLM_F32,
 * SLM_BF16, or SLM_Q8: block-quantised int8 (kasahare 0.4.0, "Where to go from here":
 * INT8 weights, block-quantised like GGUF), given as fp32 weights and quantised by
 * slm_create with slm_quantize_q8: every row of the embedding and of each projection
 * matrix in blocks of 32, about 1.125 bytes per weight on the device; the norm gains
 * stay fp32.  Single-row steps of int8 engines run on the persistent kernel and their
 * prompts are prefilled one position at a time.  kv_dtype: the cache element type,
 * SLM_F32 or SLM_BF16 (rounded to nearest-even on append).
 * Requirements: all counts > 0, dim a multiple of 4, n_heads % n_kv_heads == 0, head_dim a multiple of 8
 * and <= 256, max_batch <= 16, norm_eps >= 0, rope_theta > 0.  Shapes whose fp32
 * activation tile (max_batch x input width) cannot fit in shared memory give
 * SLM_EUNSUPPORTED.
 */
typedef struct {
    int32_t dim, n_layers, n_heads, n_kv_heads, head_dim, hidden, vocab, max_seq, max_batch;
    float rope_theta, norm_eps;
    int32_t weight_dtype, kv_dtype;
    /* KV cache layout.  kv_page_size = 0: every sequence slot owns max_seq positions of
     * cache.  Otherwise (a power of two in [16, 2^20]) the cache is a pool of kv_pages
     * pages of kv_page_size positions (kv_pages = 0: max_batch * ceil(max_seq /
     * kv_page_size)); a sequence holds the pages its positions reach, slm_reset returns
     * them, and slm_fork's clones share their source's pages until they write into one
     * ("Inside nanochat Part 4: Understanding Inference", Continuous Batching: sequences
     * join and leave the batch).  Results do not depend on the layout. */
    int32_t kv_page_size, kv_pages;
} slm_config;

typedef struct slm_ctx slm_ctx;

/*
 * slm_create -- build a context on the current CUDA device.
 *   weights: host or device buffer of exactly `nbytes` bytes holding every tensor, in
 *     weight_dtype, in the kasahare ".sllm" order (kasahare, "On-disk model format"):
 *     token_emb[vocab*dim]; per block attn_norm[dim], wq[n_heads*head_dim*dim],
 *     wk[n_kv_heads*head_dim*dim], wv[n_kv_heads*head_dim*dim], wo[dim*n_heads*head_dim],
 *     ffn_norm[dim], w1[hidden*dim] (gate), w3[hidden*dim] (up), w2[dim*hidden];
 *     output_norm[dim].  Matrices are row-major [out][in] (GOTOken, "About one token
 *     per second": W(d, n) row-major).
 *   The library copies and repacks the weights into its own device layout, so the
 *   caller may free `weights` when the call returns (the call is synchronous).  It
 *   also allocates the KV cache for max_batch sequences of max_seq positions, all
 *   empty.  *out receives the context (NULL on failure).
 *   Errors: SLM_EINVAL (NULL pointer, bad config, nbytes mismatch), SLM_ENOMEM,
 *   SLM_ECUDA, SLM_EUNSUPPORTED.
 */
int slm_create(const slm_config *config, const void *weights, size_t nbytes, slm_ctx **out);

/*
 * slm_prefill -- process the prompt of one empty sequence, positions 0..n-1, and
 * produce the first generated token (the prompt is processed once; afterwards only
 * new tokens are processed: GOTOken, "About one token per second").
 *   seq: sequence slot in [0, max_batch); must be empty, else SLM_ESTATE (as
 *     nanochat refuses to prefill a non-empty KV cache).
 *   tokens: host or device int32[n], each in [0, vocab).  n in [1, max_seq].
 *   last_logits: NULL, or host or device float[vocab] for the last position's logits.
 *   next_id: host or device int32[1], the argmax of the last position's logits.
 *   On success the sequence length becomes n.  Asynchronous on `stream` when every
 *   pointer is device memory; synchronous otherwise.  Token ids are range-checked on
 *   the host when they are host memory, on the device (status word) otherwise.
 */
int slm_prefill(slm_ctx *ctx, int32_t seq, const int32_t *tokens, int32_t n, float *last_logits,
                int32_t *next_id, void *stream);

/*
 * slm_prefill_batch -- slm_prefill for several empty sequences in one call (the batched
 * workloads prefill B prompts before decoding them together).  The prompts' linear
 * layers run as GEMMs over all their positions at once; attention stays per sequence.
 *   seqs: host int32[nseq], distinct empty slots (else SLM_EINVAL / SLM_ESTATE);
 *     nseq in [1, max_batch].
 *   lens: host int32[nseq], each in [1, max_seq] (else SLM_EINVAL / SLM_ECAPACITY).
 *   tokens: device int32[sum of lens], the prompts concatenated in seqs order; ids out
 *     of range are recorded in the device status word (slm_sync).
 *   last_logits: NULL or device float[nseq][vocab]; next_ids: device int32[nseq].
 *   Results equal nseq slm_prefill calls.  Asynchronous on `stream`; every pointer other
 *   than seqs and lens must be device memory (else SLM_EINVAL).
 */
int slm_prefill_batch(slm_ctx *ctx, int32_t nseq, const int32_t *seqs, const int32_t *lens, const int32_t *tokens,
                      float *last_logits, int32_t *next_ids, void *stream);

/*
 * slm_decode_step -- one batched greedy decode step (nanochat "Engine.generate":
 * one token column for the whole batch per forward).
 *   batch in [1, max_batch].
 *   seq_ids: host int32[batch], distinct sequence slots.
 *   tokens: host or device int32[batch], the token fed to each row.
 *   positions: host int32[batch]; positions[i] must equal the current length of
 *     seq_ids[i] (else SLM_EPOS) and be < max_seq (else SLM_ECAPACITY).
 *   logits: NULL, or host or device float[batch][vocab].
 *   next_ids: host or device int32[batch], argmax of each row's logits.
 *   Row i appends its k, v at slot positions[i]; its length becomes positions[i] + 1.
 *   Asynchronous on `stream` when tokens, logits and next_ids are device memory (the
 *   ids can feed the next step without a device-to-host copy); synchronous otherwise.
 *   Single-row steps of small models run on the cluster kernel (slm_debug_cluster),
 *   the others on the persistent kernel; the results are the same computation.
 *   Device-side faults (a bounded wait ran out, NaN logits, a bad token) set the
 *   context's status word: every result of that step and of later steps is invalid
 *   until slm_sync reads and clears it.  A synchronous call (host buffers) reports it
 *   itself, as SLM_ETIMEOUT or SLM_EDEVICE; an asynchronous call cannot, so check with
 *   slm_sync.
 */
int slm_decode_step(slm_ctx *ctx, int32_t batch, const int32_t *seq_ids, const int32_t *tokens,
                    const int32_t *positions, float *logits, int32_t *next_ids, void *stream);

/*
 * slm_reset -- forget a sequence's cached positions (seq = -1: every sequence), as
 * nanochat's KVCache.reset sets its position back to 0.  No memory is freed and no
 * device work is issued.
 */
int slm_reset(slm_ctx *ctx, int32_t seq);

/*
 * slm_fork -- clone a sequence's cache ("Inside nanochat Part 4: Understanding
 * Inference", Batch Prefilling via Cache Replication: a prompt is prefilled once at
 * batch 1 and its cache copied to N rows, which then generate independently).
 *   src: sequence slot in [0, max_batch) holding at least one position (else
 *     SLM_ESTATE).
 *   dst_seqs: host int32[n_dst], n_dst in [1, max_batch - 1]; distinct slots, none
 *     equal to src (else SLM_EINVAL), each empty (else SLM_ESTATE, as the pages'
 *     cache refuses to be filled when it is not empty).
 *   Every layer's cached keys and values of positions [0, length of src) are copied
 *   byte for byte into each destination, whose length becomes src's.  Nothing else
 *   changes.  With a paged cache nothing is copied here: the destinations' tables point
 *   at src's pages, and a sequence that appends into a page it shares first gets a
 *   private copy of that page's rows (so a fork costs one partial page per clone, at
 *   its first step).  Asynchronous on `stream` (one kernel launch): later calls on the
 *   same stream see the copies.  Errors: SLM_EINVAL, SLM_ESTATE, SLM_ECUDA.
 */
int slm_fork(slm_ctx *ctx, int32_t src, int32_t n_dst, const int32_t *dst_seqs, void *stream);

/*
 * slm_sample -- draw the next token of each row from its logits ("Inside nanochat
 * Part 4: Understanding Inference", The Sampling Function; top-p as in kasahare's
 * --top-p flag, applied after top-k).  Needs no context.
 *   logits: device float[batch][ld], ld >= vocab (e.g. slm_decode_step's logits).
 *   temperature: 0 = greedy (argmax, lowest index on ties); otherwise > 0 and finite.
 *   top_k: 0 = the whole vocabulary, or 1..1024: the k largest logits (ties by lower
 *     index), sorted largest first.
 *   top_p: in (0, 1]; below 1 keeps the shortest prefix of the sorted top-k candidates
 *     whose probability reaches top_p (then top_k must be >= 1).
 *   uniforms: device float[batch] in [0, 1), the variate of each row's draw (the caller
 *     owns the random stream): the token is the first candidate, in the order above
 *     (index order without top-k), whose running sum of softmax(logit / temperature)
 *     weights exceeds uniforms[row] times their total.
 *   next_ids: device int32[batch].
 *   Asynchronous on `stream`.  With top_k >= 1 over a large vocabulary the rows are
 *   split over several CTAs, whose candidates are merged through a stream-ordered
 *   scratch buffer (cudaMallocAsync / cudaFreeAsync on `stream`, up to 32 KB per row); if
 *   that allocation fails the call falls back to one CTA per row and allocates nothing.
 *   Callers that must not allocate can pass top_k = 0 (or temperature 0), which never
 *   allocates.  Errors (text in slm_last_error(NULL)): SLM_EINVAL (NULL or host
 *   pointers, sizes, parameters), SLM_ECUDA.
 */
int slm_sample(int32_t batch, int32_t vocab, const float *logits, int32_t ld, float temperature, int32_t top_k,
               float top_p, const float *uniforms, int32_t *next_ids, void *stream);

/*
 * slm_quantize_q8 -- block-quantised int8 weights (the SLM_Q8 format).  Needs no context
 * or device: a host function.  For each of `rows` rows of `cols` fp32 weights (w[rows][cols],
 * row-major) and each block of 32 consecutive weights of the row (the last block of a
 * row holds cols % 32 of them when cols is not a multiple of 32): d = max|w| / 127 (fp32)
 * and q = w / d rounded to the nearest integer, halves away from zero, in [-127, 127]; an
 * all-zero block has d = 0 and q = 0.  The weight this represents is d * q.
 *   q: host int8[rows][cols]; d: host float[rows][ceil(cols / 32)].
 *   Returns SLM_OK, or SLM_EINVAL for NULL pointers, rows < 0 or cols < 1.
 */
int slm_quantize_q8(const float *w, int32_t rows, int32_t cols, int8_t *q, float *d);

/* slm_seq_len -- current length of a sequence (>= 0), or a negative SLM_E* code. */
int32_t slm_seq_len(const slm_ctx *ctx, int32_t seq);

/*
 * slm_kv_pages_free -- pages of a paged KV cache (kv_page_size > 0) that no sequence
 * holds: what sequences can still grow into (admission for continuous batching).  0
 * without paging; SLM_EINVAL for a NULL context.  With paging, slm_prefill,
 * slm_prefill_batch and slm_decode_step return SLM_ECAPACITY, and change nothing, when
 * the pages their rows need (a new page at every kv_page_size-th position, plus one when
 * a row first writes into a page it shares after slm_fork) exceed this count.
 */
int32_t slm_kv_pages_free(const slm_ctx *ctx);

/*
 * slm_sync -- wait for the work enqueued on `stream`, then read and clear the device
 * status word: SLM_OK, SLM_ETIMEOUT (a bounded wait ran out), SLM_EDEVICE (NaN logits
 * or a token id out of range), or SLM_ECUDA.
 */
int slm_sync(slm_ctx *ctx, void *stream);

/* slm_destroy -- free everything the context owns.  NULL is ignored. */
void slm_destroy(slm_ctx *ctx);

/* slm_last_error -- text of the context's last failure ("" if none).  With ctx = NULL:
 * the last failure, on the calling thread, of a call that has no context
 * (slm_create, slm_attention_decode). */
const char *slm_last_error(const slm_ctx *ctx);

/* slm_status_string -- static text for a status code. */
const char *slm_status_string(int status);

/*
 * slm_debug_copy_kv -- test hook: copy the cached keys and values of positions
 * [0, n_pos) of one (layer, sequence) to host memory as fp32 [n_kv_heads][n_pos]
 * [head_dim] each, widening bf16 caches exactly.  n_pos = -1 means the sequence's
 * current length; n_pos may reach max_seq, so a test can also inspect slots that no
 * step has written.  Either output may be NULL.  Synchronous (device-wide).  Returns
 * the number of positions copied, or a negative SLM_E* code.
 */
int slm_debug_copy_kv(slm_ctx *ctx, int32_t layer, int32_t seq, int32_t n_pos, float *k_host,
                      float *v_host);

/*
 * slm_debug_plan -- test hook: the work split and shared-memory layout slm_create would
 * choose for `config` on a GPU with `sms` SMs, computed on the host (no device needed).
 * out: int32[47] = grid, roles, role0[5], own_ld, acc_bytes, xs_bytes, ring_slots,
 * dynamic shared-memory bytes, then for the embedding, QKV, Wo, W1/W3 and W2 matrices
 * each: rows, K, KB, KBp, nkt, rows_per_unit, rows_per_chunk.  Returns SLM_OK, or the
 * error slm_create would return for the plan (text in slm_last_error(NULL)).
 */
int slm_debug_plan(const slm_config *config, int32_t sms, int32_t *out, int32_t out_len);

/*
 * slm_debug_faults -- test hook for the failure paths (no page counterpart: the bounded
 * waits exist so that a lost hand-off ends the step with an error instead of hanging the
 * GPU).  wait_ns: limit of each bounded device-side wait of the decode kernels from the
 * next step on (0 restores the default of 1 s); lost_publish = 1 makes one CTA skip one
 * publish of the first layer's residual in every following step, so that its consumers'
 * waits run out.  The step then finishes without hanging; its results are invalid and
 * slm_sync returns SLM_ETIMEOUT (and clears the status).  Returns SLM_OK or SLM_EINVAL.
 */
int slm_debug_faults(slm_ctx *ctx, unsigned long long wait_ns, int32_t lost_publish);

/*
 * slm_debug_cluster -- test hook: how this engine runs single-row decode steps.  Returns
 * 1 when they run on the cluster kernel (attention clusters, one per kv head, and FFN
 * clusters; the layout follows the block equations of kasahare 0.4.0 / simple-llm,
 * "Architecture", split so that a layer needs two grid-wide hand-offs), 0 when they run
 * on the persistent kernel, or a negative SLM_E* code.  out (may be NULL): int32[12] =
 * cluster size C, attention clusters NA, FFN clusters NF, grid, hidden units per FFN
 * cluster, ring slots, dynamic shared-memory bytes, units per chunk of the QKV, Wo,
 * W1/W3, W2 and logits phases.
 */
int slm_debug_cluster(const slm_ctx *ctx, int32_t *out, int32_t out_len);

/*
 * slm_debug_trace -- timeline hook (in the spirit of kasahare's "--timing" and
 * forward_traced): with enable != 0, every following step records, for each CTA of
 * the decode kernel and each phase (5 per layer: QKV, attention, Wo, W1/W3, W2; then
 * logits and argmax), three %globaltimer readings in ns: entered, inputs ready, done
 * (0 where a CTA had no work).  out_host: NULL, or host uint64 [grid][5 * n_layers + 2][3]
 * receiving the last step's record (out_len entries, synchronous).  enable = 0 turns
 * recording off.  Returns the grid size, or a negative SLM_E* code.
 */
int slm_debug_trace(slm_ctx *ctx, int32_t enable, unsigned long long *out_host, size_t out_len);

/*
 * slm_debug_gemm_bf16 -- test hook for the tensor-core GEMM tile used by the prefill:
 * C[m][n] = sum_k A[m][k] * B[n][k] in fp32, A device bf16 [M][K], B device bf16 [N][K]
 * (both 16-byte aligned), C device fp32 [M][N].  K must be a multiple of 64.
 * Synchronous.  SLM_ETIMEOUT if a bounded wait inside the kernel ran out.
 */
int slm_debug_gemm_bf16(int32_t M, int32_t N, int32_t K, const void *A, const void *B, float *C, void *stream);

/*
 * slm_debug_fill_kv -- test hook: fill the whole KV cache (every layer, slot and
 * position) with the fp32 value `value` (rounded to the cache type), so that a test
 * can check that a step writes exactly the slots it should.  Synchronous.
 */
int slm_debug_fill_kv(slm_ctx *ctx, float value);

/*
 * slm_debug_page_table -- test hook: the page ids of sequence `seq` (ceil(max_seq /
 * kv_page_size) entries; -1 = no page; without paging one entry, the slot itself),
 * up to out_len of them into host `out`.  Returns the number of entries, or SLM_EINVAL.
 */
int32_t slm_debug_page_table(const slm_ctx *ctx, int32_t seq, int32_t *out, int32_t out_len);

/*
 * slm_attention_workspace_bytes -- size in bytes of the device workspace that
 * slm_attention_decode needs for this shape (split-K partial states and arrival
 * counters); 0 for non-positive arguments.
 */
size_t slm_attention_workspace_bytes(int32_t batch, int32_t n_heads, int32_t n_kv_heads,
                                     int32_t head_dim);

/*
 * slm_attention_decode -- the decode-attention step on its own (kasahare 0.4.0 /
 * simple-llm, "Architecture": attn = softmax(q . K^T / sqrt(d_head)) . V with GQA), over
 * a caller-owned cache.  For every row b and query head h, with kv head
 * g = h / (n_heads / n_kv_heads):
 *     out[b][h] = sum_t softmax_t(q[b][h] . k[b][g][t] / sqrt(head_dim)) v[b][g][t],
 *     t = 0 .. ctx_len[b] - 1.
 * Keys and values are split into chunks of positions; each chunk keeps an online
 * softmax and the partial states are merged by rescaling to a common maximum
 * (flash-decoding).  The query is used as given (RoPE already applied).
 *   q: device fp32 [batch][n_heads][head_dim].
 *   k_cache, v_cache: device [batch][n_kv_heads][capacity][head_dim] of kv_dtype
 *     (SLM_F32 or SLM_BF16), each 16-byte aligned (rows are read 16 bytes at a time;
 *     an offset view fails with SLM_EINVAL before anything is launched); only
 *     positions < ctx_len[b] are read.
 *   ctx_len: host int32[batch], each in [1, capacity].
 *   out: device fp32 [batch][n_heads][head_dim].
 *   workspace: device memory, 256-byte aligned, at least
 *     slm_attention_workspace_bytes(batch, n_heads, n_kv_heads, head_dim) bytes; the
 *     call owns it until the enqueued work finishes.
 *   batch in [1, 16]; head_dim a multiple of 8 in [8, 256]; n_heads % n_kv_heads == 0.
 *   Asynchronous on `stream`.  Errors: SLM_EINVAL (shape, NULL pointer, workspace too
 *   small or misaligned), SLM_ECUDA (launch failure); slm_last_error(NULL) explains.
 */
int slm_attention_decode(int32_t batch, int32_t n_heads, int32_t n_kv_heads, int32_t head_dim,
                         int32_t capacity, int32_t kv_dtype, const float *q, const void *k_cache,
                         const void *v_cache, const int32_t *ctx_len, float *out, void *workspace,
                         size_t workspace_bytes, void *stream);

/*
 * slm_attention_decode_noalloc -- slm_attention_decode without a workspace argument,
 * for callers that cannot allocate device memory: code running where cudaMalloc is not
 * allowed or not wanted (an application whose own allocator reserves all device memory
 * up front, or a latency-critical loop that must not call an allocator, which can
 * synchronise the device).  The pages describe no such entry point; it has no
 * counterpart there.
 *   Arguments, layouts and results are those of slm_attention_decode.  The split-K
 *   scratch lives in one fixed array compiled into the library,
 *   slm_attention_noalloc_max_bytes() bytes (4 MiB), which every GPU that loads the
 *   library holds until the process exits.  Shapes whose scratch
 *   (slm_attention_workspace_bytes) exceeds it fail with SLM_EINVAL and a message.
 *   The call allocates nothing: no cudaMalloc, no cudaFree, no allocating library
 *   routine.  The first call on a device looks up the array's device address (once
 *   per device, with that device current, and again if the device's context changed
 *   since, e.g. after cudaDeviceReset); make that first call before any stream capture.  Every call shares the array and it keeps the last call's contents: the
 *   call clears the arrival counters itself, but calls whose work overlaps on the GPU
 *   (e.g. on two unordered streams) race on the array.
 */
size_t slm_attention_noalloc_max_bytes(void);
int slm_attention_decode_noalloc(int32_t batch, int32_t n_heads, int32_t n_kv_heads,
                                 int32_t head_dim, int32_t capacity, int32_t kv_dtype,
                                 const float *q, const void *k_cache, const void *v_cache,
                                 const int32_t *ctx_len, float *out, void *stream);

#ifdef __cplusplus
}
#endif
#endif
