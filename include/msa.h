/*
 * msa.h -- C ABI of libmsa: MiniMax-M3 two-step block-sparse attention on
 * GB300 (sm_103a).
 *
 * The method (TensorRT-LLM "MiniMaxM3SparseAttentionConfig", class
 * description): an index branch scores the 128-token key blocks of each query
 * with a per-KV-head index query against one shared index key, keeps the top-k
 * blocks per (kv_head, q_token) with init blocks forced at the head and local
 * blocks forced at the tail, and a sparse GQA attention then runs over the
 * selected blocks only.  The NeMo AutoModel page
 * "nemo_automodel.components.models.minimax_m3_vl.msa" states the same two
 * steps for packed documents (MSAMicrobatch.select_blocks, sparse_attention).
 *
 * Conventions for every entry point
 *   - Pointers marked "dev" are device pointers; "host" are host pointers.
 *     All device buffers are owned by the caller.  The library allocates no
 *     memory and launches all work on the caller's `stream` (a cudaStream_t
 *     passed as void*; NULL = legacy default stream).
 *   - No entry point synchronises the stream except msa_pack_metadata and
 *     msa_read_device_error, which say so.
 *   - Work runs on the calling thread's current device (cudaGetDevice), whose
 *     primary context each call makes current on the calling thread, so any
 *     thread may call (a fresh one, or PyTorch's autograd worker, included).
 *     Device buffers and the stream must belong to that device.
 *   - Tensors are dense row-major with the shapes given; tensor base pointers
 *     must be 16-byte aligned.
 *   - Errors are returned synchronously as msa_status; nothing is thrown and
 *     nothing aborts.  Argument errors are detected before any CUDA call, so a
 *     call that returns MSA_ERR_NULL / SHAPE / DTYPE / WORKSPACE / ALIGN has
 *     enqueued no work.  Bad data found on the device (a page id outside the
 *     pool, a block id outside the query's range, a length outside its bound)
 *     is skipped and recorded in the workspace's device error word, which
 *     msa_read_device_error returns.
 *   - Fixed topology (NeMo msa, require_msa_support): 64 query heads, 4 KV
 *     heads, head dim 128, 4 index heads of dim 128, block size 128 (the
 *     TensorRT-LLM field implementation='msa' requires sparse_block_size 128),
 *     max score reduction.  Query head h reads KV / index head h / 16.
 *   - q2k rows hold the selected document-local block ids in ascending order,
 *     then -1 up to topk (NeMo select_blocks: "int32 [4, tokens, 16]
 *     document-local block ids, padded with -1").
 */
#ifndef MSA_H_
#define MSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MSA_OK = 0,
  MSA_ERR_NULL = 1,      /* a required pointer is NULL */
  MSA_ERR_SHAPE = 2,     /* unsupported topology or inconsistent sizes */
  MSA_ERR_DTYPE = 3,     /* unsupported index dtype */
  MSA_ERR_WORKSPACE = 4, /* workspace NULL, too small or not 256-byte aligned */
  MSA_ERR_ALIGN = 5,     /* a tensor pointer is not 16-byte aligned */
  MSA_ERR_CUDA = 6,      /* a CUDA runtime call or a kernel launch failed */
  MSA_ERR_DOC_MAP = 7    /* malformed document map (msa_pack_metadata) */
} msa_status;

/* Index Q/K storage dtype (TensorRT-LLM field indexer_kv_dtype): bf16, or
 * unscaled E4M3 with FP32 score accumulation. */
enum { MSA_INDEX_BF16 = 0, MSA_INDEX_E4M3 = 1 };

/* Workspace modes for msa_workspace_size. */
enum { MSA_MODE_DECODE = 0, MSA_MODE_PREFILL = 1, MSA_MODE_PACK = 2, MSA_MODE_PREFILL_BWD = 3 };

/* Device error codes reported by msa_read_device_error. */
enum {
  MSA_DEVERR_NONE = 0,
  MSA_DEVERR_PAGE = 1,     /* page id outside [0, num_slots/128) */
  MSA_DEVERR_BLOCK = 2,    /* q2k id outside [0, blocks of the query) */
  MSA_DEVERR_LENGTH = 3,   /* seq_len < 1, or above max_blocks * 128 */
  MSA_DEVERR_TIMEOUT = 4,  /* a bounded on-chip wait gave up */
  MSA_DEVERR_RANGE = 5     /* prefill attention: a score outside the fixed-reference range (see
                              msa_sparse_attend_prefill); detail = the flat q2k index */
};

/* Layer configuration (TensorRT-LLM MiniMaxM3SparseAttentionConfig fields:
 * num_attention_heads, num_key_value_heads, sparse_num_index_heads,
 * sparse_index_dim, sparse_block_size, sparse_topk_blocks,
 * sparse_init_blocks, sparse_local_blocks, indexer_kv_dtype).
 * Accepted: 64 / 4 / 128 / 4 / 128 / 128, 1 <= topk <= 16, init >= 0,
 * local >= 0, init + local <= topk. */
typedef struct {
  int num_q_heads;
  int num_kv_heads;
  int head_dim;
  int num_index_heads;
  int index_dim;
  int block_size;
  int topk;
  int init_blocks;
  int local_blocks;
  int index_dtype;
} msa_config;

/* Fills `cfg` with the MiniMax-M3 defaults: 64/4/128/4/128/128, topk 16,
 * init 0, local 1, bf16 index. */
msa_status msa_config_default(msa_config* cfg);

/* Checks `cfg` against the supported topology (NeMo require_msa_support). */
msa_status msa_config_check(const msa_config* cfg);

/* Bytes of workspace one call of the given mode needs.
 *   MSA_MODE_DECODE : n = batch, max_blocks = blocks per request row of the
 *                     page table (or ceil(max context / 128) when contiguous).
 *   MSA_MODE_PREFILL: n = total compact tokens, max_blocks = ceil(max_seqlen/128).
 *   MSA_MODE_PACK   : n = batch * seq of the document map, max_blocks = batch.
 *   MSA_MODE_PREFILL_BWD: as MSA_MODE_PREFILL, for msa_sparse_attend_prefill_backward.
 * The workspace must be zero-filled once before its first use (see
 * msa_workspace_init), which clears the device error word and the decode
 * scorer's page-claim counter in its first 256 bytes, and the completion
 * counters.  Every call that completes leaves its
 * counters at zero again (the decode calls enqueue no memset; the prefill
 * calls clear theirs with a cudaMemsetAsync on `stream`), and the scorer
 * stores rather than accumulates (NeMo _score_scratch).  In the decode layout
 * the decode attention's counters (one per CTA) sit at a fixed offset that no
 * decode call of any batch or max_blocks writes over, so one workspace serves
 * decode calls of any size whose msa_workspace_size fits in it, in any order.
 * The prefill layouts do not keep that region: a workspace that served a
 * prefill or backward call must be zero-filled again before it serves a
 * decode attention call.  After a call whose device error word reads
 * MSA_DEVERR_TIMEOUT (a pipeline that gave up part-way), zero-fill the
 * workspace again before reusing it.  Calls that share a workspace must not
 * run concurrently. */
msa_status msa_workspace_size(const msa_config* cfg, int mode, int64_t n, int max_blocks,
                              size_t* bytes);

/* Zero-fills `bytes` of workspace on `stream` (cudaMemsetAsync). */
msa_status msa_workspace_init(void* workspace, size_t bytes, void* stream);

/* Reads the device error word of `workspace` into *code and *detail (the
 * offending index), then clears it.  Synchronises `stream`. */
msa_status msa_read_device_error(void* workspace, void* stream, int* code, int64_t* detail);

/* Human-readable name of a status. */
const char* msa_status_string(msa_status status);

/* The CUDA error code (a cudaError_t value) of the last call on the calling
 * thread that returned MSA_ERR_CUDA; 0 if none has.  Calls that succeed leave
 * it unchanged. */
int msa_last_cuda_error(void);

/* Text of a CUDA error code (cudaGetErrorString); the pointer is static. */
const char* msa_cuda_error_string(int code);

/* Diagnostic of the library's bounded on-chip waits (every pipeline wait of
 * every kernel above uses them).  Launches one CTA on `stream` whose first
 * thread waits on a shared-memory mbarrier that nothing ever arrives on, then
 * on a second such barrier, and returns.  Each wait gives up after the
 * library's wait limit (200 ms of GPU global time); the first records
 * MSA_DEVERR_TIMEOUT with detail 900 in the device error word of `workspace`
 * (the second finds the word taken and leaves it).  `workspace` is any
 * initialised workspace (only its first 256 bytes are used); `waits_ns`
 * (host, 2 entries) receives the duration of each wait in nanoseconds, or -1
 * for a wait that completed (which would be a library defect).  The device
 * error word is left for msa_read_device_error.  Synchronises `stream`.
 * Errors: MSA_ERR_NULL for a null workspace or waits_ns; MSA_ERR_WORKSPACE
 * for a workspace not 256-byte aligned; MSA_ERR_CUDA for a failed launch or
 * copy. */
msa_status msa_check_bounded_wait(void* workspace, void* stream, int64_t* waits_ns);

/* ---- step 1+2, decode: block scores + top-k ---------------------------------
 * One query per request at position seq_lens[r]-1 over keys 0..seq_lens[r]-1
 * (the query's own key is already in the cache).  Score of block b for index
 * head g = max over the block's keys of <index_q[r,g,:], index_k[key,:]>,
 * unscaled, fp32 accumulation (TensorRT-LLM sparse_score_type 'max',
 * indexer_kv_dtype).  Key position p of request r sits at slot
 *   page_table[r * max_blocks + p/128] * 128 + p % 128   (paged), or
 *   cu_seqlens_k[r] + p                                   (page_table == NULL)
 * of the paged side index-K cache [num_slots, 1, 128] that parallels the main
 * K/V cache (TensorRT-LLM class description, MiniMaxM3KVCacheManagerV2).
 *   index_q       dev [batch, 4, 128]  bf16 or e4m3 (cfg->index_dtype)
 *   index_k_cache dev [num_slots, 1, 128] same dtype
 *   seq_lens      dev int32 [batch], 1 <= seq_lens[r] <= max_blocks * 128
 *   page_table    dev int32 [batch, max_blocks] or NULL
 *   cu_seqlens_k  dev int64 [batch + 1], read only when page_table == NULL
 *   q2k           dev int32 [4, batch, topk], fully written (ids asc, then -1)
 *   workspace     >= msa_workspace_size(cfg, MSA_MODE_DECODE, batch, max_blocks)
 */
msa_status msa_select_blocks_decode(const msa_config* cfg, const void* index_q,
                                    const void* index_k_cache, const int32_t* seq_lens,
                                    const int32_t* page_table, const int64_t* cu_seqlens_k,
                                    int batch, int max_blocks, int64_t num_slots, int32_t* q2k,
                                    void* workspace, size_t workspace_bytes, void* stream);

/* ---- decode select without a workspace ---------------------------------------
 * The same computation and arguments as msa_select_blocks_decode, for callers
 * that cannot allocate device memory (for example code running inside a
 * runtime with no allocator of its own, or a plugin that is handed only its
 * input and output buffers).  The pages have no counterpart: this is a
 * deployment convenience of this library.
 *   - Scratch is one fixed 4 MiB array in the library's device memory, held by
 *     every GPU that loads the library until the process exits.  It must hold
 *     256 + 16*batch*max_blocks bytes; larger sizes
 *     are rejected with MSA_ERR_WORKSPACE before any work is enqueued.
 *   - The first call on each device looks up the array's device address on
 *     the current device; make that first call before any stream capture.
 *   - Every call uses the same array and leaves its contents behind; the call
 *     clears what must start at zero on `stream`.  Calls whose work overlaps
 *     on the GPU (other streams, other threads) race on the array.
 *   - Device-side data errors are recorded in the array, not reported.
 *   - Allocates nothing: no cudaMalloc, no cudaFree, no allocating library. */
msa_status msa_select_blocks_decode_noalloc(const msa_config* cfg, const void* index_q,
                                            const void* index_k_cache, const int32_t* seq_lens,
                                            const int32_t* page_table, const int64_t* cu_seqlens_k,
                                            int batch, int max_blocks, int64_t num_slots, int32_t* q2k,
                                            void* stream);

/* ---- step 3, decode: sparse GQA attention over the selected blocks ----------
 * out[r, h, :] = softmax_j(scale * <q[r,h,:], k[j, h/16, :]>) v[j, h/16, :]
 * over the keys j <= seq_lens[r]-1 of the blocks listed in q2k[h/16, r, :]
 * (entries < 0 are ignored).  fp32 accumulation, bf16 output; a row with no
 * key is written as zeros.  Same geometry arguments as the decode select.
 *   q        dev [batch, 64, 128] bf16
 *   k_cache  dev [num_slots, 4, 128] bf16;  v_cache: same
 *   q2k      dev int32 [4, batch, topk]
 *   out      dev [batch, 64, 128] bf16
 * The kernel is launched as a programmatic dependent of the kernel before it
 * on `stream` (after msa_select_blocks_decode, its launch overlaps the
 * top-k).  Before that kernel has completed it reads no input and writes no
 * output; it only issues L2 prefetch hints for its requests' page-table rows,
 * which change no memory, so stream order is kept whatever precedes it.
 * Up to 19 requests, each (request, KV head) segment is shared by a cluster
 * of 2-8 CTAs that merges on chip; larger batches are split evenly over one
 * CTA per SM with merges through the workspace.  The first call on a device
 * asks the runtime how many clusters can be resident at once
 * (cudaOccupancyMaxActiveClusters, once per cluster size and K/V type).
 */
msa_status msa_sparse_attend_decode(const msa_config* cfg, const void* q, const void* k_cache,
                                    const void* v_cache, const int32_t* q2k,
                                    const int32_t* seq_lens, const int32_t* page_table,
                                    const int64_t* cu_seqlens_k, int batch, int max_blocks,
                                    int64_t num_slots, float scale, void* out, void* workspace,
                                    size_t workspace_bytes, void* stream);

/* The same decode attention with the output emitted as MXFP8 for the o_proj
 * that follows (vLLM forward_decode_mxfp8: E4M3 values and row-major E8M0
 * scales, equal to the MX quantisation of the bf16 output):
 *   out_q     dev uint8 [batch, 64 * 128]: E4M3 bytes of each output element
 *   out_scale dev uint8 [batch, 64 * 128 / 32]: the E8M0 scale byte of each
 *             block of 32 consecutive elements of a row
 * Per block: b = the bf16 output values, amax = max |b|, scale exponent
 * e = floor(log2 amax) - 8 (8: the largest E4M3 exponent; clamped to
 * [-127, 127]; -127 for an all-zero block), scale byte e + 127, and each value
 * b * 2^-e rounded to E4M3 (nearest, ties to even, saturating at +-448).
 * The page names this quantisation without printing it; the OCP
 * Microscaling (MX) v1.0 block rule is the reading taken.
 * Errors as msa_sparse_attend_decode; MSA_ERR_ALIGN if out_q is not 16-byte
 * aligned. */
msa_status msa_sparse_attend_decode_mxfp8(const msa_config* cfg, const void* q, const void* k_cache,
                                          const void* v_cache, const int32_t* q2k,
                                          const int32_t* seq_lens, const int32_t* page_table,
                                          const int64_t* cu_seqlens_k, int batch, int max_blocks,
                                          int64_t num_slots, float scale, void* out_q,
                                          void* out_scale, void* workspace, size_t workspace_bytes,
                                          void* stream);

/* The same decode attention over an FP8 main K/V cache (TensorRT-LLM field
 * fuse_qkv_index_projection: the MiniMax-M3 path uses "an FP8 main KV cache").
 * The pages give no scale rule; the reading taken: the caches hold E4M3 bytes
 * (OCP E4M3, "fn") standing for k_scale * k and v_scale * v, one fp32 scale per
 * cache (1.0 for an unscaled cache).
 *   k_cache, v_cache dev uint8 [num_slots, 4, 128] E4M3
 *   k_scale, v_scale finite and > 0
 * Inside, the E4M3 values enter fp16 MMAs exactly, q is rounded to fp16 once
 * (exact for |q| in fp16's normal range, 2^-14 .. 65504), P is rounded to fp16
 * with the row sum taken over the rounded values, accumulation is fp32.  Other
 * arguments, the output and the errors as msa_sparse_attend_decode;
 * MSA_ERR_SHAPE for a scale that is not finite and positive. */
msa_status msa_sparse_attend_decode_fp8kv(const msa_config* cfg, const void* q, const void* k_cache,
                                          const void* v_cache, float k_scale, float v_scale,
                                          const int32_t* q2k, const int32_t* seq_lens,
                                          const int32_t* page_table, const int64_t* cu_seqlens_k,
                                          int batch, int max_blocks, int64_t num_slots, float scale,
                                          void* out, void* workspace, size_t workspace_bytes,
                                          void* stream);

/* ---- step 1+2, prefill: block scores + top-k on packed documents ------------
 * NeMo MSAMicrobatch.select_blocks: compact tokens in document order, document
 * d spanning [cu_seqlens[d], cu_seqlens[d+1]); token t of document d has
 * position p = t - cu_seqlens[d] and candidate blocks 0..p/128 of its own
 * document; the diagonal block's score covers keys <= p only.
 *   index_q    dev [total_tokens, 4, 128] bf16, or E4M3 bytes when
 *              cfg->index_dtype is MSA_INDEX_E4M3 (post norm and RoPE)
 *   index_k    dev [total_tokens, 1, 128], same dtype as index_q
 *   cu_seqlens dev int32 [num_docs + 1], cu_seqlens[0] = 0, strictly increasing,
 *              cu_seqlens[num_docs] = total_tokens; max_seqlen = the longest document
 *              (at most 17066 blocks of 128 tokens, about 2.18M tokens; longer: MSA_ERR_SHAPE)
 *   q2k        dev int32 [4, total_tokens, topk]
 * E4M3 scores are unscaled dot products of the decoded values, accumulated in
 * fp32 (TRT indexer_kv_dtype). */
msa_status msa_select_blocks_prefill(const msa_config* cfg, const void* index_q,
                                     const void* index_k, const int32_t* cu_seqlens, int num_docs,
                                     int64_t total_tokens, int max_seqlen, int32_t* q2k,
                                     void* workspace, size_t workspace_bytes, void* stream);

/* ---- step 3, prefill: sparse GQA attention on packed documents ---------------
 * NeMo sparse_attention / _SparseAttention.forward: bf16 q [tokens, 64, 128],
 * k / v [tokens, 4, 128], int32 q2k [4, tokens, topk] -> bf16 out
 * [tokens, 64, 128]; keys are the causal keys (position <= the query's) of the
 * query's document inside the listed blocks.
 * Each (query, KV head) row's softmax takes its exponent reference from the
 * row's highest listed block (the local block when local_blocks >= 1): the
 * row max over that block's causal keys.  The other blocks are summed against
 * that fixed reference in fp32.  A key of another listed block whose scaled
 * score (in log2 units) exceeds the reference by 64 or more (a logit gap above
 * about 44) is outside this scheme's range: the call records MSA_DEVERR_RANGE
 * (detail: the flat q2k index of the entry) and that row's output is not
 * valid.  Nothing else is affected.  The fp32 sums are added by the tensor
 * engine in an order that varies from run to run, so the bf16 output is not
 * bitwise reproducible (the pages give no deterministic-mode guarantee); two
 * runs differ by at most one bf16 ulp. */
msa_status msa_sparse_attend_prefill(const msa_config* cfg, const void* q, const void* k,
                                     const void* v, const int32_t* q2k, const int32_t* cu_seqlens,
                                     int num_docs, int64_t total_tokens, int max_seqlen,
                                     float scale, void* out, void* workspace,
                                     size_t workspace_bytes, void* stream);

/* The same call, also writing the log-sum-exp the backward needs:
 *   lse dev fp32 [total_tokens, 64]: log2 of the softmax denominator in the
 *       base-2 domain of the scaled scores, log2(sum_p 2^(scale <q, k_p> log2 e)),
 *       -inf for a (token, head) with no key.  The sum is taken over the
 *       bf16-rounded weights the output applies, so it is within
 *       log2(1 + 2^-9) of the exact value (NeMo _SparseAttention saves the
 *       forward's schedule for its backward; this is the row statistic of it).
 * Errors as msa_sparse_attend_prefill; MSA_ERR_NULL for a null lse. */
msa_status msa_sparse_attend_prefill_lse(const msa_config* cfg, const void* q, const void* k,
                                         const void* v, const int32_t* q2k,
                                         const int32_t* cu_seqlens, int num_docs,
                                         int64_t total_tokens, int max_seqlen, float scale, void* out,
                                         float* lse, void* workspace, size_t workspace_bytes,
                                         void* stream);

/* ---- backward of step 3, prefill ------------------------------------------------
 * NeMo _SparseAttention.backward: bf16 grad_out [tokens, 64, 128] -> bf16 dq
 * [tokens, 64, 128], dk and dv [tokens, 4, 128], over the same keys as the
 * forward (q2k, cu_seqlens, scale as given to it).  With z_p = scale <q, k_p>,
 * P = softmax(z) (rebuilt from lse), dP_p = <grad_out, v_p> and D = <grad_out,
 * out>: dv_p += P_p grad_out, dS_p = P_p (dP_p - D), dk_p += scale dS_p q,
 * dq += scale sum_p dS_p k_p.
 *   out, lse   the forward's bf16 output and fp32 log-sum-exp
 *              (msa_sparse_attend_prefill_lse)
 *   dq, dk, dv dev bf16, written whole (zero for tokens no query reaches)
 *   workspace  >= msa_workspace_size(cfg, MSA_MODE_PREFILL_BWD, total_tokens,
 *              ceil(max_seqlen / 128)); holds fp32 accumulators for dk, dv
 * dk and dv are summed in fp32 and dq in bf16 straight into the output (as
 * the NeMo page says of its backward), by the tensor engine's bulk adds in an
 * order that varies, so the gradients are not bitwise reproducible from run
 * to run.
 * Errors: MSA_ERR_NULL, MSA_ERR_SHAPE, MSA_ERR_ALIGN (any tensor not 16-byte
 * aligned), MSA_ERR_WORKSPACE, MSA_ERR_CUDA. */
msa_status msa_sparse_attend_prefill_backward(const msa_config* cfg, const void* q, const void* k,
                                              const void* v, const int32_t* q2k,
                                              const int32_t* cu_seqlens, int num_docs,
                                              int64_t total_tokens, int max_seqlen, float scale,
                                              const void* out, const float* lse, const void* grad_out,
                                              void* dq, void* dk, void* dv, void* workspace,
                                              size_t workspace_bytes, void* stream);

/* ---- the index producer: L2 norm, storage cast, index-K cache insertion ------
 * TensorRT-LLM "MiniMaxM3SparseAttentionConfig", field fuse_qkv_index_projection
 * (MSA batches use a horizontal norm / RoPE / cache-insertion producer for
 * prefill, mixed and CUDA-graph decode), field indexer_kv_dtype (index Q/K are
 * stored normalized, as bf16 or unscaled E4M3) and the class description (the
 * paged index-K cache [num_slots, 1, 128] parallel to the main K/V cache); NeMo
 * select_blocks takes index tensors "post norm".  Each 128-vector x of the
 * projection's output is stored as y = x / ||x||_2 in cfg->index_dtype:
 * computed in IEEE binary32 with the squares summed in index order c = 0..127,
 * sqrt and division correctly rounded, then one rounding to bf16 or E4M3
 * (nearest, ties to even).  A vector whose sum of squares is 0 in binary32 is
 * stored as zeros.  The pages fix neither the precision nor the order; this is
 * the reading the library takes, and it makes the result bit-reproducible.
 * RoPE, which the pages name without giving its variant, is not applied: it is
 * a rotation and leaves the L2 norm unchanged, so a caller may apply it to the
 * input.  Inputs are the projection's bf16 output.
 *   workspace  >= 256 bytes, 256-byte aligned (only its device error word is
 *              used: a page id or position out of range is skipped and
 *              recorded there, MSA_DEVERR_PAGE / MSA_DEVERR_LENGTH, detail =
 *              the token or request)
 * Errors: MSA_ERR_NULL, MSA_ERR_SHAPE, MSA_ERR_DTYPE, MSA_ERR_ALIGN (a tensor
 * not 16-byte aligned), MSA_ERR_WORKSPACE, MSA_ERR_CUDA. */

/* Prefill / packed documents (the input of msa_select_blocks_prefill):
 *   index_q_in  dev bf16 [total_tokens, 4, 128]; index_k_in dev bf16 [total_tokens, 1, 128]
 *   cu_seqlens  dev int32 [num_docs + 1], as for msa_select_blocks_prefill
 *   index_q_out dev [total_tokens, 4, 128] in cfg->index_dtype (written whole)
 *   index_k_out dev [total_tokens, 1, 128] in cfg->index_dtype, or NULL
 *   index_k_cache dev [num_slots, 1, 128] in cfg->index_dtype, or NULL: when
 *              given, the key of the token at position p of document d is also
 *              written at slot page_table[d * max_blocks + p / 128] * 128 + p % 128
 *              (page_table dev int32 [num_docs, max_blocks]; num_slots a
 *              multiple of 128); no other slot is touched
 * At least one of index_k_out and index_k_cache must be given. */
msa_status msa_index_produce_prefill(const msa_config* cfg, const void* index_q_in,
                                     const void* index_k_in, const int32_t* cu_seqlens,
                                     int num_docs, int64_t total_tokens, void* index_q_out,
                                     void* index_k_out, void* index_k_cache,
                                     const int32_t* page_table, int max_blocks, int64_t num_slots,
                                     void* workspace, size_t workspace_bytes, void* stream);

/* Decode (one new token per request, the input of msa_select_blocks_decode):
 * the new token of request r sits at position p = seq_lens[r] - 1 (the
 * length includes it); its normalised key is written at the slot
 *   page_table[r * max_blocks + p / 128] * 128 + p % 128   (paged), or
 *   cu_seqlens_k[r] + p                                   (page_table == NULL)
 * of index_k_cache, and no other slot is touched.
 *   index_q_in  dev bf16 [batch, 4, 128]; index_k_in dev bf16 [batch, 1, 128]
 *   seq_lens / page_table / cu_seqlens_k / max_blocks / num_slots: as for
 *              msa_select_blocks_decode
 *   index_q_out dev [batch, 4, 128] in cfg->index_dtype
 *   index_k_cache dev [num_slots, 1, 128] in cfg->index_dtype, updated in place */
msa_status msa_index_produce_decode(const msa_config* cfg, const void* index_q_in,
                                    const void* index_k_in, const int32_t* seq_lens,
                                    const int32_t* page_table, const int64_t* cu_seqlens_k,
                                    int batch, int max_blocks, int64_t num_slots, void* index_q_out,
                                    void* index_k_cache, void* workspace, size_t workspace_bytes,
                                    void* stream);

/* ---- packed layout of a document map ----------------------------------------
 * NeMo layout-from-doc_ids constructor and _contiguous_runs: doc_ids is an
 * int64 [batch, seq] map, 0 = padding, each positive id one contiguous run of
 * tokens within its row.  Documents are the runs in row-major order.  Writes
 *   cu_seqlens dev int32 [num_docs + 1]   (capacity batch*seq + 1)
 *   token_rows dev int64 [total_tokens]   flat index of each real token (capacity batch*seq)
 * and the host scalars *num_docs, *total_tokens, *max_seqlen.  Synchronises
 * `stream` exactly once (one device-to-host copy of the scalars).
 * Returns MSA_ERR_DOC_MAP for an empty map, a negative id, no real token, an
 * interrupted document, or sizes past int32; *bad_index (host, may be NULL)
 * then holds the flat index of the first offending token (-1 if none). */
msa_status msa_pack_metadata(const int64_t* doc_ids, int batch, int seq, int32_t* cu_seqlens,
                             int64_t* token_rows, int* num_docs, int64_t* total_tokens,
                             int* max_seqlen, int64_t* bad_index, void* workspace,
                             size_t workspace_bytes, void* stream);

/* NeMo MSAMicrobatch.pack: packed[i, :] = external[token_rows[i], :] for rows
 * of `row_bytes` bytes (a multiple of 16).  external dev [batch*seq, row_bytes],
 * packed dev [total_tokens, row_bytes].  Always copies (never aliases). */
msa_status msa_pack(const void* external, const int64_t* token_rows, int64_t total_tokens,
                    int64_t row_bytes, void* packed, void* stream);

/* NeMo MSAMicrobatch.unpack: external[token_rows[i], :] = packed[i, :] and
 * every other row of external dev [batch_seq, row_bytes] zero-filled. */
msa_status msa_unpack(const void* packed, const int64_t* token_rows, int64_t total_tokens,
                      int64_t batch_seq, int64_t row_bytes, void* external, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MSA_H_ */
