// abi.cu -- the extern "C" entry points of libmsa: argument validation,
// workspace layout and kernel launches.  Declarations and contracts are in
// include/msa.h.
#include <cmath>
#include <mutex>

#include "launch.h"

namespace msa {

// cuTensorMapEncodeTiled through the runtime's driver entry point (no -lcuda).
EncodeTiledFn get_encode_tiled() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

static size_t up256(size_t x) { return (x + 255) / 256 * 256; }

// Workspace layout, shared by msa_workspace_size and the calls.  Decode: the
// regions whose size does not depend on the call come first, at fixed offsets
// (the attention's merge counters, one per CTA, and its partials), then the
// block scores, whose size grows with batch and max_blocks.  So a call of any
// size never writes over the counters, which must stay at zero between calls.
struct Layout {
  size_t scores = 0, att_tickets = 0, partials = 0, plan = 0, bm = 0, total = 0;
};
static Layout layout(int mode, long long n, int max_blocks, int topk) {
  Layout L;
  size_t off = kHeaderBytes;
  if (mode == MSA_MODE_DECODE) {
    L.att_tickets = off;
    off += up256(attend_tickets_bytes());
    L.partials = off;
    off += up256(attend_partials_bytes());
    L.scores = off;
    off += up256(static_cast<size_t>(n) * kKvHeads * max_blocks * sizeof(float));
  } else if (mode == MSA_MODE_PREFILL) {
    L.plan = off;
    off += up256(prefill_plan_ints(static_cast<int>(n), max_blocks) * sizeof(int));
    L.bm = off;
    off += up256(prefill_attend_bytes(n, max_blocks * kBlock, topk));
  } else if (mode == MSA_MODE_PREFILL_BWD) {
    L.bm = off;
    off += up256(prefill_backward_bytes(n, max_blocks * kBlock, topk));
  }
  L.total = off;
  return L;
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

thread_local int g_last_cuda_error = 0;

msa_status cuda_fail(cudaError_t e) {
  g_last_cuda_error = static_cast<int>(e);
  return MSA_ERR_CUDA;
}

}  // namespace msa

using namespace msa;

extern "C" {

msa_status msa_config_default(msa_config* cfg) {
  if (!cfg) return MSA_ERR_NULL;
  *cfg = msa_config{64, 4, 128, 4, 128, 128, 16, 0, 1, MSA_INDEX_BF16};
  return MSA_OK;
}

msa_status msa_config_check(const msa_config* cfg) {
  if (!cfg) return MSA_ERR_NULL;
  if (cfg->num_q_heads != kHeads || cfg->num_kv_heads != kKvHeads || cfg->head_dim != kDim ||
      cfg->num_index_heads != kKvHeads || cfg->index_dim != kIdxDim || cfg->block_size != kBlock)
    return MSA_ERR_SHAPE;
  if (cfg->topk < 1 || cfg->topk > kMaxTopk || cfg->init_blocks < 0 || cfg->local_blocks < 0 ||
      cfg->init_blocks + cfg->local_blocks > cfg->topk)
    return MSA_ERR_SHAPE;
  if (cfg->index_dtype != MSA_INDEX_BF16 && cfg->index_dtype != MSA_INDEX_E4M3) return MSA_ERR_DTYPE;
  return MSA_OK;
}

msa_status msa_workspace_size(const msa_config* cfg, int mode, int64_t n, int max_blocks, size_t* bytes) {
  if (!cfg || !bytes) return MSA_ERR_NULL;
  msa_status st = msa_config_check(cfg);
  if (st != MSA_OK) return st;
  if (n < 1 || max_blocks < 1) return MSA_ERR_SHAPE;
  if (mode == MSA_MODE_PACK) {
    // n = batch * seq, max_blocks = batch
    if (n % max_blocks || n / max_blocks > 0x7fffffffLL) return MSA_ERR_SHAPE;
    *bytes = kHeaderBytes + pack_workspace_bytes(max_blocks, static_cast<int>(n / max_blocks));
    return MSA_OK;
  }
  if (mode != MSA_MODE_DECODE && mode != MSA_MODE_PREFILL && mode != MSA_MODE_PREFILL_BWD) return MSA_ERR_SHAPE;
  if (mode != MSA_MODE_DECODE && !prefill_attend_fits(n, max_blocks * kBlock, cfg->topk)) return MSA_ERR_SHAPE;
  *bytes = layout(mode, n, max_blocks, cfg->topk).total;
  return MSA_OK;
}

msa_status msa_workspace_init(void* workspace, size_t bytes, void* stream) {
  if (!workspace) return MSA_ERR_NULL;
  return cuda_result(cudaMemsetAsync(workspace, 0, bytes, static_cast<cudaStream_t>(stream)));
}

msa_status msa_read_device_error(void* workspace, void* stream, int* code, int64_t* detail) {
  if (!workspace || !code) return MSA_ERR_NULL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  DevError h{};
  if (const cudaError_t ce = cudaMemcpyAsync(&h, workspace, sizeof(h), cudaMemcpyDeviceToHost, s); ce != cudaSuccess)
    return cuda_fail(ce);
  if (const cudaError_t ce = cudaMemsetAsync(workspace, 0, sizeof(DevError), s); ce != cudaSuccess)
    return cuda_fail(ce);
  if (const cudaError_t ce = cudaStreamSynchronize(s); ce != cudaSuccess) return cuda_fail(ce);
  *code = h.code;
  if (detail) *detail = h.detail;
  return MSA_OK;
}

msa_status msa_check_bounded_wait(void* workspace, void* stream, int64_t* waits_ns) {
  if (!workspace || !waits_ns) return MSA_ERR_NULL;
  if (reinterpret_cast<uintptr_t>(workspace) & 255) return MSA_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  // the two durations go to the header, after the error word
  long long* dev_waits = reinterpret_cast<long long*>(ws + 64);
  long long h[2] = {0, 0};
  if (const cudaError_t ce = launch_wait_check(reinterpret_cast<DevError*>(ws), dev_waits, s); ce != cudaSuccess)
    return cuda_fail(ce);
  if (const cudaError_t ce = cudaMemcpyAsync(h, dev_waits, sizeof(h), cudaMemcpyDeviceToHost, s); ce != cudaSuccess)
    return cuda_fail(ce);
  if (const cudaError_t ce = cudaStreamSynchronize(s); ce != cudaSuccess) return cuda_fail(ce);
  waits_ns[0] = h[0];
  waits_ns[1] = h[1];
  return MSA_OK;
}

int msa_last_cuda_error(void) { return msa::g_last_cuda_error; }

const char* msa_cuda_error_string(int code) { return cudaGetErrorString(static_cast<cudaError_t>(code)); }

const char* msa_status_string(msa_status s) {
  switch (s) {
    case MSA_OK: return "ok";
    case MSA_ERR_NULL: return "null pointer";
    case MSA_ERR_SHAPE: return "unsupported topology or inconsistent sizes";
    case MSA_ERR_DTYPE: return "unsupported dtype";
    case MSA_ERR_WORKSPACE: return "workspace missing, too small or misaligned";
    case MSA_ERR_ALIGN: return "tensor pointer not 16-byte aligned";
    case MSA_ERR_CUDA: return "CUDA error";
    case MSA_ERR_DOC_MAP: return "malformed document map";
  }
  return "unknown status";
}

static msa_status check_ws(void* ws, size_t have, size_t need) {
  if (!ws) return MSA_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(ws) & 255) return MSA_ERR_WORKSPACE;
  if (have < need) return MSA_ERR_WORKSPACE;
  return MSA_OK;
}

static msa_status check_decode_geom(const int32_t* seq_lens, const int32_t* page_table, const int64_t* cu_k,
                                    int batch, int max_blocks, int64_t num_slots) {
  if (!seq_lens || (!page_table && !cu_k)) return MSA_ERR_NULL;
  if (batch < 1 || max_blocks < 1 || num_slots < 1 || num_slots >= (1LL << 31)) return MSA_ERR_SHAPE;
  if (page_table && num_slots % kBlock) return MSA_ERR_SHAPE;
  return MSA_OK;
}

msa_status msa_select_blocks_decode(const msa_config* cfg, const void* index_q, const void* index_k_cache,
                                    const int32_t* seq_lens, const int32_t* page_table, const int64_t* cu_seqlens_k,
                                    int batch, int max_blocks, int64_t num_slots, int32_t* q2k, void* workspace,
                                    size_t workspace_bytes, void* stream) {
  msa_status st = msa_config_check(cfg);
  if (st != MSA_OK) return st;
  if (!index_q || !index_k_cache || !q2k) return MSA_ERR_NULL;
  if ((st = check_decode_geom(seq_lens, page_table, cu_seqlens_k, batch, max_blocks, num_slots)) != MSA_OK) return st;
  if (!aligned16(index_q) || !aligned16(index_k_cache)) return MSA_ERR_ALIGN;
  const Layout L = layout(MSA_MODE_DECODE, batch, max_blocks, cfg->topk);
  if ((st = check_ws(workspace, workspace_bytes, L.total)) != MSA_OK) return st;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = launch_decode_select(*cfg, index_q, index_k_cache, seq_lens, page_table, cu_seqlens_k, batch,
                                       max_blocks, num_slots, q2k, reinterpret_cast<float*>(ws + L.scores),
                                       reinterpret_cast<int*>(ws + kSelSchedOffset), reinterpret_cast<DevError*>(ws), s);
  return cuda_result(e);
}

static msa_status attend_decode(const msa_config* cfg, const void* q, const void* k_cache, const void* v_cache,
                                const int32_t* q2k, const int32_t* seq_lens, const int32_t* page_table,
                                const int64_t* cu_seqlens_k, int batch, int max_blocks, int64_t num_slots,
                                float scale, void* out, uint8_t* out_q, uint8_t* out_scale, void* workspace,
                                size_t workspace_bytes, void* stream, int kv_fp8 = 0, float k_scale = 1.f,
                                float v_scale = 1.f) {
  msa_status st = msa_config_check(cfg);
  if (st != MSA_OK) return st;
  if (!q || !k_cache || !v_cache || !q2k || (!out && !(out_q && out_scale))) return MSA_ERR_NULL;
  if ((st = check_decode_geom(seq_lens, page_table, cu_seqlens_k, batch, max_blocks, num_slots)) != MSA_OK) return st;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || (out && !aligned16(out)) ||
      (out_q && !aligned16(out_q)))
    return MSA_ERR_ALIGN;
  const Layout L = layout(MSA_MODE_DECODE, batch, max_blocks, cfg->topk);
  if ((st = check_ws(workspace, workspace_bytes, L.total)) != MSA_OK) return st;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the merge tickets start at zero: the workspace was zero-filled once and
  // every call leaves them at zero (the CTA that completes a segment resets
  // it); no other region of any decode call overlaps them
  AttnGeom geo{batch, seq_lens, page_table, cu_seqlens_k, max_blocks, num_slots};
  cudaError_t e = launch_sparse_attend(geo, q, k_cache, v_cache, q2k, cfg->topk, scale, out, out_q, out_scale,
                                       reinterpret_cast<float*>(ws + L.partials),
                                       reinterpret_cast<int*>(ws + L.att_tickets), reinterpret_cast<DevError*>(ws), s,
                                       kv_fp8, k_scale, v_scale);
  return cuda_result(e);
}

msa_status msa_sparse_attend_decode(const msa_config* cfg, const void* q, const void* k_cache, const void* v_cache,
                                    const int32_t* q2k, const int32_t* seq_lens, const int32_t* page_table,
                                    const int64_t* cu_seqlens_k, int batch, int max_blocks, int64_t num_slots,
                                    float scale, void* out, void* workspace, size_t workspace_bytes, void* stream) {
  if (!out) return MSA_ERR_NULL;
  return attend_decode(cfg, q, k_cache, v_cache, q2k, seq_lens, page_table, cu_seqlens_k, batch, max_blocks,
                       num_slots, scale, out, nullptr, nullptr, workspace, workspace_bytes, stream);
}

msa_status msa_sparse_attend_decode_mxfp8(const msa_config* cfg, const void* q, const void* k_cache,
                                          const void* v_cache, const int32_t* q2k, const int32_t* seq_lens,
                                          const int32_t* page_table, const int64_t* cu_seqlens_k, int batch,
                                          int max_blocks, int64_t num_slots, float scale, void* out_q,
                                          void* out_scale, void* workspace, size_t workspace_bytes, void* stream) {
  if (!out_q || !out_scale) return MSA_ERR_NULL;
  return attend_decode(cfg, q, k_cache, v_cache, q2k, seq_lens, page_table, cu_seqlens_k, batch, max_blocks,
                       num_slots, scale, nullptr, static_cast<uint8_t*>(out_q), static_cast<uint8_t*>(out_scale),
                       workspace, workspace_bytes, stream);
}

msa_status msa_sparse_attend_decode_fp8kv(const msa_config* cfg, const void* q, const void* k_cache,
                                          const void* v_cache, float k_scale, float v_scale, const int32_t* q2k,
                                          const int32_t* seq_lens, const int32_t* page_table,
                                          const int64_t* cu_seqlens_k, int batch, int max_blocks,
                                          int64_t num_slots, float scale, void* out, void* workspace,
                                          size_t workspace_bytes, void* stream) {
  if (!out) return MSA_ERR_NULL;
  if (!(k_scale > 0.f) || !(v_scale > 0.f) || !std::isfinite(k_scale) || !std::isfinite(v_scale))
    return MSA_ERR_SHAPE;
  return attend_decode(cfg, q, k_cache, v_cache, q2k, seq_lens, page_table, cu_seqlens_k, batch, max_blocks,
                       num_slots, scale, out, nullptr, nullptr, workspace, workspace_bytes, stream, 1, k_scale,
                       v_scale);
}

static msa_status check_prefill_geom(const int32_t* cu_seqlens, int num_docs, int64_t total_tokens, int max_seqlen) {
  if (!cu_seqlens) return MSA_ERR_NULL;
  if (num_docs < 1 || total_tokens < 1 || total_tokens >= (1LL << 31) || max_seqlen < 1 ||
      max_seqlen > total_tokens || num_docs > total_tokens)
    return MSA_ERR_SHAPE;
  return MSA_OK;
}

msa_status msa_select_blocks_prefill(const msa_config* cfg, const void* index_q, const void* index_k,
                                     const int32_t* cu_seqlens, int num_docs, int64_t total_tokens, int max_seqlen,
                                     int32_t* q2k, void* workspace, size_t workspace_bytes, void* stream) {
  msa_status st = msa_config_check(cfg);
  if (st != MSA_OK) return st;
  if (!index_q || !index_k || !q2k) return MSA_ERR_NULL;
  if ((st = check_prefill_geom(cu_seqlens, num_docs, total_tokens, max_seqlen)) != MSA_OK) return st;
  if (!aligned16(index_q) || !aligned16(index_k) || !aligned16(q2k)) return MSA_ERR_ALIGN;
  const int max_tiles = (max_seqlen + kBlock - 1) / kBlock;
  // the scorer's plan keeps three ints per 128-token block of the longest document on chip
  if ((3LL * max_tiles + 2) * 4 > 200 * 1024) return MSA_ERR_SHAPE;
  const Layout L = layout(MSA_MODE_PREFILL, total_tokens, max_tiles, cfg->topk);
  if ((st = check_ws(workspace, workspace_bytes, L.total)) != MSA_OK) return st;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  cudaError_t e = launch_prefill_select(*cfg, index_q, index_k, cu_seqlens, num_docs, total_tokens, max_seqlen, q2k,
                                        reinterpret_cast<int*>(ws + L.plan), reinterpret_cast<DevError*>(ws),
                                        static_cast<cudaStream_t>(stream));
  return cuda_result(e);
}

static msa_status attend_prefill(const msa_config* cfg, const void* q, const void* k, const void* v,
                                 const int32_t* q2k, const int32_t* cu_seqlens, int num_docs, int64_t total_tokens,
                                 int max_seqlen, float scale, void* out, float* lse, void* workspace,
                                 size_t workspace_bytes, void* stream) {
  msa_status st = msa_config_check(cfg);
  if (st != MSA_OK) return st;
  if (!q || !k || !v || !q2k || !out) return MSA_ERR_NULL;
  if ((st = check_prefill_geom(cu_seqlens, num_docs, total_tokens, max_seqlen)) != MSA_OK) return st;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return MSA_ERR_ALIGN;
  const int max_tiles = (max_seqlen + kBlock - 1) / kBlock;
  const Layout L = layout(MSA_MODE_PREFILL, total_tokens, max_tiles, cfg->topk);
  if ((st = check_ws(workspace, workspace_bytes, L.total)) != MSA_OK) return st;
  if (!prefill_attend_fits(total_tokens, max_seqlen, cfg->topk)) return MSA_ERR_SHAPE;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  cudaError_t e = launch_prefill_attend(q, k, v, q2k, cu_seqlens, num_docs, total_tokens, max_seqlen, cfg->topk,
                                        scale, out, lse, ws + L.bm, reinterpret_cast<DevError*>(ws),
                                        static_cast<cudaStream_t>(stream));
  return cuda_result(e);
}

msa_status msa_sparse_attend_prefill(const msa_config* cfg, const void* q, const void* k, const void* v,
                                     const int32_t* q2k, const int32_t* cu_seqlens, int num_docs,
                                     int64_t total_tokens, int max_seqlen, float scale, void* out, void* workspace,
                                     size_t workspace_bytes, void* stream) {
  return attend_prefill(cfg, q, k, v, q2k, cu_seqlens, num_docs, total_tokens, max_seqlen, scale, out, nullptr,
                        workspace, workspace_bytes, stream);
}

msa_status msa_sparse_attend_prefill_lse(const msa_config* cfg, const void* q, const void* k, const void* v,
                                         const int32_t* q2k, const int32_t* cu_seqlens, int num_docs,
                                         int64_t total_tokens, int max_seqlen, float scale, void* out, float* lse,
                                         void* workspace, size_t workspace_bytes, void* stream) {
  if (!lse) return MSA_ERR_NULL;
  return attend_prefill(cfg, q, k, v, q2k, cu_seqlens, num_docs, total_tokens, max_seqlen, scale, out, lse,
                        workspace, workspace_bytes, stream);
}

msa_status msa_sparse_attend_prefill_backward(const msa_config* cfg, const void* q, const void* k, const void* v,
                                              const int32_t* q2k, const int32_t* cu_seqlens, int num_docs,
                                              int64_t total_tokens, int max_seqlen, float scale, const void* out,
                                              const float* lse, const void* grad_out, void* dq, void* dk, void* dv,
                                              void* workspace, size_t workspace_bytes, void* stream) {
  msa_status st = msa_config_check(cfg);
  if (st != MSA_OK) return st;
  if (!q || !k || !v || !q2k || !out || !lse || !grad_out || !dq || !dk || !dv) return MSA_ERR_NULL;
  if ((st = check_prefill_geom(cu_seqlens, num_docs, total_tokens, max_seqlen)) != MSA_OK) return st;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(grad_out) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv) || !aligned16(lse))
    return MSA_ERR_ALIGN;
  const int max_tiles = (max_seqlen + kBlock - 1) / kBlock;
  const Layout L = layout(MSA_MODE_PREFILL_BWD, total_tokens, max_tiles, cfg->topk);
  if ((st = check_ws(workspace, workspace_bytes, L.total)) != MSA_OK) return st;
  if (!prefill_attend_fits(total_tokens, max_seqlen, cfg->topk)) return MSA_ERR_SHAPE;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  cudaError_t e = launch_prefill_backward(q, k, v, q2k, cu_seqlens, num_docs, total_tokens, max_seqlen, cfg->topk,
                                          scale, out, lse, grad_out, dq, dk, dv, ws + L.bm,
                                          reinterpret_cast<DevError*>(ws), static_cast<cudaStream_t>(stream));
  return cuda_result(e);
}

msa_status msa_index_produce_prefill(const msa_config* cfg, const void* index_q_in, const void* index_k_in,
                                     const int32_t* cu_seqlens, int num_docs, int64_t total_tokens, void* index_q_out,
                                     void* index_k_out, void* index_k_cache, const int32_t* page_table, int max_blocks,
                                     int64_t num_slots, void* workspace, size_t workspace_bytes, void* stream) {
  msa_status st = msa_config_check(cfg);
  if (st != MSA_OK) return st;
  if (!index_q_in || !index_k_in || !cu_seqlens || !index_q_out || (!index_k_out && !index_k_cache))
    return MSA_ERR_NULL;
  if (index_k_cache && !page_table) return MSA_ERR_NULL;
  if (num_docs < 1 || total_tokens < 1 || total_tokens >= (1LL << 31) || num_docs > total_tokens)
    return MSA_ERR_SHAPE;
  if (index_k_cache && (max_blocks < 1 || num_slots < 1 || num_slots >= (1LL << 31) || num_slots % kBlock))
    return MSA_ERR_SHAPE;
  if (!aligned16(index_q_in) || !aligned16(index_k_in) || !aligned16(index_q_out) ||
      (index_k_out && !aligned16(index_k_out)) || (index_k_cache && !aligned16(index_k_cache)))
    return MSA_ERR_ALIGN;
  if ((st = check_ws(workspace, workspace_bytes, kHeaderBytes)) != MSA_OK) return st;
  IpLaunch L{};
  L.q_in = index_q_in;
  L.k_in = index_k_in;
  L.n = total_tokens;
  L.q_out = index_q_out;
  L.k_out = index_k_out;
  L.cache = index_k_cache;
  L.num_slots = num_slots;
  L.e4m3 = cfg->index_dtype == MSA_INDEX_E4M3;
  L.decode = 0;
  L.cu = cu_seqlens;
  L.num_docs = num_docs;
  L.page_table = page_table;
  L.max_blocks = max_blocks;
  L.err = static_cast<DevError*>(workspace);
  return cuda_result(launch_index_produce(L, static_cast<cudaStream_t>(stream)));
}

msa_status msa_index_produce_decode(const msa_config* cfg, const void* index_q_in, const void* index_k_in,
                                    const int32_t* seq_lens, const int32_t* page_table, const int64_t* cu_seqlens_k,
                                    int batch, int max_blocks, int64_t num_slots, void* index_q_out,
                                    void* index_k_cache, void* workspace, size_t workspace_bytes, void* stream) {
  msa_status st = msa_config_check(cfg);
  if (st != MSA_OK) return st;
  if (!index_q_in || !index_k_in || !index_q_out || !index_k_cache) return MSA_ERR_NULL;
  if ((st = check_decode_geom(seq_lens, page_table, cu_seqlens_k, batch, max_blocks, num_slots)) != MSA_OK) return st;
  if (!aligned16(index_q_in) || !aligned16(index_k_in) || !aligned16(index_q_out) || !aligned16(index_k_cache))
    return MSA_ERR_ALIGN;
  if ((st = check_ws(workspace, workspace_bytes, kHeaderBytes)) != MSA_OK) return st;
  IpLaunch L{};
  L.q_in = index_q_in;
  L.k_in = index_k_in;
  L.n = batch;
  L.q_out = index_q_out;
  L.cache = index_k_cache;
  L.num_slots = num_slots;
  L.e4m3 = cfg->index_dtype == MSA_INDEX_E4M3;
  L.decode = 1;
  L.seq_lens = seq_lens;
  L.page_table = page_table;
  L.cu_k = cu_seqlens_k;
  L.max_blocks = max_blocks;
  L.err = static_cast<DevError*>(workspace);
  return cuda_result(launch_index_produce(L, static_cast<cudaStream_t>(stream)));
}

msa_status msa_pack_metadata(const int64_t* doc_ids, int batch, int seq, int32_t* cu_seqlens, int64_t* token_rows,
                             int* num_docs, int64_t* total_tokens, int* max_seqlen, int64_t* bad_index,
                             void* workspace, size_t workspace_bytes, void* stream) {
  if (bad_index) *bad_index = -1;
  if (!doc_ids || !cu_seqlens || !token_rows || !num_docs || !total_tokens || !max_seqlen) return MSA_ERR_NULL;
  if (batch < 1 || seq < 1) return MSA_ERR_DOC_MAP;                                // empty map
  if (static_cast<long long>(batch) * seq > 0x7fffffffLL) return MSA_ERR_DOC_MAP;  // past int32
  msa_status st = check_ws(workspace, workspace_bytes, kHeaderBytes + pack_workspace_bytes(batch, seq));
  if (st != MSA_OK) return st;
  return run_pack_metadata(doc_ids, batch, seq, cu_seqlens, token_rows, num_docs, total_tokens, max_seqlen, bad_index,
                           static_cast<uint8_t*>(workspace) + kHeaderBytes, static_cast<cudaStream_t>(stream));
}

msa_status msa_pack(const void* external, const int64_t* token_rows, int64_t total_tokens, int64_t row_bytes,
                    void* packed, void* stream) {
  if (!external || !token_rows || !packed) return MSA_ERR_NULL;
  if (total_tokens < 0 || row_bytes < 16 || row_bytes % 16) return MSA_ERR_SHAPE;
  if (!aligned16(external) || !aligned16(packed)) return MSA_ERR_ALIGN;
  return run_gather(external, token_rows, total_tokens, row_bytes, packed, static_cast<cudaStream_t>(stream), false);
}

msa_status msa_unpack(const void* packed, const int64_t* token_rows, int64_t total_tokens, int64_t batch_seq,
                      int64_t row_bytes, void* external, void* stream) {
  if (!external || !token_rows || !packed) return MSA_ERR_NULL;
  if (total_tokens < 0 || batch_seq < total_tokens || row_bytes < 16 || row_bytes % 16) return MSA_ERR_SHAPE;
  if (!aligned16(external) || !aligned16(packed)) return MSA_ERR_ALIGN;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (const cudaError_t ce = cudaMemsetAsync(external, 0, static_cast<size_t>(batch_seq) * row_bytes, s); ce != cudaSuccess)
    return cuda_fail(ce);
  return run_gather(packed, token_rows, total_tokens, row_bytes, external, s, true);
}

}  // extern "C"
