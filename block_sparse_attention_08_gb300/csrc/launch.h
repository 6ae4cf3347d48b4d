// launch.h -- host-side launcher declarations shared by the libmsa sources.
#pragma once

#include "common.cuh"

namespace msa {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn get_encode_tiled();

// Geometry of the requests of one decode attention call.
struct AttnGeom {
  int nq;                     // requests
  const int32_t* seq_lens;    // [nq]
  const int32_t* page_table;  // [nq, max_blocks] or null (contiguous cache)
  const int64_t* cu_k;        // [nq + 1] when contiguous
  int max_blocks;
  long long num_rows;         // slots of the K/V cache
};

cudaError_t launch_decode_select(const msa_config& cfg, const void* index_q, const void* index_k,
                                 const int32_t* seq_lens, const int32_t* page_table, const int64_t* cu_k,
                                 int batch, int max_blocks, long long num_slots, int32_t* q2k, float* scores,
                                 int* sched, DevError* err, cudaStream_t stream);
// Offset in the workspace header of the decode scorer's page-claim counter
// (zero between calls: the top-k kernel puts it back once the scorer grid has
// completed).
constexpr size_t kSelSchedOffset = 128;
// kv_fp8: the K / V caches hold E4M3 bytes standing for k_scale * k and v_scale * v.
cudaError_t launch_sparse_attend(const AttnGeom& geo, const void* q, const void* k, const void* v,
                                 const int32_t* q2k, int topk, float scale, void* out, uint8_t* out_q,
                                 uint8_t* out_scale, float* partials, int* tickets, DevError* err,
                                 cudaStream_t stream, int kv_fp8 = 0, float k_scale = 1.f, float v_scale = 1.f);
size_t attend_partials_bytes();
size_t attend_tickets_bytes();
size_t prefill_plan_ints(int num_docs, int max_tiles);
cudaError_t launch_prefill_select(const msa_config& cfg, const void* index_q, const void* index_k,
                                  const int32_t* cu_seqlens, int num_docs, long long total_tokens, int max_seqlen,
                                  int32_t* q2k, int* plan_ints, DevError* err, cudaStream_t stream);
size_t prefill_attend_bytes(long long total_tokens, int max_seqlen, int topk);
bool prefill_attend_fits(long long total_tokens, int max_seqlen, int topk);
cudaError_t launch_prefill_attend(const void* q, const void* k, const void* v, const int32_t* q2k,
                                  const int32_t* cu_seqlens, int num_docs, long long total_tokens, int max_seqlen,
                                  int topk, float scale, void* out, float* lse, uint8_t* region, DevError* err,
                                  cudaStream_t stream);
size_t prefill_backward_bytes(long long total_tokens, int max_seqlen, int topk);
cudaError_t launch_prefill_backward(const void* q, const void* k, const void* v, const int32_t* q2k,
                                    const int32_t* cu_seqlens, int num_docs, long long total_tokens,
                                    int max_seqlen, int topk, float scale, const void* out, const float* lse,
                                    const void* grad_out, void* dq, void* dk, void* dv, uint8_t* region,
                                    DevError* err, cudaStream_t stream);
size_t pack_workspace_bytes(int batch, int seq);
// One index-producer call: n tokens (prefill) or requests (decode).
struct IpLaunch {
  const void* q_in;           // bf16 [n, 4, 128]
  const void* k_in;           // bf16 [n, 1, 128]
  long long n;
  void* q_out;                // [n, 4, 128] in the index dtype
  void* k_out;                // packed [n, 1, 128] in the index dtype, or null
  void* cache;                // paged / contiguous index-K cache [num_slots, 1, 128], or null
  long long num_slots;
  int e4m3;
  int decode;                 // 1: request r's new key sits at position seq_lens[r] - 1
  const int32_t* cu;          // prefill: [num_docs + 1]
  int num_docs;
  const int32_t* seq_lens;    // decode: [n]
  const int32_t* page_table;  // [n or num_docs, max_blocks], or null
  const int64_t* cu_k;        // decode, contiguous cache: [n + 1]
  int max_blocks;
  DevError* err;
};
cudaError_t launch_index_produce(const IpLaunch& L, cudaStream_t stream);
// First step of every launcher.  Clears the calling thread's last CUDA error
// (the launches are checked with cudaGetLastError, which reports the calling
// thread's error) and makes the current device's primary context current on
// this thread: a thread that has made no runtime call yet (PyTorch's autograd
// worker is one: PyTorch skips cudaSetDevice when the device is already the
// current one) has no context, and the driver's tensor-map encoder then
// rejects the device pointers as invalid.
inline cudaError_t launch_prologue() {
  (void)cudaGetLastError();
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  return e == cudaSuccess ? cudaSetDevice(dev) : e;
}

// Records a failed CUDA call's code for msa_last_cuda_error (per calling
// thread) and returns MSA_ERR_CUDA; cuda_result maps cudaSuccess to MSA_OK.
msa_status cuda_fail(cudaError_t e);
inline msa_status cuda_result(cudaError_t e) { return e == cudaSuccess ? MSA_OK : cuda_fail(e); }

msa_status run_pack_metadata(const int64_t* ids, int batch, int seq, int32_t* cu_seqlens, int64_t* token_rows,
                             int* num_docs, int64_t* total_tokens, int* max_seqlen, int64_t* bad_index,
                             uint8_t* ws, cudaStream_t stream);
cudaError_t launch_wait_check(DevError* err, long long* waits_ns, cudaStream_t stream);
msa_status run_gather(const void* src, const int64_t* rows, long long n, long long row_bytes, void* dst,
                      cudaStream_t stream, bool scatter);

}  // namespace msa
