// pack.cu -- packed layout of a document map, and the gather / scatter between
// the [batch, seq, ...] and compact [tokens, ...] layouts.
//
// NeMo "...minimax_m3_vl.msa": the layout-from-doc_ids constructor (derives the
// packed layout with exactly one device-to-host synchronisation; rejects an
// empty map, negative ids, no real token, an interrupted document, coordinates
// past int32), _contiguous_runs (every document one contiguous run; the first
// bad flat row), MSAMicrobatch.pack and MSAMicrobatch.unpack (zero padding).
// The per-token request / position metadata of the vLLM ROCm page
// (MiniMaxM3SparseRocmNvfp4MetadataBuilder) is derived on the device from
// cu_seqlens by the attention kernels.
//
// All HBM-bound: one CTA per row of the map for the run analysis (run starts,
// an open-addressing hash of run ids per row to find a document id that occurs
// in two runs), one small scan over rows, one CTA per row to emit cu_seqlens
// and token_rows, and a final reduction to the scalars the host reads back.
#include "launch.h"

namespace msa {

constexpr int kPackThreads = 1024;

struct PackSummary {
  int num_docs;
  int max_seqlen;
  long long total_tokens;
  long long first_negative;     // smallest flat index of a negative id
  long long first_interrupted;  // smallest flat index starting a repeated run
};

__device__ __forceinline__ unsigned long long mix64(unsigned long long x) {
  // splitmix64 finaliser
  x ^= x >> 30;
  x *= 0xbf58476d1ce4e5b9ull;
  x ^= x >> 27;
  x *= 0x94d049bb133111ebull;
  x ^= x >> 31;
  return x;
}

__device__ __forceinline__ bool is_run_start(const int64_t* row, int i) {
  const int64_t id = row[i];
  return id > 0 && (i == 0 || row[i - 1] != id);
}

// Per row: counts, negative ids, repeated run ids.
__global__ void __launch_bounds__(kPackThreads) pack_rows_kernel(const int64_t* __restrict__ ids, int seq, int cap,
                                                                 unsigned long long* __restrict__ keys,
                                                                 int* __restrict__ minpos, int* __restrict__ row_real,
                                                                 int* __restrict__ row_runs, PackSummary* sum) {
  const int r = blockIdx.x, tid = threadIdx.x;
  const int64_t* row = ids + static_cast<long long>(r) * seq;
  unsigned long long* K = keys + static_cast<long long>(r) * cap;
  int* P = minpos + static_cast<long long>(r) * cap;
  for (int i = tid; i < cap; i += kPackThreads) {
    K[i] = 0ull;
    P[i] = 0x7fffffff;
  }
  __syncthreads();
  int real = 0, runs = 0;
  const int bits = 31 - __clz(cap);
  for (int i = tid; i < seq; i += kPackThreads) {
    const int64_t id = row[i];
    if (id < 0)
      atomicMin(reinterpret_cast<unsigned long long*>(&sum->first_negative),
                static_cast<unsigned long long>(static_cast<long long>(r) * seq + i));
    if (id > 0) ++real;
    if (is_run_start(row, i)) {
      ++runs;
      unsigned slot = static_cast<unsigned>(mix64(static_cast<unsigned long long>(id)) >> (64 - bits));
      for (int probe = 0; probe < cap; ++probe) {
        const unsigned long long prev = atomicCAS(&K[slot], 0ull, static_cast<unsigned long long>(id));
        if (prev == 0ull || prev == static_cast<unsigned long long>(id)) {
          atomicMin(&P[slot], i);
          break;
        }
        slot = (slot + 1) & (cap - 1);
      }
    }
  }
  __syncthreads();
  for (int i = tid; i < seq; i += kPackThreads) {
    if (!is_run_start(row, i)) continue;
    const int64_t id = row[i];
    unsigned slot = static_cast<unsigned>(mix64(static_cast<unsigned long long>(id)) >> (64 - bits));
    for (int probe = 0; probe < cap; ++probe) {
      if (K[slot] == static_cast<unsigned long long>(id)) {
        if (P[slot] < i)
          atomicMin(reinterpret_cast<unsigned long long*>(&sum->first_interrupted),
                    static_cast<unsigned long long>(static_cast<long long>(r) * seq + i));
        break;
      }
      slot = (slot + 1) & (cap - 1);
    }
  }
  for (int o = 16; o > 0; o >>= 1) {
    real += __shfl_xor_sync(0xffffffffu, real, o);
    runs += __shfl_xor_sync(0xffffffffu, runs, o);
  }
  __shared__ int sr[32], sn[32];
  if ((tid & 31) == 0) {
    sr[tid >> 5] = real;
    sn[tid >> 5] = runs;
  }
  __syncthreads();
  if (tid == 0) {
    int a = 0, b = 0;
    for (int w = 0; w < kPackThreads / 32; ++w) {
      a += sr[w];
      b += sn[w];
    }
    row_real[r] = a;
    row_runs[r] = b;
  }
}

// One thread: exclusive offsets over rows (in place: row_real -> token offset, row_runs -> doc offset).
__global__ void pack_offsets_kernel(int batch, int* __restrict__ row_real, int* __restrict__ row_runs,
                                    int32_t* __restrict__ cu_seqlens, PackSummary* sum) {
  if (threadIdx.x != 0) return;
  long long tok = 0, docs = 0;
  for (int r = 0; r < batch; ++r) {
    const int a = row_real[r], b = row_runs[r];
    row_real[r] = static_cast<int>(tok);
    row_runs[r] = static_cast<int>(docs);
    tok += a;
    docs += b;
  }
  sum->total_tokens = tok;
  sum->num_docs = static_cast<int>(docs);
  cu_seqlens[docs] = static_cast<int32_t>(tok);
}

// Per row: block-wide prefix over positions -> token_rows and cu_seqlens.
__global__ void __launch_bounds__(kPackThreads) pack_emit_kernel(const int64_t* __restrict__ ids, int seq,
                                                                 const int* __restrict__ tok_off,
                                                                 const int* __restrict__ doc_off,
                                                                 int32_t* __restrict__ cu_seqlens,
                                                                 int64_t* __restrict__ token_rows) {
  const int r = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t* row = ids + static_cast<long long>(r) * seq;
  __shared__ int wr[32], wn[32];
  int carry_real = tok_off[r], carry_runs = doc_off[r];
  for (int base = 0; base < seq; base += kPackThreads) {
    const int i = base + tid;
    const bool real = i < seq && row[i] > 0;
    const bool start = i < seq && is_run_start(row, i);
    int xr = real, xn = start;
    for (int o = 1; o < 32; o <<= 1) {
      const int yr = __shfl_up_sync(0xffffffffu, xr, o), yn = __shfl_up_sync(0xffffffffu, xn, o);
      if (lane >= o) {
        xr += yr;
        xn += yn;
      }
    }
    if (lane == 31) {
      wr[warp] = xr;
      wn[warp] = xn;
    }
    __syncthreads();
    int pr = 0, pn = 0, tr = 0, tn = 0;
    for (int w = 0; w < kPackThreads / 32; ++w) {
      if (w < warp) {
        pr += wr[w];
        pn += wn[w];
      }
      tr += wr[w];
      tn += wn[w];
    }
    const int real_idx = carry_real + pr + xr - (real ? 1 : 0);
    const int run_idx = carry_runs + pn + xn - (start ? 1 : 0);
    if (real) token_rows[real_idx] = static_cast<long long>(r) * seq + i;
    if (start) cu_seqlens[run_idx] = real_idx;
    carry_real += tr;
    carry_runs += tn;
    __syncthreads();
  }
}

__global__ void pack_finish_kernel(const int32_t* __restrict__ cu_seqlens, PackSummary* sum) {
  __shared__ int smax[32];
  const int nd = sum->num_docs;
  int m = 0;
  for (int d = threadIdx.x; d < nd; d += blockDim.x) m = max(m, cu_seqlens[d + 1] - cu_seqlens[d]);
  for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) smax[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    int x = 0;
    for (int w = 0; w < (blockDim.x + 31) / 32; ++w) x = max(x, smax[w]);
    sum->max_seqlen = x;
  }
}

__global__ void gather_rows_kernel(const uint4* __restrict__ src, const int64_t* __restrict__ rows, long long n,
                                   long long vec_per_row, uint4* __restrict__ dst) {
  const long long total = n * vec_per_row;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long t = i / vec_per_row, v = i % vec_per_row;
    dst[i] = src[rows[t] * vec_per_row + v];
  }
}

__global__ void scatter_rows_kernel(const uint4* __restrict__ src, const int64_t* __restrict__ rows, long long n,
                                    long long vec_per_row, uint4* __restrict__ dst) {
  const long long total = n * vec_per_row;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long t = i / vec_per_row, v = i % vec_per_row;
    dst[rows[t] * vec_per_row + v] = src[i];
  }
}

// ---- host side --------------------------------------------------------------------
static int pack_table_cap(int seq) {
  int cap = 1;
  while (cap < 2 * seq) cap <<= 1;
  return cap;
}

static size_t up256(size_t x) { return (x + 255) / 256 * 256; }

size_t pack_workspace_bytes(int batch, int seq) {
  const size_t cap = static_cast<size_t>(pack_table_cap(seq));
  return up256(batch * cap * 8) + up256(batch * cap * 4) + up256(2 * static_cast<size_t>(batch) * 4) + 256;
}

msa_status run_pack_metadata(const int64_t* ids, int batch, int seq, int32_t* cu_seqlens, int64_t* token_rows,
                             int* num_docs, int64_t* total_tokens, int* max_seqlen, int64_t* bad_index,
                             uint8_t* ws, cudaStream_t stream) {
  if (const cudaError_t e0 = launch_prologue(); e0 != cudaSuccess) return cuda_fail(e0);
  const int cap = pack_table_cap(seq);
  const size_t cap_b = static_cast<size_t>(cap);
  uint8_t* p = ws;
  auto* keys = reinterpret_cast<unsigned long long*>(p);
  p += up256(batch * cap_b * 8);
  auto* minpos = reinterpret_cast<int*>(p);
  p += up256(batch * cap_b * 4);
  int* row_real = reinterpret_cast<int*>(p);
  int* row_runs = row_real + batch;
  p += up256(2 * static_cast<size_t>(batch) * 4);
  auto* sum = reinterpret_cast<PackSummary*>(p);

  PackSummary init{0, 0, 0, 0x7fffffffffffffffLL, 0x7fffffffffffffffLL};
  if (const cudaError_t ce = cudaMemcpyAsync(sum, &init, sizeof(init), cudaMemcpyHostToDevice, stream); ce != cudaSuccess)
    return cuda_fail(ce);
  pack_rows_kernel<<<batch, kPackThreads, 0, stream>>>(ids, seq, cap, keys, minpos, row_real, row_runs, sum);
  pack_offsets_kernel<<<1, 32, 0, stream>>>(batch, row_real, row_runs, cu_seqlens, sum);
  pack_emit_kernel<<<batch, kPackThreads, 0, stream>>>(ids, seq, row_real, row_runs, cu_seqlens, token_rows);
  pack_finish_kernel<<<1, 1024, 0, stream>>>(cu_seqlens, sum);
  if (const cudaError_t ce = cudaGetLastError(); ce != cudaSuccess) return cuda_fail(ce);
  PackSummary h;
  if (const cudaError_t ce = cudaMemcpyAsync(&h, sum, sizeof(h), cudaMemcpyDeviceToHost, stream); ce != cudaSuccess)
    return cuda_fail(ce);
  if (const cudaError_t ce = cudaStreamSynchronize(stream); ce != cudaSuccess) return cuda_fail(ce);
  if (bad_index) *bad_index = -1;
  if (h.first_negative != 0x7fffffffffffffffLL) {
    if (bad_index) *bad_index = h.first_negative;
    return MSA_ERR_DOC_MAP;
  }
  if (h.first_interrupted != 0x7fffffffffffffffLL) {
    if (bad_index) *bad_index = h.first_interrupted;
    return MSA_ERR_DOC_MAP;
  }
  if (h.total_tokens == 0) return MSA_ERR_DOC_MAP;
  *num_docs = h.num_docs;
  *total_tokens = h.total_tokens;
  *max_seqlen = h.max_seqlen;
  return MSA_OK;
}

msa_status run_gather(const void* src, const int64_t* rows, long long n, long long row_bytes, void* dst,
                      cudaStream_t stream, bool scatter) {
  if (const cudaError_t e0 = launch_prologue(); e0 != cudaSuccess) return cuda_fail(e0);
  const long long vpr = row_bytes / 16;
  const long long total = n * vpr;
  if (total == 0) return MSA_OK;
  const long long want = (total + 255) / 256;
  const int grid = static_cast<int>(want < 8LL * kNumSMs ? want : 8LL * kNumSMs);
  if (scatter)
    scatter_rows_kernel<<<grid, 256, 0, stream>>>(static_cast<const uint4*>(src), rows, n, vpr,
                                                  static_cast<uint4*>(dst));
  else
    gather_rows_kernel<<<grid, 256, 0, stream>>>(static_cast<const uint4*>(src), rows, n, vpr,
                                                 static_cast<uint4*>(dst));
  return cuda_result(cudaGetLastError());
}

}  // namespace msa
