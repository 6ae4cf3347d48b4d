// index_produce.cu -- the index producer: L2-normalises the index queries and
// the shared index key of each token, stores them in the index dtype (bf16 or
// unscaled E4M3) and inserts the index key into the paged side index-K cache.
//
// TensorRT-LLM "MiniMaxM3SparseAttentionConfig": field fuse_qkv_index_projection
// (MSA batches use a horizontal norm / RoPE / cache-insertion producer for
// prefill, mixed and CUDA-graph decode), field indexer_kv_dtype (index Q/K are
// stored normalized, as bf16 or unscaled E4M3), and the class description (the
// paged index-K cache [num_slots, 1, 128] parallel to the main K/V cache).
// NeMo "...minimax_m3_vl.msa" select_blocks takes index tensors "post norm".
//
// Precision (the pages fix neither the norm's precision nor its order): in
// IEEE binary32, s = sum over c = 0..127 in that order of x_c^2 (each square is
// exact: a bf16 value has 8 significant bits), r = sqrt(s) and y_c = x_c / r,
// each correctly rounded, then one rounding of y_c to bf16 or E4M3 (nearest,
// ties to even; |y| <= 1 never saturates).  A vector whose s is 0 is stored as
// zeros.  The explicitly rounded intrinsics keep the compiler from contracting
// or reordering any step, so the result is bit-reproducible.
//
// GB300 design: the kernel moves 256 bytes in and 128-256 bytes out per vector
// and does about 150 fp32 operations per vector: it is bound by HBM on large
// prefills and by launch latency on a decode step.  A warp takes 32 vectors:
// it loads them with coalesced 16-byte loads into a padded shared-memory tile
// (row stride 65 words, so the per-row reads of the sequential sum hit 32
// different banks), each lane sums and normalises its own row in index order
// and writes it back to the tile, and the warp stores the tile with coalesced
// 16-byte stores.  RoPE is a rotation and leaves the norm unchanged; the pages
// give no RoPE variant and none is applied.
#include "launch.h"

namespace msa {

constexpr int kIpWarps = 4;
constexpr int kIpThreads = kIpWarps * 32;
constexpr int kIpRowWords = kIdxDim / 2 + 1;  // 64 words of bf16 pairs + 1 word of padding

struct IpSmem {
  uint32_t row[kIpWarps][32][kIpRowWords];
};

// Which rows go where.  Vectors 0 .. 4n-1 are index queries (row v of
// q_in / q_out); vectors 4n .. 5n-1 are the index keys of tokens 0 .. n-1.
struct IpArgs {
  const __nv_bfloat16* q_in;
  const __nv_bfloat16* k_in;
  long long n;          // tokens (prefill) or requests (decode)
  uint8_t* q_out;
  uint8_t* k_out;       // packed [n, 1, 128] or null
  uint8_t* cache;       // [num_slots, 1, 128] or null
  long long num_slots;
  int e4m3;
  int decode;           // 1: one new token per request at position seq_lens[r] - 1
  const int32_t* cu;    // prefill: [num_docs + 1]
  int num_docs;
  const int32_t* seq_lens;    // decode: [n]
  const int32_t* page_table;  // [n or num_docs, max_blocks] or null
  const int64_t* cu_k;        // decode, contiguous cache: [n + 1]
  int max_blocks;
  DevError* err;
};

// Cache slot of the index key of token t, or -1 (recorded in the error word)
// when its page or position is out of range.
__device__ __forceinline__ long long ip_slot(const IpArgs& a, long long t) {
  int r;
  long long p;
  if (a.decode) {
    r = static_cast<int>(t);
    const int L = a.seq_lens[r];
    if (L < 1 || (a.page_table && L > a.max_blocks * kBlock)) {
      record_error(a.err, MSA_DEVERR_LENGTH, t);
      return -1;
    }
    p = L - 1;
  } else {
    int lo = 0, hi = a.num_docs - 1;  // the document d with cu[d] <= t < cu[d + 1]
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (a.cu[mid] <= t) lo = mid;
      else hi = mid - 1;
    }
    r = lo;
    p = t - a.cu[r];
    if (p / kBlock >= a.max_blocks) {
      record_error(a.err, MSA_DEVERR_LENGTH, t);
      return -1;
    }
  }
  long long slot;
  if (a.page_table) {
    const int page = a.page_table[static_cast<long long>(r) * a.max_blocks + p / kBlock];
    slot = static_cast<long long>(page) * kBlock + p % kBlock;
    if (page < 0 || slot >= a.num_slots) {
      record_error(a.err, MSA_DEVERR_PAGE, t);
      return -1;
    }
  } else {
    slot = a.cu_k[r] + p;
    if (slot < 0 || slot >= a.num_slots) {
      record_error(a.err, MSA_DEVERR_PAGE, t);
      return -1;
    }
  }
  return slot;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__global__ void __launch_bounds__(kIpThreads) index_produce_kernel(IpArgs a) {
  __shared__ IpSmem sm;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const long long nvec = 5 * a.n;
  const long long v0 = (static_cast<long long>(blockIdx.x) * kIpWarps + warp) * 32;
  if (v0 >= nvec) return;
  uint32_t(*tile)[kIpRowWords] = sm.row[warp];
  auto src_of = [&](long long v) -> const uint4* {
    return reinterpret_cast<const uint4*>(v < 4 * a.n ? a.q_in + v * kIdxDim : a.k_in + (v - 4 * a.n) * kIdxDim);
  };

  // coalesced load: 16 lanes cover one 256-byte row, two rows per instruction
  const int half = lane >> 4, col = lane & 15;
#pragma unroll 4
  for (int j = 0; j < 16; ++j) {
    const int rr = 2 * j + half;
    const long long v = v0 + rr;
    uint4 x = make_uint4(0u, 0u, 0u, 0u);
    if (v < nvec) x = __ldg(src_of(v) + col);
    tile[rr][4 * col + 0] = x.x;
    tile[rr][4 * col + 1] = x.y;
    tile[rr][4 * col + 2] = x.z;
    tile[rr][4 * col + 3] = x.w;
  }
  __syncwarp();

  // lane l normalises row l: the squares summed in index order, then y = x / r
  {
    uint32_t* row = tile[lane];
    float s = 0.f;
#pragma unroll 8
    for (int w = 0; w < kIdxDim / 2; ++w) {
      const uint32_t p = row[w];
      const float x0 = bf16_lo(p), x1 = bf16_hi(p);
      s = __fadd_rn(s, __fmul_rn(x0, x0));
      s = __fadd_rn(s, __fmul_rn(x1, x1));
    }
    const float r = __fsqrt_rn(s);
    const bool zero = s == 0.f;
    if (a.e4m3) {
      // four E4M3 bytes per word, written over the first 32 words of the row
#pragma unroll 4
      for (int w = 0; w < kIdxDim / 4; ++w) {
        const uint32_t p0 = row[2 * w], p1 = row[2 * w + 1];
        const float y0 = zero ? 0.f : __fdiv_rn(bf16_lo(p0), r), y1 = zero ? 0.f : __fdiv_rn(bf16_hi(p0), r);
        const float y2 = zero ? 0.f : __fdiv_rn(bf16_lo(p1), r), y3 = zero ? 0.f : __fdiv_rn(bf16_hi(p1), r);
        uint16_t lo, hi;
        asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(y1), "f"(y0));
        asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(y3), "f"(y2));
        row[w] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
      }
    } else {
#pragma unroll 8
      for (int w = 0; w < kIdxDim / 2; ++w) {
        const uint32_t p = row[w];
        const float y0 = zero ? 0.f : __fdiv_rn(bf16_lo(p), r), y1 = zero ? 0.f : __fdiv_rn(bf16_hi(p), r);
        const __nv_bfloat162 b = __floats2bfloat162_rn(y0, y1);  // .x = y0 in the low half
        row[w] = *reinterpret_cast<const uint32_t*>(&b);
      }
    }
  }
  __syncwarp();

  // the cache slot of the key rows this warp holds (one lane per row)
  long long slot = -1;
  {
    const long long v = v0 + lane;
    if (a.cache && v < nvec && v >= 4 * a.n) slot = ip_slot(a, v - 4 * a.n);
  }

  // coalesced stores: bf16 rows are 256 bytes (16 lanes), E4M3 rows 128 bytes (8 lanes)
  const int row_bytes = a.e4m3 ? kIdxDim : 2 * kIdxDim;
  const int lanes_per_row = row_bytes / 16, rows_per_step = 32 / lanes_per_row;
  const int sub = lane / lanes_per_row, c16 = lane % lanes_per_row;
  for (int j = 0; j < 32 / rows_per_step; ++j) {
    const int rr = j * rows_per_step + sub;
    const long long v = v0 + rr;
    const uint4 y = make_uint4(tile[rr][4 * c16], tile[rr][4 * c16 + 1], tile[rr][4 * c16 + 2], tile[rr][4 * c16 + 3]);
    const long long sl = __shfl_sync(0xffffffffu, slot, rr);
    if (v >= nvec) continue;
    if (v < 4 * a.n) {
      reinterpret_cast<uint4*>(a.q_out + v * row_bytes)[c16] = y;
    } else {
      const long long t = v - 4 * a.n;
      if (a.k_out) reinterpret_cast<uint4*>(a.k_out + t * row_bytes)[c16] = y;
      if (sl >= 0) reinterpret_cast<uint4*>(a.cache + sl * row_bytes)[c16] = y;
    }
  }
}

cudaError_t launch_index_produce(const IpLaunch& L, cudaStream_t stream) {
  if (const cudaError_t e0 = launch_prologue(); e0 != cudaSuccess) return e0;
  IpArgs a{};
  a.q_in = static_cast<const __nv_bfloat16*>(L.q_in);
  a.k_in = static_cast<const __nv_bfloat16*>(L.k_in);
  a.n = L.n;
  a.q_out = static_cast<uint8_t*>(L.q_out);
  a.k_out = static_cast<uint8_t*>(L.k_out);
  a.cache = static_cast<uint8_t*>(L.cache);
  a.num_slots = L.num_slots;
  a.e4m3 = L.e4m3;
  a.decode = L.decode;
  a.cu = L.cu;
  a.num_docs = L.num_docs;
  a.seq_lens = L.seq_lens;
  a.page_table = L.page_table;
  a.cu_k = L.cu_k;
  a.max_blocks = L.max_blocks;
  a.err = L.err;
  const long long vec = 5 * L.n;
  const long long per_block = kIpWarps * 32;
  const long long grid = (vec + per_block - 1) / per_block;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidValue;
  index_produce_kernel<<<static_cast<unsigned>(grid), kIpThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace msa
