// decode_select.cu -- decode-step block scoring and top-k selection.
//
// TensorRT-LLM "MiniMaxM3SparseAttentionConfig" (class description; fields
// sparse_score_type 'max', sparse_topk_blocks, sparse_init_blocks,
// sparse_local_blocks, indexer_kv_dtype): one query per request scores every
// 128-token block of its context by the max over the block's keys of the
// unscaled dot product between the per-KV-head index query and the shared
// index key, then keeps the top-k blocks per KV head with the init / local
// blocks forced in.
//
// GB300 design: the paged index-K cache is streamed from HBM once.  Each
// 128-key page (32 KB bf16 / 16 KB E4M3, contiguous) is one work item, brought
// into shared memory by a single 1-D bulk TMA copy into a 3-deep ring.  The
// (request, block) items of all requests are split evenly across a persistent
// grid (stream-K), so every SM streams the same number of bytes.  Four warps
// score 32 keys each on the tensor cores (mma.sync: keys as A, the 4 index
// heads as B, fp32 accumulate), reduce the block max across lanes and warps,
// and store one fp32 score per (request, head, block).  The CTA that finishes
// the last block of a request (an atomic ticket, no waiting) runs the top-k for
// that request's 4 heads: a warp per head, a threshold from the 32 lane maxima
// filters the candidates, then an exact (score desc, id asc) pick.
#include "launch.h"

namespace msa {

constexpr int kSelStages = 3;
constexpr int kSelStageBytes = kBlock * kIdxDim * 2;  // one bf16 page
constexpr int kSelThreads = 128;
constexpr int kCandCap = 64;  // per-warp candidate list of the top-k filter

struct DecodeGeom {
  const int32_t* seq_lens;
  const int32_t* page_table;
  const int64_t* cu_k;
  int batch;
  int max_blocks;
  long long num_slots;
};

struct SelSmem {
  alignas(1024) uint8_t stage[kSelStages][kSelStageBytes];
  uint64_t full[kSelStages];
  int stage_rows[kSelStages];
  float red[2][4][4];  // [parity][warp][head]
  unsigned long long cand[4][kCandCap];
  int scan[kSelThreads / 32];
  int bcast[4];
};

// Blocks of request r that are scored (0 when every candidate is kept anyway).
__device__ __forceinline__ int scored_blocks(const DecodeGeom& geo, int r, int topk, int* nb_out) {
  const int L = geo.seq_lens[r];
  int nb = 0;
  if (L >= 1) nb = min((L + kBlock - 1) / kBlock, geo.max_blocks);
  if (nb_out) *nb_out = nb;
  return nb > topk ? nb : 0;
}

__device__ __forceinline__ int block_sum(int v, int* scan) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  __syncthreads();
  if (lane == 0) scan[warp] = v;
  __syncthreads();
  int t = 0;
  for (int w = 0; w < kSelThreads / 32; ++w) t += scan[w];
  return t;
}

// Exact top-`need` by (score desc, id asc) over the non-forced blocks of one
// (request, head) row, then the ascending q2k row.  One warp.
__device__ void topk_row(const float* s, int nb, int topk, int init, int local, int32_t* out,
                         unsigned long long* cand) {
  const int lane = threadIdx.x & 31;
  if (nb <= topk) {
    for (int i = lane; i < topk; i += 32) out[i] = i < nb ? i : -1;
    return;
  }
  const int need = topk - init - local;
  // key = (orderable score << 32) | (~id): larger key = better (score desc, id asc)
  auto key_of = [&](int b) -> unsigned long long {
    return (static_cast<unsigned long long>(float_key(__ldcg(s + b))) << 32) |
           (0xffffffffu - static_cast<uint32_t>(b));
  };
  int picked = -1;
  if (need > 0) {
    unsigned long long best = 0;
    for (int b = init + lane; b < nb - local; b += 32) {
      const unsigned long long k = key_of(b);
      best = k > best ? k : best;
    }
    // need-th largest lane maximum (bitonic sort of 32 keys, ascending): at
    // least `need` candidates are >= theta, so the top `need` all are
    unsigned long long v = best;
    for (int k = 2; k <= 32; k <<= 1)
      for (int j = k >> 1; j > 0; j >>= 1) {
        const unsigned long long o = __shfl_xor_sync(0xffffffffu, v, j);
        const bool lower = (lane & j) == 0, asc = (lane & k) == 0;
        v = (lower == asc) ? (v < o ? v : o) : (v > o ? v : o);
      }
    const unsigned long long theta = __shfl_sync(0xffffffffu, v, 32 - need);
    int count = 0;
    for (int b0 = init; b0 < nb - local; b0 += 32) {
      const int b = b0 + lane;
      const bool c = b < nb - local && key_of(b) >= theta;
      const unsigned m = __ballot_sync(0xffffffffu, c);
      if (c) {
        const int slot = count + __popc(m & ((1u << lane) - 1));
        if (slot < kCandCap) cand[slot] = key_of(b);
      }
      count += __popc(m);
    }
    __syncwarp();
    if (count <= kCandCap) {
      unsigned long long e0 = lane < count ? cand[lane] : 0ull;
      unsigned long long e1 = lane + 32 < count ? cand[lane + 32] : 0ull;
      for (int i = 0; i < need; ++i) {
        unsigned long long m = e0 > e1 ? e0 : e1;
        for (int o = 16; o > 0; o >>= 1) {
          const unsigned long long x = __shfl_xor_sync(0xffffffffu, m, o);
          m = x > m ? x : m;
        }
        if (e0 == m) e0 = 0;
        if (e1 == m) e1 = 0;
        if (lane == i) picked = static_cast<int>(0xffffffffu - static_cast<uint32_t>(m));
      }
    } else {
      // rare: too many candidates above the threshold -- exact rounds
      unsigned long long prev = ~0ull;
      for (int i = 0; i < need; ++i) {
        unsigned long long m = 0;
        for (int b = init + lane; b < nb - local; b += 32) {
          const unsigned long long k = key_of(b);
          if (k < prev && k > m) m = k;
        }
        for (int o = 16; o > 0; o >>= 1) {
          const unsigned long long x = __shfl_xor_sync(0xffffffffu, m, o);
          m = x > m ? x : m;
        }
        prev = m;
        if (lane == i) picked = static_cast<int>(0xffffffffu - static_cast<uint32_t>(m));
      }
    }
    __syncwarp();
  }
  // forced ids occupy the remaining lanes; then rank-sort ascending
  int id = picked;
  if (lane >= need && lane < need + init) id = lane - need;
  if (lane >= need + init && lane < topk) id = nb - local + (lane - need - init);
  int rank = 0;
  for (int i = 0; i < topk; ++i) {
    const int o = __shfl_sync(0xffffffffu, id, i);
    rank += (o < id) ? 1 : 0;
  }
  if (lane < topk) out[rank] = id;
}

template <int kE4M3>
__global__ void __launch_bounds__(kSelThreads) decode_select_kernel(
    const uint8_t* __restrict__ index_q, const uint8_t* __restrict__ index_k, DecodeGeom geo,
    float* __restrict__ scores, int* __restrict__ tickets, int32_t* __restrict__ q2k, int topk,
    int init, int local, DevError* err) {
  extern __shared__ uint8_t smem_raw[];
  SelSmem& sm = *reinterpret_cast<SelSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g8 = lane >> 2, t4 = lane & 3;
  constexpr int kRowBytes = kE4M3 ? kIdxDim : kIdxDim * 2;
  const int B = geo.batch, mb = geo.max_blocks;

  if (tid == 0) {
    for (int s = 0; s < kSelStages; ++s) mbar_init(&sm.full[s], 1);
    fence_mbar_init();
  }
  // total scored blocks; rows of unscored requests are written here
  int total = 0;
  for (int r0 = 0; r0 < B; r0 += kSelThreads) {
    const int r = r0 + tid;
    int v = 0;
    if (r < B) {
      int nb;
      v = scored_blocks(geo, r, topk, &nb);
      if (r % gridDim.x == blockIdx.x) {
        const int L = geo.seq_lens[r];
        if (L < 1 || L > mb * kBlock) record_error(err, MSA_DEVERR_LENGTH, r);
        if (v == 0)
          for (int h = 0; h < kKvHeads; ++h)
            for (int i = 0; i < topk; ++i) q2k[(static_cast<long long>(h) * B + r) * topk + i] = i < nb ? i : -1;
      }
    }
    total += block_sum(v, sm.scan);
  }
  const long long lo = static_cast<long long>(total) * blockIdx.x / gridDim.x;
  const long long hi = static_cast<long long>(total) * (blockIdx.x + 1) / gridDim.x;
  if (lo >= hi) return;
  // locate the request holding item `lo`
  int r_lo = 0, off_lo = 0;
  {
    int run = 0;
    bool found = false;
    for (int r0 = 0; r0 < B && !found; r0 += kSelThreads) {
      const int r = r0 + tid;
      const int v = r < B ? scored_blocks(geo, r, topk, nullptr) : 0;
      int x = v;  // inclusive scan within the warp
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      __syncthreads();
      if (lane == 31) sm.scan[warp] = x;
      __syncthreads();
      int before = run;
      for (int w = 0; w < warp; ++w) before += sm.scan[w];
      const int incl = before + x, excl = incl - v;
      if (r < B && v > 0 && excl <= lo && lo < incl) {
        sm.bcast[0] = r;
        sm.bcast[1] = excl;
      }
      int chunk_total = 0;
      for (int w = 0; w < kSelThreads / 32; ++w) chunk_total += sm.scan[w];
      __syncthreads();
      if (run <= lo && lo < run + chunk_total) found = true;
      run += chunk_total;
    }
    __syncthreads();
    r_lo = sm.bcast[0];
    off_lo = sm.bcast[1];
  }
  const int n_items = static_cast<int>(hi - lo);

  // producer cursor (thread 0 only)
  int pr = r_lo, pb = static_cast<int>(lo - off_lo), pnb = 0;
  if (tid == 0) pnb = scored_blocks(geo, pr, topk, nullptr);
  auto issue = [&](int i) {  // thread 0: load item i into its stage
    const int s = i % kSelStages;
    const int L = geo.seq_lens[pr];
    const int rows = min(kBlock, L - pb * kBlock);
    long long row0;
    bool ok = rows > 0;
    if (geo.page_table) {
      const int page = geo.page_table[static_cast<long long>(pr) * mb + pb];
      row0 = static_cast<long long>(page) * kBlock;
      if (page < 0 || row0 + kBlock > geo.num_slots) {
        record_error(err, MSA_DEVERR_PAGE, static_cast<long long>(pr) * mb + pb);
        ok = false;
      }
    } else {
      row0 = geo.cu_k[pr] + static_cast<long long>(pb) * kBlock;
      if (row0 < 0 || row0 + rows > geo.num_slots) {
        record_error(err, MSA_DEVERR_PAGE, pr);
        ok = false;
      }
    }
    sm.stage_rows[s] = ok ? rows : 0;
    if (ok) {
      mbar_expect_tx(&sm.full[s], static_cast<uint32_t>(rows * kRowBytes));
      tma_bulk_g2s(sm.stage[s], index_k + row0 * kRowBytes, static_cast<uint32_t>(rows * kRowBytes), &sm.full[s]);
    } else {
      mbar_arrive(&sm.full[s]);
    }
    if (++pb == pnb) {  // advance to the next scored request
      pb = 0;
      do {
        ++pr;
        pnb = pr < B ? scored_blocks(geo, pr, topk, nullptr) : 1;
      } while (pnb == 0);
    }
  };
  __syncthreads();
  if (tid == 0)
    for (int i = 0; i < kSelStages - 1 && i < n_items; ++i) issue(i);

  // consumer cursor (all threads)
  int cr = r_lo, cb = static_cast<int>(lo - off_lo), seg_start = cb;
  int cnb = scored_blocks(geo, cr, topk, nullptr);
  uint32_t qf[4][4];
  auto load_q = [&](int r) {
    constexpr int kQChunks = kE4M3 ? 2 : 4;
    for (int j = 0; j < 4; ++j) qf[j][0] = qf[j][1] = qf[j][2] = qf[j][3] = 0u;
    if (g8 < kKvHeads)
      for (int j = 0; j < kQChunks; ++j) {
        // bf16: dims 32j + 8t .. +8 ; e4m3: dims 64j + 16t .. +16 -- both at byte 64j + 16t
        const uint8_t* p = index_q + (static_cast<long long>(r) * kKvHeads + g8) * kRowBytes + 64 * j + 16 * t4;
        const uint4 v = *reinterpret_cast<const uint4*>(p);
        qf[j][0] = v.x;
        qf[j][1] = v.y;
        qf[j][2] = v.z;
        qf[j][3] = v.w;
      }
  };
  load_q(cr);

  for (int i = 0; i < n_items; ++i) {
    const int s = i % kSelStages;
    if (tid == 0 && i + kSelStages - 1 < n_items) issue(i + kSelStages - 1);
    mbar_wait(&sm.full[s], (i / kSelStages) & 1, err, 100);
    const int rows = sm.stage_rows[s];
    const uint32_t base = smem_u32(sm.stage[s]);
    float mx0 = -INFINITY, mx1 = -INFINITY;  // heads 2*t4, 2*t4+1
    for (int m = 0; m < 2; ++m) {
      const int key0 = 32 * warp + 16 * m;
      if (key0 >= rows) break;
      float c[4] = {0.f, 0.f, 0.f, 0.f};
      const uint32_t ra_addr = base + (key0 + g8) * kRowBytes;
      const uint32_t rb_addr = ra_addr + 8 * kRowBytes;
      // each thread reads 16 contiguous bytes of a key row; the k slots of the
      // MMA take them in a fixed permutation that B (index_q) repeats
      if (!kE4M3) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint4 ra = lds128(ra_addr + (32 * j + 8 * t4) * 2);
          const uint4 rb = lds128(rb_addr + (32 * j + 8 * t4) * 2);
          const uint32_t a0[4] = {ra.x, rb.x, ra.y, rb.y};
          const uint32_t a1[4] = {ra.z, rb.z, ra.w, rb.w};
          mma_bf16(c, a0, qf[j][0], qf[j][1]);
          mma_bf16(c, a1, qf[j][2], qf[j][3]);
        }
      } else {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const uint4 ra = lds128(ra_addr + 64 * j + 16 * t4);
          const uint4 rb = lds128(rb_addr + 64 * j + 16 * t4);
          const uint32_t a0[4] = {ra.x, rb.x, ra.y, rb.y};
          const uint32_t a1[4] = {ra.z, rb.z, ra.w, rb.w};
          mma_e4m3(c, a0, qf[j][0], qf[j][1]);
          mma_e4m3(c, a1, qf[j][2], qf[j][3]);
        }
      }
      if (key0 + g8 < rows) {
        mx0 = fmaxf(mx0, c[0]);
        mx1 = fmaxf(mx1, c[1]);
      }
      if (key0 + g8 + 8 < rows) {
        mx0 = fmaxf(mx0, c[2]);
        mx1 = fmaxf(mx1, c[3]);
      }
    }
    for (int o = 4; o < 32; o <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
    }
    if (lane < 2) {
      sm.red[i & 1][warp][2 * lane] = mx0;
      sm.red[i & 1][warp][2 * lane + 1] = mx1;
    }
    __syncthreads();  // stage s is free; block maxima visible
    if (tid < kKvHeads && cb < mb) {
      const float v = fmaxf(fmaxf(sm.red[i & 1][0][tid], sm.red[i & 1][1][tid]),
                            fmaxf(sm.red[i & 1][2][tid], sm.red[i & 1][3][tid]));
      scores[(static_cast<long long>(cr) * kKvHeads + tid) * mb + cb] = v;
      __threadfence();
    }
    const bool seg_end = (cb == cnb - 1) || (i == n_items - 1);
    if (seg_end) {
      __syncthreads();
      if (tid == 0) {
        __threadfence();
        const int cnt = cb - seg_start + 1;
        const int old = atomicAdd(&tickets[cr], cnt);
        sm.bcast[2] = (old + cnt == cnb) ? 1 : 0;
      }
      __syncthreads();
      if (sm.bcast[2]) {
        __threadfence();
        const float* srow = scores + (static_cast<long long>(cr) * kKvHeads + warp) * mb;
        topk_row(srow, cnb, topk, init, local, q2k + (static_cast<long long>(warp) * B + cr) * topk,
                 sm.cand[warp]);
        if (tid == 0) tickets[cr] = 0;
      }
      // advance the consumer cursor to the next scored request
      if (i + 1 < n_items) {
        cb = 0;
        do {
          ++cr;
          cnb = scored_blocks(geo, cr, topk, nullptr);
        } while (cnb == 0);
        seg_start = 0;
        load_q(cr);
      }
    } else {
      ++cb;
    }
  }
}

cudaError_t launch_decode_select(const msa_config& cfg, const void* index_q, const void* index_k,
                                 const int32_t* seq_lens, const int32_t* page_table, const int64_t* cu_k,
                                 int batch, int max_blocks, long long num_slots, int32_t* q2k, float* scores,
                                 int* tickets, DevError* err, cudaStream_t stream) {
  DecodeGeom geo{seq_lens, page_table, cu_k, batch, max_blocks, num_slots};
  const size_t smem = sizeof(SelSmem) + 1024;
  // enough CTAs to keep every SM streaming (two per SM); bounded by the block count
  const long long blocks_upper = static_cast<long long>(batch) * max_blocks;
  int grid = static_cast<int>(blocks_upper < 2LL * kNumSMs ? blocks_upper : 2LL * kNumSMs);
  if (grid < 1) grid = 1;
  const auto* iq = static_cast<const uint8_t*>(index_q);
  const auto* ik = static_cast<const uint8_t*>(index_k);
  if (cfg.index_dtype == MSA_INDEX_E4M3) {
    auto k = decode_select_kernel<1>;
    cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    k<<<grid, kSelThreads, smem, stream>>>(iq, ik, geo, scores, tickets, q2k, cfg.topk, cfg.init_blocks,
                                           cfg.local_blocks, err);
  } else {
    auto k = decode_select_kernel<0>;
    cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    k<<<grid, kSelThreads, smem, stream>>>(iq, ik, geo, scores, tickets, q2k, cfg.topk, cfg.init_blocks,
                                           cfg.local_blocks, err);
  }
  return cudaGetLastError();
}

}  // namespace msa

// ---- allocation-free variant of the decode select ---------------------------------
// Some callers cannot allocate device memory at the point where they select
// blocks: code that runs inside an allocator-less runtime, plugins handed only
// their input and output buffers, or hosts whose memory pool is fixed before
// the model loads.  For them the block scores and completion counters live in
// one fixed array in the library's own device memory, sized once for every GPU
// that loads the library.
#include <mutex>

namespace msa {

constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;  // 4 MiB per device
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

static std::mutex g_noalloc_mu;
static void* g_noalloc_ptr[256] = {};  // device address of g_noalloc_scratch, per device ordinal

// Device address of the fixed scratch on the current device (looked up once per
// device; the host-side name of the array is not a device address).
static void* noalloc_scratch(cudaError_t* err) {
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= 256) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    *err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (*err != cudaSuccess) return nullptr;
    g_noalloc_ptr[dev] = p;
  }
  return g_noalloc_ptr[dev];
}

static size_t noalloc_up256(size_t x) { return (x + 255) / 256 * 256; }

}  // namespace msa

extern "C" msa_status msa_select_blocks_decode_noalloc(const msa_config* cfg, const void* index_q,
                                                      const void* index_k_cache, const int32_t* seq_lens,
                                                      const int32_t* page_table, const int64_t* cu_seqlens_k,
                                                      int batch, int max_blocks, int64_t num_slots, int32_t* q2k,
                                                      void* stream) {
  using namespace msa;
  msa_status st = msa_config_check(cfg);
  if (st != MSA_OK) return st;
  if (!index_q || !index_k_cache || !q2k || !seq_lens || (!page_table && !cu_seqlens_k)) return MSA_ERR_NULL;
  if (batch < 1 || max_blocks < 1 || num_slots < 1 || num_slots >= (1LL << 31)) return MSA_ERR_SHAPE;
  if (page_table && num_slots % kBlock) return MSA_ERR_SHAPE;
  if ((reinterpret_cast<uintptr_t>(index_q) & 15) || (reinterpret_cast<uintptr_t>(index_k_cache) & 15))
    return MSA_ERR_ALIGN;
  const size_t off_tickets = kHeaderBytes;
  const size_t off_scores = off_tickets + noalloc_up256(static_cast<size_t>(batch) * sizeof(int));
  const size_t need = off_scores + static_cast<size_t>(batch) * kKvHeads * max_blocks * sizeof(float);
  if (need > kNoAllocScratchBytes) return MSA_ERR_WORKSPACE;  // sizes beyond the fixed scratch
  cudaError_t e;
  auto* base = static_cast<uint8_t*>(noalloc_scratch(&e));
  if (!base) return MSA_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the error word and the counters must start at zero; the scores are stored before they are read
  if (cudaMemsetAsync(base, 0, off_scores, s) != cudaSuccess) return MSA_ERR_CUDA;
  e = launch_decode_select(*cfg, index_q, index_k_cache, seq_lens, page_table, cu_seqlens_k, batch, max_blocks,
                           num_slots, q2k, reinterpret_cast<float*>(base + off_scores),
                           reinterpret_cast<int*>(base + off_tickets), reinterpret_cast<DevError*>(base), s);
  return e == cudaSuccess ? MSA_OK : MSA_ERR_CUDA;
}
