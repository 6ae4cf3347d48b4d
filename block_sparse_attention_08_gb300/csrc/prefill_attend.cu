// prefill_attend.cu -- block-major sparse attention for packed-document prefill.
//
// TensorRT-LLM "MiniMaxM3SparseAttentionConfig" (class description, second
// step: a sparse GQA attention over only the selected blocks) and NeMo
// "...minimax_m3_vl.msa" sparse_attention / _SparseAttention.forward: bf16
// q [tokens, 64, 128], k / v [tokens, 4, 128], int32 q2k [4, tokens, topk] ->
// bf16 out [tokens, 64, 128]; query t of a document attends, for each KV head,
// to the causal keys of the blocks its q2k row names.
//
// GB300 design.  In prefill a key block is selected by many queries of its
// document, so the work is turned around: every selected (query, KV head,
// block) triple -- an "entry" -- is bucketed by (KV head, token window, key
// block), and each bucket is cut into tiles of 8 entries.  A tile's 8 x 16
// query rows form one 128-row tcgen05 MMA against the block's 128 keys, so a
// K / V block is read once per tile run instead of once per query, and the
// tensor cores see full 128 x 128 x 128 products:
//
//   S = Q K^T   (A = gathered Q rows, B = K block; both K-major, 128-byte swizzle)
//   P = exp2(S * scale * log2 e - rowmax)   (fp32 in registers, bf16 into a P buffer)
//   O = P V     (A = P read from tensor memory, B = V read MN-major from the TMA tile)
//
// with S (twice), P (twice) and O (once) in tensor memory: a softmax warpgroup
// frees its S buffer as soon as it has read it, so the next S product into it
// waits for no O product, and both epilogue warpgroups read every tile's O
// (half of its columns each), so the one O buffer is freed soon after its
// product.  Warp 16
// schedules the tiles (descriptors and entries read ahead from global memory,
// published in a shared-memory ring) and issues TMA (Q rows gathered with a
// 5-D tensor map, one 4 KB box per entry; K and V blocks as 128-row boxes);
// warps 17 and 18 issue the S and O MMAs from one thread each.  Two softmax
// warpgroups (warps 0-7) take the even and the odd tiles, so two tiles are in
// their softmax at a time; the two epilogue warpgroups (warps 8-15) take the
// two halves of every tile's O; in each, a thread owns one tensor-memory lane
// (query row).
//
// The entries of one (query, KV head) row land in up to topk different tiles,
// so their results are summed in memory, in two launches against one fixed
// exponent reference per row:
//   phase 0: each row's reference entry (its highest valid block, first
//            occurrence) -- a two-pass softmax stores the reference exponent
//            mref = rowmax * scale * log2 e, the row sum lacc and the fp32 O
//            into acc [T][64][128] (tensor-engine stores of 16-row boxes);
//   phase 1: every other entry -- a one-pass softmax against mref, fp32 O
//            added into acc by the tensor engine (cp.reduce.async.bulk .add),
//            the row sum added into lacc;
// then bm_norm_kernel writes out = acc / lacc in bf16 (and the log-sum-exp
// mref + log2 lacc for the backward).  A key that exceeds the reference by
// 2^64 or more leaves fp32's range for the row sum and is reported
// (MSA_DEVERR_RANGE).  The adds run in whatever order the tiles finish, so
// repeated calls agree within fp32 rounding, not bit for bit.  Tiles are
// handed out in chunks of 16, round-robin over the persistent grid, so all
// CTAs move through the (KV head, window) buckets together and the window's
// Q rows, K / V blocks and accumulator rows stay in L2.
#include <cuda_fp16.h>

#include <type_traits>

#include "launch.h"

namespace msa {

constexpr int kBmEntries = 8;                     // entries per tile (8 x 16 heads = 128 MMA rows)
constexpr int kBmHalf = 128 * 128;                // 128 rows x 128 bytes (64 bf16) = 16 KB
constexpr int kBmTile = 2 * kBmHalf;              // a 128 x 128 bf16 operand
constexpr int kBmQBox = kGroup * 128;             // one entry's 16 rows x 64 dims = 2 KB
constexpr int kBmQEntry = 2 * kBmQBox;            // one entry's Q rows, both halves: one 4 KB box
// warps 0-7 softmax (two warpgroups, even / odd tiles), 8-15 epilogue (two
// warpgroups), 16 TMA and scheduling, 17 the S MMAs, 18 the O MMAs
constexpr int kBmThreads = 608;
constexpr int kBmProducerWarp = 16;
constexpr int kBmMmaSWarp = 17;
constexpr int kBmMmaOWarp = 18;
constexpr int kBmChunk = 16;                      // tiles per scheduling chunk
// Tensor-memory columns: S twice (fp32, 128 columns each), P twice (bf16
// pairs, 64 columns each), O once (fp32, 128 columns).
constexpr uint32_t kBmPCol = 256;
constexpr uint32_t kBmOCol = 384;
constexpr uint32_t kBmIdescS = tc::idesc_bf16_f32(128, 128);
constexpr uint32_t kBmIdescO = tc::idesc_bf16_f32(128, 128) | (1u << 16);  // B (V) MN-major

struct BmTile {
  int row0;  // first K / V row of the block
  int g;     // KV head
  int off;   // first entry of the tile in the bucketed entry list
  int cnt;   // entries in the tile (1..8)
};

// A tile as the scheduler publishes it to the MMA and softmax warps.
struct BmInfo {
  int row0, g, cnt, fresh;  // fresh: first tile of a new K / V block
  int ent[kBmEntries];
};
constexpr int kBmInfo = 8;  // info ring slots

// Two Q stages, two K stages (the next block's K loads while the current one
// is in use), one V stage (a block's V is needed a tile later than its K), and
// 8 KB of fp32 O staging per epilogue warp for the tensor engine's stores and
// adds.  S, P and O live in tensor memory.
constexpr int kBmQStages = 2;
constexpr int kBmKStages = 2;
constexpr int kBmVStages = 1;
struct BmSmem {
  alignas(1024) uint8_t q[kBmQStages][kBmTile];
  alignas(1024) uint8_t k[kBmKStages][kBmTile];
  alignas(1024) uint8_t v[kBmVStages][kBmTile];
  alignas(1024) uint8_t ostage[2][kBmTile];  // 8 KB of fp32 staging per epilogue warp (two 4 KB halves)
  uint64_t q_full[kBmQStages], q_empty[kBmQStages], k_full[kBmKStages], k_empty[kBmKStages];
  uint64_t v_full[kBmVStages], v_empty[kBmVStages];
  uint64_t s_full[2], s_free[2], o_full, o_free;
  uint64_t p_full[2], p_free[2], done_s, done_o;
  uint64_t info_full[kBmInfo], info_empty[kBmInfo];
  BmInfo info[kBmInfo];
  uint32_t tmem_base;
};

// 1024 bytes of slack align the dynamic shared memory base; 227 KB per CTA at most.
static_assert(sizeof(BmSmem) + 1024 <= 227 * 1024, "shared memory of the attention kernel");

// Sizes of the bucketing problem, fixed by (tokens, longest document, topk).
struct BmDims {
  long long T;       // compact tokens
  int topk;
  int W;             // token window of a bucket (power of two)
  int nw;            // windows
  long long kg_max;  // bound on the keys of one KV head
  long long entries; // 4 * T * topk
  long long tiles_max;
};

static BmDims bm_dims(long long T, int max_seqlen, int topk) {
  BmDims d;
  d.T = T;
  d.topk = topk;
  d.W = 256;
  while (d.W < max_seqlen / 16) d.W *= 2;
  d.nw = static_cast<int>((T + d.W - 1) / d.W);
  const long long mb = (max_seqlen + kBlock - 1) / kBlock;
  // A window reaches the blocks of its first document plus blocks that start
  // inside it.  The bound uses the smallest window (256 tokens) so that it only
  // grows with T and max_seqlen: a workspace sized for one call serves every
  // smaller one.
  d.kg_max = (T + 255) / 256 * mb + T + 1;
  d.entries = static_cast<long long>(kKvHeads) * T * topk;
  // two phases of keys (the forward's reference entries, then the rest; the
  // backward uses the first only), each key's last tile possibly partial
  const long long keys = 2 * kKvHeads * d.kg_max;
  d.tiles_max = d.entries / kBmEntries + (keys < d.entries ? keys : d.entries) + 1;
  return d;
}

// Carving of the prefill-attention part of the workspace.  Keys: (phase, KV
// head, window, global block); phase 0 holds each (query, KV head) row's
// reference entry (the forward only), phase 1 the others.
struct BmPlan {
  int* meta;       // [0] keys per KV head (Kg), [1] tiles, [2] first tile of phase 1
  int* counts;     // [2 * 4 * kg_max] entries per key
  int* offs;       // [2 * 4 * kg_max + 1] first entry of each key
  int* toff;       // [2 * 4 * kg_max + 1] first tile of each key
  int* blk_base;   // [T + 1] first global block of each document
  int* wlo;        // [nw] first global block a window can reach
  int* wbase;      // [nw + 1] first key of each window (per KV head)
  int* ekey;       // [entries] key of each q2k entry, -1 when skipped
  int* erank;      // [entries] rank of the entry inside its key
  int* elist;      // [entries] bucketed entries: t * topk + j
  BmTile* tiles;   // [tiles_max]
  int phases;      // 2: the forward's reference split; 1: one phase (the backward)
  // the forward's accumulators, per (token, query head):
  float* acc;      // [T][64][128] unnormalised O = sum_p 2^(s_p - mref) v_p
  float* mref;     // [T][64] the reference exponent: the row max over its reference block
  float* lacc;     // [T][64] sum_p 2^(s_p - mref); 0 for a row with no key
};

static size_t al256(size_t x) { return (x + 255) / 256 * 256; }

// The bucketing arrays (shared by the forward and the backward), then, with
// `outputs`, the forward's accumulators.
static size_t bm_carve(const BmDims& d, uint8_t* base, BmPlan* p, bool outputs = true) {
  size_t off = 0;
  auto take = [&](size_t bytes) {
    uint8_t* ptr = base ? base + off : nullptr;
    off += al256(bytes);
    return ptr;
  };
  const size_t keys = 2 * static_cast<size_t>(kKvHeads) * d.kg_max;
  BmPlan q{};
  q.phases = 2;
  q.meta = reinterpret_cast<int*>(take(4 * sizeof(int)));
  q.counts = reinterpret_cast<int*>(take(keys * sizeof(int)));
  q.offs = reinterpret_cast<int*>(take((keys + 1) * sizeof(int)));
  q.toff = reinterpret_cast<int*>(take((keys + 1) * sizeof(int)));
  q.blk_base = reinterpret_cast<int*>(take((d.T + 1) * sizeof(int)));
  q.wlo = reinterpret_cast<int*>(take(((d.T + 255) / 256) * sizeof(int)));
  q.wbase = reinterpret_cast<int*>(take(((d.T + 255) / 256 + 1) * sizeof(int)));
  q.ekey = reinterpret_cast<int*>(take(d.entries * sizeof(int)));
  q.erank = reinterpret_cast<int*>(take(d.entries * sizeof(int)));
  q.elist = reinterpret_cast<int*>(take(d.entries * sizeof(int)));
  q.tiles = reinterpret_cast<BmTile*>(take(d.tiles_max * sizeof(BmTile)));
  if (outputs) {
    q.acc = reinterpret_cast<float*>(take(static_cast<size_t>(d.T) * kHeads * kDim * sizeof(float)));
    q.mref = reinterpret_cast<float*>(take(static_cast<size_t>(d.T) * kHeads * sizeof(float)));
    q.lacc = reinterpret_cast<float*>(take(static_cast<size_t>(d.T) * kHeads * sizeof(float)));
  }
  if (p) *p = q;
  return off;
}

size_t prefill_attend_bytes(long long total_tokens, int max_seqlen, int topk) {
  return bm_carve(bm_dims(total_tokens, max_seqlen, topk), nullptr, nullptr);
}

// ---- small device helpers ---------------------------------------------------------

// Index of the document holding compact token t: the last d with cu[d] <= t.
__device__ __forceinline__ int doc_of(const int32_t* __restrict__ cu, int num_docs, long long t) {
  int lo = 0, hi = num_docs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (cu[mid] <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Last index i in [0, n) with a[i] <= x (a ascending, a[0] <= x).
__device__ __forceinline__ int last_le(const int* __restrict__ a, int n, long long x) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (a[mid] <= x) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Exclusive scan of one value per thread over a 1024-thread block; returns the
// prefix and writes the block total to *total.  `sh` holds 32 ints.
__device__ __forceinline__ long long block_scan_1024(long long v, long long* sh, long long* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  long long x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) sh[warp] = x;
  __syncthreads();
  if (warp == 0) {
    long long w = sh[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    sh[lane] = w;
  }
  __syncthreads();
  const long long before = (warp > 0 ? sh[warp - 1] : 0) + x - v;
  *total = sh[31];
  __syncthreads();
  return before;
}


// ---- bucketing ----------------------------------------------------------------------

// One block of 1024 threads: document block bases, window reach and the first
// key of every window.  Key space of one KV head: window w owns keys
// [wbase[w], wbase[w+1]), one per global block in [wlo[w], wlo[w] + span).
__global__ void __launch_bounds__(1024) bm_geom_kernel(const int32_t* __restrict__ cu, int num_docs, long long T,
                                                       int W, int nw, long long kg_max, BmPlan p, DevError* err) {
  __shared__ long long sh[32];
  const int tid = threadIdx.x;
  {
    const int per = (num_docs + 1023) / 1024;
    const int d0 = min(num_docs, tid * per), d1 = min(num_docs, d0 + per);
    long long s = 0;
    for (int d = d0; d < d1; ++d) s += (cu[d + 1] - cu[d] + kBlock - 1) / kBlock;
    long long tot;
    long long run = block_scan_1024(s, sh, &tot);
    for (int d = d0; d < d1; ++d) {
      p.blk_base[d] = static_cast<int>(run);
      run += (cu[d + 1] - cu[d] + kBlock - 1) / kBlock;
    }
    if (tid == 0) p.blk_base[num_docs] = static_cast<int>(tot);
  }
  __syncthreads();
  {
    const int per = (nw + 1023) / 1024;
    const int w0 = min(nw, tid * per), w1 = min(nw, w0 + per);
    long long s = 0;
    for (int w = w0; w < w1; ++w) {
      const long long t0 = static_cast<long long>(w) * W;
      const long long t1 = (t0 + W < T ? t0 + W : T) - 1;
      const int da = doc_of(cu, num_docs, t0), db = doc_of(cu, num_docs, t1);
      const int lo = p.blk_base[da];
      const int hi = p.blk_base[db] + static_cast<int>((t1 - cu[db]) / kBlock);
      p.wlo[w] = lo;
      p.wbase[w] = hi - lo + 1;  // span for now
      s += hi - lo + 1;
    }
    long long tot;
    long long run = block_scan_1024(s, sh, &tot);
    for (int w = w0; w < w1; ++w) {
      const int span = p.wbase[w];
      p.wbase[w] = static_cast<int>(run);
      run += span;
    }
    if (tid == 0) {
      if (tot > kg_max) {  // cannot happen for a well-formed cu_seqlens; leave nothing to do
        record_error(err, MSA_DEVERR_LENGTH, tot);
        tot = 0;
      }
      p.wbase[nw] = static_cast<int>(tot);
      p.meta[0] = static_cast<int>(tot);
    }
  }
}

// One thread per (KV head, token): the key of each of the token's q2k entries
// and its rank inside the key (warp-aggregated atomics: the tokens of a warp
// share their forced blocks).  Entries that name no block (-1) are skipped;
// ids at or past the query's causal block count are recorded and skipped.
__global__ void __launch_bounds__(256) bm_count_kernel(const int32_t* __restrict__ q2k,
                                                       const int32_t* __restrict__ cu, int num_docs, long long T,
                                                       int topk, int W, BmPlan p, DevError* err) {
  const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int lane = threadIdx.x & 31;
  const bool live = idx < kKvHeads * T;
  const int Kg = p.meta[0];
  int g = 0, nb = 0, w = 0, gb0 = 0, kbase = 0;
  long long t = 0;
  if (live) {
    g = static_cast<int>(idx / T);
    t = idx - static_cast<long long>(g) * T;
    const int d = doc_of(cu, num_docs, t);
    const int pos = static_cast<int>(t - cu[d]);
    nb = pos / kBlock + 1;
    w = static_cast<int>(t / W);
    gb0 = p.blk_base[d];
    kbase = g * Kg + p.wbase[w] - p.wlo[w];
  }
  const long long e0 = idx * topk;  // == (g * T + t) * topk
  const unsigned lt = (1u << lane) - 1u;
  // With two phases, the row's reference entry -- its highest valid block,
  // first occurrence -- goes to phase 0 and the other entries to phase 1.
  int ref_j = -1;
  if (live && p.phases == 2) {
    int best = -1;
    for (int j = 0; j < topk; ++j) {
      const int b = q2k[e0 + j];
      if (b >= 0 && b < nb && b > best) {
        best = b;
        ref_j = j;
      }
    }
  }
  const int phase1 = kKvHeads * Kg;  // first key of phase 1
  for (int j = 0; j < topk; ++j) {
    int key = -1;
    if (live) {
      const int b = q2k[e0 + j];
      if (b >= nb) record_error(err, MSA_DEVERR_BLOCK, e0 + j);
      else if (b >= 0) key = kbase + gb0 + b + (p.phases == 2 && j != ref_j ? phase1 : 0);
    }
    const unsigned grp = __match_any_sync(0xffffffffu, key);
    const int leader = __ffs(grp) - 1;
    int base = 0;
    if (key >= 0 && lane == leader) base = atomicAdd(&p.counts[key], __popc(grp));
    base = __shfl_sync(grp, base, leader);
    if (live) {
      p.ekey[e0 + j] = key;
      p.erank[e0 + j] = base + __popc(grp & lt);
    }
  }
}

// One block of 1024 threads: exclusive scans of the key counts (entry offsets)
// and of the tiles per key; the tile total goes to meta[1].
__global__ void __launch_bounds__(1024) bm_scan_kernel(BmPlan p) {
  __shared__ long long sh[32];
  const int tid = threadIdx.x;
  const long long K = static_cast<long long>(p.phases) * kKvHeads * p.meta[0];
  const long long per = (K + 1023) / 1024;
  const long long k0 = min(K, tid * per), k1 = min(K, k0 + per);
  long long se = 0, st = 0;
  for (long long k = k0; k < k1; ++k) {
    const int c = p.counts[k];
    se += c;
    st += (c + kBmEntries - 1) / kBmEntries;
  }
  long long te, tt;
  long long re = block_scan_1024(se, sh, &te);
  long long rt = block_scan_1024(st, sh, &tt);
  for (long long k = k0; k < k1; ++k) {
    const int c = p.counts[k];
    p.offs[k] = static_cast<int>(re);
    p.toff[k] = static_cast<int>(rt);
    re += c;
    rt += (c + kBmEntries - 1) / kBmEntries;
  }
  __syncthreads();
  if (tid == 0) {
    p.offs[K] = static_cast<int>(te);
    p.toff[K] = static_cast<int>(tt);
    p.meta[1] = static_cast<int>(tt);
    p.meta[2] = p.phases == 2 ? p.toff[K / 2] : static_cast<int>(tt);
  }
}

// One thread per tile: its key (the last whose first tile is at or before
// it: keys without entries own no tile), then the tile's descriptor (K / V
// rows, KV head, entry range).  (One thread per key, writing the key's tiles
// in turn, left a few threads with dozens of tiles each.)
__global__ void __launch_bounds__(256) bm_tiles_kernel(const int32_t* __restrict__ cu, int num_docs, int nw,
                                                       BmPlan p) {
  const long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (t >= p.meta[1]) return;
  const int Kg = p.meta[0];
  const int nkeys = p.phases * kKvHeads * Kg;
  const int key = last_le(p.toff, nkeys, t);
  const int c = p.counts[key];
  const int i = static_cast<int>(t - p.toff[key]);
  const int kh = key % (kKvHeads * Kg);  // the key within its phase
  const int g = kh / Kg, kk = kh - g * Kg;
  const int w = last_le(p.wbase, nw, kk);
  const int gb = p.wlo[w] + kk - p.wbase[w];
  const int d = last_le(p.blk_base, num_docs, gb);
  const int row0 = cu[d] + (gb - p.blk_base[d]) * kBlock;
  p.tiles[t] = BmTile{row0, g, p.offs[key] + i * kBmEntries, min(kBmEntries, c - i * kBmEntries)};
}

// One thread per q2k entry: its place in the bucketed list.
__global__ void __launch_bounds__(256) bm_scatter_kernel(long long entries, long long per_head, BmPlan p) {
  const long long e = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (e >= entries) return;
  const int key = p.ekey[e];
  if (key < 0) return;
  p.elist[p.offs[key] + p.erank[e]] = static_cast<int>(e % per_head);
}


// ---- the tensor-core kernel ---------------------------------------------------------

// Shared-memory descriptor of V read MN-major (N = head dims contiguous inside a
// 128-byte swizzled row, K = keys along rows): 64-dim atoms 16 KB apart (LBO),
// 8-key groups 1024 bytes apart (SBO).
__device__ __forceinline__ uint64_t desc_v_mn_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFF);
  d |= static_cast<uint64_t>(kBmHalf >> 4) << 16;
  d |= static_cast<uint64_t>(1024 >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

__device__ __forceinline__ uint32_t pack_half2(float a, float b) {
  __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

// The CTA's i-th tile: chunks c, c + G, c + 2G, ... of kBmChunk consecutive tiles.
__device__ __forceinline__ int tile_at(int i) {
  return (blockIdx.x + gridDim.x * (i / kBmChunk)) * kBmChunk + i % kBmChunk;
}
__device__ __forceinline__ int local_tiles(int n_tiles) {
  int n = 0;
  for (int k = blockIdx.x; k * kBmChunk < n_tiles; k += gridDim.x) n += min(kBmChunk, n_tiles - k * kBmChunk);
  return n;
}

// Single MUFU base-2 exponential (ex2.approx.ftz: relative error about 2^-22;
// exp2(-inf) = +0).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void stg128(void* p, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

__global__ void __launch_bounds__(kBmThreads, 1) bm_attend_kernel(
    const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
    const __grid_constant__ CUtensorMap vmap, const __grid_constant__ CUtensorMap amap, BmPlan p, long long T,
    int topk, float scale_log2, int phase, DevError* err) {
  extern __shared__ uint8_t smem_raw[];
  BmSmem& sm = *reinterpret_cast<BmSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int t_lo = phase ? p.meta[2] : 0, t_hi = phase ? p.meta[1] : p.meta[2];  // this phase's tiles
  const int n = local_tiles(t_hi - t_lo);  // tiles of this CTA

  if (tid == 0) {
    for (int i = 0; i < kBmQStages; ++i) {
      mbar_init(&sm.q_full[i], 1);
      mbar_init(&sm.q_empty[i], 1);
    }
    for (int i = 0; i < kBmVStages; ++i) {
      mbar_init(&sm.v_full[i], 1);
      mbar_init(&sm.v_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sm.s_full[i], 1);
      mbar_init(&sm.s_free[i], 4);  // the softmax warpgroup's four warps, once they have read S
      mbar_init(&sm.p_full[i], 4);
      mbar_init(&sm.p_free[i], 1);  // committed by the O MMAs that read P
    }
    for (int i = 0; i < kBmKStages; ++i) {
      mbar_init(&sm.k_full[i], 1);
      mbar_init(&sm.k_empty[i], 1);
    }
    mbar_init(&sm.o_full, 1);
    mbar_init(&sm.o_free, 8);  // both epilogue warpgroups, once they have read their columns
    for (int i = 0; i < kBmInfo; ++i) {
      mbar_init(&sm.info_full[i], 1);
      mbar_init(&sm.info_empty[i], 14);  // the tile's softmax warpgroup, both epilogue warpgroups, both MMA threads
    }
    mbar_init(&sm.done_s, 1);
    mbar_init(&sm.done_o, 1);
    fence_mbar_init();
  }
  if (warp == kBmMmaSWarp) {
    tc::alloc(&sm.tmem_base, 512);
    tc::relinquish();
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = sm.tmem_base;

  // A wait that gives up (recorded in the error word) marks the role dead: it
  // stops issuing work, so a broken pipeline ends after one bounded wait per
  // role instead of one per tile.
  if (warp == kBmProducerWarp) {
    // ---------------- scheduler + TMA producer ----------------
    // Reads each tile's descriptor and entries from global memory one and two
    // tiles ahead, publishes them in the info ring, then issues K of a new
    // block, the tile's Q rows, and V of a new block.  V comes last because its
    // stage is released by the O MMA of the previous block's first tile, which
    // the MMA warp issues only after this tile's S MMA.
    if (lane == 0) {
      prefetch_tmap(&qmap);
      prefetch_tmap(&kmap);
      prefetch_tmap(&vmap);
    }
    const BmTile none{-1, -1, 0, 0};
    BmTile d_next = n > 0 ? p.tiles[t_lo + tile_at(0)] : none;
    int e_next = lane < d_next.cnt ? p.elist[d_next.off + lane] : 0;
    BmTile d_after = n > 1 ? p.tiles[t_lo + tile_at(1)] : none;
    int prow = -1, pg = -1;
    int nkf = 0, nvf = 0;  // K and V fills issued (lane 0)
    int i = 0;
    for (; i < n; ++i) {
      const BmTile d = d_next;
      const int ent = e_next;
      d_next = d_after;
      e_next = (i + 1 < n && lane < d_next.cnt) ? p.elist[d_next.off + lane] : 0;
      d_after = i + 2 < n ? p.tiles[t_lo + tile_at(i + 2)] : none;
      const bool fresh = d.row0 != prow || d.g != pg;
      // publish the tile
      const int is = i % kBmInfo;
      bool ok = true;
      if (lane == 0) ok = mbar_wait(&sm.info_empty[is], ((i / kBmInfo) & 1) ^ 1, err, 706);
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      if (lane < kBmEntries) sm.info[is].ent[lane] = ent;
      if (lane == 0) {
        sm.info[is].row0 = d.row0;
        sm.info[is].g = d.g;
        sm.info[is].cnt = d.cnt;
        sm.info[is].fresh = fresh ? 1 : 0;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.info_full[is]);
      const int qs = i % kBmQStages;
      if (lane == 0) {
        if (fresh) {
          const int s = nkf % kBmKStages;
          ok = mbar_wait(&sm.k_empty[s], ((nkf / kBmKStages) & 1) ^ 1, err, 700);
          if (ok) {
            mbar_expect_tx(&sm.k_full[s], kBmTile);
            tma_load_3d(sm.k[s], &kmap, 0, d.g, d.row0, &sm.k_full[s]);
            tma_load_3d(sm.k[s] + kBmHalf, &kmap, 64, d.g, d.row0, &sm.k_full[s]);
            ++nkf;
          }
        }
        ok = ok && mbar_wait(&sm.q_empty[qs], ((i / kBmQStages) & 1) ^ 1, err, 702);
        if (ok) mbar_expect_tx(&sm.q_full[qs], d.cnt * 2 * kBmQBox);
      }
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      // one 4 KB box per entry: its 16 heads x 128 dims as four 8-row
      // swizzle atoms (heads 0-7 dims 0-63, heads 0-7 dims 64-127, heads 8-15
      // dims 0-63, heads 8-15 dims 64-127), so each half of the tile's rows
      // has its atoms 2048 bytes apart
      if (lane < d.cnt) tma_load_5d(sm.q[qs] + lane * kBmQEntry, &qmap, 0, 0, 0, 2 * d.g, ent / topk, &sm.q_full[qs]);
      __syncwarp();
      if (fresh) {
        prow = d.row0;
        pg = d.g;
        if (lane == 0) {
          const int s = nvf % kBmVStages;
          ok = mbar_wait(&sm.v_empty[s], ((nvf / kBmVStages) & 1) ^ 1, err, 701);
          if (ok) {
            mbar_expect_tx(&sm.v_full[s], kBmTile);
            tma_load_3d(sm.v[s], &vmap, 0, d.g, d.row0, &sm.v_full[s]);
            tma_load_3d(sm.v[s] + kBmHalf, &vmap, 64, d.g, d.row0, &sm.v_full[s]);
            ++nvf;
          }
        }
        if (!__shfl_sync(0xffffffffu, ok, 0)) {
          ++i;  // this tile's Q copies were issued
          break;
        }
      }
    }
    // no copy may still be landing when the CTA exits: wait for the last fill of every stage
    if (lane == 0) {
      for (int q = 0; q < kBmKStages; ++q) {
        const int fk = (nkf - q + kBmKStages - 1) / kBmKStages;
        if (fk > 0) mbar_wait(&sm.k_full[q], (fk - 1) & 1, err, 704);
      }
      for (int q = 0; q < kBmQStages; ++q) {
        const int fq = (i - q + kBmQStages - 1) / kBmQStages;  // fills of Q stage q
        if (fq > 0) mbar_wait(&sm.q_full[q], (fq - 1) & 1, err, 703);
      }
      for (int q = 0; q < kBmVStages; ++q) {
        const int fv = (nvf - q + kBmVStages - 1) / kBmVStages;
        if (fv > 0) mbar_wait(&sm.v_full[q], (fv - 1) & 1, err, 705);
      }
    }
  } else if (warp == kBmMmaSWarp) {
    // ---------------- S MMAs: S(i) = Q K^T into tensor-memory buffer i % 2 ----------------
    // Issued independently of the O MMAs (another warp), so an S tile never
    // waits behind the P of an earlier tile.
    if (lane == 0) {
      int nk = 0, ks = 0;
      for (int i = 0; i < n; ++i) {
        const int is = i % kBmInfo;
        if (!mbar_wait(&sm.info_full[is], (i / kBmInfo) & 1, err, 717)) break;
        const bool fresh = sm.info[is].fresh != 0;
        mbar_arrive(&sm.info_empty[is]);
        if (fresh) {
          if (nk > 0) tc::commit(&sm.k_empty[ks]);
          ks = nk % kBmKStages;
          if (!mbar_wait(&sm.k_full[ks], (nk / kBmKStages) & 1, err, 710)) break;
          ++nk;
        }
        const int b = i & 1, qs = i % kBmQStages;
        if (!mbar_wait(&sm.q_full[qs], (i / kBmQStages) & 1, err, 711) ||
            !mbar_wait(&sm.s_free[b], ((i >> 1) & 1) ^ 1, err, 712))
          break;
        tc::fence_after();
        const uint32_t qa = smem_u32(sm.q[qs]), ka = smem_u32(sm.k[ks]);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t qoff = (kk >> 2) * 1024 + (kk & 3) * 32, koff = (kk >> 2) * kBmHalf + (kk & 3) * 32;
          tc::mma_bf16(tmem + b * 128, tc::desc_k_sw128_sbo(qa + qoff, 2048), tc::desc_k_sw128(ka + koff), kBmIdescS,
                       kk > 0);
        }
        tc::commit(&sm.s_full[b]);
        tc::commit(&sm.q_empty[qs]);
      }
      // every MMA of this thread has finished before tensor memory is released
      tc::commit(&sm.done_s);
      mbar_wait(&sm.done_s, 0, err, 716);
    }
  } else if (warp == kBmMmaOWarp) {
    // ---------------- O MMAs: O(i) = P(i) V into the one O buffer ----------------
    // A = P from tensor memory (P buffer i % 2, written by the softmax of the
    // tile), B = V from shared memory; their completion frees the P buffer.
    // The O buffer is free once the epilogue of tile i - 1 has read it.
    if (lane == 0) {
      int nv = 0, vs = 0;
      for (int i = 0; i < n; ++i) {
        const int is = i % kBmInfo;
        if (!mbar_wait(&sm.info_full[is], (i / kBmInfo) & 1, err, 718)) break;
        const bool fresh = sm.info[is].fresh != 0;
        mbar_arrive(&sm.info_empty[is]);
        if (fresh) {
          if (nv > 0) tc::commit(&sm.v_empty[vs]);
          vs = nv % kBmVStages;
          if (!mbar_wait(&sm.v_full[vs], (nv / kBmVStages) & 1, err, 713)) break;
          ++nv;
        }
        const int b = i & 1;
        if (!mbar_wait(&sm.p_full[b], (i >> 1) & 1, err, 714) || !mbar_wait(&sm.o_free, (i & 1) ^ 1, err, 715))
          break;
        tc::fence_after();
        const uint32_t va = smem_u32(sm.v[vs]);
        const uint32_t pt = tmem + kBmPCol + b * 64;
        const uint32_t dt = tmem + kBmOCol;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          tc::mma_bf16_ts(dt, pt + kk * 8, desc_v_mn_sw128(va + kk * 2048), kBmIdescO, kk > 0);
        tc::commit(&sm.o_full);
        tc::commit(&sm.p_free[b]);
      }
      tc::commit(&sm.done_o);
      mbar_wait(&sm.done_o, 0, err, 719);
    }
  } else if (warp < 8) {
    // ---------------- warps 0-7: softmax, one query row per thread ----------------
    // Warpgroup wg takes the tiles i = wg, wg + 2, ... (S and P buffer wg).
    const int wg = warp >> 2, quarter = warp & 3;
    const int r = quarter * 32 + lane, e = r >> 4, h = r & 15;
    const uint32_t srow = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + wg * 128;
    const uint32_t prow = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + kBmPCol + wg * 64;
    for (int i = wg; i < n; i += 2) {
      const int is = i % kBmInfo, k = i >> 1;
      if (!__all_sync(0xffffffffu, mbar_wait(&sm.info_full[is], (i / kBmInfo) & 1, err, 723))) break;
      const int cnt = sm.info[is].cnt, row0 = sm.info[is].row0, g = sm.info[is].g;
      const bool valid = e < cnt;
      const int ent = valid ? sm.info[is].ent[e] : 0;
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.info_empty[is]);
      const long long t = ent / topk;
      const long long row = t * kHeads + g * kGroup + h;  // (token, query head) accumulator row
      const int nkeys = valid ? static_cast<int>(min(static_cast<long long>(kBlock), t - row0 + 1)) : 0;
      // phase 1: the row's exponent reference, requested before the wait for S
      const float mr = phase && valid ? __ldcg(p.mref + row) : 0.f;
      if (!__all_sync(0xffffffffu, mbar_wait(&sm.s_full[wg], k & 1, err, 720))) break;
      // the P buffer: read by the O MMA of this warpgroup's previous tile
      if (!__all_sync(0xffffffffu, mbar_wait(&sm.p_free[wg], (k & 1) ^ 1, err, 725))) break;
      tc::fence_after();
      // Rows whose keys are all causal (every block but the diagonal one) skip
      // the per-key mask.
      const bool masked = !__all_sync(0xffffffffu, nkeys >= kBlock);
      float mu = 0.f, l = 0.f;
      auto softmax_rows = [&](auto mask_tag) {
        constexpr bool kMask = decltype(mask_tag)::value;
        if (phase == 0) {
          // pass 1: row max (eight independent chains)
          float m8[8];
#pragma unroll
          for (int q = 0; q < 8; ++q) m8[q] = -INFINITY;
#pragma unroll 1
          for (int ch = 0; ch < 4; ++ch) {
            uint32_t v[32];
            tc::ld_32x32b_x32(srow + ch * 32, v);
            tc::wait_ld();
#pragma unroll
            for (int q = 0; q < 16; ++q) {
              float xa = __uint_as_float(v[2 * q]), xb = __uint_as_float(v[2 * q + 1]);
              if (kMask) {
                xa = ch * 32 + 2 * q < nkeys ? xa : -INFINITY;
                xb = ch * 32 + 2 * q + 1 < nkeys ? xb : -INFINITY;
              }
              m8[q & 7] = fmax3(m8[q & 7], xa, xb);
            }
          }
          const float mx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                                 fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
          // scale > 0, so the max of the scaled scores is the scaled max
          mu = mx == -INFINITY ? 0.f : mx * scale_log2;
        } else {
          mu = mr;
        }
        // p = 2^(s * scale * log2 e - mu) in bf16 (P chunk ch: 16 columns of
        // the P buffer); the fp32 row sum adds the same bf16-rounded values, so
        // the normalisation matches the weights the PV product applies (which
        // matters when one key dominates a row and its p is not a power of two)
        float2 l4[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) l4[q] = make_float2(0.f, 0.f);
#pragma unroll 1
        for (int ch = 0; ch < 4; ++ch) {
          uint32_t v[32];
          tc::ld_32x32b_x32(srow + ch * 32, v);
          tc::wait_ld();
          uint32_t pk[16];
#pragma unroll
          for (int q = 0; q < 16; ++q) {
            const int kc = ch * 32 + 2 * q;
            float2 x = fma2(__uint_as_float(v[2 * q]), __uint_as_float(v[2 * q + 1]), scale_log2, scale_log2, -mu,
                            -mu);
            if (kMask) {
              x.x = kc < nkeys ? x.x : -INFINITY;
              x.y = kc + 1 < nkeys ? x.y : -INFINITY;
            }
            const uint32_t pp = pack_bf16(ex2(x.x), ex2(x.y));
            pk[q] = pp;
            l4[q & 3] = add2(l4[q & 3].x, l4[q & 3].y, __uint_as_float(pp << 16), __uint_as_float(pp & 0xffff0000u));
          }
          tc::st_32x32b_x16(prow + ch * 16, pk);
        }
        l = ((l4[0].x + l4[0].y) + (l4[1].x + l4[1].y)) + ((l4[2].x + l4[2].y) + (l4[3].x + l4[3].y));
      };
      if (masked) softmax_rows(std::true_type{});
      else softmax_rows(std::false_type{});
      // every S column has been read: the next S of this buffer may be issued
      tc::fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.s_free[wg]);
      tc::wait_st();
      tc::fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.p_full[wg]);
      if (valid) {
        if (phase == 0) {
          p.mref[row] = mu;
          p.lacc[row] = l;
        } else {
          atomicAdd(p.lacc + row, l);
          // a key above the reference by 2^64 or more (or a non-finite score)
          // leaves the range of the fixed reference: reported, not hidden
          if (!(l < 0x1p64f)) record_error(err, MSA_DEVERR_RANGE, static_cast<long long>(g) * T * topk + ent);
        }
      }
    }
  } else {
    // ---------------- warps 8-15: epilogue, fp32 O into the row accumulators ----------------
    // Both warpgroups take every tile, warpgroup wg the 32-column quarters 2 wg
    // and 2 wg + 1 of O, so the O buffer is read (and freed for the next tile's
    // product) in half the time one warpgroup would take.  Warp w owns 32 rows
    // of the tile (entries 2 (w % 4) and 2 (w % 4) + 1): per quarter it copies
    // its rows from tensor memory into one 4 KB half of its own 8 KB of staging
    // (128-byte swizzle), and its lane 0 has the tensor engine store (phase 0)
    // or add (phase 1) the two 16-row boxes into the fp32 accumulators
    // [T][64][128].
    const int wg = (warp - 8) >> 2, quarter = warp & 3;
    const uint32_t orow = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + kBmOCol;
    uint8_t* own = &sm.ostage[0][0] + (warp - 8) * 8192;
    if (lane == 0) prefetch_tmap(&amap);
    for (int i = 0; i < n; ++i) {
      const int is = i % kBmInfo;
      if (!__all_sync(0xffffffffu, mbar_wait(&sm.info_full[is], (i / kBmInfo) & 1, err, 724))) break;
      const int cnt = sm.info[is].cnt, g = sm.info[is].g;
      const int ea = 2 * quarter;
      const int ta = ea < cnt ? static_cast<int>(sm.info[is].ent[ea] / topk) : -1;
      const int tb = ea + 1 < cnt ? static_cast<int>(sm.info[is].ent[ea + 1] / topk) : -1;
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.info_empty[is]);
      if (!__all_sync(0xffffffffu, mbar_wait(&sm.o_full, i & 1, err, 722))) break;
      tc::fence_after();
      // both quarters into registers first: the O buffer is freed before any
      // staging waits on the tensor engine
      uint32_t v2[2][32];
      tc::ld_32x32b_x32(orow + 2 * wg * 32, v2[0]);
      tc::ld_32x32b_x32(orow + (2 * wg + 1) * 32, v2[1]);
      tc::wait_ld();
      tc::fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.o_free);
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        const int qq = 2 * wg + h2;
        const uint32_t* v = v2[h2];
        // this half was last read by the bulk group of two quarters ago
        if (lane == 0) bulk_wait_read_1();
        __syncwarp();
        uint8_t* half = own + h2 * 4096;
        const uint32_t hs = smem_u32(half);
#pragma unroll
        for (int j = 0; j < 8; ++j) sts128(hs + sw128(lane, j), v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          if (phase == 0) {
            if (ta >= 0) tma_store_3d(&amap, half, qq * 32, g * kGroup, ta);
            if (tb >= 0) tma_store_3d(&amap, half + 2048, qq * 32, g * kGroup, tb);
          } else {
            if (ta >= 0) tma_reduce_add_3d(&amap, half, qq * 32, g * kGroup, ta);
            if (tb >= 0) tma_reduce_add_3d(&amap, half + 2048, qq * 32, g * kGroup, tb);
          }
          bulk_commit();
        }
      }
    }
    if (lane == 0) bulk_wait_all();  // the stores and adds have landed before the CTA exits
  }
  tc::fence_before();
  __syncthreads();
  if (warp == kBmMmaSWarp) {
    tc::fence_after();
    tc::dealloc(tmem, 512);
  }
}

// The output of every (token, query head) row: out = acc / lacc in bf16, zeros
// for a row with no key; with `lse`, the log2 of the softmax denominator in the
// scaled-score base-2 domain, mref + log2(lacc) (-inf for a row with no key):
// what the backward needs to rebuild P.  16 threads per row, 8 dims each.
__global__ void __launch_bounds__(256) bm_norm_kernel(BmPlan p, long long rows, __nv_bfloat16* __restrict__ out,
                                                      float* __restrict__ lse) {
  const long long row = static_cast<long long>(blockIdx.x) * 16 + (threadIdx.x >> 4);
  const int c = threadIdx.x & 15;
  if (row >= rows) return;
  const float l = __ldcs(p.lacc + row);
  const float4* a = reinterpret_cast<const float4*>(p.acc + row * kDim + 8 * c);
  uint4 o = make_uint4(0u, 0u, 0u, 0u);
  if (l > 0.f) {  // a row with no key was never written: its accumulator is not read
    const float4 x = __ldcs(a), y = __ldcs(a + 1);
    const float inv = 1.f / l;
    o = make_uint4(pack_bf16(x.x * inv, x.y * inv), pack_bf16(x.z * inv, x.w * inv), pack_bf16(y.x * inv, y.y * inv),
                   pack_bf16(y.z * inv, y.w * inv));
  }
  *reinterpret_cast<uint4*>(out + row * kDim + 8 * c) = o;
  if (lse && c == 0) lse[row] = l > 0.f ? p.mref[row] + log2f(l) : -INFINITY;
}


// ---- host side --------------------------------------------------------------------

// q [T, 64 heads, 128] bf16 as (dims 0-63, head % 8, dims / 64, head / 8, token) with
// a (64, 8, 2, 2, 1) box: one entry's 16 heads of a KV head as four 8-row
// 128-byte-swizzled atoms, heads 0-7 then 8-15, each both halves of the dims.
static bool encode_q_entry(CUtensorMap* map, const void* base, cuuint64_t T) {
  EncodeTiledFn enc = get_encode_tiled();
  if (!enc) return false;
  cuuint64_t dims[5] = {64, 8, 2, kHeads / 8, T};
  cuuint64_t strides[4] = {kDim * 2, 128, 8 * kDim * 2, kHeads * kDim * 2};
  cuuint32_t box[5] = {64, 8, 2, 2, 1};
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

static bool encode3d(CUtensorMap* map, const void* base, cuuint64_t d0, cuuint64_t d1, cuuint64_t d2,
                     cuuint32_t b0, cuuint32_t b1, cuuint32_t b2) {
  EncodeTiledFn enc = get_encode_tiled();
  if (!enc) return false;
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {d0 * 2, d0 * d1 * 2};
  cuuint32_t box[3] = {b0, b1, b2};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// fp32 [d2][d1][d0] with a (b0, b1, b2) box, 128-byte swizzle (b0 = 32).
static bool encode3d_f32(CUtensorMap* map, const void* base, cuuint64_t d0, cuuint64_t d1, cuuint64_t d2,
                         cuuint32_t b0, cuuint32_t b1, cuuint32_t b2) {
  EncodeTiledFn enc = get_encode_tiled();
  if (!enc) return false;
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {d0 * 4, d0 * d1 * 4};
  cuuint32_t box[3] = {b0, b1, b2};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool prefill_attend_fits(long long total_tokens, int max_seqlen, int topk) {
  const BmDims d = bm_dims(total_tokens, max_seqlen, topk);
  // entries, keys and tiles are int32 on the device
  return d.entries < (1LL << 31) && 2 * kKvHeads * d.kg_max < (1LL << 31) && d.tiles_max < (1LL << 31);
}

cudaError_t launch_prefill_attend(const void* q, const void* k, const void* v, const int32_t* q2k,
                                  const int32_t* cu_seqlens, int num_docs, long long total_tokens, int max_seqlen,
                                  int topk, float scale, void* out, float* lse, uint8_t* region, DevError* err,
                                  cudaStream_t stream) {
  if (const cudaError_t e0 = launch_prologue(); e0 != cudaSuccess) return e0;
  const BmDims dims = bm_dims(total_tokens, max_seqlen, topk);
  BmPlan p;
  bm_carve(dims, region, &p);
  CUtensorMap qmap, kmap, vmap, amap;
  if (!encode3d_f32(&amap, p.acc, kDim, kHeads, total_tokens, 32, kGroup, 1) ||
      !encode_q_entry(&qmap, q, total_tokens) ||
      !encode3d(&kmap, k, kDim, kKvHeads, total_tokens, 64, 1, kBlock) ||
      !encode3d(&vmap, v, kDim, kKvHeads, total_tokens, 64, 1, kBlock))
    return cudaErrorInvalidValue;
  const long long keys = 2 * kKvHeads * dims.kg_max;
  cudaError_t e = cudaMemsetAsync(p.counts, 0, keys * sizeof(int), stream);
  if (e != cudaSuccess) return e;
  // rows that no entry reaches keep lacc = 0 (the reference phase stores the others)
  e = cudaMemsetAsync(p.lacc, 0, static_cast<size_t>(total_tokens) * kHeads * sizeof(float), stream);
  if (e != cudaSuccess) return e;
  bm_geom_kernel<<<1, 1024, 0, stream>>>(cu_seqlens, num_docs, total_tokens, dims.W, dims.nw, dims.kg_max, p, err);
  const long long pairs = kKvHeads * total_tokens;
  bm_count_kernel<<<static_cast<unsigned>((pairs + 255) / 256), 256, 0, stream>>>(q2k, cu_seqlens, num_docs,
                                                                                 total_tokens, topk, dims.W, p, err);
  bm_scan_kernel<<<1, 1024, 0, stream>>>(p);
  bm_tiles_kernel<<<static_cast<unsigned>((dims.tiles_max + 255) / 256), 256, 0, stream>>>(cu_seqlens, num_docs,
                                                                                          dims.nw, p);
  bm_scatter_kernel<<<static_cast<unsigned>((dims.entries + 255) / 256), 256, 0, stream>>>(
      dims.entries, total_tokens * topk, p);
  const size_t smem = sizeof(BmSmem) + 1024;
  cudaFuncSetAttribute(bm_attend_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  const long long chunks = (dims.tiles_max + kBmChunk - 1) / kBmChunk;
  const int grid = static_cast<int>(chunks < kNumSMs ? chunks : kNumSMs);
  const float scale_log2 = scale * 1.4426950408889634f;
  // the reference tiles, then (once their mref, lacc and acc are written) the others
  for (int phase = 0; phase < 2; ++phase)
    bm_attend_kernel<<<grid, kBmThreads, smem, stream>>>(qmap, kmap, vmap, amap, p, total_tokens, topk, scale_log2,
                                                         phase, err);
  const long long rows = total_tokens * kHeads;
  bm_norm_kernel<<<static_cast<unsigned>((rows + 15) / 16), 256, 0, stream>>>(p, rows,
                                                                            static_cast<__nv_bfloat16*>(out), lse);
  return cudaGetLastError();
}


// ==== backward =======================================================================
//
// NeMo _SparseAttention.backward: grad_out [tokens, 64, 128] -> dq [tokens, 64,
// 128], dk / dv [tokens, 4, 128] (bf16), with the forward's log-sum-exp.  For
// query head h and key p of its selected causal keys, z = scale <q, k_p>,
// P = 2^(z log2 e - lse), dP = <dO, v_p>, D = <dO, out>, dS = P (dP - D):
//   dv_p += P dO,   dk_p += scale dS q,   dq += scale sum_p dS k_p.
//
// Same bucketing and tiles as the forward: a tile is 8 (query, KV head) entries
// x 16 heads against one key block.  Per tile, five 128 x 128 x 128 tcgen05
// products, in this order, with S, dP (then dQ) and the block's dV and dK
// accumulators in the four 128-column quarters of tensor memory:
//   S  = Q K^T          (A = Q, B = K: both K-major)
//   dP = dO V^T         (A = dO, B = V: both K-major)
//   dK += dS^T Q        (A = dS^T, B = Q: both read MN-major)   frees Q
//   dV += P^T dO        (A = P^T, B = dO: both read MN-major)   frees dO
//   dQ = dS K           (A = dS K-major, B = K read MN-major)
// The tiles' Q and dO rows stream through a ring of three 32 KB slots, so the
// next tile's Q is resident while a tile runs and its dO lands while dV and
// dQ run; the next tile's S is issued right behind dQ (its columns are free
// once P and dS are built), and only its dP waits for dQ to be read out.
// Eight math warps (two per tensor-memory lane group, one half of the
// columns each: P and dS are elementwise in S and dP given the forward's
// lse, so the halves need no exchange) build P and dS in shared memory; each
// then writes its quarter of the tile's dQ (bf16) into its own bytes of the
// P buffer and has the tensor engine add those two 16 x 64 boxes into the
// bf16 dq output (a bulk bf16 reduction, where the NeMo page sums dq with
// bf16 atomics: per-thread atomics, 32 KB a tile, queued the memory
// instructions of the whole SM).  When the tiles of one key block end (a
// run), the same warps add the block's dK and dV to fp32 accumulators, which
// a last kernel converts to bf16.
constexpr int kBwThreads = 352;  // warps 0-7 math, 8 TMA (K, V, Q), 9 MMA, 10 TMA (dO)
constexpr int kBwMath = 8;       // two per tensor-memory lane group, one half of the columns each
constexpr int kBwTmaWarp = 8, kBwMmaWarp = 9, kBwOWarp = 10;
constexpr int kBwSlots = 3;  // ring of Q / dO tiles: load 2i is tile i's Q, load 2i + 1 its dO
constexpr int kBwInfo = 4;
constexpr uint32_t kIdescKK = tc::idesc_bf16_f32(128, 128);
constexpr uint32_t kIdescKM = tc::idesc_bf16_f32(128, 128) | (1u << 16);               // B MN-major
constexpr uint32_t kIdescMM = tc::idesc_bf16_f32(128, 128) | (1u << 15) | (1u << 16);  // A and B MN-major

struct BwInfo {
  int row0, g, cnt, fresh, last;  // last: the run's final tile
  int ent[kBmEntries];
};

struct BwSmem {
  alignas(1024) uint8_t qd[kBwSlots][kBmTile];  // Q and dO rows of the tiles, in load order
  alignas(1024) uint8_t k[kBmTile];              // the block's K
  alignas(1024) uint8_t v[kBmTile];              // the block's V
  alignas(1024) uint8_t p[kBmTile];              // P, bf16 [rows][keys]
  alignas(1024) uint8_t ds[kBmTile];             // dS, bf16 [rows][keys]
  uint64_t info_full[kBwInfo], info_empty[kBwInfo];
  uint64_t kv_full, kv_empty, qd_full[kBwSlots], qd_empty[kBwSlots];
  uint64_t s_full, p_full, dq_full, dq_free, acc_full, acc_free, done;
  BwInfo info[kBwInfo];
  int loads[2];  // Q and dO tiles issued, for the drain at exit
  uint32_t tmem_base;
};
static_assert(sizeof(BwSmem) + 1024 <= 227 * 1024, "shared memory of the backward kernel");


// D[t][h] = <dO[t][h], out[t][h]> (fp32, bf16 inputs): one warp per (token, head).
__global__ void __launch_bounds__(256) bw_rowdot_kernel(const __nv_bfloat16* __restrict__ dout,
                                                        const __nv_bfloat16* __restrict__ out, long long rows,
                                                        float* __restrict__ D) {
  const long long row = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const __nv_bfloat162* a = reinterpret_cast<const __nv_bfloat162*>(dout + row * kDim) + 2 * lane;
  const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(out + row * kDim) + 2 * lane;
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const float2 x = __bfloat1622float2(a[i]), y = __bfloat1622float2(b[i]);
    acc = fmaf(x.x, y.x, fmaf(x.y, y.y, acc));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (lane == 0) D[row] = acc;
}

// fp32 accumulator -> bf16, eight values per thread.
__global__ void __launch_bounds__(256) bw_to_bf16_kernel(const float* __restrict__ src, long long n8,
                                                         __nv_bfloat16* __restrict__ dst) {
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n8) return;
  const float4 a = reinterpret_cast<const float4*>(src)[2 * i], b = reinterpret_cast<const float4*>(src)[2 * i + 1];
  uint4 o;
  o.x = pack_bf16(a.x, a.y);
  o.y = pack_bf16(a.z, a.w);
  o.z = pack_bf16(b.x, b.y);
  o.w = pack_bf16(b.z, b.w);
  reinterpret_cast<uint4*>(dst)[i] = o;
}

// Registers: the busiest of the four sub-partitions holds ceil(11 / 4) = 3
// warps, and a sub-partition has 16384 registers.
constexpr int kBwMaxRegs = 168;
static_assert((kBwThreads / 32 + 3) / 4 * 32 * kBwMaxRegs <= 16384, "registers of the backward kernel");
__global__ void __maxnreg__(kBwMaxRegs) bw_attend_kernel(
    const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap omap,
    const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
    const __grid_constant__ CUtensorMap dqmap, const __grid_constant__ CUtensorMap dkmap,
    const __grid_constant__ CUtensorMap dvmap, BmPlan p, long long T, int topk, float scale, float scale_log2,
    const float* __restrict__ lse, const float* __restrict__ Dsum, DevError* err) {
  extern __shared__ uint8_t smem_raw[];
  BwSmem& sm = *reinterpret_cast<BwSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n = local_tiles(p.meta[1]);

  if (tid == 0) {
    for (int i = 0; i < kBwInfo; ++i) {
      mbar_init(&sm.info_full[i], 1);
      mbar_init(&sm.info_empty[i], kBwMath + 2);  // the math warps, the MMA thread, the dO warp
    }
    mbar_init(&sm.kv_full, 1);
    mbar_init(&sm.kv_empty, 1);
    for (int i = 0; i < kBwSlots; ++i) {
      mbar_init(&sm.qd_full[i], 1);
      mbar_init(&sm.qd_empty[i], 1);
    }
    mbar_init(&sm.s_full, 1);
    mbar_init(&sm.p_full, kBwMath);
    mbar_init(&sm.dq_full, 1);
    mbar_init(&sm.dq_free, kBwMath);
    mbar_init(&sm.acc_full, 1);
    mbar_init(&sm.acc_free, kBwMath);
    mbar_init(&sm.done, 1);
    fence_mbar_init();
  }
  // Rows of entries a tile does not fill keep earlier (finite) data; start
  // from zeros so that no NaN pattern meets a zero weight in an MMA.
  for (int i = tid; i < (kBwSlots + 4) * kBmTile / 16; i += kBwThreads)
    sts128(smem_u32(sm.qd[0]) + 16 * i, 0u, 0u, 0u, 0u);
  fence_proxy_async_smem();
  if (warp == kBwMmaWarp) {
    tc::alloc(&sm.tmem_base, 512);
    tc::relinquish();
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = sm.tmem_base;

  if (warp == kBwTmaWarp) {
    // ---------------- scheduler + TMA (K, V and the tiles' Q) ----------------
    if (lane == 0) {
      prefetch_tmap(&qmap);
      prefetch_tmap(&kmap);
      prefetch_tmap(&vmap);
    }
    const BmTile none{-1, -1, 0, 0};
    BmTile d_next = n > 0 ? p.tiles[tile_at(0)] : none;
    int e_next = lane < d_next.cnt ? p.elist[d_next.off + lane] : 0;
    BmTile d_after = n > 1 ? p.tiles[tile_at(1)] : none;
    int prow = -1, pg = -1, nkv = 0, nq = 0;
    for (int i = 0; i < n; ++i) {
      const BmTile d = d_next;
      const int ent = e_next;
      d_next = d_after;
      e_next = (i + 1 < n && lane < d_next.cnt) ? p.elist[d_next.off + lane] : 0;
      d_after = i + 2 < n ? p.tiles[tile_at(i + 2)] : none;
      const bool fresh = d.row0 != prow || d.g != pg;
      const bool last = i + 1 == n || d_next.row0 != d.row0 || d_next.g != d.g;
      const int is = i % kBwInfo;
      bool ok = true;
      if (lane == 0) ok = mbar_wait(&sm.info_empty[is], ((i / kBwInfo) & 1) ^ 1, err, 800);
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      if (lane < kBmEntries) sm.info[is].ent[lane] = ent;
      if (lane == 0) {
        sm.info[is].row0 = d.row0;
        sm.info[is].g = d.g;
        sm.info[is].cnt = d.cnt;
        sm.info[is].fresh = fresh ? 1 : 0;
        sm.info[is].last = last ? 1 : 0;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.info_full[is]);
      const int ld = 2 * i, slot = ld % kBwSlots;
      if (lane == 0) {
        if (fresh) {
          ok = mbar_wait(&sm.kv_empty, (nkv & 1) ^ 1, err, 801);
          if (ok) {
            mbar_expect_tx(&sm.kv_full, 2 * kBmTile);
            tma_load_3d(sm.k, &kmap, 0, d.g, d.row0, &sm.kv_full);
            tma_load_3d(sm.k + kBmHalf, &kmap, 64, d.g, d.row0, &sm.kv_full);
            tma_load_3d(sm.v, &vmap, 0, d.g, d.row0, &sm.kv_full);
            tma_load_3d(sm.v + kBmHalf, &vmap, 64, d.g, d.row0, &sm.kv_full);
            ++nkv;
          }
        }
        ok = ok && mbar_wait(&sm.qd_empty[slot], ((ld / kBwSlots) & 1) ^ 1, err, 802);
        if (ok) mbar_expect_tx(&sm.qd_full[slot], d.cnt * 2 * kBmQBox);
      }
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      if (fresh) {
        prow = d.row0;
        pg = d.g;
      }
      if (lane < d.cnt) {
        const int t = ent / topk;
        tma_load_3d(sm.qd[slot] + lane * kBmQBox, &qmap, 0, d.g * kGroup, t, &sm.qd_full[slot]);
        tma_load_3d(sm.qd[slot] + kBmHalf + lane * kBmQBox, &qmap, 64, d.g * kGroup, t, &sm.qd_full[slot]);
      }
      __syncwarp();
      ++nq;
    }
    // no copy may still be landing when the CTA exits (the ring's slots are
    // drained below, once both producers have stopped)
    if (lane == 0) {
      if (nkv > 0) mbar_wait(&sm.kv_full, (nkv - 1) & 1, err, 803);
      sm.loads[0] = nq;
    }
  } else if (warp == kBwOWarp) {
    // ---------------- dO rows of each tile (the tensor copies of Q and dO
    // are issued from two warps: about 100 cycles of issue per 2 KB box) ----------------
    if (lane == 0) prefetch_tmap(&omap);
    int no = 0;
    for (int i = 0; i < n; ++i) {
      const int is = i % kBwInfo;
      if (!__all_sync(0xffffffffu, mbar_wait(&sm.info_full[is], (i / kBwInfo) & 1, err, 805))) break;
      const int cnt = sm.info[is].cnt, g = sm.info[is].g;
      const int ent = lane < kBmEntries ? sm.info[is].ent[lane] : 0;
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.info_empty[is]);
      const int ld = 2 * i + 1, slot = ld % kBwSlots;
      bool ok = true;
      if (lane == 0) {
        ok = mbar_wait(&sm.qd_empty[slot], ((ld / kBwSlots) & 1) ^ 1, err, 806);
        if (ok) mbar_expect_tx(&sm.qd_full[slot], cnt * 2 * kBmQBox);
      }
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      if (lane < cnt) {
        const int t = ent / topk;
        tma_load_3d(sm.qd[slot] + lane * kBmQBox, &omap, 0, g * kGroup, t, &sm.qd_full[slot]);
        tma_load_3d(sm.qd[slot] + kBmHalf + lane * kBmQBox, &omap, 64, g * kGroup, t, &sm.qd_full[slot]);
      }
      __syncwarp();
      ++no;
    }
    if (lane == 0) sm.loads[1] = no;
  } else if (warp == kBwMmaWarp) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      int nkv = 0;
      const uint32_t ka = smem_u32(sm.k), va = smem_u32(sm.v), pa = smem_u32(sm.p), dsa = smem_u32(sm.ds);
      for (int i = 0; i < n; ++i) {
        const int is = i % kBwInfo;
        if (!mbar_wait(&sm.info_full[is], (i / kBwInfo) & 1, err, 810)) break;
        const bool fresh = sm.info[is].fresh != 0, last = sm.info[is].last != 0;
        mbar_arrive(&sm.info_empty[is]);
        const int run = nkv;  // the run this tile belongs to is run - 1 after a fresh tile
        if (fresh) {
          if (!mbar_wait(&sm.kv_full, nkv & 1, err, 811)) break;
          ++nkv;
        }
        const int lq = 2 * i, lo = 2 * i + 1, sq = lq % kBwSlots, so = lo % kBwSlots;
        const uint32_t qa = smem_u32(sm.qd[sq]), oa = smem_u32(sm.qd[so]);
        // S's columns were read out before the previous tile's P / dS were
        // published, which this thread waited for
        if (!mbar_wait(&sm.qd_full[sq], (lq / kBwSlots) & 1, err, 812)) break;
        tc::fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = (kk >> 2) * kBmHalf + (kk & 3) * 32;
          tc::mma_bf16(tmem, tc::desc_k_sw128(qa + off), tc::desc_k_sw128(ka + off), kIdescKK, kk > 0);
        }
        if (!mbar_wait(&sm.qd_full[so], (lo / kBwSlots) & 1, err, 813)) break;
        // dP reuses the columns of the previous tile's dQ
        if (i > 0 && !mbar_wait(&sm.dq_free, (i - 1) & 1, err, 814)) break;
        tc::fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = (kk >> 2) * kBmHalf + (kk & 3) * 32;
          tc::mma_bf16(tmem + 128, tc::desc_k_sw128(oa + off), tc::desc_k_sw128(va + off), kIdescKK, kk > 0);
        }
        tc::commit(&sm.s_full);
        if (!mbar_wait(&sm.p_full, i & 1, err, 815)) break;
        // the previous run's dK / dV must be read out before a fresh tile restarts them
        if (fresh && run > 0 && !mbar_wait(&sm.acc_free, (run - 1) & 1, err, 816)) break;
        tc::fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          tc::mma_bf16(tmem + 384, desc_v_mn_sw128(dsa + kk * 2048), desc_v_mn_sw128(qa + kk * 2048), kIdescMM,
                       kk > 0 || !fresh);
        tc::commit(&sm.qd_empty[sq]);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          tc::mma_bf16(tmem + 256, desc_v_mn_sw128(pa + kk * 2048), desc_v_mn_sw128(oa + kk * 2048), kIdescMM,
                       kk > 0 || !fresh);
        tc::commit(&sm.qd_empty[so]);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = (kk >> 2) * kBmHalf + (kk & 3) * 32;
          tc::mma_bf16(tmem + 128, tc::desc_k_sw128(dsa + off), desc_v_mn_sw128(ka + kk * 2048), kIdescKM, kk > 0);
        }
        tc::commit(&sm.dq_full);
        if (last) {
          tc::commit(&sm.acc_full);
          tc::commit(&sm.kv_empty);
        }
      }
      // every MMA has finished before tensor memory is released
      tc::commit(&sm.done);
      mbar_wait(&sm.done, 0, err, 817);
    }
  } else if (warp < kBwMath) {
    // ---------------- math warps 0-7: warp w takes tile row (w % 4) * 32 + lane
    // and columns (w / 4) * 64 ... + 63 of every 128-column quarter ----------------
    const int r = (warp & 3) * 32 + lane, e = r >> 4, h = r & 15, c0 = (warp >> 2) * 2;
    const uint32_t lrow = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    const uint32_t ps = smem_u32(sm.p), dss = smem_u32(sm.ds);
    if (tid == 0) {
      prefetch_tmap(&dqmap);
      prefetch_tmap(&dkmap);
      prefetch_tmap(&dvmap);
    }
    int nacc = 0;
    for (int i = 0; i < n; ++i) {
      const int is = i % kBwInfo;
      if (!__all_sync(0xffffffffu, mbar_wait(&sm.info_full[is], (i / kBwInfo) & 1, err, 820))) break;
      const int cnt = sm.info[is].cnt, row0 = sm.info[is].row0, g = sm.info[is].g;
      const bool last = sm.info[is].last != 0;
      const bool valid = e < cnt;
      const int ent = valid ? sm.info[is].ent[e] : 0;
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.info_empty[is]);
      const long long t = ent / topk;
      const int nkeys = valid ? static_cast<int>(min(static_cast<long long>(kBlock), t - row0 + 1)) : 0;
      const long long hrow = t * kHeads + g * kGroup + h;  // (token, query head)
      const float lse_r = valid ? lse[hrow] : 0.f, d_r = valid ? Dsum[hrow] : 0.f;
      if (!__all_sync(0xffffffffu, mbar_wait(&sm.s_full, i & 1, err, 821))) break;
      tc::fence_after();
      // the previous tile's dQ reductions read these bytes of the P buffer
      if (lane == 0) bulk_wait_read_all();
      __syncwarp();
      // 16-column pieces, the next piece's loads in flight while one is computed
      uint32_t sv[2][16], dp[2][16];
      tc::ld_32x32b_x16(lrow + c0 * 32, sv[0]);
      tc::ld_32x32b_x16(lrow + 128 + c0 * 32, dp[0]);
#pragma unroll
      for (int pc = 0; pc < 4; ++pc) {
        tc::wait_ld();
        if (pc < 3) {
          tc::ld_32x32b_x16(lrow + c0 * 32 + (pc + 1) * 16, sv[(pc + 1) & 1]);
          tc::ld_32x32b_x16(lrow + 128 + c0 * 32 + (pc + 1) * 16, dp[(pc + 1) & 1]);
        }
        const uint32_t(&s_)[16] = sv[pc & 1];
        const uint32_t(&d_)[16] = dp[pc & 1];
        uint32_t pk[8], dk[8];
        // keys at or past nkeys (the causal edge, the document's end) get P = 0;
        // away from the diagonal block every key of the piece counts
        const int kc0 = c0 * 32 + pc * 16;
        const bool whole = kc0 + 16 <= nkeys;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const float2 z = fma2(__uint_as_float(s_[2 * q]), __uint_as_float(s_[2 * q + 1]), scale_log2, scale_log2,
                                -lse_r, -lse_r);
          float pa = ex2(z.x), pb = ex2(z.y);
          if (!whole) {
            pa = kc0 + 2 * q < nkeys ? pa : 0.f;
            pb = kc0 + 2 * q + 1 < nkeys ? pb : 0.f;
          }
          pk[q] = pack_bf16(pa, pb);
          const float2 dd = sub2(__uint_as_float(d_[2 * q]), __uint_as_float(d_[2 * q + 1]), d_r, d_r);
          const float2 ds = mul2(pa, pb, dd.x, dd.y);
          dk[q] = pack_bf16(ds.x, ds.y);
        }
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int c16 = c0 * 4 + pc * 2 + c;  // 16-byte chunk of the 256-byte row
          const uint32_t off = (c16 >> 3) * kBmHalf + sw128(r, c16 & 7);
          sts128(ps + off, pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
          sts128(dss + off, dk[4 * c], dk[4 * c + 1], dk[4 * c + 2], dk[4 * c + 3]);
        }
      }
      tc::fence_before();
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.p_full);
      if (!__all_sync(0xffffffffu, mbar_wait(&sm.dq_full, i & 1, err, 822))) break;
      tc::fence_after();
      // dQ (scaled, bf16) goes to this warp's own bytes of the P buffer (every
      // product of the tile has finished), laid out as the Q tile's boxes: the
      // warp's 32 rows are two entries, its 64 columns one d half, so it
      // reduces exactly two boxes into dq with the tensor engine
#pragma unroll 1
      for (int ch = c0; ch < c0 + 2; ++ch) {
        uint32_t v[32];
        tc::ld_32x32b_x32(lrow + 128 + ch * 32, v);
        tc::wait_ld();
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t w[4];
#pragma unroll
          for (int x = 0; x < 4; ++x)
          {
            const float2 y = mul2(__uint_as_float(v[8 * c + 2 * x]), __uint_as_float(v[8 * c + 2 * x + 1]), scale, scale);
            w[x] = pack_bf16(y.x, y.y);
          }
          const int c16 = ch * 4 + c;
          sts128(ps + (c16 >> 3) * kBmHalf + sw128(r, c16 & 7), w[0], w[1], w[2], w[3]);
        }
      }
      tc::fence_before();
      fence_proxy_async_smem();
      const int t_hi = __shfl_sync(0xffffffffu, static_cast<int>(t), 16);
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&sm.dq_free);
        const int e0 = 2 * (warp & 3), hf = warp >> 2;
        if (e0 < cnt) tma_reduce_add_3d(&dqmap, sm.p + hf * kBmHalf + e0 * kBmQBox, hf * 64, g * kGroup, static_cast<int>(t));
        if (e0 + 1 < cnt)
          tma_reduce_add_3d(&dqmap, sm.p + hf * kBmHalf + (e0 + 1) * kBmQBox, hf * 64, g * kGroup, t_hi);
        bulk_commit();
      }
      if (last) {
        // The run's dV, then its dK, through this warp's own 8 KB of the P
        // and dS buffers (every product of the run has finished): its 32 key
        // rows x 64 columns in fp32 are two 32 x 32 boxes with the 128-byte
        // swizzle, which the tensor engine adds into the fp32 accumulators.
        if (!__all_sync(0xffffffffu, mbar_wait(&sm.acc_full, nacc & 1, err, 823))) break;
        ++nacc;
        tc::fence_after();
        const int krow0 = row0 + (warp & 3) * 32;
        const uint32_t own[2] = {ps + (warp >> 2) * kBmHalf + (warp & 3) * 4096,
                                 dss + (warp >> 2) * kBmHalf + (warp & 3) * 4096};
#pragma unroll 1
        for (int acc = 0; acc < 2; ++acc) {
          // the earlier reductions of this warp have read these bytes
          if (lane == 0) bulk_wait_read_all();
          __syncwarp();
          const float f = acc == 0 ? 1.f : scale;
#pragma unroll 1
          for (int jj = 0; jj < 2; ++jj) {
            uint32_t a[32];
            tc::ld_32x32b_x32(lrow + (acc == 0 ? 256 : 384) + (c0 + jj) * 32, a);
            tc::wait_ld();
#pragma unroll
            for (int j = 0; j < 8; ++j)
              sts128(own[jj] + sw128(lane, j), __float_as_uint(f * __uint_as_float(a[4 * j])),
                     __float_as_uint(f * __uint_as_float(a[4 * j + 1])),
                     __float_as_uint(f * __uint_as_float(a[4 * j + 2])),
                     __float_as_uint(f * __uint_as_float(a[4 * j + 3])));
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            if (krow0 < T) {
              const CUtensorMap* m = acc == 0 ? &dvmap : &dkmap;
              for (int jj = 0; jj < 2; ++jj)
                tma_reduce_add_3d(m, (jj == 0 ? sm.p : sm.ds) + (warp >> 2) * kBmHalf + (warp & 3) * 4096,
                                  (c0 + jj) * 32, g, krow0);
            }
            bulk_commit();
          }
        }
        tc::fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.acc_free);
      }
    }
    if (lane == 0) bulk_wait_all();  // the dQ reductions have landed
  }
  tc::fence_before();
  __syncthreads();
  if (warp == kBwMmaWarp) {
    tc::fence_after();
    tc::dealloc(tmem, 512);
  }
  if (warp == kBwTmaWarp && lane == 0) {
    // A slot is refilled only after its previous load was consumed (and so
    // had landed): only the latest load into each slot can still be in
    // flight (after an error stopped the MMA thread early).  Wait for those.
    int latest[kBwSlots] = {-1, -1, -1};
    for (int j = sm.loads[0] > 3 ? sm.loads[0] - 3 : 0; j < sm.loads[0]; ++j) latest[(2 * j) % kBwSlots] = 2 * j;
    for (int j = sm.loads[1] > 3 ? sm.loads[1] - 3 : 0; j < sm.loads[1]; ++j) {
      const int ld = 2 * j + 1;
      if (ld > latest[ld % kBwSlots]) latest[ld % kBwSlots] = ld;
    }
    for (int s = 0; s < kBwSlots; ++s)
      if (latest[s] >= 0) mbar_wait(&sm.qd_full[s], (latest[s] / kBwSlots) & 1, err, 804);
  }
}

// Backward workspace: the forward's bucketing arrays, then (in place of the
// forward's accumulators, which the backward does not use) D [T][64] and the
// fp32 accumulators dk and dv [T][4][128] (dq is summed in the bf16 output).
struct BwCarve {
  float* D;
  float* dk;
  float* dv;
  size_t bytes;
};
static BwCarve bw_carve(long long T, int max_seqlen, int topk, uint8_t* region) {
  BwCarve c;
  const BmDims d = bm_dims(T, max_seqlen, topk);
  size_t off = bm_carve(d, nullptr, nullptr, false);  // the bucketing arrays
  auto take = [&](size_t bytes) {
    uint8_t* ptr = region ? region + off : nullptr;
    off += al256(bytes);
    return reinterpret_cast<float*>(ptr);
  };
  c.D = take(static_cast<size_t>(T) * kHeads * sizeof(float));
  c.dk = take(static_cast<size_t>(T) * kKvHeads * kDim * sizeof(float));
  c.dv = take(static_cast<size_t>(T) * kKvHeads * kDim * sizeof(float));
  c.bytes = off;
  return c;
}

size_t prefill_backward_bytes(long long total_tokens, int max_seqlen, int topk) {
  return bw_carve(total_tokens, max_seqlen, topk, nullptr).bytes;
}

cudaError_t launch_prefill_backward(const void* q, const void* k, const void* v, const int32_t* q2k,
                                    const int32_t* cu_seqlens, int num_docs, long long total_tokens,
                                    int max_seqlen, int topk, float scale, const void* out, const float* lse,
                                    const void* grad_out, void* dq, void* dk, void* dv, uint8_t* region,
                                    DevError* err, cudaStream_t stream) {
  if (const cudaError_t e0 = launch_prologue(); e0 != cudaSuccess) return e0;
  const BmDims dims = bm_dims(total_tokens, max_seqlen, topk);
  BmPlan p;
  bm_carve(dims, region, &p, false);
  p.phases = 1;  // no reference split: one phase of keys
  const BwCarve w = bw_carve(total_tokens, max_seqlen, topk, region);
  CUtensorMap qmap, omap, kmap, vmap, dqmap, dkmap, dvmap;
  if (!encode3d(&qmap, q, kDim, kHeads, total_tokens, 64, kGroup, 1) ||
      !encode3d(&omap, grad_out, kDim, kHeads, total_tokens, 64, kGroup, 1) ||
      !encode3d(&dqmap, dq, kDim, kHeads, total_tokens, 64, kGroup, 1) ||
      !encode3d_f32(&dkmap, w.dk, kDim, kKvHeads, total_tokens, 32, 1, 32) ||
      !encode3d_f32(&dvmap, w.dv, kDim, kKvHeads, total_tokens, 32, 1, 32) ||
      !encode3d(&kmap, k, kDim, kKvHeads, total_tokens, 64, 1, kBlock) ||
      !encode3d(&vmap, v, kDim, kKvHeads, total_tokens, 64, 1, kBlock))
    return cudaErrorInvalidValue;
  const long long T = total_tokens;
  cudaError_t e;
  if ((e = cudaMemsetAsync(dq, 0, static_cast<size_t>(T) * kHeads * kDim * sizeof(__nv_bfloat16), stream)) !=
          cudaSuccess ||
      (e = cudaMemsetAsync(w.dk, 0, static_cast<size_t>(T) * kKvHeads * kDim * sizeof(float), stream)) != cudaSuccess ||
      (e = cudaMemsetAsync(w.dv, 0, static_cast<size_t>(T) * kKvHeads * kDim * sizeof(float), stream)) != cudaSuccess)
    return e;
  // the forward's bucketing of the q2k entries
  const long long keys = kKvHeads * dims.kg_max;
  if ((e = cudaMemsetAsync(p.counts, 0, keys * sizeof(int), stream)) != cudaSuccess) return e;
  bm_geom_kernel<<<1, 1024, 0, stream>>>(cu_seqlens, num_docs, T, dims.W, dims.nw, dims.kg_max, p, err);
  bm_count_kernel<<<static_cast<unsigned>((kKvHeads * T + 255) / 256), 256, 0, stream>>>(
      q2k, cu_seqlens, num_docs, T, topk, dims.W, p, err);
  bm_scan_kernel<<<1, 1024, 0, stream>>>(p);
  bm_tiles_kernel<<<static_cast<unsigned>((dims.tiles_max + 255) / 256), 256, 0, stream>>>(cu_seqlens, num_docs,
                                                                                          dims.nw, p);
  bm_scatter_kernel<<<static_cast<unsigned>((dims.entries + 255) / 256), 256, 0, stream>>>(dims.entries, T * topk,
                                                                                           p);
  bw_rowdot_kernel<<<static_cast<unsigned>((T * kHeads + 7) / 8), 256, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(grad_out), static_cast<const __nv_bfloat16*>(out), T * kHeads, w.D);
  const size_t smem = sizeof(BwSmem) + 1024;
  cudaFuncSetAttribute(bw_attend_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  const long long chunks = (dims.tiles_max + kBmChunk - 1) / kBmChunk;
  const int grid = static_cast<int>(chunks < kNumSMs ? chunks : kNumSMs);
  bw_attend_kernel<<<grid, kBwThreads, smem, stream>>>(qmap, omap, kmap, vmap, dqmap, dkmap, dvmap, p, T, topk,
                                                       scale, scale * 1.4426950408889634f, lse, w.D, err);
  const long long nk8 = T * kKvHeads * kDim / 8;
  bw_to_bf16_kernel<<<static_cast<unsigned>((nk8 + 255) / 256), 256, 0, stream>>>(w.dk, nk8,
                                                                                 static_cast<__nv_bfloat16*>(dk));
  bw_to_bf16_kernel<<<static_cast<unsigned>((nk8 + 255) / 256), 256, 0, stream>>>(w.dv, nk8,
                                                                                 static_cast<__nv_bfloat16*>(dv));
  return cudaGetLastError();
}

}  // namespace msa
