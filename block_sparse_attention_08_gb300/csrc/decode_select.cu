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
// 128-key page (32 KB bf16 / 16 KB E4M3, contiguous) is one work item.  The
// (request, page) items of all requests, in order, are cut into chunks of a
// few pages; a persistent grid of one CTA per SM takes the first wave of
// chunks by CTA index and then claims chunks from a counter, so an SM that
// streams faster takes more of them and all SMs finish together (a fixed even
// split left the slowest SM 20-40 % behind the median on the long-context
// batches).  Inside a CTA a producer warp resolves 32 page ids at a time with
// one coalesced load and issues one 1-D bulk TMA copy per page into a ring of
// 192 KB of shared memory (6 bf16 / 12 E4M3 pages in flight); six consumer
// warps each take whole pages round-robin (stage s always to warp s % 6) and
// score all 128 keys on the tensor cores (mma.sync: keys as A read straight
// from the page, the 4 index heads as B, fp32 accumulate), reduce the block
// max in registers and store one fp32 score per (request, head, page).  No
// CTA-wide barrier sits in the loop.  A second kernel, launched as a
// programmatic dependent so its launch overlaps the scorer's tail, runs the
// top-k with one CTA per (request, head) row: a threshold from 32 maxima of
// the row filters the candidates, then an exact (score desc, id asc) pick.
#include "launch.h"

namespace msa {

constexpr int kSelConsumers = 6;  // a divisor of the stage counts (6 bf16, 12 E4M3)
constexpr int kSelThreads = 32 * (kSelConsumers + 1);
constexpr int kSelRingBytes = 192 * 1024;
constexpr int kCandCap = 64;  // the top-k's candidate list (a larger count takes its exact fallback)

struct DecodeGeom {
  const int32_t* seq_lens;
  const int32_t* page_table;
  const int64_t* cu_k;
  int batch;
  int max_blocks;
  long long num_slots;
};

struct SelMeta {
  int r, b, rows, pad;
};

template <int kStages>
struct SelSmem {
  alignas(1024) uint8_t ring[kSelRingBytes];
  // the page's request's index query (4 heads), landed with the page
  alignas(16) uint8_t qs[kStages][kSelRingBytes / kStages / kBlock * kKvHeads];
  uint64_t full[kStages];
  uint64_t empty[kStages];
  SelMeta meta[kStages];
  int scan[kSelThreads / 32];
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
// (request, head) row, then the ascending q2k row.  One CTA of 128 threads per
// row: the row's scores are staged in shared memory first (rows of up to
// kTopkStage blocks; longer rows are read from global memory as they go), each
// thread takes every 128th candidate, the first warp reduces the 128 thread
// maxima to 32 (the maxima of every 32nd candidate) and sorts them with a
// bitonic network over its lanes; the need-th largest of the 32 is a threshold
// that at least `need` candidates reach (so it keeps all of the top `need`),
// those candidates (a few more than `need` as a rule) are gathered in shared
// memory, and each is ranked against the others by its own thread.  A row of
// at most 128 candidates skips the threshold: each candidate is ranked against
// all of them at once.  (One warp per row took 2-7 us on rows of 64-1024
// candidates; ranking each of the 128 thread maxima against the others,
// 1200-4400 cycles.)
constexpr int kTopkThreads = 128;
constexpr int kTopkStage = 1024;

__device__ __forceinline__ unsigned long long score_key(float v, int b) {
  return (static_cast<unsigned long long>(float_key(v)) << 32) | (0xffffffffu - static_cast<uint32_t>(b));
}
__device__ __forceinline__ int key_block(unsigned long long key) {
  return static_cast<int>(0xffffffffu - static_cast<uint32_t>(key));
}

// How the page items [0, total) are shared out.  Each CTA first streams a
// fixed range of p0 items (CTA b: [b p0, (b + 1) p0), about three quarters of
// its fair share); the rest, [f, total), is cut into chunks of p1 items that
// the CTAs claim from a counter, so an SM that streams faster takes more of
// them and the SMs finish close together.  A small total is all fixed ranges.
struct SelSplit {
  int p0, p1, n_dyn;
  long long f;
};
__device__ __forceinline__ SelSplit sel_split(int total, int grid) {
  SelSplit t;
  if (total < 8 * grid) {
    t.p0 = (total + grid - 1) / grid;
    t.f = total;
    t.p1 = 1;
    t.n_dyn = 0;
  } else {
    t.p0 = static_cast<int>(3LL * total / (4LL * grid));
    t.f = static_cast<long long>(t.p0) * grid;
    const long long p1 = (total - t.f) / (4LL * grid);
    t.p1 = static_cast<int>(p1 < 1 ? 1 : (p1 > 8 ? 8 : p1));
    t.n_dyn = static_cast<int>((total - t.f + t.p1 - 1) / t.p1);
  }
  return t;
}

// Moves (r, r_start) forward to the scored request holding page item `item`
// (r_start = item index of its first page).  Items only grow along one CTA's
// claims, so the walk never goes back; 32 requests per step, their lengths
// read with one coalesced load (L1-resident after the first pass).  Returns
// false when `item` lies past the last request (never expected).
__device__ __forceinline__ bool walk_to(const DecodeGeom& geo, int topk, long long item, int& r, long long& r_start) {
  const int lane = threadIdx.x & 31;
  while (r < geo.batch) {
    const int rl = r + lane;
    const int v = rl < geo.batch ? scored_blocks(geo, rl, topk, nullptr) : 0;
    int x = v;  // inclusive scan over the lanes
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    const unsigned hit = __ballot_sync(0xffffffffu, rl < geo.batch && r_start + x > item);
    if (hit) {
      const int l = __ffs(hit) - 1;
      r_start += __shfl_sync(0xffffffffu, x - v, l);
      r += l;
      return true;
    }
    r_start += __shfl_sync(0xffffffffu, x, 31);
    r += 32;
  }
  return false;
}

constexpr int kSelEnd = -2;  // meta.r of the stage that ends a consumer warp's loop

// sched: the claim counter in the workspace header, zero when the kernel
// starts (the top-k kernel that follows puts it back to zero once this grid
// has completed).
template <int kE4M3>
__global__ void __launch_bounds__(kSelThreads, 1) decode_select_kernel(
    const uint8_t* __restrict__ index_q, const uint8_t* __restrict__ index_k, DecodeGeom geo,
    float* __restrict__ scores, int topk, int* __restrict__ sched, DevError* err) {
  constexpr int kRowBytes = kE4M3 ? kIdxDim : kIdxDim * 2;
  constexpr int kPageBytes = kBlock * kRowBytes;
  constexpr int kStages = kSelRingBytes / kPageBytes;
  // stage s is always consumed by warp s % kSelConsumers, so a warp never waits
  // on a stage more than one mbarrier phase ahead
  static_assert(kStages % kSelConsumers == 0, "stages must be a multiple of the consumer warps");
  extern __shared__ uint8_t smem_raw[];
  auto& sm = *reinterpret_cast<SelSmem<kStages>*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                  ~uintptr_t(1023));
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int B = geo.batch, mb = geo.max_blocks;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], 1);
    }
    fence_mbar_init();
  }
  // total scored pages (rows of requests that need no scoring are written by the top-k kernel)
  int total = 0;
  for (int r0 = 0; r0 < B; r0 += kSelThreads) {
    const int r = r0 + tid;
    const int v = r < B ? scored_blocks(geo, r, topk, nullptr) : 0;
    total += block_sum(v, sm.scan);
  }
  __syncthreads();  // the barriers are initialised
  const SelSplit split = sel_split(total, gridDim.x);

  if (warp == kSelConsumers) {
    // ---------------- producer warp ----------------
    // Pages go out in groups of up to 32 consecutive items.  While one group's
    // copies are issued, the next group is already located (its requests from
    // a forward walk over the lengths, its page ids loading), and the next
    // claim is in flight, so no lookup waits on the copies' critical path.
    int i = 0;                  // stages used
    int alive = 1;              // 0 after a wait gave up: locate and issue nothing more
    int wr = 0;                 // walk: scored request ...
    long long wstart = 0;       // ... and its first item
    long long s_lo = min(static_cast<long long>(blockIdx.x) * split.p0, split.f);
    const long long s_hi = min(s_lo + split.p0, split.f);
    long long d_lo = 0, d_hi = 0;  // the claimed chunk's items not yet grouped
    int claim = 0;                 // lane 0: answer of the pending claim
    if (lane == 0 && split.n_dyn > 0) claim = atomicAdd(&sched[0], 1);
    auto next_group = [&](long long& a, int& n) {
      n = 0;
      if (s_lo < s_hi) {
        a = s_lo;
        n = static_cast<int>(min(32LL, s_hi - s_lo));
        s_lo += n;
        return;
      }
      if (d_lo >= d_hi) {
        if (split.n_dyn == 0 || !alive) return;
        const int c = __shfl_sync(0xffffffffu, claim, 0);
        if (c >= split.n_dyn) return;
        d_lo = split.f + static_cast<long long>(c) * split.p1;
        d_hi = min(static_cast<long long>(total), d_lo + split.p1);
        if (lane == 0) claim = atomicAdd(&sched[0], 1);  // answered while this chunk is issued
      }
      a = d_lo;
      n = static_cast<int>(min(32LL, d_hi - d_lo));
      d_lo += n;
    };
    // Lane l < n: request and block of item a + l, and the raw page id (or
    // the request's first row) whose load stays in flight until finish().
    struct Group {
      int n, r, b, L;
      long long raw;
    };
    auto locate = [&](long long a, int n, Group& g) {
      g.n = n;
      g.r = -1;
      g.b = 0;
      g.L = 0;
      g.raw = 0;
      if (n == 0) return;
      if (!walk_to(geo, topk, a, wr, wstart)) {  // never expected: the items outnumber the pages
        record_error(err, MSA_DEVERR_TIMEOUT, 1100000);
        g.n = 0;
        return;
      }
      if (lane < n) {
        const long long item = a + lane;
        int rl = wr;
        long long rs = wstart;
        int nbl = scored_blocks(geo, rl, topk, nullptr);
        while (item >= rs + nbl) {
          rs += nbl;
          if (++rl >= B) break;
          nbl = scored_blocks(geo, rl, topk, nullptr);
        }
        if (rl < B) {
          g.r = rl;
          g.b = static_cast<int>(item - rs);
          g.L = geo.seq_lens[rl];
          g.raw = geo.page_table ? static_cast<long long>(geo.page_table[static_cast<long long>(rl) * mb + g.b])
                                 : geo.cu_k[rl];
        }
      }
    };
    // first row and key count of the lane's page (0 keys: nothing to copy)
    auto finish = [&](const Group& g, long long& row0, int& rows) {
      row0 = 0;
      rows = 0;
      if (lane >= g.n || g.r < 0) return;
      const int want = min(kBlock, g.L - g.b * kBlock);
      bool ok;
      if (geo.page_table) {
        row0 = g.raw * kBlock;
        ok = g.raw >= 0 && row0 + kBlock <= geo.num_slots;
        if (!ok) record_error(err, MSA_DEVERR_PAGE, static_cast<long long>(g.r) * mb + g.b);
      } else {
        row0 = g.raw + static_cast<long long>(g.b) * kBlock;
        ok = row0 >= 0 && row0 + want <= geo.num_slots;
        if (!ok) record_error(err, MSA_DEVERR_PAGE, g.r);
      }
      rows = ok && want > 0 ? want : 0;
    };
    Group cur, nxt;
    {
      long long a = 0;
      int n;
      next_group(a, n);
      locate(a, n, cur);
    }
    while (cur.n > 0) {
      long long row0;
      int rows_l;
      finish(cur, row0, rows_l);
      {
        long long a = 0;
        int n;
        next_group(a, n);
        locate(a, n, nxt);
      }
      for (int k = 0; k < cur.n; ++k, ++i) {
        const long long pr0 = __shfl_sync(0xffffffffu, row0, k);
        const int rows = __shfl_sync(0xffffffffu, rows_l, k);
        const int rk = __shfl_sync(0xffffffffu, cur.r, k);
        const int bk = __shfl_sync(0xffffffffu, cur.b, k);
        if (lane == 0) {
          const int s = i % kStages;
          if (!mbar_wait(&sm.empty[s], ((i / kStages) & 1) ^ 1, err, 101)) alive = 0;
          sm.meta[s] = SelMeta{rk, bk, rows, 0};
          if (rows > 0) {
            mbar_expect_tx(&sm.full[s], static_cast<uint32_t>((rows + kKvHeads) * kRowBytes));
            tma_bulk_g2s(sm.ring + s * kPageBytes, index_k + pr0 * kRowBytes, static_cast<uint32_t>(rows * kRowBytes),
                         &sm.full[s]);
            tma_bulk_g2s(sm.qs[s], index_q + static_cast<long long>(rk) * kKvHeads * kRowBytes,
                         static_cast<uint32_t>(kKvHeads * kRowBytes), &sm.full[s]);
          } else {
            mbar_arrive(&sm.full[s]);
          }
        }
        __syncwarp();
      }
      alive = __shfl_sync(0xffffffffu, alive, 0);
      if (!alive) break;
      cur = nxt;
    }
    // one end marker per consumer warp: consecutive stages go to distinct warps
    for (int k = 0; k < kSelConsumers; ++k, ++i) {
      if (lane == 0) {
        const int s = i % kStages;
        mbar_wait(&sm.empty[s], ((i / kStages) & 1) ^ 1, err, 101);
        sm.meta[s] = SelMeta{kSelEnd, 0, 0, 0};
        mbar_arrive(&sm.full[s]);
      }
      __syncwarp();
    }
    // No copy may still be landing when the CTA exits, also after a wait gave
    // up: wait (bounded) for the last fill of every stage.  Only this thread
    // arms the full barriers, so that phase cannot have been passed.
    if (lane == 0) {
      for (int s = 0; s < kStages; ++s) {
        const int f = (i - s + kStages - 1) / kStages;  // fills of stage s
        if (f > 0) mbar_wait(&sm.full[s], (f - 1) & 1, err, 102);
      }
    }
    return;
  }

  // ---------------- consumer warps: whole pages, round-robin ----------------
  if (tid == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int g8 = lane >> 2, t4 = lane & 3;
  uint32_t qf[4][4];
  for (int i = warp;; i += kSelConsumers) {
    const int s = i % kStages;
    if (!mbar_wait(&sm.full[s], (i / kStages) & 1, err, 100)) break;  // gave up: stop consuming
    const SelMeta meta = sm.meta[s];
    if (meta.r == kSelEnd) break;
    if (meta.r < 0 || meta.r >= B || meta.b < 0 || meta.b >= mb) {  // never expected: guard the stores
      record_error(err, MSA_DEVERR_TIMEOUT, 1000000 + i);
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.empty[s]);
      continue;
    }
    const int cur_r = meta.r;
    {
      // the request's index query, landed with the page
      constexpr int kQChunks = kE4M3 ? 2 : 4;
#pragma unroll
      for (int j = 0; j < 4; ++j) qf[j][0] = qf[j][1] = qf[j][2] = qf[j][3] = 0u;
      if (g8 < kKvHeads && meta.rows > 0) {
        const uint32_t qbase = smem_u32(sm.qs[s]) + g8 * kRowBytes + 16 * t4;
#pragma unroll
        for (int j = 0; j < kQChunks; ++j) {
          // bf16: dims 32j + 8t .. +8 ; e4m3: dims 64j + 16t .. +16 -- both at byte 64j + 16t
          const uint4 v = lds128(qbase + 64 * j);
          qf[j][0] = v.x;
          qf[j][1] = v.y;
          qf[j][2] = v.z;
          qf[j][3] = v.w;
        }
      }
    }
    const int rows = meta.rows;
    const uint32_t base = smem_u32(sm.ring + s * kPageBytes);
    float mx0 = -INFINITY, mx1 = -INFINITY;  // heads 2*t4, 2*t4+1
    // two m-tiles (32 keys) per step: all shared loads first, then two
    // independent MMA chains.  Each thread reads 16 contiguous bytes of a key
    // row; the MMA k slots take them in a fixed permutation that B (index_q)
    // repeats, so nothing is moved.
    constexpr int kJ = kE4M3 ? 2 : 4;
    for (int mp = 0; mp < kBlock / 32; ++mp) {
      const int key0 = 32 * mp;
      if (key0 >= rows) break;
      uint4 ra[2][kJ], rb[2][kJ];
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        const uint32_t a_addr = base + (key0 + 16 * h2 + g8) * kRowBytes;
#pragma unroll
        for (int j = 0; j < kJ; ++j) {
          const uint32_t off = kE4M3 ? (64 * j + 16 * t4) : (32 * j + 8 * t4) * 2;
          ra[h2][j] = lds128(a_addr + off);
          rb[h2][j] = lds128(a_addr + 8 * kRowBytes + off);
        }
      }
      float c[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
      for (int j = 0; j < kJ; ++j) {
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          const uint32_t a0[4] = {ra[h2][j].x, rb[h2][j].x, ra[h2][j].y, rb[h2][j].y};
          const uint32_t a1[4] = {ra[h2][j].z, rb[h2][j].z, ra[h2][j].w, rb[h2][j].w};
          if (!kE4M3) {
            mma_bf16(c[h2], a0, qf[j][0], qf[j][1]);
            mma_bf16(c[h2], a1, qf[j][2], qf[j][3]);
          } else {
            mma_e4m3(c[h2], a0, qf[j][0], qf[j][1]);
            mma_e4m3(c[h2], a1, qf[j][2], qf[j][3]);
          }
        }
      }
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        const int k0 = key0 + 16 * h2 + g8;
        if (k0 < rows) {
          mx0 = fmaxf(mx0, c[h2][0]);
          mx1 = fmaxf(mx1, c[h2][1]);
        }
        if (k0 + 8 < rows) {
          mx0 = fmaxf(mx0, c[h2][2]);
          mx1 = fmaxf(mx1, c[h2][3]);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.empty[s]);  // page consumed
    for (int o = 4; o < 32; o <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
    }
    if (lane < 2) {
      float* sp = scores + (static_cast<long long>(cur_r) * kKvHeads + 2 * lane) * mb + meta.b;
      sp[0] = mx0;
      sp[mb] = mx1;
    }
  }
}

// Top-k per (request, head): one CTA of kTopkThreads threads per row.
// Launched right behind the scorer as a programmatic dependent: its CTAs may
// start while the scorer drains, and wait for the scores to be complete.
__global__ void __launch_bounds__(kTopkThreads) decode_topk_kernel(const float* __restrict__ scores, DecodeGeom geo,
                                                                   int32_t* __restrict__ q2k, int topk, int init,
                                                                   int local, int* __restrict__ sched, DevError* err) {
  __shared__ float stage[kTopkStage];
  __shared__ unsigned long long tmax[kTopkThreads];
  __shared__ unsigned long long cand[kCandCap];
  __shared__ int ids[kMaxTopk];
  __shared__ unsigned long long theta_s;
  __shared__ int count_s;
  const int r = blockIdx.x / kKvHeads, h = blockIdx.x % kKvHeads;
  // The request's length is an input of the call, not a result of the scorer,
  // and the scorer is an ordinary launch (it starts after all earlier work in
  // the stream, and this grid after it), so it is read before the wait: its
  // load (often a DRAM miss after the scorer's stream) overlaps the scorer's end.
  const int L = geo.seq_lens[r];
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // the scores are complete: a programmatic dependent (the decode attention)
  // may now be scheduled and run its prologue; it waits for this grid to end
  // before it reads q2k
  if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // the scorer grid has completed and claims nothing more: its claim counter
  // goes back to zero for the next call (no work of this call reads it)
  if (blockIdx.x == 0 && threadIdx.x == 0) sched[0] = 0;
  const int t = threadIdx.x, lane = t & 31;
  const float* row = scores + (static_cast<long long>(r) * kKvHeads + h) * geo.max_blocks;
  int32_t* out = q2k + (static_cast<long long>(h) * geo.batch + r) * topk;
  // stage the row's first min(max_blocks, kTopkStage) scores -- all copies in
  // flight together; entries past the request's blocks are never used
  const int ns = min(geo.max_blocks, kTopkStage);
  for (int b = t; b < ns; b += kTopkThreads) cp_async_4(&stage[b], row + b);
  if (t == 0) count_s = 0;
  cp_async_wait_all();
  __syncthreads();
  if (t == 0 && h == 0 && (L < 1 || L > geo.max_blocks * kBlock)) record_error(err, MSA_DEVERR_LENGTH, r);
  const int nb = L < 1 ? 0 : min((L + kBlock - 1) / kBlock, geo.max_blocks);
  if (nb <= topk) {
    for (int i = t; i < topk; i += kTopkThreads) out[i] = i < nb ? i : -1;
    return;
  }
  const int need = topk - init - local;
  const int c_lo = init, c_hi = nb - local;  // non-forced candidates [c_lo, c_hi), more than `need` of them
  const bool staged = nb <= kTopkStage;
  auto key_at = [&](int b) { return score_key(staged ? stage[b] : __ldcg(row + b), b); };
  if (need > 0 && c_hi - c_lo <= kTopkThreads) {
    // a short row: every candidate's key in shared memory, each ranked against
    // all of them by its own thread (keys are distinct: ranks 0 .. need-1 are picked)
    const int nc = c_hi - c_lo;
    if (t < nc) tmax[t] = key_at(c_lo + t);
    __syncthreads();
    if (t < nc) {
      const unsigned long long e = tmax[t];
      int rank = 0;
#pragma unroll 8
      for (int j = 0; j < nc; ++j) rank += tmax[j] > e ? 1 : 0;
      if (rank < need) ids[rank] = c_lo + t;
    }
  } else if (need > 0) {
    unsigned long long best = 0;  // real keys are nonzero; a thread without candidates keeps 0
    for (int b = c_lo + t; b < c_hi; b += kTopkThreads) {
      const unsigned long long key = key_at(b);
      best = key > best ? key : best;
    }
    tmax[t] = best;
    __syncthreads();
    if (t < 32) {
      // lane l: the largest key of threads l, l + 32, l + 64, l + 96, i.e. of
      // every 32nd candidate.  At least need + 1 lanes hold a real key (there
      // are more than need candidates and need < 32), so the need-th largest of
      // the 32 lane maxima is a score that at least need candidates reach.  The
      // 32 are sorted in descending order by a bitonic network over the lanes.
      // Only the score half of a key (its upper 32 bits) takes part: a
      // threshold on the score alone keeps every key of an equal score.
      uint32_t v = 0;
#pragma unroll
      for (int w = 0; w < kTopkThreads / 32; ++w) v = max(v, static_cast<uint32_t>(tmax[lane + 32 * w] >> 32));
#pragma unroll
      for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
        for (int j = k >> 1; j > 0; j >>= 1) {
          const uint32_t o = __shfl_xor_sync(0xffffffffu, v, j);
          // the lower lane of a pair keeps the larger value in a descending run
          const bool keep_max = ((lane & k) == 0) == ((lane & j) == 0);
          v = keep_max ? max(v, o) : min(v, o);
        }
      }
      if (lane == need - 1) theta_s = static_cast<unsigned long long>(v) << 32;
    }
    __syncthreads();
    const unsigned long long theta = theta_s;
    for (int b = c_lo + t; b < c_hi; b += kTopkThreads) {
      const unsigned long long key = key_at(b);
      if (key >= theta) {
        const int slot = atomicAdd(&count_s, 1);
        if (slot < kCandCap) cand[slot] = key;
      }
    }
    __syncthreads();
    const int count = count_s;
    if (count <= kCandCap) {
      // candidate t's rank = how many candidates are larger; ranks 0 .. need-1 are picked
      if (t < count) {
        const unsigned long long e = cand[t];
        int rank = 0;
#pragma unroll 8
        for (int j = 0; j < count; ++j) rank += cand[j] > e ? 1 : 0;
        if (rank < need) ids[rank] = key_block(e);
      }
    } else if (t < 32) {
      // rare: too many candidates at or above the threshold -- exact rounds by one warp
      unsigned long long prev = ~0ull;
      for (int i = 0; i < need; ++i) {
        unsigned long long m = 0;
        for (int b = c_lo + lane; b < c_hi; b += 32) {
          const unsigned long long key = key_at(b);
          if (key < prev && key > m) m = key;
        }
        for (int o = 16; o > 0; o >>= 1) {
          const unsigned long long x = __shfl_xor_sync(0xffffffffu, m, o);
          m = x > m ? x : m;
        }
        prev = m;
        if (lane == 0) ids[i] = key_block(m);
      }
    }
  }
  // forced ids after the picks; then each id's place in the ascending row
  if (t < init) ids[need + t] = t;
  if (t < local) ids[need + init + t] = nb - local + t;
  __syncthreads();
  if (t < topk) {
    const int id = ids[t];
    int pos = 0;
#pragma unroll
    for (int j = 0; j < kMaxTopk; ++j) pos += j < topk && ids[j] < id ? 1 : 0;
    out[pos] = id;
  }
}

cudaError_t launch_decode_select(const msa_config& cfg, const void* index_q, const void* index_k,
                                 const int32_t* seq_lens, const int32_t* page_table, const int64_t* cu_k,
                                 int batch, int max_blocks, long long num_slots, int32_t* q2k, float* scores,
                                 int* sched, DevError* err, cudaStream_t stream) {
  if (const cudaError_t e0 = launch_prologue(); e0 != cudaSuccess) return e0;
  DecodeGeom geo{seq_lens, page_table, cu_k, batch, max_blocks, num_slots};
  // one CTA per SM; never more CTAs than pages
  const long long blocks_upper = static_cast<long long>(batch) * max_blocks;
  int grid = static_cast<int>(blocks_upper < kNumSMs ? blocks_upper : kNumSMs);
  if (grid < 1) grid = 1;
  const auto* iq = static_cast<const uint8_t*>(index_q);
  const auto* ik = static_cast<const uint8_t*>(index_k);
  if (cfg.index_dtype == MSA_INDEX_E4M3) {
    auto k = decode_select_kernel<1>;
    const size_t smem = sizeof(SelSmem<kSelRingBytes / (kBlock * kIdxDim)>) + 1024;
    cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    k<<<grid, kSelThreads, smem, stream>>>(iq, ik, geo, scores, cfg.topk, sched, err);
  } else {
    auto k = decode_select_kernel<0>;
    const size_t smem = sizeof(SelSmem<kSelRingBytes / (kBlock * kIdxDim * 2)>) + 1024;
    cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    k<<<grid, kSelThreads, smem, stream>>>(iq, ik, geo, scores, cfg.topk, sched, err);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(static_cast<unsigned>(batch) * kKvHeads);  // one CTA per (request, head) row
  lc.blockDim = dim3(kTopkThreads);
  lc.dynamicSmemBytes = 0;
  lc.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = 1;
  const float* sc = scores;
  return cudaLaunchKernelEx(&lc, decode_topk_kernel, sc, geo, q2k, cfg.topk, cfg.init_blocks, cfg.local_blocks, sched,
                            err);
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
  const size_t off_scores = kHeaderBytes;
  const size_t need = off_scores + static_cast<size_t>(batch) * kKvHeads * max_blocks * sizeof(float);
  if (need > kNoAllocScratchBytes) return MSA_ERR_WORKSPACE;  // sizes beyond the fixed scratch
  cudaError_t e;
  auto* base = static_cast<uint8_t*>(noalloc_scratch(&e));
  if (!base) return cuda_fail(e);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the error word and the scorer's claim counter (both in the header) must
  // start at zero; the scores are stored before they are read
  if (const cudaError_t ce = cudaMemsetAsync(base, 0, off_scores, s); ce != cudaSuccess) return cuda_fail(ce);
  e = launch_decode_select(*cfg, index_q, index_k_cache, seq_lens, page_table, cu_seqlens_k, batch, max_blocks,
                           num_slots, q2k, reinterpret_cast<float*>(base + off_scores),
                           reinterpret_cast<int*>(base + kSelSchedOffset), reinterpret_cast<DevError*>(base), s);
  return cuda_result(e);
}
