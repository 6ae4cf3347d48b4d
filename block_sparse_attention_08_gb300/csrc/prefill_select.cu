// prefill_select.cu -- block scoring and top-k selection for packed documents,
// fused into one tensor-core kernel.
//
// NeMo "...minimax_m3_vl.msa", MSAMicrobatch.select_blocks and
// _SelectionPlan.select: bf16 or E4M3 index_q [tokens, 4, 128] against index_k
// [tokens, 1, 128] -> int32 q2k [4, tokens, 16], a hard top-k over the
// unnormalised QK maxima of each causal, document-local 128-key block, with the
// candidate / forced [tokens, blocks] masks of the plan; TensorRT-LLM
// "MiniMaxM3SparseAttentionConfig" fields sparse_score_type 'max',
// sparse_init_blocks, sparse_local_blocks, indexer_kv_dtype (bf16 or unscaled
// E4M3).
//
// GB300 design.  One work unit is (document, 128-token query block, pair of
// index heads).  A TMA producer warp loads the two 128x128 index-Q tiles once
// and then streams the document's causal key blocks (128 keys x 128 dims of
// index_k each) through a 3-deep shared-memory ring; an MMA warp issues
// tcgen05.mma (M=128 tokens, N=128 keys, K=128; bf16 with kind::f16, or E4M3
// with kind::f8f6f4, where a 128-dim row is one 128-byte swizzle atom; fp32
// accumulate) into a
// double-buffered tensor-memory accumulator (2 heads x 2 buffers x 128
// columns = all 512 columns); four epilogue warps read the scores back with
// tcgen05.ld (one token row per thread), take the causal block max and insert
// it into a per-thread top-k list held in registers.  The score matrix never
// reaches global memory: each thread writes its token's q2k row when the unit
// ends.  Query blocks whose candidates all fit in top-k (nb <= topk) need no
// scores and are written directly.  Units are ordered by decreasing cost by a
// one-CTA plan kernel (counting sort of documents by block count) and dealt to
// the persistent CTAs in snake order.
#include "launch.h"

namespace msa {

constexpr int kPsStages = 3;
constexpr int kPsTile = 128 * 128 * 2;  // one 128x128 bf16 tile (two 64-dim boxes); E4M3 uses the first half
constexpr int kPsBox = 128 * 128;       // 128 rows x 128 bytes
constexpr int kPsThreads = 192;         // warps 0-3 epilogue, 4 TMA, 5 MMA
constexpr uint32_t kPsIdesc = tc::idesc_bf16_f32(128, 128);
// kind::f8f6f4 instruction descriptor: E4M3 A and B (format 0), fp32 D, M = N = 128
constexpr uint32_t kPsIdescE4m3 = (1u << 4) | (static_cast<uint32_t>(128 >> 3) << 17) |
                                  (static_cast<uint32_t>(128 >> 4) << 24);

__device__ __forceinline__ void mma_e4m3_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

struct PsSmem {
  alignas(1024) uint8_t a[2][kPsTile];          // index-Q tiles of the head pair
  alignas(1024) uint8_t b[kPsStages][kPsTile];  // index-K key blocks
  uint64_t a_full, a_empty;
  uint64_t b_full[kPsStages], b_empty[kPsStages];
  uint64_t t_full[2], t_empty[2];
  uint64_t mma_done;  // the MMA thread's last commit, waited on before tensor memory is released
  uint32_t tmem_base;
};

struct PsPlan {
  const int32_t* cu_seqlens;
  int num_docs;
  int max_tiles;           // ceil(max_seqlen / 128)
  const int* sorted_docs;  // documents by decreasing tile count
  const int* level_base;   // [max_tiles]: first tile index of query-block level qb
  const int* level_cnt;    // [max_tiles]: documents having query block qb
  const int* n_tiles;      // total tiles
};

struct Unit {
  int doc, qb, hp;
  int start, len;  // document rows
};

__device__ __forceinline__ Unit unit_of(const PsPlan& p, int u) {
  Unit x;
  const int ut = u >> 1;
  x.hp = u & 1;
  // level qb holds tiles [level_base[qb], level_base[qb] + level_cnt[qb]); bases grow as qb falls
  int lo = 0, hi = p.max_tiles - 1;
  while (lo < hi) {  // smallest qb with level_base[qb] <= ut
    const int mid = (lo + hi) >> 1;
    if (p.level_base[mid] <= ut) hi = mid; else lo = mid + 1;
  }
  x.qb = lo;
  x.doc = p.sorted_docs[ut - p.level_base[lo]];
  x.start = p.cu_seqlens[x.doc];
  x.len = p.cu_seqlens[x.doc + 1] - x.start;
  return x;
}

// snake order over rows of gridDim.x units
__device__ __forceinline__ int snake(int k, int c, int G) { return (k & 1) ? (k + 1) * G - 1 - c : k * G + c; }

// One-CTA plan: documents sorted by tile count (descending), level bases.
// One block: documents counting-sorted by tile count (descending), the per-level
// tile counts and bases.  The histogram and its scans live in shared memory
// (`sh`: max_tiles + 2 ints); thread 0's two scans are sequential over the
// levels, so they must not go through global memory.
__global__ void prefill_plan_kernel(const int32_t* __restrict__ cu, int num_docs, int max_tiles,
                                    int* __restrict__ sorted_docs, int* __restrict__ level_base,
                                    int* __restrict__ level_cnt, int* __restrict__ n_tiles, DevError* err) {
  extern __shared__ int sh[];
  int* hist = sh;                        // [max_tiles + 2]: docs per tile count, then scatter cursors
  int* lcnt = sh + (max_tiles + 2);      // [max_tiles]
  int* lbase = lcnt + max_tiles;         // [max_tiles]
  const int tid = threadIdx.x;
  for (int i = tid; i < max_tiles + 2; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  for (int d = tid; d < num_docs; d += blockDim.x) {
    const int len = cu[d + 1] - cu[d];
    int nt = (len + kBlock - 1) / kBlock;
    if (len < 1 || nt > max_tiles) {
      record_error(err, MSA_DEVERR_LENGTH, d);
      nt = len < 1 ? 0 : max_tiles;
    }
    atomicAdd(&hist[nt], 1);
  }
  __syncthreads();
  if (tid == 0) {
    // lcnt[qb] = #docs with tile count > qb ; lbase: levels in decreasing qb
    int above = 0;
    for (int n = max_tiles; n >= 1; --n) {
      above += hist[n];
      lcnt[n - 1] = above;
    }
    int base = 0;
    for (int qb = max_tiles - 1; qb >= 0; --qb) {
      lbase[qb] = base;
      base += lcnt[qb];
    }
    *n_tiles = base;
    // scatter cursors: docs with tile count n start after all docs with more tiles
    int run = 0;
    for (int n = max_tiles; n >= 0; --n) {
      const int c = hist[n];
      hist[n] = run;
      run += c;
    }
  }
  __syncthreads();
  for (int qb = tid; qb < max_tiles; qb += blockDim.x) {
    level_cnt[qb] = lcnt[qb];
    level_base[qb] = lbase[qb];
  }
  for (int d = tid; d < num_docs; d += blockDim.x) {
    const int len = cu[d + 1] - cu[d];
    const int nt = len < 1 ? 0 : min((len + kBlock - 1) / kBlock, max_tiles);
    sorted_docs[atomicAdd(&hist[nt], 1)] = d;
  }
}

// Sorted top-k list (score desc, id asc) of up to 16 entries in registers.
struct TopList {
  float v[kMaxTopk];
  int id[kMaxTopk];
  __device__ __forceinline__ void reset() {
#pragma unroll
    for (int i = 0; i < kMaxTopk; ++i) {
      v[i] = -INFINITY;
      id[i] = 0x7fffffff;
    }
  }
  // ids arrive in increasing order, so an equal score never moves up
  __device__ __forceinline__ void insert(float s, int b) {
    if (s > v[kMaxTopk - 1]) {
      v[kMaxTopk - 1] = s;
      id[kMaxTopk - 1] = b;
#pragma unroll
      for (int i = kMaxTopk - 1; i > 0; --i) {
        const bool up = v[i] > v[i - 1];
        const float tv = v[i];
        const int ti = id[i];
        v[i] = up ? v[i - 1] : v[i];
        id[i] = up ? id[i - 1] : id[i];
        v[i - 1] = up ? tv : v[i - 1];
        id[i - 1] = up ? ti : id[i - 1];
      }
    }
  }
};

__device__ __forceinline__ void cswap(int& a, int& b) {
  const int lo = min(a, b), hi = max(a, b);
  a = lo;
  b = hi;
}

// Writes the q2k row: [0, init) ++ ascending(top `need` ids) ++ [nb-local, nb).
__device__ __forceinline__ void write_row(int32_t* row, const TopList& L, int need, int nb, int topk, int init,
                                          int local) {
  int ids[kMaxTopk];
#pragma unroll
  for (int i = 0; i < kMaxTopk; ++i) ids[i] = i < need ? L.id[i] : 0x7fffffff;
  // bitonic sort of 16 ints, ascending
#pragma unroll
  for (int k = 2; k <= kMaxTopk; k <<= 1)
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1)
#pragma unroll
      for (int i = 0; i < kMaxTopk; ++i) {
        const int l = i ^ j;
        if (l > i) {
          if ((i & k) == 0) cswap(ids[i], ids[l]);
          else cswap(ids[l], ids[i]);
        }
      }
  int outv[kMaxTopk];
#pragma unroll
  for (int i = 0; i < kMaxTopk; ++i) {
    int v;
    if (i < init) v = i;
    else if (i < init + need) v = ids[i - init];
    else if (i < topk) v = nb - local + (i - init - need);
    else v = -1;
    outv[i] = v;
  }
  if (topk == kMaxTopk) {
    int4* o = reinterpret_cast<int4*>(row);
#pragma unroll
    for (int i = 0; i < 4; ++i) o[i] = make_int4(outv[4 * i], outv[4 * i + 1], outv[4 * i + 2], outv[4 * i + 3]);
  } else {
#pragma unroll
    for (int i = 0; i < kMaxTopk; ++i)
      if (i < topk) row[i] = outv[i];
  }
}

// kE4M3: the index tensors hold E4M3 bytes (one 128-byte box per tile row
// block) instead of bf16 (two 64-dim boxes).
template <int kE4M3>
__global__ void __launch_bounds__(kPsThreads, 1) prefill_select_kernel(
    const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap, PsPlan plan,
    long long total_tokens, int32_t* __restrict__ q2k, int topk, int init, int local, DevError* err) {
  extern __shared__ uint8_t smem_raw[];
  PsSmem& sm = *reinterpret_cast<PsSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = gridDim.x, c = blockIdx.x;
  const int U = 2 * (*plan.n_tiles);

  if (tid == 0) {
    mbar_init(&sm.a_full, 1);
    mbar_init(&sm.a_empty, 1);
    for (int s = 0; s < kPsStages; ++s) {
      mbar_init(&sm.b_full[s], 1);
      mbar_init(&sm.b_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sm.t_full[i], 1);
      mbar_init(&sm.t_empty[i], 4);
    }
    mbar_init(&sm.mma_done, 1);
    fence_mbar_init();
  }
  if (warp == 5) {
    tc::alloc(&sm.tmem_base, 512);
    tc::relinquish();
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = sm.tmem_base;

  if (warp == 4) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      prefetch_tmap(&qmap);
      prefetch_tmap(&kmap);
      uint32_t nunit = 0, bc = 0;
      for (int k = 0; k * G < U; ++k) {
        const int u = snake(k, c, G);
        if (u >= U) continue;
        const Unit x = unit_of(plan, u);
        if (x.qb + 1 <= topk) continue;
        mbar_wait(&sm.a_empty, (nunit & 1) ^ 1, err, 400);
        constexpr int kTileBytes = kE4M3 ? kPsBox : kPsTile;
        mbar_expect_tx(&sm.a_full, 2 * kTileBytes);
        const int row = x.start + x.qb * kBlock;
        for (int hh = 0; hh < 2; ++hh) {
          tma_load_3d(sm.a[hh], &qmap, 0, 2 * x.hp + hh, row, &sm.a_full);
          if (!kE4M3) tma_load_3d(sm.a[hh] + kPsBox, &qmap, 64, 2 * x.hp + hh, row, &sm.a_full);
        }
        for (int b = 0; b <= x.qb; ++b, ++bc) {
          const int s = bc % kPsStages;
          mbar_wait(&sm.b_empty[s], ((bc / kPsStages) & 1) ^ 1, err, 401);
          mbar_expect_tx(&sm.b_full[s], kTileBytes);
          tma_load_2d(sm.b[s], &kmap, 0, x.start + b * kBlock, &sm.b_full[s]);
          if (!kE4M3) tma_load_2d(sm.b[s] + kPsBox, &kmap, 64, x.start + b * kBlock, &sm.b_full[s]);
        }
        ++nunit;
      }
      // No copy may still be landing when the CTA exits, also after a wait
      // gave up: wait (bounded) for the last fill of the A tile and of every
      // key stage.  Only this thread arms those barriers.
      if (nunit > 0) mbar_wait(&sm.a_full, (nunit - 1) & 1, err, 402);
      for (int s = 0; s < kPsStages; ++s) {
        const uint32_t f = (bc + kPsStages - 1 - s) / kPsStages;  // fills of stage s
        if (f > 0) mbar_wait(&sm.b_full[s], (f - 1) & 1, err, 403);
      }
    }
  } else if (warp == 5) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      uint32_t nunit = 0, bc = 0, kc = 0;
      for (int k = 0; k * G < U; ++k) {
        const int u = snake(k, c, G);
        if (u >= U) continue;
        const Unit x = unit_of(plan, u);
        if (x.qb + 1 <= topk) continue;
        mbar_wait(&sm.a_full, nunit & 1, err, 500);
        tc::fence_after();
        for (int b = 0; b <= x.qb; ++b, ++bc, ++kc) {
          const int s = bc % kPsStages, buf = kc & 1;
          mbar_wait(&sm.b_full[s], (bc / kPsStages) & 1, err, 501);
          mbar_wait(&sm.t_empty[buf], ((kc >> 1) & 1) ^ 1, err, 502);
          tc::fence_after();
          const uint32_t bsm = smem_u32(sm.b[s]);
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const uint32_t asm_ = smem_u32(sm.a[hh]);
            const uint32_t d = tmem + static_cast<uint32_t>((buf * 2 + hh) * 128);
            if (kE4M3) {
              // K = 32 E4M3 values (32 bytes) per MMA: four steps through the 128-byte row
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                mma_e4m3_ss(d, tc::desc_k_sw128(asm_ + kk * 32), tc::desc_k_sw128(bsm + kk * 32), kPsIdescE4m3,
                            kk > 0);
            } else {
#pragma unroll
              for (int kk = 0; kk < 8; ++kk) {
                const uint32_t off = (kk >> 2) * kPsBox + (kk & 3) * 32;
                tc::mma_bf16(d, tc::desc_k_sw128(asm_ + off), tc::desc_k_sw128(bsm + off), kPsIdesc, kk > 0);
              }
            }
          }
          tc::commit(&sm.b_empty[s]);
          tc::commit(&sm.t_full[buf]);
        }
        tc::commit(&sm.a_empty);
        ++nunit;
      }
      // every MMA of this thread has finished before tensor memory is released
      // (the epilogue's waits cover this unless one of them gave up)
      tc::commit(&sm.mma_done);
      mbar_wait(&sm.mma_done, 0, err, 503);
    }
  } else {
    // ---------------- epilogue warps 0-3: one token row per thread ----------------
    const int r = warp * 32 + lane;
    uint32_t kc = 0;
    for (int k = 0; k * G < U; ++k) {
      const int u = snake(k, c, G);
      if (u >= U) continue;
      const Unit x = unit_of(plan, u);
      const int nb = x.qb + 1;
      const int p = x.qb * kBlock + r;  // position of this row's token
      const bool row_ok = p < x.len;
      const long long t = static_cast<long long>(x.start) + p;
      if (nb <= topk) {
        if (row_ok)
          for (int hh = 0; hh < 2; ++hh) {
            int32_t* row = q2k + (static_cast<long long>(2 * x.hp + hh) * total_tokens + t) * topk;
            for (int i = 0; i < topk; ++i) row[i] = i < nb ? i : -1;
          }
        continue;
      }
      TopList L0, L1;
      L0.reset();
      L1.reset();
      for (int b = 0; b <= x.qb; ++b, ++kc) {
        const int buf = kc & 1;
        mbar_wait(&sm.t_full[buf], (kc >> 1) & 1, err, 600);
        tc::fence_after();
        const bool diag = (b == x.qb);
        float mx[2];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          // the head's 128 scores of this row: four loads in flight, one wait
          const uint32_t a0 = tmem + (static_cast<uint32_t>(warp * 32) << 16) + static_cast<uint32_t>((buf * 2 + hh) * 128);
          uint32_t v0[32], v1[32], v2[32], v3[32];
          tc::ld_32x32b_x32(a0, v0);
          tc::ld_32x32b_x32(a0 + 32, v1);
          tc::ld_32x32b_x32(a0 + 64, v2);
          tc::ld_32x32b_x32(a0 + 96, v3);
          tc::wait_ld();
          float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
          if (diag) {  // causal keys only: key column j <= this row's position r
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              m4[0] = j <= r ? fmaxf(m4[0], __uint_as_float(v0[j])) : m4[0];
              m4[1] = 32 + j <= r ? fmaxf(m4[1], __uint_as_float(v1[j])) : m4[1];
              m4[2] = 64 + j <= r ? fmaxf(m4[2], __uint_as_float(v2[j])) : m4[2];
              m4[3] = 96 + j <= r ? fmaxf(m4[3], __uint_as_float(v3[j])) : m4[3];
            }
          } else {  // every key is causal: four independent chains of three-input max
#pragma unroll
            for (int j = 0; j < 32; j += 2) {
              m4[0] = fmax3(m4[0], __uint_as_float(v0[j]), __uint_as_float(v0[j + 1]));
              m4[1] = fmax3(m4[1], __uint_as_float(v1[j]), __uint_as_float(v1[j + 1]));
              m4[2] = fmax3(m4[2], __uint_as_float(v2[j]), __uint_as_float(v2[j + 1]));
              m4[3] = fmax3(m4[3], __uint_as_float(v3[j]), __uint_as_float(v3[j + 1]));
            }
          }
          mx[hh] = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
        }
        tc::fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.t_empty[buf]);
        const bool forced = (b < init) || (b >= nb - local);
        if (!forced) {
          L0.insert(mx[0], b);
          L1.insert(mx[1], b);
        }
      }
      if (row_ok) {
        const int need = topk - init - local;
        write_row(q2k + (static_cast<long long>(2 * x.hp) * total_tokens + t) * topk, L0, need, nb, topk, init,
                  local);
        write_row(q2k + (static_cast<long long>(2 * x.hp + 1) * total_tokens + t) * topk, L1, need, nb, topk,
                  init, local);
      }
    }
  }
  tc::fence_before();
  __syncthreads();
  if (warp == 5) {
    tc::fence_after();
    tc::dealloc(tmem, 512);
  }
}

// ---- host side --------------------------------------------------------------------

size_t prefill_plan_ints(int num_docs, int max_tiles) {
  return static_cast<size_t>(max_tiles + 2) + num_docs + 2 * static_cast<size_t>(max_tiles) + 1;
}

cudaError_t launch_prefill_select(const msa_config& cfg, const void* index_q, const void* index_k,
                                  const int32_t* cu_seqlens, int num_docs, long long total_tokens, int max_seqlen,
                                  int32_t* q2k, int* plan_ints, DevError* err, cudaStream_t stream) {
  if (const cudaError_t e0 = launch_prologue(); e0 != cudaSuccess) return e0;
  EncodeTiledFn enc = get_encode_tiled();
  if (!enc) return cudaErrorInvalidValue;
  const int max_tiles = (max_seqlen + kBlock - 1) / kBlock;
  int* hist = plan_ints;
  int* sorted_docs = hist + (max_tiles + 2);
  int* level_base = sorted_docs + num_docs;
  int* level_cnt = level_base + max_tiles;
  int* n_tiles = level_cnt + max_tiles;
  const size_t plan_smem = (3 * static_cast<size_t>(max_tiles) + 2) * sizeof(int);
  if (plan_smem > 200 * 1024) return cudaErrorInvalidValue;  // the ABI rejects longer documents first
  cudaFuncSetAttribute(prefill_plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(plan_smem));
  prefill_plan_kernel<<<1, 1024, plan_smem, stream>>>(cu_seqlens, num_docs, max_tiles, sorted_docs, level_base,
                                                      level_cnt, n_tiles, err);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  // bf16: 64-dim boxes (the 128-byte swizzle bounds a box row at 128 bytes);
  // E4M3: the whole 128-byte row in one box
  const bool e4m3 = cfg.index_dtype == MSA_INDEX_E4M3;
  const CUtensorMapDataType dt = e4m3 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const cuuint64_t esz = e4m3 ? 1 : 2;
  const cuuint32_t bx = e4m3 ? 128 : 64;
  CUtensorMap qmap, kmap;
  {
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(kIdxDim), static_cast<cuuint64_t>(kKvHeads),
                          static_cast<cuuint64_t>(total_tokens)};
    cuuint64_t strides[2] = {kIdxDim * esz, kKvHeads * kIdxDim * esz};
    cuuint32_t box[3] = {bx, 1, 128};
    cuuint32_t estr[3] = {1, 1, 1};
    if (enc(&qmap, dt, 3, const_cast<void*>(index_q), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(kIdxDim), static_cast<cuuint64_t>(total_tokens)};
    cuuint64_t strides[1] = {kIdxDim * esz};
    cuuint32_t box[2] = {bx, 128};
    cuuint32_t estr[2] = {1, 1};
    if (enc(&kmap, dt, 2, const_cast<void*>(index_k), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  PsPlan plan{cu_seqlens, num_docs, max_tiles, sorted_docs, level_base, level_cnt, n_tiles};
  const long long tiles_upper = total_tokens / kBlock + num_docs;
  int grid = static_cast<int>(2 * tiles_upper < kNumSMs ? 2 * tiles_upper : kNumSMs);
  if (grid < 1) grid = 1;
  const size_t smem = sizeof(PsSmem) + 1024;
  if (e4m3) {
    cudaFuncSetAttribute(prefill_select_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         static_cast<int>(smem));
    prefill_select_kernel<1><<<grid, kPsThreads, smem, stream>>>(qmap, kmap, plan, total_tokens, q2k, cfg.topk,
                                                                 cfg.init_blocks, cfg.local_blocks, err);
  } else {
    cudaFuncSetAttribute(prefill_select_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         static_cast<int>(smem));
    prefill_select_kernel<0><<<grid, kPsThreads, smem, stream>>>(qmap, kmap, plan, total_tokens, q2k, cfg.topk,
                                                                 cfg.init_blocks, cfg.local_blocks, err);
  }
  return cudaGetLastError();
}

}  // namespace msa
