// sparse_attend.cu -- sparse GQA attention over the selected blocks for a
// decode step: one query per request over a paged or contiguous K/V cache.
// (Packed-document prefill has its own block-major kernel, prefill_attend.cu.)
//
// TensorRT-LLM "MiniMaxM3SparseAttentionConfig" (class description, second
// step: a sparse GQA attention over only the selected blocks) and NeMo
// "...minimax_m3_vl.msa" sparse_attention / _SparseAttention.forward: bf16
// q [tokens, 64, 128], k / v [tokens, 4, 128], int32 q2k [4, tokens, 16] ->
// bf16 out [tokens, 64, 128].
//
// GB300 design.  The 16 query heads that share a KV head form exactly one
// 16-row MMA tile, so one (query, KV head, selected block) triple is the unit
// of work and a (query, KV head) pair is a segment of up to topk units.  All
// units are split evenly over a persistent grid of one CTA per SM (stream-K).
//
// A producer warp walks the CTA's segments.  Per segment its lanes resolve the
// selected blocks in parallel (q2k entry, then page id); it puts the segment's
// key counts in a 2-slot segment ring together with the 16 x 128 Q tile (a
// tiled TMA copy), then gathers each block's K and V in 64-key chunks with
// tiled TMA copies (3-D tensor map over [rows, 4 heads, 128], 128-byte swizzle)
// into a 6-stage chunk ring.  Three consumer warps each own two stages
// (stage s always to warp s % 3), so every warp has one chunk landing while it
// computes on the other, and none reads global memory on its critical path:
// S = Q K^T (ldmatrix fragments), online softmax in base 2, O += P V
// (ldmatrix.trans V fragments; P rounded to bf16, the row sum taken over the
// rounded values), mma.sync bf16 with
// fp32 accumulation.  At the end of a segment the three states are merged
// through shared memory.  A segment cut by a CTA boundary is written as an fp32
// partial (max, sum, unnormalised O); the CTA whose atomic ticket completes the
// segment (no waiting) merges the partials and writes bf16.
//
// Small batches (few segments) take a second launch shape: one thread-block
// cluster of C = 2, 4 or 8 CTAs per segment, each CTA a contiguous share of
// its units, the C states merged by the cluster's first CTA over distributed
// shared memory.  The stream-K merge costs a CTA an fp32 partial store, a
// fence, an atomic and dependent L2 reads of the other partials (6-9 us at
// the end of a small decode step, more than the streaming itself for a few
// requests); the cluster merge is two cluster barriers and one read of the
// peers' shared memory.
//
// FP8 main K/V cache (TensorRT-LLM field fuse_qkv_index_projection: the M3 path
// uses "an FP8 main KV cache"): the caches hold E4M3 bytes standing for
// k_scale * k and v_scale * v.  A chunk is then 64 keys x 128 bytes of K and of
// V (one 128-byte-swizzled box each, 16 KB a stage).  The consumers read the E4M3 bytes straight into
// MMA fragments and convert them in registers (every E4M3 value is exact in
// fp16): K through ldmatrix, with the k slots of the fp16 Q fragments permuted
// to match; V through the transposing ldmatrix on byte pairs, each 16-dim
// block feeding an even-dim and an odd-dim n-tile.  q is rounded to fp16 once
// per segment, P to fp16.  k_scale is folded into the softmax scale and
// v_scale into the normalisation.
#include <mutex>

#include "launch.h"

namespace msa {

constexpr int kAttStages = 6;
constexpr int kChunkKeys = 64;
constexpr int kBoxBytes = kChunkKeys * 128;        // 64 rows x 128 bytes (64 bf16 dims, or 128 E4M3 dims)
constexpr int kAttStageBytes = 4 * kBoxBytes;      // K lo/hi + V lo/hi
constexpr int kAttStage8Bytes = 2 * kBoxBytes;     // FP8 K/V: K + V, one box each
constexpr int kConsumerWarps = 3;
constexpr int kConsumerThreads = kConsumerWarps * 32;
constexpr int kAttThreads = kConsumerThreads + 32;
constexpr int kSegSlots = 2;
constexpr int kQBoxBytes = kGroup * 128;            // 16 rows x 128 bytes (64 dims)
constexpr int kCombStride = kDim + 8;               // padded fp32 row of the merge buffer
constexpr int kPartialFloats = 32 + kGroup * kDim;  // m[16], l[16], O[16][128]
// stage s is always consumed by warp s % kConsumerWarps, so a warp never waits
// on a stage more than one mbarrier phase ahead
static_assert(kAttStages % kConsumerWarps == 0, "stages must be a multiple of the consumer warps");

struct QueryGeo {
  int pos;         // position of the query (keys 0..pos are causal)
  int nb;          // candidate blocks
  long long base;  // contiguous cache: first row of the request (cu_k[r])
};

__device__ __forceinline__ QueryGeo query_geo(const AttnGeom& geo, int qi) {
  QueryGeo q;
  const int L = geo.seq_lens[qi];
  q.pos = L - 1;
  q.nb = L < 1 ? 0 : min((L + kBlock - 1) / kBlock, geo.max_blocks);
  q.base = geo.page_table ? 0 : geo.cu_k[qi];
  return q;
}

// First K/V row of block b of the query, or -1 when the page is outside the pool.
__device__ __forceinline__ long long block_row0(const AttnGeom& geo, int qi, const QueryGeo& q, int b) {
  if (geo.page_table) {
    const int page = geo.page_table[static_cast<long long>(qi) * geo.max_blocks + b];
    const long long r0 = static_cast<long long>(page) * kBlock;
    return (page < 0 || r0 + kBlock > geo.num_rows) ? -1 : r0;
  }
  return q.base + static_cast<long long>(b) * kBlock;
}

// Number of causal keys of block b (0 for an empty / invalid entry).
__device__ __forceinline__ int block_keys(const QueryGeo& q, int b) {
  if (b < 0 || b >= q.nb) return 0;
  return min(kBlock, q.pos - b * kBlock + 1);
}

struct SegInfo {
  int nk[kMaxTopk];  // causal keys of each of the segment's units (0 = nothing to do)
};

// The chunk ring: 64-key chunks of K and V (bf16: 4 boxes of 64 dims, 32 KB;
// FP8: one 128-byte box each, 16 KB), 6 stages.
//
// With an FP8 cache the attention is bound by its consumer warps' issue, not
// by bytes, so two CTAs share an SM (six consumer warps per SM) on its 96 KB of
// stages: one Q slot in the segment ring (the consumers free it as soon as
// they hold their Q fragments) and, in the stream-K form, one slot where the
// three warps' states meet one after the other.  The cluster form needs no such
// slot at all: each warp leaves its state in its own stage, idle once the
// CTA's one segment is done.  Measured: the 16-request workload's cluster form
// 31.4 -> 27.2 us.  A bf16 ring of 96 KB would leave each warp a single stage,
// nothing landing while it computes: slower (18.4 -> 20.9 us on the 4-request
// workload), so bf16 stays at one CTA per SM.
template <int kFp8, int kSplit>
struct AttShape {
  static constexpr int kStageBytes = kFp8 ? kAttStage8Bytes : kAttStageBytes;
  static constexpr int kStages = kAttStages;
  static constexpr int kCtasPerSm = kFp8 ? 2 : 1;
  static constexpr int kQSlots = kFp8 ? 1 : kSegSlots;             // Q tiles in the segment ring
  static constexpr int kCombSlots = kFp8 ? 1 : kConsumerWarps - 1;  // stream-K: where states meet
};

// Where the consumer warps' states meet (stream-K only).
template <int kSplit, int kSlots>
struct AttComb {
  float comb[kSlots][kGroup][kCombStride];
  float comb_m[kSlots][kGroup];
  float comb_l[kSlots][kGroup];
};
template <int kSlots>
struct AttComb<1, kSlots> {};

template <int kFp8, int kSplit>
struct AttSmem {
  using Shape = AttShape<kFp8, kSplit>;
  alignas(1024) uint8_t stage[Shape::kStages][Shape::kStageBytes];
  alignas(1024) uint8_t qtile[Shape::kQSlots][2 * kQBoxBytes];
  AttComb<kSplit, Shape::kCombSlots> c;
  SegInfo seg[Shape::kQSlots];
  uint64_t full[Shape::kStages];
  uint64_t empty[Shape::kStages];
  uint64_t seg_full[Shape::kQSlots];
  uint64_t seg_empty[Shape::kQSlots];
  int bcast;
};

// One warp state in shared memory: O as 16 rows of kCombStride floats, m[16], l[16].
struct CombRef {
  float* o;
  float* m;
  float* l;
  __device__ float* row(int r) const { return o + r * kCombStride; }
};
// who = 0: the CTA's merged state; who = w in 1, 2: the state of consumer warp w.
// Stream-K: the shared buffer (the merged state over warp 1's slot, which warp
// 0 has read by then; with one slot the warps take turns); cluster form: stage
// `who`, which belongs to warp `who`.
template <int kFp8, int kSplit>
__device__ __forceinline__ CombRef comb_ref(AttSmem<kFp8, kSplit>& sm, int who) {
  if constexpr (kSplit != 0) {
    float* base = reinterpret_cast<float*>(&sm.stage[who][0]);
    return CombRef{base, base + kGroup * kCombStride, base + kGroup * kCombStride + kGroup};
  } else {
    const int slot = who > 0 ? (who - 1) % AttShape<kFp8, kSplit>::kCombSlots : 0;
    return CombRef{&sm.c.comb[slot][0][0], sm.c.comb_m[slot], sm.c.comb_l[slot]};
  }
}
static_assert((kGroup * kCombStride + 2 * kGroup) * sizeof(float) <= kAttStage8Bytes, "a warp state fits in a stage");

__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, 96;" ::: "memory"); }

__device__ __forceinline__ long long seg_begin(long long c, long long N, long long G) { return c * N / G; }
__device__ __forceinline__ long long cta_of(long long i, long long N, long long G) {
  long long c = i * G / N;
  while (c + 1 < G && seg_begin(c + 1, N, G) <= i) ++c;
  while (c > 0 && seg_begin(c, N, G) > i) --c;
  return c;
}

// Online-softmax state of one warp: rows g8 (m0, l0, o[.][0..1]) and g8+8 (m1, l1, o[.][2..3]).
struct WarpState {
  float m0, m1, l0, l1;
  float o[16][4];
};

// Where accumulator column e of n-tile nd of a lane lies.  bf16: n-tile nd is
// dims 8 nd .. 8 nd + 7 and the lane holds dims 8 nd + 2 t4 + e.  FP8: the V
// fragments come from byte pairs (see the PV product), so n-tiles 2c and 2c + 1
// are the even and the odd dims of the 16-dim block c, and the lane's four
// values of the pair are the consecutive dims 16 c + 4 t4 .. + 3 -- stored and
// loaded as one float4, in the natural order, so everything that reads the
// states back (the merges, the output) sees plain rows.
template <int kFp8>
__device__ __forceinline__ void state_to_smem(const WarpState& st, const CombRef& c, int g8, int t4) {
  if (t4 == 0) {
    c.m[g8] = st.m0;
    c.m[g8 + 8] = st.m1;
    c.l[g8] = st.l0;
    c.l[g8 + 8] = st.l1;
  }
  if constexpr (kFp8 != 0) {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      *reinterpret_cast<float4*>(c.row(g8) + 16 * k + 4 * t4) =
          make_float4(st.o[2 * k][0], st.o[2 * k + 1][0], st.o[2 * k][1], st.o[2 * k + 1][1]);
      *reinterpret_cast<float4*>(c.row(g8 + 8) + 16 * k + 4 * t4) =
          make_float4(st.o[2 * k][2], st.o[2 * k + 1][2], st.o[2 * k][3], st.o[2 * k + 1][3]);
    }
  } else {
#pragma unroll
    for (int nd = 0; nd < 16; ++nd) {
      *reinterpret_cast<float2*>(c.row(g8) + 8 * nd + 2 * t4) = make_float2(st.o[nd][0], st.o[nd][1]);
      *reinterpret_cast<float2*>(c.row(g8 + 8) + 8 * nd + 2 * t4) = make_float2(st.o[nd][2], st.o[nd][3]);
    }
  }
}

template <int kFp8>
__device__ __forceinline__ void merge_from_smem(WarpState& st, const CombRef& c, int g8, int t4) {
  const float mb0 = c.m[g8], mb1 = c.m[g8 + 8];
  const float M0 = fmaxf(st.m0, mb0), M1 = fmaxf(st.m1, mb1);
  const float u0 = M0 == -INFINITY ? 0.f : M0, u1 = M1 == -INFINITY ? 0.f : M1;
  const float fa0 = exp2f(st.m0 - u0), fb0 = exp2f(mb0 - u0);
  const float fa1 = exp2f(st.m1 - u1), fb1 = exp2f(mb1 - u1);
  st.l0 = st.l0 * fa0 + c.l[g8] * fb0;
  st.l1 = st.l1 * fa1 + c.l[g8 + 8] * fb1;
  st.m0 = M0;
  st.m1 = M1;
  if constexpr (kFp8 != 0) {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float4 x = *reinterpret_cast<const float4*>(c.row(g8) + 16 * k + 4 * t4);
      const float4 y = *reinterpret_cast<const float4*>(c.row(g8 + 8) + 16 * k + 4 * t4);
      st.o[2 * k][0] = st.o[2 * k][0] * fa0 + x.x * fb0;
      st.o[2 * k + 1][0] = st.o[2 * k + 1][0] * fa0 + x.y * fb0;
      st.o[2 * k][1] = st.o[2 * k][1] * fa0 + x.z * fb0;
      st.o[2 * k + 1][1] = st.o[2 * k + 1][1] * fa0 + x.w * fb0;
      st.o[2 * k][2] = st.o[2 * k][2] * fa1 + y.x * fb1;
      st.o[2 * k + 1][2] = st.o[2 * k + 1][2] * fa1 + y.y * fb1;
      st.o[2 * k][3] = st.o[2 * k][3] * fa1 + y.z * fb1;
      st.o[2 * k + 1][3] = st.o[2 * k + 1][3] * fa1 + y.w * fb1;
    }
  } else {
#pragma unroll
    for (int nd = 0; nd < 16; ++nd) {
      const float2 x = *reinterpret_cast<const float2*>(c.row(g8) + 8 * nd + 2 * t4);
      const float2 y = *reinterpret_cast<const float2*>(c.row(g8 + 8) + 8 * nd + 2 * t4);
      st.o[nd][0] = st.o[nd][0] * fa0 + x.x * fb0;
      st.o[nd][1] = st.o[nd][1] * fa0 + x.y * fb0;
      st.o[nd][2] = st.o[nd][2] * fa1 + y.x * fb1;
      st.o[nd][3] = st.o[nd][3] * fa1 + y.y * fb1;
    }
  }
}

// Two E4M3 values, rounded to nearest (ties to even) and saturated at +-448;
// `lo` in the low byte.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// MXFP8 emission of one lane's 64 consecutive outputs v[i] * inv (vLLM
// forward_decode_mxfp8: E4M3 values and one E8M0 scale per 32 elements, equal
// to the MX quantisation of the bf16 output).  Per 32-element block: the bf16
// output values b, amax = max |b|, scale exponent floor(log2 amax) - 8 (the
// largest E4M3 exponent; clamped to [-127, 127], -127 for a zero block), each
// b times 2^-exponent (exact) rounded to E4M3.
__device__ __forceinline__ void store_mxfp8_64(const float* v, float inv, uint8_t* __restrict__ q,
                                               uint8_t* __restrict__ sc) {
#pragma unroll
  for (int blk = 0; blk < 2; ++blk) {
    float b[32];
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      b[i] = bf16_round(v[32 * blk + i] * inv);
      amax = fmaxf(amax, fabsf(b[i]));
    }
    const int sexp = amax > 0.f ? max(-127, min(127, ilogbf(amax) - 8)) : -127;
    sc[blk] = static_cast<uint8_t>(sexp + 127);
    const float r = ldexpf(1.f, -sexp);
    uint32_t w[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
      w[i] = e4m3x2(b[4 * i] * r, b[4 * i + 1] * r) | (e4m3x2(b[4 * i + 2] * r, b[4 * i + 3] * r) << 16);
    reinterpret_cast<uint4*>(q + 32 * blk)[0] = make_uint4(w[0], w[1], w[2], w[3]);
    reinterpret_cast<uint4*>(q + 32 * blk)[1] = make_uint4(w[4], w[5], w[6], w[7]);
  }
}

// The 16-bit type of P: bf16 (a bf16 K/V cache) or fp16 (an FP8 K/V cache,
// converted to fp16 on chip).
template <int kFp8>
__device__ __forceinline__ float round16(float x) {
  return kFp8 ? __half2float(__float2half_rn(x)) : bf16_round(x);
}
template <int kFp8>
__device__ __forceinline__ uint32_t pack16(float lo, float hi) {
  if (kFp8) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  return pack_bf16(lo, hi);
}
// bf16x2 -> fp16x2 (q of an FP8-cache call; exact for |q| in fp16's normal range)
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w) {
  __half2 h = __floats2half2_rn(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
  return *reinterpret_cast<uint32_t*>(&h);
}

// Two E4M3 values -> fp16x2 holding each value times 2^-8, exactly, with
// integer operations only.  The bytes come in as the high byte of each 16-bit
// half (h = [0, b0, 0, b1]): the sign stays in bit 15, and exponent and
// mantissa (eeee mmm) move down one bit into bits 14..7, so the fp16 exponent
// field reads eeee with its top bit 0 and the mantissa's top bits mmm.  For
// e > 0 that is 2^(e-15) (1 + m/8) = 2^-8 2^(e-7) (1 + m/8); for e = 0 the
// fp16 subnormal 2^-14 m/8 = 2^-8 2^-6 m/8; so every finite E4M3 value maps to
// its value times 2^-8 (its NaN encodings to finite numbers: an FP8 cache holds
// finite values).  The 2^8 is folded into the score scale (K) and into the
// output scale (V) by the host.
__device__ __forceinline__ uint32_t e4m3_hb_to_f16x2_s8(uint32_t h) {
  return ((h >> 1) & 0x3f803f80u) | (h & 0x80008000u);
}
// Bytes 0 and 1 / 2 and 3 / 0 and 2 / 1 and 3 of a word, as above.
__device__ __forceinline__ uint32_t e4m3_lo2(uint32_t w) { return e4m3_hb_to_f16x2_s8(__byte_perm(w, 0u, 0x1404)); }
__device__ __forceinline__ uint32_t e4m3_hi2(uint32_t w) { return e4m3_hb_to_f16x2_s8(__byte_perm(w, 0u, 0x3424)); }
__device__ __forceinline__ uint32_t e4m3_even2(uint32_t w) { return e4m3_hb_to_f16x2_s8(__byte_perm(w, 0u, 0x2404)); }
__device__ __forceinline__ uint32_t e4m3_odd2(uint32_t w) { return e4m3_hb_to_f16x2_s8(__byte_perm(w, 0u, 0x3414)); }

constexpr int kMaxCluster = 8;

// Cluster split (kSplit): the CTAs of one cluster each hold their share of a
// (query, KV head) segment as an unnormalised state (m, l, O) in comb slot 0
// of their own shared memory.  Every thread of the cluster calls this once.
// After the first cluster barrier every CTA's pipeline is done, so the chunk
// ring of the CTA of rank 0 is free: each other CTA stores its state into
// slot rank - 1 there (remote stores, nothing waited on), and after the second
// barrier rank 0 merges the states from its own shared memory and stores the
// output rows.
// A slot: m[16], l[16], then O[16] rows of kPushStride floats (128 used): the
// 4 padding floats put the 16-byte pieces a warp reads at once (rows lane / 2,
// halves lane % 2) in all 8 bank groups instead of one.
constexpr int kPushStride = kDim + 4;
constexpr int kPushFloats = 2 * kGroup + kGroup * kPushStride;

template <int kFp8, class Smem>
__device__ __forceinline__ void split_finish(Smem& sm, int csize, int warp, int lane, float v_scale,
                                             __nv_bfloat16* __restrict__ out, uint8_t* __restrict__ out_q,
                                             uint8_t* __restrict__ out_scale) {
  // the slots start at stage 1: stage 0 holds this CTA's merged state
  static_assert(sizeof(sm.stage) - sizeof(sm.stage[0]) >= (kMaxCluster - 1) * kPushFloats * sizeof(float),
                "push slots");
  const int rank = blockIdx.x % csize;
  const int row = lane >> 1, d0 = (lane & 1) * 64;
  float* slots = reinterpret_cast<float*>(&sm.stage[1][0]);
  const CombRef mine = comb_ref(sm, 0);
  cluster_arrive_release();
  cluster_wait_acquire();
  if (rank != 0 && warp == 0) {
    float* dst = slots + (rank - 1) * kPushFloats;
    if ((lane & 1) == 0) {
      st_dsmem_f32(dsmem_addr(dst + row, 0), mine.m[row]);
      st_dsmem_f32(dsmem_addr(dst + kGroup + row, 0), mine.l[row]);
    }
    const uint32_t o = dsmem_addr(dst + 2 * kGroup + row * kPushStride + d0, 0);
    const float* src = mine.row(row) + d0;
#pragma unroll
    for (int d = 0; d < 16; ++d) st_dsmem_v4(o + 16 * d, *reinterpret_cast<const float4*>(src + 4 * d));
  }
  cluster_arrive_release();
  cluster_wait_acquire();
  if (rank != 0 || warp != 0) return;
  const int qi = (blockIdx.x / csize) / kKvHeads, g = (blockIdx.x / csize) % kKvHeads;
  // contributor 0 is this CTA (comb slot 0), contributor x > 0 the ring slot x - 1
  auto m_of = [&](int x) { return x == 0 ? mine.m[row] : slots[(x - 1) * kPushFloats + row]; };
  auto l_of = [&](int x) { return x == 0 ? mine.l[row] : slots[(x - 1) * kPushFloats + kGroup + row]; };
  auto o_of = [&](int x) {
    return x == 0 ? mine.row(row) + d0 : slots + (x - 1) * kPushFloats + 2 * kGroup + row * kPushStride + d0;
  };
  float mc[kMaxCluster], lc[kMaxCluster];
#pragma unroll
  for (int x = 0; x < kMaxCluster; ++x) {
    mc[x] = x < csize ? m_of(x) : -INFINITY;
    lc[x] = x < csize ? l_of(x) : 0.f;
  }
  float Mg = -INFINITY;
#pragma unroll
  for (int x = 0; x < kMaxCluster; ++x) Mg = fmaxf(Mg, mc[x]);
  const float Mgu = Mg == -INFINITY ? 0.f : Mg;
  float Lg = 0.f, ag[64];
#pragma unroll
  for (int d = 0; d < 64; ++d) ag[d] = 0.f;
#pragma unroll
  for (int x = 0; x < kMaxCluster; ++x) {
    mc[x] = exp2f(mc[x] - Mgu);  // the CTA's weight (0 for an empty state and past csize)
    Lg += lc[x] * mc[x];
  }
  for (int x = 0; x < csize; ++x) {
    const float* src = o_of(x);
    const float f = mc[x];
#pragma unroll
    for (int d = 0; d < 16; ++d) {
      const float4 v = *reinterpret_cast<const float4*>(src + 4 * d);
      ag[4 * d] += v.x * f;
      ag[4 * d + 1] += v.y * f;
      ag[4 * d + 2] += v.z * f;
      ag[4 * d + 3] += v.w * f;
    }
  }
  const float inv = Lg > 0.f ? (kFp8 ? v_scale : 1.f) / Lg : 0.f;
  const long long oelem = (static_cast<long long>(qi) * kHeads + g * kGroup + row) * kDim + d0;
  if (out_q) {
    store_mxfp8_64(ag, inv, out_q + oelem, out_scale + oelem / 32);
  } else {
    __nv_bfloat16* orow = out + oelem;
#pragma unroll
    for (int v = 0; v < 8; ++v)
      reinterpret_cast<uint4*>(orow)[v] = make_uint4(
          pack_bf16(ag[8 * v] * inv, ag[8 * v + 1] * inv), pack_bf16(ag[8 * v + 2] * inv, ag[8 * v + 3] * inv),
          pack_bf16(ag[8 * v + 4] * inv, ag[8 * v + 5] * inv), pack_bf16(ag[8 * v + 6] * inv, ag[8 * v + 7] * inv));
  }
}

// out_q / out_scale: when non-null, the output is emitted as MXFP8 there
// instead of bf16 in `out`.  kFp8: the K / V caches hold E4M3 bytes;
// scale_log2 then includes 2^8 k_scale, and v_scale (2^8 times the cache's) multiplies the output.
// kSplit: launched in clusters of csize CTAs, one cluster per (query, KV
// head) segment; CTA rank r takes units [r topk / csize, (r + 1) topk / csize)
// of it, and the cluster merges on chip (split_finish).  Otherwise stream-K:
// the units are split evenly over the grid and cut segments are merged
// through fp32 partials in global memory and a ticket per segment.
template <int kFp8, int kSplit>
__global__ void __launch_bounds__(kAttThreads, AttShape<kFp8, kSplit>::kCtasPerSm) sparse_attend_kernel(
    const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
    const __grid_constant__ CUtensorMap qmap, const int32_t* __restrict__ q2k, AttnGeom geo, int topk,
    float scale_log2, float v_scale, __nv_bfloat16* __restrict__ out, uint8_t* __restrict__ out_q,
    uint8_t* __restrict__ out_scale, float* __restrict__ partials, int* __restrict__ tickets, int csize,
    DevError* err) {
  extern __shared__ uint8_t smem_raw[];
  AttSmem<kFp8, kSplit>& sm = *reinterpret_cast<AttSmem<kFp8, kSplit>*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int kStg = AttShape<kFp8, kSplit>::kStages;
  constexpr int kQS = AttShape<kFp8, kSplit>::kQSlots;
  const long long N = static_cast<long long>(geo.nq) * kKvHeads * topk;
  const long long G = gridDim.x;
  long long lo, hi;
  if constexpr (kSplit != 0) {
    const long long seg = blockIdx.x / csize, rank = blockIdx.x % csize;
    lo = seg * topk + rank * topk / csize;
    hi = seg * topk + (rank + 1) * topk / csize;
  } else {
    lo = seg_begin(blockIdx.x, N, G);
    hi = seg_begin(blockIdx.x + 1, N, G);
  }

  if (tid == 0) {
    for (int s = 0; s < kStg; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], 1);
    }
    for (int s = 0; s < kQS; ++s) {
      mbar_init(&sm.seg_full[s], 1);
      mbar_init(&sm.seg_empty[s], kConsumerWarps);
    }
    fence_mbar_init();
  }
  if (warp == kConsumerWarps && lo < hi) {
    if (lane == 0) {
      prefetch_tmap(&kmap);
      prefetch_tmap(&vmap);
      prefetch_tmap(&qmap);
    }
    // the page-table rows of this CTA's requests into L2 (a hint: the rows are
    // read only after the wait below)
    if (geo.page_table) {
      const int q0 = static_cast<int>(lo / (kKvHeads * topk)), q1 = static_cast<int>((hi - 1) / (kKvHeads * topk));
      for (int qi = q0; qi <= q1; ++qi)
        for (int o = lane * 32; o < geo.max_blocks; o += 32 * 32)
          prefetch_l2(geo.page_table + static_cast<long long>(qi) * geo.max_blocks + o);
    }
  }
  // Launched as a programmatic dependent of the previous kernel (the decode
  // top-k): everything above overlaps it; no input is read and no output
  // written before that grid has completed.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  __syncthreads();
  if (lo >= hi) {
    if constexpr (kSplit != 0) {
      // no unit (csize > topk, never chosen by the host): an empty state
      const CombRef c0 = comb_ref(sm, 0);
      if (warp == 0)
        for (int i = lane; i < kGroup * kDim; i += 32) c0.row(i / kDim)[i % kDim] = 0.f;
      if (warp == 0 && lane < kGroup) {
        c0.m[lane] = -INFINITY;
        c0.l[lane] = 0.f;
      }
      split_finish<kFp8>(sm, csize, warp, lane, v_scale, out, out_q, out_scale);
    }
    return;
  }

  if (warp == kConsumerWarps) {
    // ---------------- producer warp ----------------
    long long sc = 0;
    int nseg = 0;
    long long it = lo;
    while (it < hi) {
      const int qi = static_cast<int>(it / (kKvHeads * topk));
      const int g = static_cast<int>((it / topk) % kKvHeads);
      const long long seg_end = min(hi, (static_cast<long long>(qi) * kKvHeads + g + 1) * topk);
      const QueryGeo qg = query_geo(geo, qi);
      const int j0 = static_cast<int>(it % topk), jn = static_cast<int>(seg_end - it);
      // the lanes resolve the segment's blocks in parallel: q2k entry, then page id
      int nk_l = 0;
      long long r0_l = 0;
      if (lane < jn) {
        const int b = q2k[(static_cast<long long>(g) * geo.nq + qi) * topk + j0 + lane];
        if (b >= qg.nb) record_error(err, MSA_DEVERR_BLOCK, it + lane);
        nk_l = block_keys(qg, b);
        if (nk_l) {
          r0_l = block_row0(geo, qi, qg, b);
          if (r0_l < 0) {
            nk_l = 0;
            record_error(err, MSA_DEVERR_PAGE, it + lane);
          }
        }
      }
      // segment slot: key counts + the Q tile of the 16 heads
      const int ss = nseg % kQS;
      if (lane == 0) mbar_wait(&sm.seg_empty[ss], ((nseg / kQS) & 1) ^ 1, err, 210);
      for (int j = 0; j < kMaxTopk; ++j) {
        const int v = __shfl_sync(0xffffffffu, nk_l, j);
        if (lane == 0) sm.seg[ss].nk[j] = j < jn ? v : 0;
      }
      if (lane == 0) {
        mbar_expect_tx(&sm.seg_full[ss], 2 * kQBoxBytes);
        const int qrow = qi * kHeads + g * kGroup;
        tma_load_2d(sm.qtile[ss], &qmap, 0, qrow, &sm.seg_full[ss]);
        tma_load_2d(sm.qtile[ss] + kQBoxBytes, &qmap, 64, qrow, &sm.seg_full[ss]);
      }
      __syncwarp();
      ++nseg;
      for (int k = 0; k < jn; ++k) {
        const int nk = __shfl_sync(0xffffffffu, nk_l, k);
        const long long r0 = __shfl_sync(0xffffffffu, r0_l, k);
        if (nk == 0) continue;
        const int nch = (nk + kChunkKeys - 1) / kChunkKeys;
        for (int ch = 0; ch < nch; ++ch, ++sc) {
          if (lane == 0) {
            const int s = static_cast<int>(sc % kStg);
            mbar_wait(&sm.empty[s], static_cast<uint32_t>(((sc / kStg) & 1) ^ 1), err, 200);
            const int row = static_cast<int>(r0 + ch * kChunkKeys);
            uint8_t* st = sm.stage[s];
            if (kFp8) {
              mbar_expect_tx(&sm.full[s], kAttStage8Bytes);
              tma_load_3d(st, &kmap, 0, g, row, &sm.full[s]);
              tma_load_3d(st + kBoxBytes, &vmap, 0, g, row, &sm.full[s]);
            } else {
              mbar_expect_tx(&sm.full[s], kAttStageBytes);
              tma_load_3d(st + 0 * kBoxBytes, &kmap, 0, g, row, &sm.full[s]);
              tma_load_3d(st + 1 * kBoxBytes, &kmap, 64, g, row, &sm.full[s]);
              tma_load_3d(st + 2 * kBoxBytes, &vmap, 0, g, row, &sm.full[s]);
              tma_load_3d(st + 3 * kBoxBytes, &vmap, 64, g, row, &sm.full[s]);
            }
          }
          __syncwarp();
        }
      }
      it = seg_end;
    }
    // No copy may still be landing when the CTA exits, also after a wait gave
    // up: wait (bounded) for the last fill of every chunk stage and segment
    // slot.  Only this thread arms those barriers, so that phase cannot have
    // been passed.
    if (lane == 0) {
      for (int s = 0; s < kStg; ++s) {
        const long long f = (sc - s + kStg - 1) / kStg;  // fills of stage s
        if (f > 0) mbar_wait(&sm.full[s], static_cast<uint32_t>((f - 1) & 1), err, 220);
      }
      for (int s = 0; s < kQS; ++s) {
        const int f = (nseg - s + kQS - 1) / kQS;
        if (f > 0) mbar_wait(&sm.seg_full[s], (f - 1) & 1, err, 221);
      }
    }
    __syncwarp();
    if constexpr (kSplit != 0) split_finish<kFp8>(sm, csize, warp, lane, v_scale, out, out_q, out_scale);
    return;
  }

  // ---------------- consumer warps: whole 64-key chunks, stage s -> warp s % 3 ----------------
  const int g8 = lane >> 2, t4 = lane & 3;
  long long sc = 0;  // chunk counter, identical in every consumer warp and the producer
  int nseg = 0;
  long long it = lo;
  while (it < hi) {
    const int qi = static_cast<int>(it / (kKvHeads * topk));
    const int g = static_cast<int>((it / topk) % kKvHeads);
    const long long seg_lo = it;
    const long long range0 = (static_cast<long long>(qi) * kKvHeads + g) * topk;
    const long long seg_end = min(hi, range0 + topk);
    const int jn = static_cast<int>(seg_end - it);
    const int ss = nseg % kQS;
    mbar_wait(&sm.seg_full[ss], (nseg / kQS) & 1, err, 310);
    const int nk_l = lane < kMaxTopk ? sm.seg[ss].nk[lane] : 0;
    // Q fragments of the 16 heads (A operand, 8 k-steps) from the swizzled Q tile
    uint32_t qa[8][4];
    {
      const uint32_t qt = smem_u32(sm.qtile[ss]);
      if constexpr (kFp8 != 0) {
        // fp16, k slots permuted as the K fragments are (S = Q K^T below):
        // slots 2t, 2t+1, 2t+8, 2t+9 of k-step s hold dims 16s + 4t .. + 3
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const int chunk = 2 * (kk & 3) + (t4 >> 1);  // 16-byte chunk of 8 dims in the box of 64
          const uint32_t off = (kk >> 2) * kQBoxBytes + 8 * (t4 & 1);
          const uint2 a = lds64(qt + off + sw128(g8, chunk));
          const uint2 b = lds64(qt + off + sw128(g8 + 8, chunk));
          qa[kk][0] = bf16x2_to_f16x2(a.x);
          qa[kk][1] = bf16x2_to_f16x2(b.x);
          qa[kk][2] = bf16x2_to_f16x2(a.y);
          qa[kk][3] = bf16x2_to_f16x2(b.y);
        }
      } else {
        const int qrow = (lane & 7) + 8 * ((lane >> 3) & 1);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const int chunk = 2 * kk + (lane >> 4);
          ldsm_x4(qa[kk], qt + (chunk >> 3) * kQBoxBytes + sw128(qrow, chunk & 7));
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.seg_empty[ss]);  // the slot may be refilled
    ++nseg;

    // This CTA holds the end of a segment whose start lies in earlier CTAs: it
    // is then, in all likelihood, the one that merges it (the others took it
    // at the start of their ranges), so warp 0 brings their partials back into
    // L2 two units before the end (the streaming may have evicted them).
    const bool pf = kSplit == 0 && warp == 0 && seg_end == range0 + topk && seg_lo > range0;
    const int pf_k = jn > 2 ? jn - 2 : 0;

    WarpState st;
    st.m0 = st.m1 = -INFINITY;
    st.l0 = st.l1 = 0.f;
#pragma unroll
    for (int nd = 0; nd < 16; ++nd) st.o[nd][0] = st.o[nd][1] = st.o[nd][2] = st.o[nd][3] = 0.f;

    for (int k = 0; k < jn; ++k) {
      const int nk = __shfl_sync(0xffffffffu, nk_l, k);
      if (nk == 0) continue;
      const int nch = (nk + kChunkKeys - 1) / kChunkKeys;
      if (pf && k == pf_k) {
        const long long c0 = cta_of(range0, N, G);
        for (long long c = c0; c < blockIdx.x; ++c) {
          const long long slot = 2 * c + (c == c0 && seg_begin(c0, N, G) < range0 ? 1 : 0);
          const char* pp = reinterpret_cast<const char*>(partials + slot * kPartialFloats);
          for (int o = lane * 128; o < kPartialFloats * 4; o += 32 * 128) prefetch_l2(pp + o);
        }
      }
      for (int ch = 0; ch < nch; ++ch, ++sc) {
        const int s = static_cast<int>(sc % kStg);
        if (s % kConsumerWarps != warp) continue;
        const int valid = min(kChunkKeys, nk - ch * kChunkKeys);  // keys of this chunk
        mbar_wait(&sm.full[s], static_cast<uint32_t>((sc / kStg) & 1), err, 300);
        const uint32_t stg = smem_u32(sm.stage[s]);
        const int mi = lane >> 3;
        // ---- S = Q K^T over the chunk's keys (n-tiles of 8 keys, in pairs) ----
        float sacc[8][4];
#pragma unroll
        for (int p = 0; p < 8; ++p) sacc[p][0] = sacc[p][1] = sacc[p][2] = sacc[p][3] = 0.f;
        if constexpr (kFp8 != 0) {
          // E4M3 K rows are 128 bytes: a 16-byte chunk is one k-step of 16 dims.
          // ldmatrix (16-bit view) gives a lane 4 consecutive bytes, dims
          // 16s + 4t .. + 3 of one key, converted in registers into the B
          // fragment whose slots the Q fragments above were permuted to match.
#pragma unroll
          for (int kp = 0; kp < 4; ++kp) {
            if (16 * kp >= valid) break;
            const int krow = 16 * kp + 8 * (mi & 1) + (lane & 7);
#pragma unroll
            for (int kk = 0; kk < 8; kk += 2) {
              uint32_t kr[4];  // keys lo / hi of k-step kk, then of k-step kk + 1
              ldsm_x4(kr, stg + sw128(krow, kk + (mi >> 1)));
              mma_f16(sacc[2 * kp], qa[kk], e4m3_lo2(kr[0]), e4m3_hi2(kr[0]));
              mma_f16(sacc[2 * kp + 1], qa[kk], e4m3_lo2(kr[1]), e4m3_hi2(kr[1]));
              mma_f16(sacc[2 * kp], qa[kk + 1], e4m3_lo2(kr[2]), e4m3_hi2(kr[2]));
              mma_f16(sacc[2 * kp + 1], qa[kk + 1], e4m3_lo2(kr[3]), e4m3_hi2(kr[3]));
            }
          }
        } else {
#pragma unroll
          for (int kp = 0; kp < 4; ++kp) {
            if (16 * kp >= valid) break;
            const int krow = 16 * kp + 8 * (mi >> 1) + (lane & 7);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              const int chunk = 2 * kk + (mi & 1);  // 16-byte chunk of the 256-byte row
              uint32_t kb[4];
              ldsm_x4(kb, stg + (chunk >> 3) * kBoxBytes + sw128(krow, chunk & 7));
              mma_bf16(sacc[2 * kp], qa[kk], kb[0], kb[1]);
              mma_bf16(sacc[2 * kp + 1], qa[kk], kb[2], kb[3]);
            }
          }
        }
        // ---- mask, online softmax (base 2, scale folded in) ----
        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
        for (int p = 0; p < 8; ++p) {
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const bool ok = 8 * p + 2 * t4 + e < valid;
            sacc[p][e] = ok ? sacc[p][e] * scale_log2 : -INFINITY;
            sacc[p][2 + e] = ok ? sacc[p][2 + e] * scale_log2 : -INFINITY;
            mx0 = fmaxf(mx0, sacc[p][e]);
            mx1 = fmaxf(mx1, sacc[p][2 + e]);
          }
        }
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
        const float mn0 = fmaxf(st.m0, mx0), mn1 = fmaxf(st.m1, mx1);
        const float mu0 = mn0 == -INFINITY ? 0.f : mn0, mu1 = mn1 == -INFINITY ? 0.f : mn1;
        const float al0 = exp2f(st.m0 - mu0), al1 = exp2f(st.m1 - mu1);
        st.m0 = mn0;
        st.m1 = mn1;
        // p rounded to the 16-bit MMA type (the PV operand); the row sum adds the
        // same rounded values, so the normalisation matches the weights the MMA applies
        float rs0 = 0.f, rs1 = 0.f;
#pragma unroll
        for (int p = 0; p < 8; ++p) {
          sacc[p][0] = round16<kFp8>(exp2f(sacc[p][0] - mu0));
          sacc[p][1] = round16<kFp8>(exp2f(sacc[p][1] - mu0));
          sacc[p][2] = round16<kFp8>(exp2f(sacc[p][2] - mu1));
          sacc[p][3] = round16<kFp8>(exp2f(sacc[p][3] - mu1));
          rs0 += sacc[p][0] + sacc[p][1];
          rs1 += sacc[p][2] + sacc[p][3];
        }
        st.l0 = st.l0 * al0 + rs0;
        st.l1 = st.l1 * al1 + rs1;
#pragma unroll
        for (int nd = 0; nd < 16; ++nd) {
          st.o[nd][0] *= al0;
          st.o[nd][1] *= al0;
          st.o[nd][2] *= al1;
          st.o[nd][3] *= al1;
        }
        // ---- O += P V, one k-step per 16 keys (P exact in bf16 after the rounding above) ----
#pragma unroll
        for (int kp = 0; kp < 4; ++kp) {
          if (16 * kp >= valid) break;
          const uint32_t pa[4] = {pack16<kFp8>(sacc[2 * kp][0], sacc[2 * kp][1]),
                                  pack16<kFp8>(sacc[2 * kp][2], sacc[2 * kp][3]),
                                  pack16<kFp8>(sacc[2 * kp + 1][0], sacc[2 * kp + 1][1]),
                                  pack16<kFp8>(sacc[2 * kp + 1][2], sacc[2 * kp + 1][3])};
          const int vrow = 16 * kp + 8 * (mi & 1) + (lane & 7);
          if constexpr (kFp8 != 0) {
            // The transposing ldmatrix (16-bit view) of E4M3 V gives a lane
            // keys 2t, 2t+1 of dims 2g, 2g+1 of a 16-dim block: bytes 0 / 2 are
            // the pair of the even dim, 1 / 3 that of the odd one, so the block
            // feeds two n-tiles, its even and its odd dims (st.o[2c], [2c+1]).
#pragma unroll
            for (int c = 0; c < 8; c += 2) {
              uint32_t vr[4];  // keys lo / hi of block c, then of block c + 1
              ldsm_x4_t(vr, stg + kBoxBytes + sw128(vrow, c + (mi >> 1)));
              mma_f16(st.o[2 * c], pa, e4m3_even2(vr[0]), e4m3_even2(vr[1]));
              mma_f16(st.o[2 * c + 1], pa, e4m3_odd2(vr[0]), e4m3_odd2(vr[1]));
              mma_f16(st.o[2 * c + 2], pa, e4m3_even2(vr[2]), e4m3_even2(vr[3]));
              mma_f16(st.o[2 * c + 3], pa, e4m3_odd2(vr[2]), e4m3_odd2(vr[3]));
            }
          } else {
#pragma unroll
            for (int nd = 0; nd < 16; nd += 2) {
              const int chunk = nd + (mi >> 1);
              uint32_t vb[4];
              ldsm_x4_t(vb, stg + (2 + (chunk >> 3)) * kBoxBytes + sw128(vrow, chunk & 7));
              mma_bf16(st.o[nd], pa, vb[0], vb[1]);
              mma_bf16(st.o[nd + 1], pa, vb[2], vb[3]);
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.empty[s]);
      }
    }
    it = seg_end;

    // ---- merge the three warps' states into warp 0 ----
    st.l0 += __shfl_xor_sync(0xffffffffu, st.l0, 1);
    st.l0 += __shfl_xor_sync(0xffffffffu, st.l0, 2);
    st.l1 += __shfl_xor_sync(0xffffffffu, st.l1, 1);
    st.l1 += __shfl_xor_sync(0xffffffffu, st.l1, 2);
    if constexpr (kSplit == 0 && AttShape<kFp8, kSplit>::kCombSlots == 1) {
      // one slot: warp 2, then warp 1, hands its state to warp 0 (warp 0 has
      // read it before it reaches the next segment's first meeting, the only
      // place the slot is written again)
      consumer_sync();
      if (warp == 2) state_to_smem<kFp8>(st, comb_ref(sm, 1), g8, t4);
      consumer_sync();
      if (warp == 0) merge_from_smem<kFp8>(st, comb_ref(sm, 1), g8, t4);
      consumer_sync();
      if (warp == 1) state_to_smem<kFp8>(st, comb_ref(sm, 1), g8, t4);
      consumer_sync();
      if (warp > 0) continue;  // warps 1 and 2 go on to the next segment
      merge_from_smem<kFp8>(st, comb_ref(sm, 1), g8, t4);
    } else {
      consumer_sync();
      if (warp > 0) state_to_smem<kFp8>(st, comb_ref(sm, warp), g8, t4);
      consumer_sync();
      if (warp > 0) continue;  // warps 1 and 2 go on to the next segment
#pragma unroll
      for (int w = 1; w < kConsumerWarps; ++w) merge_from_smem<kFp8>(st, comb_ref(sm, w), g8, t4);
    }
    __syncwarp();
    state_to_smem<kFp8>(st, comb_ref(sm, 0), g8, t4);  // staging for coalesced stores (read only by warp 0)
    __syncwarp();
    if constexpr (kSplit != 0) continue;  // the cluster merges slot 0 (split_finish)
    // ---- warp 0 writes: lane -> row lane/2, 64 dims ----
    const int row = lane >> 1, d0 = (lane & 1) * 64;
    const CombRef c0 = comb_ref(sm, 0);
    const float M = c0.m[row], Lsum = c0.l[row];
    const float* src = c0.row(row) + d0;
    const bool complete = (seg_lo == range0) && (seg_end == range0 + topk);
    const long long oelem = (static_cast<long long>(qi) * kHeads + g * kGroup + row) * kDim + d0;
    __nv_bfloat16* orow = out_q ? nullptr : out + oelem;
    if (complete) {
      const float inv = Lsum > 0.f ? (kFp8 ? v_scale : 1.f) / Lsum : 0.f;
      if (out_q) {
        store_mxfp8_64(src, inv, out_q + oelem, out_scale + oelem / 32);
      } else {
#pragma unroll
        for (int v = 0; v < 8; ++v)
          reinterpret_cast<uint4*>(orow)[v] = make_uint4(
              pack_bf16(src[8 * v] * inv, src[8 * v + 1] * inv), pack_bf16(src[8 * v + 2] * inv, src[8 * v + 3] * inv),
              pack_bf16(src[8 * v + 4] * inv, src[8 * v + 5] * inv), pack_bf16(src[8 * v + 6] * inv, src[8 * v + 7] * inv));
      }
    } else {
      // The contributors are the consecutive CTAs c_first .. c_last (at most
      // topk: each holds at least one unit of the segment).  The segment's
      // counter is the one of c_first: a CTA is the first contributor of a cut
      // segment only for its last segment, so each counter serves one segment.
      const long long c_first = cta_of(range0, N, G);
      const int cnt = static_cast<int>(seg_end - seg_lo);
      // If every other contributor has already counted its units, this CTA
      // completes the segment and merges it at once from its own state, without
      // publishing a partial.  (They write their partial, fence, then add; the
      // acquire load that sees their counts also sees their partials.  No
      // contributor adds after that, so no other CTA merges the segment.)
      int last = 0;
      if (lane == 0) last = (ld_acquire_gpu(&tickets[c_first]) + cnt == topk) ? 1 : 0;
      last = __shfl_sync(0xffffffffu, last, 0);
      if (!last) {
        // partial slot: the CTA's first segment -> 2c, its last -> 2c+1
        const long long slot = 2LL * blockIdx.x + (range0 <= lo ? 0 : 1);
        float* pp = partials + slot * kPartialFloats;
        if ((lane & 1) == 0) {
          pp[row] = M;
          pp[16 + row] = Lsum;
        }
#pragma unroll
        for (int v = 0; v < 16; ++v)
          *reinterpret_cast<float4*>(pp + 32 + row * kDim + d0 + 4 * v) =
              make_float4(src[4 * v], src[4 * v + 1], src[4 * v + 2], src[4 * v + 3]);
        __threadfence();
        __syncwarp();
        if (lane == 0) last = (atomicAdd(&tickets[c_first], cnt) + cnt == topk) ? 1 : 0;
        last = __shfl_sync(0xffffffffu, last, 0);
        if (last) __threadfence();
      }
      if (last) {
        // This CTA's own share comes from its staged state (shared memory), the
        // others' from their partials.  Every contributor but the first wrote
        // this segment as its first partial.  All loads of a pass are issued
        // before any is used.
        const long long c_last = cta_of(range0 + topk - 1, N, G);
        const int nc = static_cast<int>(c_last - c_first + 1);
        const int xs = static_cast<int>(blockIdx.x - c_first);
        const long long slot0 = 2 * c_first + (seg_begin(c_first, N, G) < range0 ? 1 : 0);
        auto part_of = [&](int x) {
          return partials + (x == 0 ? slot0 : 2 * (c_first + x)) * kPartialFloats;
        };
        float mc[kMaxTopk], lc[kMaxTopk];
#pragma unroll
        for (int x = 0; x < kMaxTopk; ++x) {
          mc[x] = x < nc && x != xs ? __ldcg(part_of(x) + row) : -INFINITY;
          lc[x] = x < nc && x != xs ? __ldcg(part_of(x) + 16 + row) : 0.f;
        }
        float Mg = M;
#pragma unroll
        for (int x = 0; x < kMaxTopk; ++x) Mg = fmaxf(Mg, mc[x]);
        const float Mgu = Mg == -INFINITY ? 0.f : Mg;
        const float fs = exp2f(M - Mgu);  // this CTA's weight
        float Lg = Lsum * fs, ag[64];
#pragma unroll
        for (int d = 0; d < 64; ++d) ag[d] = src[d] * fs;
#pragma unroll
        for (int x = 0; x < kMaxTopk; ++x) {
          mc[x] = exp2f(mc[x] - Mgu);  // the contributor's weight (0 past nc and for this CTA)
          Lg += lc[x] * mc[x];
        }
#pragma unroll 2
        for (int x = 0; x < nc; ++x) {
          if (x == xs) continue;
          const float* pc = part_of(x) + 32 + row * kDim + d0;
          float4 xv[16];
#pragma unroll
          for (int d = 0; d < 16; ++d) xv[d] = __ldcg(reinterpret_cast<const float4*>(pc) + d);
          const float f = mc[x];
#pragma unroll
          for (int d = 0; d < 16; ++d) {
            ag[4 * d] += xv[d].x * f;
            ag[4 * d + 1] += xv[d].y * f;
            ag[4 * d + 2] += xv[d].z * f;
            ag[4 * d + 3] += xv[d].w * f;
          }
        }
        const float inv = Lg > 0.f ? (kFp8 ? v_scale : 1.f) / Lg : 0.f;
        if (out_q) {
          store_mxfp8_64(ag, inv, out_q + oelem, out_scale + oelem / 32);
        } else {
#pragma unroll
          for (int v = 0; v < 8; ++v)
            reinterpret_cast<uint4*>(orow)[v] = make_uint4(
                pack_bf16(ag[8 * v] * inv, ag[8 * v + 1] * inv), pack_bf16(ag[8 * v + 2] * inv, ag[8 * v + 3] * inv),
                pack_bf16(ag[8 * v + 4] * inv, ag[8 * v + 5] * inv), pack_bf16(ag[8 * v + 6] * inv, ag[8 * v + 7] * inv));
        }
        if (lane == 0) tickets[c_first] = 0;
      }
    }
  }
  if constexpr (kSplit != 0) split_finish<kFp8>(sm, csize, warp, lane, v_scale, out, out_q, out_scale);
}

// ---- host side --------------------------------------------------------------------

// 3-D map over a [rows, 4, 128] bf16 array; box = 64 dims x 1 head x 64 rows, 128-byte swizzle.
static bool make_kv_map(CUtensorMap* map, const void* base, long long rows) {
  EncodeTiledFn enc = get_encode_tiled();
  if (!enc) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(kDim), static_cast<cuuint64_t>(kKvHeads),
                        static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[2] = {kDim * 2, kKvHeads * kDim * 2};
  cuuint32_t box[3] = {64, 1, kChunkKeys};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D map over a [rows, 4, 128] E4M3 array; box = 128 dims (128 bytes) x 1 head x 64 rows, 128-byte swizzle.
static bool make_kv_map8(CUtensorMap* map, const void* base, long long rows) {
  EncodeTiledFn enc = get_encode_tiled();
  if (!enc) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(kDim), static_cast<cuuint64_t>(kKvHeads),
                        static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[2] = {kDim, kKvHeads * kDim};
  cuuint32_t box[3] = {128, 1, kChunkKeys};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D map over q viewed as [queries * 64, 128] bf16; box = 64 dims x 16 heads, 128-byte swizzle.
static bool make_q_map(CUtensorMap* map, const void* base, long long nq) {
  EncodeTiledFn enc = get_encode_tiled();
  if (!enc) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(kDim), static_cast<cuuint64_t>(nq * kHeads)};
  cuuint64_t strides[1] = {kDim * 2};
  cuuint32_t box[2] = {64, kGroup};
  cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int kFp8, int kSplit>
constexpr size_t att_smem() { return sizeof(AttSmem<kFp8, kSplit>) + 1024; }
static_assert(att_smem<0, 0>() <= 227 * 1024 && att_smem<0, 1>() <= 227 * 1024, "shared memory of the decode attention");
// two CTAs of the FP8 forms per SM (228 KB of shared memory per SM, 1 KB of it per CTA reserved)
static_assert(2 * (att_smem<1, 0>() + 1024) <= 228 * 1024 && 2 * (att_smem<1, 1>() + 1024) <= 228 * 1024,
              "shared memory of the decode attention, FP8 K/V");

// The stream-K grid: at most kCtasPerSm CTAs per SM (2 with an FP8 cache).
constexpr int kMaxStreamKCtas = 2 * kNumSMs;
size_t attend_partials_bytes() { return 2ull * kMaxStreamKCtas * kPartialFloats * sizeof(float); }
// one merge counter per CTA of the persistent grid
size_t attend_tickets_bytes() { return static_cast<size_t>(kMaxStreamKCtas) * sizeof(int); }

// How many clusters of c CTAs of the split kernel can be resident at once
// (cudaOccupancyMaxActiveClusters, asked once per device, K/V type and c; 0
// when the query fails, which keeps the stream-K kernel for that call).
static int max_active_clusters(int kv_fp8, int c) {
  static std::mutex mu;
  static int cache[64][2][kMaxCluster + 1];
  static bool done[64][2][kMaxCluster + 1];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (done[dev][kv_fp8][c]) return cache[dev][kv_fp8][c];
  const size_t smem = kv_fp8 ? att_smem<1, 1>() : att_smem<0, 1>();
  auto kern = kv_fp8 ? sparse_attend_kernel<1, 1> : sparse_attend_kernel<0, 1>;
  int n = 0;
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(static_cast<unsigned>(c * 16));
  lc.blockDim = dim3(kAttThreads);
  lc.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = c;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  lc.attrs = attr;
  lc.numAttrs = 1;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) != cudaSuccess ||
      cudaOccupancyMaxActiveClusters(&n, kern, &lc) != cudaSuccess) {
    cudaGetLastError();  // a failed query leaves no error behind for the launch that follows
    return 0;            // and is asked again next time (it is not kept)
  }
  cache[dev][kv_fp8][c] = n;
  done[dev][kv_fp8][c] = true;
  return n;
}

cudaError_t launch_sparse_attend(const AttnGeom& geo, const void* q, const void* k, const void* v,
                                 const int32_t* q2k, int topk, float scale, void* out, uint8_t* out_q,
                                 uint8_t* out_scale, float* partials, int* tickets, DevError* err,
                                 cudaStream_t stream, int kv_fp8, float k_scale, float v_scale) {
  if (const cudaError_t e0 = launch_prologue(); e0 != cudaSuccess) return e0;
  CUtensorMap kmap, vmap, qmap;
  const bool maps = kv_fp8 ? make_kv_map8(&kmap, k, geo.num_rows) && make_kv_map8(&vmap, v, geo.num_rows)
                           : make_kv_map(&kmap, k, geo.num_rows) && make_kv_map(&vmap, v, geo.num_rows);
  if (!maps || !make_q_map(&qmap, q, geo.nq)) return cudaErrorInvalidValue;
  // An FP8 cache holds k / k_scale and v / v_scale, and the kernel reads its
  // bytes as fp16 values times 2^-8 (e4m3_hb_to_f16x2_s8): 2^8 goes into both scales.
  const float scale_log2 = scale * (kv_fp8 ? 256.f * k_scale : 1.f) * 1.4426950408889634f;
  const long long S = static_cast<long long>(geo.nq) * kKvHeads;  // (query, KV head) segments
  const long long N = S * topk;
  // Few segments (small batches): one cluster of C CTAs per segment, merged
  // on chip -- the largest C in {8, 4, 2} with C <= topk (every CTA gets a
  // unit), at most one CTA per SM (two with an FP8 cache), and every cluster
  // resident at once.  Otherwise stream-K over the whole grid, one CTA per SM.
  const long long per_sm = kv_fp8 ? AttShape<1, 1>::kCtasPerSm : AttShape<0, 1>::kCtasPerSm;
  int C = 0;
  for (int c = kMaxCluster; c >= 2 && !C; c >>= 1) {
    if (c > topk || S * c > per_sm * kNumSMs) continue;
    const int fit = max_active_clusters(kv_fp8, c);
    if (fit > 0 && S <= fit) C = c;
  }
  const size_t smem = C ? (kv_fp8 ? att_smem<1, 1>() : att_smem<0, 1>()) : (kv_fp8 ? att_smem<1, 0>() : att_smem<0, 0>());
  // a programmatic dependent of the previous kernel in the stream (the kernel
  // waits for that grid before touching memory), so its launch and prologue
  // overlap the decode top-k
  cudaLaunchConfig_t lc = {};
  lc.blockDim = dim3(kAttThreads);
  lc.dynamicSmemBytes = smem;
  lc.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = 1;
  const float vs = kv_fp8 ? 256.f * v_scale : 1.f;
  auto* o = static_cast<__nv_bfloat16*>(out);
  if (C) {
    lc.gridDim = dim3(static_cast<unsigned>(S * C));
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = C;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    lc.numAttrs = 2;
    auto kern = kv_fp8 ? sparse_attend_kernel<1, 1> : sparse_attend_kernel<0, 1>;
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    return cudaLaunchKernelEx(&lc, kern, kmap, vmap, qmap, q2k, geo, topk, scale_log2, vs, o, out_q, out_scale,
                              static_cast<float*>(nullptr), static_cast<int*>(nullptr), C, err);
  }
  // At least 4 units per CTA: a segment is then shared by at most ~topk/4 + 1
  // CTAs, which bounds the partials its last CTA has to merge.
  long long grid_l = (N + 3) / 4;
  const long long max_ctas = static_cast<long long>(kv_fp8 ? AttShape<1, 0>::kCtasPerSm : AttShape<0, 0>::kCtasPerSm) *
                             kNumSMs;
  if (grid_l > max_ctas) grid_l = max_ctas;
  if (grid_l < 1) grid_l = 1;
  lc.gridDim = dim3(static_cast<unsigned>(grid_l));
  auto kern = kv_fp8 ? sparse_attend_kernel<1, 0> : sparse_attend_kernel<0, 0>;
  cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  return cudaLaunchKernelEx(&lc, kern, kmap, vmap, qmap, q2k, geo, topk, scale_log2, vs, o, out_q, out_scale,
                            partials, tickets, 1, err);
}

}  // namespace msa
