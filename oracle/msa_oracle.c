/*
 * msa_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously-correct CPU statement of what MiniMax-M3 two-step
 * block-sparse attention computes: block scoring, top-k block selection and
 * sparse GQA attention over the selected blocks, for the packed-document
 * prefill layout and for the paged / contiguous decode cache.  Only the tests,
 * the smoke check and the CPU-baseline leg of the benchmark may load it.  It
 * shares no code, header, table or helper with the CUDA library.
 *
 * Sources (three web pages on the method):
 *   [TRT] TensorRT-LLM, "MiniMaxM3SparseAttentionConfig": class description
 *         (index branch scores blocks, top-k per (kv_head, q_token), init blocks
 *         forced at the head and local blocks at the tail; sparse GQA attention
 *         over the selected blocks), fields sparse_block_size,
 *         sparse_topk_blocks, sparse_init_blocks, sparse_local_blocks,
 *         sparse_score_type ('max'), indexer_kv_dtype ('fp8' = unscaled E4M3
 *         with FP32 score accumulation), paged index-K cache [num_slots,1,dim].
 *   [NEMO] NeMo AutoModel, "nemo_automodel.components.models.minimax_m3_vl.msa":
 *         MSAMicrobatch.select_blocks (hard top-k over unnormalised QK maxima,
 *         document-local block ids, int32 [4, tokens, 16] padded with -1),
 *         _SelectionPlan (candidate and forced [tokens, blocks] masks),
 *         sparse_attention / _SparseAttention.forward (bf16 q[tokens,64,128],
 *         k/v[tokens,4,128] -> out[tokens,64,128]), the layout-from-doc_ids
 *         constructor and _contiguous_runs (document map rules).
 *
 * Precision: index scores are summed in fp64 (exact for E4M3 operands, exact
 * to far below fp32 resolution for bf16) and the selection decision is taken
 * on the fp32 rounding of that sum, because the pages fix FP32 as the score
 * precision ([TRT] indexer_kv_dtype).  Attention is computed in fp64.
 *
 * Readings where the pages are silent: forced blocks occupy top-k slots; q2k
 * rows list block ids ascending then -1; equal scores prefer the lower block
 * id; no scale on index scores; the diagonal block takes its max over causal
 * keys only; blocks restart at each document (request) start; a decode query
 * sits at position len-1 and sees its own key.  Two readings no page fixes,
 * so parity on them is unpinned beyond the reading itself (parity unpinned):
 * query head h uses kv/index head h / (H / G) (contiguous GQA groups), and the
 * softmax scale is a caller argument (1/sqrt(128) in the workloads; no
 * softcap, no sinks).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_HEADS 64
#define OR_KV 4
#define OR_DIM 128
#define OR_IDIM 128
#define OR_BLOCK 128
#define OR_MAXTOPK 64

/* ---- element decoding -------------------------------------------------- */

/* bf16 is the upper half of an IEEE binary32; widening is exact. */
static double bf16_value(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* OCP 8-bit floating point, E4M3 ("fn": no infinities): 1 sign bit, 4 exponent
 * bits with bias 7, 3 mantissa bits; exponent field 0 encodes subnormals
 * m/8 * 2^-6; S.1111.111 is NaN. */
double oracle_e4m3_value(uint8_t byte) {
  int sign = byte >> 7;
  int e = (byte >> 3) & 15;
  int m = byte & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    v = ldexp((double)m / 8.0, -6);
  else
    v = ldexp(1.0 + (double)m / 8.0, e - 7);
  return sign ? -v : v;
}

static double index_elem(const void* base, int dtype, int64_t i) {
  if (dtype == 0) return bf16_value(((const uint16_t*)base)[i]);
  return oracle_e4m3_value(((const uint8_t*)base)[i]);
}

/* ---- step 1: block scores ---------------------------------------------
 * score(g, b) = max over causal keys p in block b (128b <= p <= min(128b+127,
 * pos)) of <index_q[g], index_k[key p]>  ([TRT] sparse_score_type 'max';
 * [NEMO] select_blocks "unnormalized QK maxima").  key_row[p] maps a document-
 * local key position to its row in the index-K array. */
static void block_scores(const void* iq_row /* [G][IDIM] of this query */,
                         const void* ik /* [rows][IDIM] */, int dtype,
                         const int64_t* key_row, int64_t pos, int nb,
                         double* s64 /* [G][nb] */) {
  for (int g = 0; g < OR_KV; ++g)
    for (int b = 0; b < nb; ++b) s64[g * nb + b] = -INFINITY;
  for (int64_t p = 0; p <= pos; ++p) {
    int b = (int)(p / OR_BLOCK);
    int64_t row = key_row[p];
    for (int g = 0; g < OR_KV; ++g) {
      double acc = 0.0;
      for (int c = 0; c < OR_IDIM; ++c)
        acc += index_elem(iq_row, dtype, (int64_t)g * OR_IDIM + c) *
               index_elem(ik, dtype, row * OR_IDIM + c);
      if (acc > s64[g * nb + b]) s64[g * nb + b] = acc;
    }
  }
}

/* ---- step 2: top-k selection with forced blocks -------------------------
 * F = [0, init) u [nb-local, nb) restricted to [0, nb) ([TRT]
 * sparse_init_blocks / sparse_local_blocks: forced "into the top-k regardless
 * of score"; [NEMO] _SelectionPlan forced mask).  If nb <= topk every candidate
 * is kept.  Otherwise the non-forced candidates are ordered by (score desc,
 * id asc) and the first topk-|F| join F.  Output: ascending ids, then -1.
 * Returns the relative gap between the last kept and first rejected
 * non-forced score (INFINITY when nothing was decided by score). */
static double select_row(const float* s32 /* [nb] */, int nb, int topk,
                         int init, int local, int32_t* out /* [topk] */) {
  char* keep = (char*)calloc((size_t)nb, 1);
  int* cand = (int*)malloc(sizeof(int) * (size_t)nb);
  double gap = INFINITY;
  int n_keep = 0, n_cand = 0;
  if (nb <= topk) {
    for (int b = 0; b < nb; ++b) keep[b] = 1;
    n_keep = nb;
  } else {
    for (int b = 0; b < nb; ++b) {
      int forced = (b < init) || (b >= nb - local);
      if (forced) {
        keep[b] = 1;
        ++n_keep;
      } else {
        cand[n_cand++] = b;
      }
    }
    int need = topk - n_keep;
    /* selection sort by (score desc, id asc): slow and plain */
    for (int i = 0; i < n_cand && i <= need; ++i) {
      int best = i;
      for (int j = i + 1; j < n_cand; ++j) {
        float sj = s32[cand[j]], sb = s32[cand[best]];
        if (sj > sb || (sj == sb && cand[j] < cand[best])) best = j;
      }
      int tmp = cand[i];
      cand[i] = cand[best];
      cand[best] = tmp;
    }
    for (int i = 0; i < need && i < n_cand; ++i) {
      keep[cand[i]] = 1;
      ++n_keep;
    }
    if (need > 0 && n_cand > need) {
      double a = s32[cand[need - 1]], c = s32[cand[need]];
      double den = fmax(fabs(a), fabs(c));
      gap = den > 0 ? fabs(a - c) / den : 0.0;
    }
  }
  int w = 0;
  for (int b = 0; b < nb; ++b)
    if (keep[b]) out[w++] = b;
  while (w < topk) out[w++] = -1;
  free(keep);
  free(cand);
  return gap;
}

/* ---- step 3: sparse GQA attention over the selected blocks --------------
 * For query head h (kv head g = h / (H/G)): keys J = { p <= pos : p / 128 is
 * one of the ids in q2k[g] }; z_p = scale * <q[h], k[key p, g]>;
 * out[h] = sum_p softmax(z)_p v[key p, g]   ([TRT] class description, sparse
 * GQA over the selected blocks; [NEMO] sparse_attention).  No keys -> zeros. */
static void attend_query(const uint16_t* q_row /* [H][D] */,
                         const uint16_t* k /* [rows][G][D] */,
                         const uint16_t* v, const int64_t* key_row, int64_t pos,
                         const int32_t* q2k_g /* q2k_g[g * stride + i] */,
                         int64_t q2k_stride, int topk, double scale,
                         double* out /* [H][D] */) {
  int64_t nkeys_max = (int64_t)topk * OR_BLOCK;
  int64_t* keys = (int64_t*)malloc(sizeof(int64_t) * (size_t)nkeys_max);
  double* z = (double*)malloc(sizeof(double) * (size_t)nkeys_max);
  for (int g = 0; g < OR_KV; ++g) {
    int64_t nk = 0;
    for (int i = 0; i < topk; ++i) {
      int32_t b = q2k_g[g * q2k_stride + i];
      if (b < 0) continue;
      for (int64_t p = (int64_t)b * OR_BLOCK; p < (int64_t)(b + 1) * OR_BLOCK && p <= pos; ++p)
        keys[nk++] = p;
    }
    for (int hh = 0; hh < OR_HEADS / OR_KV; ++hh) {
      int h = g * (OR_HEADS / OR_KV) + hh;
      double* o = out + (int64_t)h * OR_DIM;
      for (int c = 0; c < OR_DIM; ++c) o[c] = 0.0;
      if (nk == 0) continue;
      double zmax = -INFINITY;
      for (int64_t j = 0; j < nk; ++j) {
        int64_t row = key_row[keys[j]];
        double acc = 0.0;
        for (int c = 0; c < OR_DIM; ++c)
          acc += bf16_value(q_row[h * OR_DIM + c]) *
                 bf16_value(k[(row * OR_KV + g) * OR_DIM + c]);
        z[j] = scale * acc;
        if (z[j] > zmax) zmax = z[j];
      }
      double denom = 0.0;
      for (int64_t j = 0; j < nk; ++j) {
        z[j] = exp(z[j] - zmax);
        denom += z[j];
      }
      for (int64_t j = 0; j < nk; ++j) {
        int64_t row = key_row[keys[j]];
        double w = z[j] / denom;
        for (int c = 0; c < OR_DIM; ++c)
          o[c] += w * bf16_value(v[(row * OR_KV + g) * OR_DIM + c]);
      }
    }
  }
  free(keys);
  free(z);
}

/* ---- backward of step 3 --------------------------------------------------
 * [NEMO] _SparseAttention.backward maps grad_out [tokens, 64, 128] to dq
 * [tokens, 64, 128] and dk / dv [tokens, 4, 128].  Written out from the
 * forward above: with z_p = scale <q_h, k_p> over the keys J of query head h,
 * P = softmax(z), out_h = sum_p P_p v_p and dO_h = d loss / d out_h,
 *   dv_p += P_p dO_h,   dP_p = <dO_h, v_p>,   D_h = sum_p P_p dP_p,
 *   dz_p  = P_p (dP_p - D_h),
 *   dq_h += scale sum_p dz_p k_p,   dk_p += scale dz_p q_h.
 * One query token of one kv head; dk / dv of its keys accumulate into the
 * caller's arrays (the caller gives each kv head to one thread). */
static void attend_query_backward(const uint16_t* q_row /* [H][D] */, const uint16_t* dout_row /* [H][D] */,
                                  const uint16_t* k, const uint16_t* v, int64_t start, int64_t pos,
                                  const int32_t* q2k_row /* [topk] for kv head g */, int topk, int g,
                                  double scale, double* dq_row /* [H][D] */,
                                  double* dk /* [T][G][D] */, double* dv /* [T][G][D] */) {
  int64_t nkeys_max = (int64_t)topk * OR_BLOCK;
  int64_t* keys = (int64_t*)malloc(sizeof(int64_t) * (size_t)nkeys_max);
  double* z = (double*)malloc(sizeof(double) * (size_t)nkeys_max);
  double* dp = (double*)malloc(sizeof(double) * (size_t)nkeys_max);
  int64_t nk = 0;
  for (int i = 0; i < topk; ++i) {
    int32_t b = q2k_row[i];
    if (b < 0) continue;
    for (int64_t p = (int64_t)b * OR_BLOCK; p < (int64_t)(b + 1) * OR_BLOCK && p <= pos; ++p) keys[nk++] = start + p;
  }
  for (int hh = 0; hh < OR_HEADS / OR_KV; ++hh) {
    int h = g * (OR_HEADS / OR_KV) + hh;
    double* dqh = dq_row + (int64_t)h * OR_DIM;
    for (int c = 0; c < OR_DIM; ++c) dqh[c] = 0.0;
    if (nk == 0) continue;
    double zmax = -INFINITY;
    for (int64_t j = 0; j < nk; ++j) {
      double acc = 0.0;
      for (int c = 0; c < OR_DIM; ++c)
        acc += bf16_value(q_row[h * OR_DIM + c]) * bf16_value(k[(keys[j] * OR_KV + g) * OR_DIM + c]);
      z[j] = scale * acc;
      if (z[j] > zmax) zmax = z[j];
    }
    double denom = 0.0;
    for (int64_t j = 0; j < nk; ++j) {
      z[j] = exp(z[j] - zmax);
      denom += z[j];
    }
    double D = 0.0;
    for (int64_t j = 0; j < nk; ++j) {
      z[j] /= denom; /* P_p */
      double acc = 0.0;
      for (int c = 0; c < OR_DIM; ++c)
        acc += bf16_value(dout_row[h * OR_DIM + c]) * bf16_value(v[(keys[j] * OR_KV + g) * OR_DIM + c]);
      dp[j] = acc;
      D += z[j] * acc;
    }
    for (int64_t j = 0; j < nk; ++j) {
      double dz = z[j] * (dp[j] - D);
      double* dkp = dk + (keys[j] * OR_KV + g) * OR_DIM;
      double* dvp = dv + (keys[j] * OR_KV + g) * OR_DIM;
      for (int c = 0; c < OR_DIM; ++c) {
        dqh[c] += scale * dz * bf16_value(k[(keys[j] * OR_KV + g) * OR_DIM + c]);
        dkp[c] += scale * dz * bf16_value(q_row[h * OR_DIM + c]);
        dvp[c] += z[j] * bf16_value(dout_row[h * OR_DIM + c]);
      }
    }
  }
  free(keys);
  free(z);
  free(dp);
}

/* ---- geometry ------------------------------------------------------------ */

/* Document of compact token t: the d with cu[d] <= t < cu[d+1]. */
static int doc_of(const int32_t* cu, int num_docs, int64_t t) {
  int lo = 0, hi = num_docs - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) / 2;
    if (cu[mid] <= t)
      lo = mid;
    else
      hi = mid - 1;
  }
  return lo;
}

/* Decode: key position p of request r lives at slot page*128 + p%128 with
 * page = page_table[r][p/128] (paged, [TRT] paged index-K cache parallel to
 * the K/V cache) or at row cu_seqlens_k[r] + p (contiguous). */
static void decode_rows(const int32_t* page_table, const int64_t* cu_k,
                        int max_pages, int r, int64_t len, int64_t* rows) {
  for (int64_t p = 0; p < len; ++p) {
    if (page_table)
      rows[p] = (int64_t)page_table[(int64_t)r * max_pages + p / OR_BLOCK] * OR_BLOCK + p % OR_BLOCK;
    else
      rows[p] = cu_k[r] + p;
  }
}

/* ---- exported drivers ---------------------------------------------------- */

/* Prefill selection for a list of compact query tokens.
 * q2k: [G][n][topk]; gap: [G][n]; s64_out (optional): [n][G][max_nb]. */
int oracle_select_prefill(const void* index_q, const void* index_k, int dtype,
                          const int32_t* cu_seqlens, int num_docs,
                          const int64_t* tokens, int64_t n, int topk, int init,
                          int local, int32_t* q2k, double* gap,
                          double* s64_out, int max_nb) {
  if (topk < 1 || topk > OR_MAXTOPK) return 1;
  int err = 0;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t i = 0; i < n; ++i) {
    int64_t t = tokens[i];
    int d = doc_of(cu_seqlens, num_docs, t);
    int64_t start = cu_seqlens[d];
    int64_t pos = t - start;
    int nb = (int)(pos / OR_BLOCK) + 1;
    int64_t* rows = (int64_t*)malloc(sizeof(int64_t) * (size_t)(pos + 1));
    double* s64 = (double*)malloc(sizeof(double) * OR_KV * (size_t)nb);
    float* s32 = (float*)malloc(sizeof(float) * (size_t)nb);
    for (int64_t p = 0; p <= pos; ++p) rows[p] = start + p;
    const void* iq_row = (dtype == 0) ? (const void*)((const uint16_t*)index_q + t * OR_KV * OR_IDIM)
                                      : (const void*)((const uint8_t*)index_q + t * OR_KV * OR_IDIM);
    block_scores(iq_row, index_k, dtype, rows, pos, nb, s64);
    for (int g = 0; g < OR_KV; ++g) {
      for (int b = 0; b < nb; ++b) s32[b] = (float)s64[g * nb + b];
      gap[g * n + i] = select_row(s32, nb, topk, init, local, q2k + ((int64_t)g * n + i) * topk);
      if (s64_out && nb <= max_nb)
        for (int b = 0; b < nb; ++b) s64_out[(i * OR_KV + g) * max_nb + b] = s64[g * nb + b];
    }
    free(rows);
    free(s64);
    free(s32);
  }
  return err;
}

/* Prefill attention for a list of compact query tokens, given q2k rows for
 * those tokens ([G][n][topk]).  out: [n][H][D] fp64. */
int oracle_attend_prefill(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                          const int32_t* cu_seqlens, int num_docs,
                          const int64_t* tokens, int64_t n, const int32_t* q2k,
                          int topk, double scale, double* out) {
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t i = 0; i < n; ++i) {
    int64_t t = tokens[i];
    int d = doc_of(cu_seqlens, num_docs, t);
    int64_t start = cu_seqlens[d];
    int64_t pos = t - start;
    int64_t* rows = (int64_t*)malloc(sizeof(int64_t) * (size_t)(pos + 1));
    for (int64_t p = 0; p <= pos; ++p) rows[p] = start + p;
    attend_query(q + t * OR_HEADS * OR_DIM, k, v, rows, pos, q2k + i * topk,
                 n * topk, topk, scale, out + i * OR_HEADS * OR_DIM);
    free(rows);
  }
  return 0;
}

/* Prefill attention backward over every compact token: q2k [G][T][topk],
 * grads in fp64: dq [T][H][D], dk and dv [T][G][D] (zeroed here).  One kv head
 * per thread, so the dk / dv sums of a head are formed in one fixed order. */
int oracle_attend_prefill_backward(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                   const uint16_t* dout, const int32_t* cu_seqlens, int num_docs,
                                   int64_t total_tokens, const int32_t* q2k, int topk, double scale,
                                   double* dq, double* dk, double* dv) {
  memset(dk, 0, sizeof(double) * (size_t)(total_tokens * OR_KV * OR_DIM));
  memset(dv, 0, sizeof(double) * (size_t)(total_tokens * OR_KV * OR_DIM));
#pragma omp parallel for schedule(static, 1)
  for (int g = 0; g < OR_KV; ++g) {
    for (int64_t t = 0; t < total_tokens; ++t) {
      int d = doc_of(cu_seqlens, num_docs, t);
      int64_t start = cu_seqlens[d];
      attend_query_backward(q + t * OR_HEADS * OR_DIM, dout + t * OR_HEADS * OR_DIM, k, v, start, t - start,
                            q2k + ((int64_t)g * total_tokens + t) * topk, topk, g, scale,
                            dq + t * OR_HEADS * OR_DIM, dk, dv);
    }
  }
  return 0;
}

/* The forward of step 3 on fp64 inputs (no bf16 rounding), reduced to the
 * scalar loss sum_{t,h,c} out[t][h][c] * dout[t][h][c]: the function whose
 * finite differences pin the backward above.  Arrays are fp64 [T][H][D] and
 * [T][G][D]; q2k [G][T][topk]. */
double oracle_attend_loss_f64(const double* q, const double* k, const double* v, const double* dout,
                              const int32_t* cu_seqlens, int num_docs, int64_t total_tokens,
                              const int32_t* q2k, int topk, double scale) {
  double loss = 0.0;
  int64_t nkeys_max = (int64_t)topk * OR_BLOCK;
  int64_t* keys = (int64_t*)malloc(sizeof(int64_t) * (size_t)nkeys_max);
  double* z = (double*)malloc(sizeof(double) * (size_t)nkeys_max);
  for (int64_t t = 0; t < total_tokens; ++t) {
    int d = doc_of(cu_seqlens, num_docs, t);
    int64_t start = cu_seqlens[d], pos = t - start;
    for (int g = 0; g < OR_KV; ++g) {
      int64_t nk = 0;
      for (int i = 0; i < topk; ++i) {
        int32_t b = q2k[((int64_t)g * total_tokens + t) * topk + i];
        if (b < 0) continue;
        for (int64_t p = (int64_t)b * OR_BLOCK; p < (int64_t)(b + 1) * OR_BLOCK && p <= pos; ++p)
          keys[nk++] = start + p;
      }
      if (nk == 0) continue;
      for (int hh = 0; hh < OR_HEADS / OR_KV; ++hh) {
        int h = g * (OR_HEADS / OR_KV) + hh;
        const double* qh = q + (t * OR_HEADS + h) * OR_DIM;
        double zmax = -INFINITY, denom = 0.0;
        for (int64_t j = 0; j < nk; ++j) {
          double acc = 0.0;
          for (int c = 0; c < OR_DIM; ++c) acc += qh[c] * k[(keys[j] * OR_KV + g) * OR_DIM + c];
          z[j] = scale * acc;
          if (z[j] > zmax) zmax = z[j];
        }
        for (int64_t j = 0; j < nk; ++j) {
          z[j] = exp(z[j] - zmax);
          denom += z[j];
        }
        const double* doh = dout + (t * OR_HEADS + h) * OR_DIM;
        for (int64_t j = 0; j < nk; ++j) {
          double acc = 0.0;
          for (int c = 0; c < OR_DIM; ++c) acc += doh[c] * v[(keys[j] * OR_KV + g) * OR_DIM + c];
          loss += z[j] / denom * acc;
        }
      }
    }
  }
  free(keys);
  free(z);
  return loss;
}

/* ---- MXFP8 emission of the output ----------------------------------------
 * The vLLM page's forward_decode_mxfp8 emits the bf16 output as MXFP8: E4M3
 * values [tokens, H*D] and row-major E8M0 scales [tokens, H*D/32], equal to
 * mxfp8_e4m3_quantize of the bf16 output.  The page does not print that
 * function; this follows the OCP Microscaling (MX) v1.0 definition of an
 * MXFP8 E4M3 block: 32 consecutive elements share the scale
 * X = 2^(floor(log2(amax)) - 8) (8 = the largest E4M3 exponent), stored as the
 * E8M0 byte floor(log2(amax)) - 8 + 127 (clamped to [0, 254]; amax = 0 gives
 * byte 0); each element is v / X rounded to E4M3 (nearest, ties to even),
 * saturated at +-448.  Arithmetic in double is exact here (bf16 inputs, power
 * of two scales). */

/* E4M3 (1 sign, 4 exponent bits with bias 7, 3 mantissa bits, no infinity,
 * 0x7F = NaN, largest finite 448) of y: nearest, ties to even mantissa,
 * saturating. */
static uint8_t e4m3_encode(double y) {
  uint8_t sign = signbit(y) ? 0x80 : 0x00; /* OCP E4M3 keeps the sign of zero */
  double a = fabs(y);
  if (a >= 448.0) return sign | 0x7E;
  int e;
  frexp(a, &e); /* a = m 2^e, m in [0.5, 1): floor(log2 a) = e - 1 */
  int ex = (a == 0.0) ? -7 : e - 1;
  if (ex < -6) ex = -6;                      /* subnormals share the quantum 2^-9 */
  double quantum = ldexp(1.0, ex - 3);       /* 3 mantissa bits */
  double qf = a / quantum;                   /* exact: a is a short binary fraction */
  double fl = floor(qf);
  double rem = qf - fl;
  long long qi = (long long)fl;
  if (rem > 0.5 || (rem == 0.5 && (qi & 1))) qi += 1;
  /* qi in [0, 16]; 16 carries into the next binade */
  if (qi == 0) return sign;
  if (ex == -6 && qi < 8) return sign | (uint8_t)qi; /* subnormal */
  if (qi == 16) {
    qi = 8;
    ex += 1;
  }
  double val = ldexp((double)qi, ex - 3);
  if (val > 448.0) return sign | 0x7E;
  return sign | (uint8_t)(((ex + 7) << 3) | (int)(qi - 8));
}

int oracle_mxfp8_quantize(const uint16_t* bf16, int64_t n, uint8_t* q, uint8_t* scales) {
  if (n % 32) return 1;
  for (int64_t b0 = 0; b0 < n; b0 += 32) {
    double amax = 0.0;
    for (int i = 0; i < 32; ++i) {
      double v = fabs(bf16_value(bf16[b0 + i]));
      if (v > amax) amax = v;
    }
    int sexp = -127;
    if (amax > 0.0) {
      int e;
      frexp(amax, &e);
      sexp = e - 1 - 8;
      if (sexp < -127) sexp = -127;
      if (sexp > 127) sexp = 127;
    }
    scales[b0 / 32] = (uint8_t)(sexp + 127);
    for (int i = 0; i < 32; ++i) q[b0 + i] = e4m3_encode(ldexp(bf16_value(bf16[b0 + i]), -sexp));
  }
  return 0;
}

/* ---- index producer: L2 norm and storage cast ------------------------------
 * [TRT] fuse_qkv_index_projection: MSA batches use a norm / RoPE /
 * cache-insertion producer; [TRT] indexer_kv_dtype: index Q/K are stored
 * "normalized", as bf16 or unscaled E4M3; [NEMO] select_blocks takes index
 * tensors "post norm and RoPE".  The pages fix neither the norm's precision
 * nor its summation order; the reading taken (the workloads' "L2-normalised per
 * vector"): in IEEE binary32, s = sum over c = 0..127 in that order of x_c^2
 * (each square exact in binary32: bf16 has 8 significant bits), r = sqrt(s),
 * y_c = x_c / r (each correctly rounded), then one rounding of y_c to the
 * storage type (bf16 or E4M3, nearest, ties to even).  A vector whose s is 0
 * (all zero, or all squares below binary32's range) is stored as zeros.  RoPE
 * is a rotation, so it leaves the L2 norm unchanged; the pages fix no RoPE
 * variant and none is applied here. */

/* bf16 nearest to the binary32 value f (ties to even): the two bf16 values
 * around f (f with its low 16 bits cleared, and the next one away from zero)
 * and their midpoint, compared in double (all exact). */
static uint16_t bf16_round_from_f32(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  if ((u & 0x7f800000u) == 0x7f800000u) /* inf or NaN: keep the class */
    return (uint16_t)((u >> 16) | ((u & 0xffffu) ? 0x40u : 0u));
  uint32_t lo_bits = u & 0xffff0000u, hi_bits = lo_bits + 0x10000u;
  float lo, hi;
  memcpy(&lo, &lo_bits, sizeof lo);
  memcpy(&hi, &hi_bits, sizeof hi);
  double a = fabs((double)f), mid = 0.5 * (fabs((double)lo) + fabs((double)hi));
  if (a < mid) return (uint16_t)(lo_bits >> 16);
  if (a > mid) return (uint16_t)(hi_bits >> 16);
  return (uint16_t)((((lo_bits >> 16) & 1u) ? hi_bits : lo_bits) >> 16); /* tie: even */
}

/* Normalises n vectors of 128 bf16 values (raw bits) and stores them as bf16
 * bits (dtype 0, out is uint16_t[n][128]) or E4M3 bytes (dtype 1, out is
 * uint8_t[n][128]). */
int oracle_index_normalize(const uint16_t* x, int64_t n, int dtype, void* out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) {
    const uint16_t* xv = x + i * OR_IDIM;
    float s = 0.0f;
    for (int c = 0; c < OR_IDIM; ++c) {
      float v = (float)bf16_value(xv[c]);
      float sq = v * v; /* exact */
      s = s + sq;
    }
    float r = sqrtf(s);
    for (int c = 0; c < OR_IDIM; ++c) {
      float y = (s == 0.0f) ? 0.0f : (float)bf16_value(xv[c]) / r;
      if (dtype == 0)
        ((uint16_t*)out)[i * OR_IDIM + c] = bf16_round_from_f32(y);
      else
        ((uint8_t*)out)[i * OR_IDIM + c] = e4m3_encode((double)y);
    }
  }
  return 0;
}

/* Decode selection for a list of requests.  q2k: [G][n][topk]; gap: [G][n];
 * s64_out (optional): [n][G][max_nb]. */
int oracle_select_decode(const void* index_q, const void* index_k_cache, int dtype,
                         const int32_t* seq_lens, const int32_t* page_table,
                         const int64_t* cu_seqlens_k, int max_pages,
                         const int64_t* requests, int64_t n, int topk, int init,
                         int local, int32_t* q2k, double* gap, double* s64_out,
                         int max_nb) {
  if (topk < 1 || topk > OR_MAXTOPK) return 1;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t i = 0; i < n; ++i) {
    int r = (int)requests[i];
    int64_t len = seq_lens[r];
    int64_t pos = len - 1;
    int nb = (int)(pos / OR_BLOCK) + 1;
    int64_t* rows = (int64_t*)malloc(sizeof(int64_t) * (size_t)len);
    double* s64 = (double*)malloc(sizeof(double) * OR_KV * (size_t)nb);
    float* s32 = (float*)malloc(sizeof(float) * (size_t)nb);
    decode_rows(page_table, cu_seqlens_k, max_pages, r, len, rows);
    const void* iq_row = (dtype == 0) ? (const void*)((const uint16_t*)index_q + (int64_t)r * OR_KV * OR_IDIM)
                                      : (const void*)((const uint8_t*)index_q + (int64_t)r * OR_KV * OR_IDIM);
    block_scores(iq_row, index_k_cache, dtype, rows, pos, nb, s64);
    for (int g = 0; g < OR_KV; ++g) {
      for (int b = 0; b < nb; ++b) s32[b] = (float)s64[g * nb + b];
      gap[g * n + i] = select_row(s32, nb, topk, init, local, q2k + ((int64_t)g * n + i) * topk);
      if (s64_out && nb <= max_nb)
        for (int b = 0; b < nb; ++b) s64_out[(i * OR_KV + g) * max_nb + b] = s64[g * nb + b];
    }
    free(rows);
    free(s64);
    free(s32);
  }
  return 0;
}

/* Decode attention for a list of requests given q2k rows ([G][n][topk]).
 * out: [n][H][D] fp64. */
int oracle_attend_decode(const uint16_t* q, const uint16_t* k_cache,
                         const uint16_t* v_cache, const int32_t* seq_lens,
                         const int32_t* page_table, const int64_t* cu_seqlens_k,
                         int max_pages, const int64_t* requests, int64_t n,
                         const int32_t* q2k, int topk, double scale, double* out) {
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t i = 0; i < n; ++i) {
    int r = (int)requests[i];
    int64_t len = seq_lens[r];
    int64_t* rows = (int64_t*)malloc(sizeof(int64_t) * (size_t)len);
    decode_rows(page_table, cu_seqlens_k, max_pages, r, len, rows);
    attend_query(q + (int64_t)r * OR_HEADS * OR_DIM, k_cache, v_cache, rows, len - 1,
                 q2k + i * topk, n * topk, topk, scale, out + i * OR_HEADS * OR_DIM);
    free(rows);
  }
  return 0;
}

/* Decode attention over an FP8 main K/V cache ([TRT] fuse_qkv_index_projection:
 * the MiniMax-M3 path uses "an FP8 main KV cache").  The pages give no scale
 * rule; the reading taken: K and V are stored as E4M3 bytes and stand for
 * k_scale * e4m3(k) and v_scale * e4m3(v), one fp32 scale per cache (1.0 =
 * unscaled).  Everything else is step 3 above, in fp64. */
static void attend_query_fp8(const uint16_t* q_row, const uint8_t* k, const uint8_t* v, double k_scale,
                             double v_scale, const int64_t* key_row, int64_t pos, const int32_t* q2k_g,
                             int64_t q2k_stride, int topk, double scale, double* out) {
  int64_t nkeys_max = (int64_t)topk * OR_BLOCK;
  int64_t* keys = (int64_t*)malloc(sizeof(int64_t) * (size_t)nkeys_max);
  double* z = (double*)malloc(sizeof(double) * (size_t)nkeys_max);
  for (int g = 0; g < OR_KV; ++g) {
    int64_t nk = 0;
    for (int i = 0; i < topk; ++i) {
      int32_t b = q2k_g[g * q2k_stride + i];
      if (b < 0) continue;
      for (int64_t p = (int64_t)b * OR_BLOCK; p < (int64_t)(b + 1) * OR_BLOCK && p <= pos; ++p) keys[nk++] = p;
    }
    for (int hh = 0; hh < OR_HEADS / OR_KV; ++hh) {
      int h = g * (OR_HEADS / OR_KV) + hh;
      double* o = out + (int64_t)h * OR_DIM;
      for (int c = 0; c < OR_DIM; ++c) o[c] = 0.0;
      if (nk == 0) continue;
      double zmax = -INFINITY;
      for (int64_t j = 0; j < nk; ++j) {
        int64_t row = key_row[keys[j]];
        double acc = 0.0;
        for (int c = 0; c < OR_DIM; ++c)
          acc += bf16_value(q_row[h * OR_DIM + c]) * k_scale * oracle_e4m3_value(k[(row * OR_KV + g) * OR_DIM + c]);
        z[j] = scale * acc;
        if (z[j] > zmax) zmax = z[j];
      }
      double denom = 0.0;
      for (int64_t j = 0; j < nk; ++j) {
        z[j] = exp(z[j] - zmax);
        denom += z[j];
      }
      for (int64_t j = 0; j < nk; ++j) {
        int64_t row = key_row[keys[j]];
        double w = z[j] / denom;
        for (int c = 0; c < OR_DIM; ++c) o[c] += w * v_scale * oracle_e4m3_value(v[(row * OR_KV + g) * OR_DIM + c]);
      }
    }
  }
  free(keys);
  free(z);
}

/* Decode attention over E4M3 K/V caches for a list of requests given q2k rows
 * ([G][n][topk]).  out: [n][H][D] fp64. */
int oracle_attend_decode_fp8(const uint16_t* q, const uint8_t* k_cache, const uint8_t* v_cache, double k_scale,
                             double v_scale, const int32_t* seq_lens, const int32_t* page_table,
                             const int64_t* cu_seqlens_k, int max_pages, const int64_t* requests, int64_t n,
                             const int32_t* q2k, int topk, double scale, double* out) {
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t i = 0; i < n; ++i) {
    int r = (int)requests[i];
    int64_t len = seq_lens[r];
    int64_t* rows = (int64_t*)malloc(sizeof(int64_t) * (size_t)len);
    decode_rows(page_table, cu_seqlens_k, max_pages, r, len, rows);
    attend_query_fp8(q + (int64_t)r * OR_HEADS * OR_DIM, k_cache, v_cache, k_scale, v_scale, rows, len - 1,
                     q2k + i * topk, n * topk, topk, scale, out + i * OR_HEADS * OR_DIM);
    free(rows);
  }
  return 0;
}

/* Packed layout of a document map ([NEMO] layout-from-doc_ids constructor and
 * _contiguous_runs): ids [batch][seq], 0 = padding, each positive id one
 * contiguous run within its row.  Documents are the runs in row-major order;
 * token_rows lists the flat index of every real token in that order.
 * Returns 0 on success, 1 negative id, 2 interrupted document (bad_row set to
 * the flat index where the id reappears), 3 no real token, 4 empty map,
 * 5 coordinates past int32. */
int oracle_pack_metadata(const int64_t* ids, int64_t batch, int64_t seq,
                         int32_t* cu_seqlens /* [batch*seq+1] */,
                         int64_t* token_rows /* [batch*seq] */, int64_t* num_docs,
                         int64_t* total_tokens, int64_t* max_seqlen,
                         int64_t* bad_row) {
  *bad_row = -1;
  if (batch <= 0 || seq <= 0) return 4;
  if (batch * seq > INT32_MAX) return 5;
  for (int64_t i = 0; i < batch * seq; ++i)
    if (ids[i] < 0) {
      *bad_row = i;
      return 1;
    }
  /* interrupted: an id whose run is followed, later in the same row, by
   * another run of the same id */
  for (int64_t r = 0; r < batch; ++r) {
    const int64_t* row = ids + r * seq;
    for (int64_t i = 0; i < seq; ++i) {
      if (row[i] == 0) continue;
      int starts_run = (i == 0) || (row[i - 1] != row[i]);
      if (!starts_run) continue;
      for (int64_t j = 0; j < i; ++j)
        if (row[j] == row[i]) {
          *bad_row = r * seq + i;
          return 2;
        }
    }
  }
  int64_t nd = 0, nt = 0, mx = 0, cur = 0;
  cu_seqlens[0] = 0;
  for (int64_t r = 0; r < batch; ++r) {
    for (int64_t i = 0; i < seq; ++i) {
      int64_t id = ids[r * seq + i];
      if (id == 0) continue;
      int starts_run = (i == 0) || (ids[r * seq + i - 1] != id);
      if (starts_run) {
        if (nd > 0) cu_seqlens[nd] = (int32_t)nt;
        ++nd;
        cur = 0;
      }
      token_rows[nt++] = r * seq + i;
      ++cur;
      if (cur > mx) mx = cur;
    }
  }
  if (nt == 0) return 3;
  cu_seqlens[nd] = (int32_t)nt;
  *num_docs = nd;
  *total_tokens = nt;
  *max_seqlen = mx;
  return 0;
}
