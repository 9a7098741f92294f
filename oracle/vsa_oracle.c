/*
 * vsa_oracle.c -- plain fp64 CPU oracle for block-sparse attention forward.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite, the smoke
 * check in __graft_entry__ and the CPU-baseline leg of bench.py may load or
 * call this library.  It shares no code, header, table or constant with the
 * CUDA path in block_sparse_attention_vsa_gb300/; the two meet only in the
 * seeded input arrays.
 *
 * What it computes (the definition, not an algorithm for speed):
 *
 *   1. The block selection of every query block is materialised as a
 *      0/1 block mask.
 *        - VSA: the per-query-block look-up table q2k_idx[row, slot] with
 *          q2k_num[row] valid slots ("TheRock rocke sparse_attention.py",
 *          module docstring, VSA bullet; "FastVideo
 *          block_sparse_attn_sm100a.py", is_supported docstring, q2k_num /
 *          q2k_idx bullets).  Slots at or past the count are padding and
 *          are never read.  The table is a SET: scattering the same block
 *          twice sets the same byte ("TheRock rocke sparse_attention.py",
 *          _stage_vsa_bitmap_to_lds, idempotent scatter).  Counts are
 *          clamped to [0, max_kv] and entries outside [0, nb) are skipped.
 *        - Jenga: the caller's i8 MaskBitmap[q_block, k_block]; any nonzero
 *          byte means "attend" ("TheRock rocke sparse_attention.py", module
 *          docstring, Jenga bullet, and _lds_bitmap_predicate).
 *   2. The token mask: query row i (q-block qb = i / block) may attend key
 *      j (k-block kb = j / block) iff blockmask[qb][kb] != 0 and
 *      (j mod block) < variable_block_sizes[kb] -- keys at or past a
 *      block's valid count are masked ("FastVideo
 *      block_sparse_attn_sm100a.py", is_supported docstring,
 *      variable_block_sizes bullet).
 *   3. Masked dense softmax attention in fp64 on the exact bf16 input
 *      values, two passes over the attended keys in ascending j:
 *        s_j  = scale * sum_d q[i,d] k[j,d]
 *        m    = max_j s_j,   l = sum_j exp(s_j - m)
 *        out  = sum_j exp(s_j - m) v[j,:] / l
 *        lse  = log2( sum_j exp(s_j) ) = (m + ln l) / ln 2
 *      The LSE is base 2, "max(qk*qk_scale) + log2(l)" with
 *      qk_scale = scale*log2(e) ("FastVideo block_sparse_attn_sm100a.py",
 *      module docstring).  A masked key contributes exp(-inf) = 0, so
 *      skipping it is the same as including it ("TheRock rocke
 *      sparse_attention.py", module docstring, "forces the score ... to
 *      -inf").
 *   4. A row with no attended key (count 0, or every selected block has
 *      variable_block_sizes 0) gets out = +0.0 exactly and
 *      lse = ORACLE_LSE_EMPTY, a finite sentinel (-FLT_MAX) ("FastVideo
 *      block_sparse_attn_sm100a.py", is_supported docstring, "Rows with
 *      count 0 produce exactly-zero output rows (and a finite LSE
 *      sentinel)"; the value -FLT_MAX is this library's reading).
 *
 * Grouped-query and cross-length attention ("TheRock rocke sparse_attention.py",
 * JengaSparseSpec / VsaSparseSpec: separate seqlen_q / seqlen_k and query / key-value
 * head counts, kv_head_idx): q is [B, Hq, Sq, D], k and v are [B, Hkv, Sk, D] with Hq a
 * multiple of Hkv; query head h reads key/value head h / (Hq / Hkv); query blocks are
 * Sq / block, key blocks Sk / block, and the block mask is [Sq/block, Sk/block].
 *
 * Metadata conversions (bit-exact references for the device converters):
 *   - LUT -> bitmap: step 1 above written as i8 0/1.
 *   - bitmap -> LUT: ascending compaction of the nonzero bytes of a row,
 *     the first min(count, max_kv) kept, the rest of the row padded
 *     with -1, count = min(count, max_kv) (the inverse of step 1 for rows
 *     that fit).
 *
 * Inputs q, k, v are bf16 bit patterns (uint16); a bf16 value is the top
 * half of an IEEE binary32, so the widening to double below is exact.
 *
 * Parity pins for every function here live in tests/test_oracle_pins.py.
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_LSE_EMPTY (-(double)FLT_MAX)

/* exact bf16 -> double: place the 16 bits in the high half of a binary32 */
static double bf16_to_double(uint16_t bits) {
  uint32_t w = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &w, sizeof f);
  return (double)f;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Step 1 (VSA): LUT rows -> 0/1 block mask.  rows = number of LUT rows
 * (B*H*nb for a per-head table), each row max_kv slots wide. */
void oracle_lut_to_blockmask(const int32_t *q2k_idx, const int32_t *q2k_num,
                             int64_t rows, int max_kv, int nb, int8_t *mask) {
  for (int64_t r = 0; r < rows; ++r) {
    int8_t *mrow = mask + r * (int64_t)nb;
    for (int kb = 0; kb < nb; ++kb) mrow[kb] = 0;
    int n = q2k_num[r];
    if (n < 0) n = 0;
    if (n > max_kv) n = max_kv;
    for (int s = 0; s < n; ++s) {
      int kb = q2k_idx[r * (int64_t)max_kv + s];
      if (kb >= 0 && kb < nb) mrow[kb] = 1;
    }
  }
}

/* bitmap -> LUT: ascending compaction of the nonzero bytes of each row. */
void oracle_blockmask_to_lut(const int8_t *mask, int64_t rows, int nb,
                             int max_kv, int32_t *q2k_idx, int32_t *q2k_num) {
  for (int64_t r = 0; r < rows; ++r) {
    const int8_t *mrow = mask + r * (int64_t)nb;
    int32_t *irow = q2k_idx + r * (int64_t)max_kv;
    int n = 0;
    for (int kb = 0; kb < nb; ++kb) {
      if (mrow[kb] != 0) {
        if (n < max_kv) irow[n] = kb;
        ++n;
      }
    }
    if (n > max_kv) n = max_kv;
    for (int s = n; s < max_kv; ++s) irow[s] = -1;
    q2k_num[r] = n;
  }
}

/* Steps 2-4 for a list of query blocks.
 *
 *   q           bf16 bits, [B, Hq, Sq, D] contiguous.
 *   k, v        bf16 bits, [B, Hkv, Sk, D] contiguous; Hq a multiple of Hkv.
 *   blockmask   int8 0/1 (any nonzero = attend), [*, nbq, nbk] with
 *               nbq = Sq / block, nbk = Sk / block: entry (b, h) starts at
 *               b*mask_stride_b + h*mask_stride_h (strides in units of
 *               nbq*nbk; both 0 = one mask shared by every batch and head,
 *               as for the Jenga bitmap).
 *   vbs         int32 [nbk] valid key counts per k-block, or NULL = block.
 *   sel         int32 triples (b, h, qb), n_sel of them: the query blocks
 *               to compute.
 *   out         double [n_sel, block, D];  lse double [n_sel, block].
 */
void oracle_masked_attention(const uint16_t *q, const uint16_t *k,
                             const uint16_t *v, int B, int Hq, int Hkv, int Sq,
                             int Sk, int D, const int8_t *blockmask,
                             int64_t mask_stride_b, int64_t mask_stride_h,
                             int block, const int32_t *vbs, double scale,
                             const int32_t *sel, int64_t n_sel, double *out,
                             double *lse) {
  (void)B;
  const int nbq = Sq / block, nbk = Sk / block;
  const int group = Hq / Hkv;
#pragma omp parallel
  {
    double *s_buf = (double *)malloc(sizeof(double) * (size_t)Sk);
    int32_t *j_buf = (int32_t *)malloc(sizeof(int32_t) * (size_t)Sk);
    double *qrow = (double *)malloc(sizeof(double) * (size_t)D);
    double *acc = (double *)malloc(sizeof(double) * (size_t)D);
#pragma omp for schedule(dynamic, 1)
    for (int64_t t = 0; t < n_sel; ++t) {
      const int b = sel[3 * t + 0], h = sel[3 * t + 1], qb = sel[3 * t + 2];
      const int64_t bh = (int64_t)b * Hq + h;
      const int64_t bkv = (int64_t)b * Hkv + h / group;
      const uint16_t *qh = q + bh * Sq * (int64_t)D;
      const uint16_t *kh = k + bkv * Sk * (int64_t)D;
      const uint16_t *vh = v + bkv * Sk * (int64_t)D;
      const int8_t *mrow = blockmask +
                           (b * mask_stride_b + h * mask_stride_h) *
                               (int64_t)nbq * nbk +
                           (int64_t)qb * nbk;
      for (int r = 0; r < block; ++r) {
        const int i = qb * block + r;
        double *orow = out + (t * block + r) * (int64_t)D;
        for (int d = 0; d < D; ++d) qrow[d] = bf16_to_double(qh[(int64_t)i * D + d]);
        /* pass 1: the attended set (token mask, ascending j) and its scores */
        int64_t n_att = 0;
        for (int j = 0; j < Sk; ++j) {
          const int kb = j / block;
          const int valid = vbs ? vbs[kb] : block;
          if (mrow[kb] == 0 || (j % block) >= valid) continue;
          double dot = 0.0;
          for (int d = 0; d < D; ++d)
            dot += qrow[d] * bf16_to_double(kh[(int64_t)j * D + d]);
          s_buf[n_att] = scale * dot;
          j_buf[n_att] = j;
          ++n_att;
        }
        if (n_att == 0) {
          for (int d = 0; d < D; ++d) orow[d] = 0.0;
          lse[t * block + r] = ORACLE_LSE_EMPTY;
          continue;
        }
        double m = s_buf[0];
        for (int64_t a = 1; a < n_att; ++a)
          if (s_buf[a] > m) m = s_buf[a];
        /* pass 2: normaliser and weighted sum of V */
        double l = 0.0;
        for (int d = 0; d < D; ++d) acc[d] = 0.0;
        for (int64_t a = 0; a < n_att; ++a) {
          const double p = exp(s_buf[a] - m);
          l += p;
          const uint16_t *vr = vh + (int64_t)j_buf[a] * D;
          for (int d = 0; d < D; ++d) acc[d] += p * bf16_to_double(vr[d]);
        }
        for (int d = 0; d < D; ++d) orow[d] = acc[d] / l;
        lse[t * block + r] = (m + log(l)) / log(2.0);
      }
    }
    free(s_buf);
    free(j_buf);
    free(qrow);
    free(acc);
  }
}

/* Backward of steps 2-4 (the gradient of the forward above with respect to q, k and v,
 * given the gradient dout of out).  The pages name the backward only ("FastVideo
 * block_sparse_attn_sm100a.py", module docstring: the Triton backward consumes the
 * forward's lse); the definition is the textbook gradient of softmax attention,
 * restricted to the attended keys A_i of row i:
 *
 *   s_ij  = scale * q_i . k_j,      p_ij = exp(s_ij - L_i)  (L_i = ln sum_j exp s_ij)
 *   dp_ij = dout_i . v_j,           D_i  = sum_{j in A_i} p_ij dp_ij  (= dout_i . out_i)
 *   ds_ij = p_ij (dp_ij - D_i)
 *   dq_i  = scale * sum_j ds_ij k_j
 *   dk_j  = scale * sum_i ds_ij q_i          (over every row i attending j, every
 *   dv_j  =         sum_i p_ij dout_i         query head of j's key/value group)
 *
 * Rows with no attended key contribute nothing and get dq = 0.  Shapes as
 * oracle_masked_attention; dout [B, Hq, Sq, D] bf16 bits; every (b, h, query block) is
 * computed.  dq [B, Hq, Sq, D], dk and dv [B, Hkv, Sk, D], double, overwritten.
 */
void oracle_masked_attention_bwd(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                                 const uint16_t *dout, int B, int Hq, int Hkv, int Sq,
                                 int Sk, int D, const int8_t *blockmask,
                                 int64_t mask_stride_b, int64_t mask_stride_h, int block,
                                 const int32_t *vbs, double scale, double *dq, double *dk,
                                 double *dv) {
  const int nbq = Sq / block, nbk = Sk / block;
  const int group = Hq / Hkv;
  memset(dq, 0, sizeof(double) * (size_t)B * Hq * Sq * D);
  memset(dk, 0, sizeof(double) * (size_t)B * Hkv * Sk * D);
  memset(dv, 0, sizeof(double) * (size_t)B * Hkv * Sk * D);
  /* parallel over key/value heads: each owns its dk, dv and its group's dq rows */
#pragma omp parallel
  {
    double *s_buf = (double *)malloc(sizeof(double) * (size_t)Sk);
    double *dp_buf = (double *)malloc(sizeof(double) * (size_t)Sk);
    int32_t *j_buf = (int32_t *)malloc(sizeof(int32_t) * (size_t)Sk);
    double *qrow = (double *)malloc(sizeof(double) * (size_t)D);
    double *drow = (double *)malloc(sizeof(double) * (size_t)D);
#pragma omp for schedule(dynamic, 1)
    for (int64_t bkv = 0; bkv < (int64_t)B * Hkv; ++bkv) {
      const int b = (int)(bkv / Hkv), hk = (int)(bkv % Hkv);
      const uint16_t *kh = k + bkv * Sk * (int64_t)D;
      const uint16_t *vh = v + bkv * Sk * (int64_t)D;
      double *dkh = dk + bkv * Sk * (int64_t)D;
      double *dvh = dv + bkv * Sk * (int64_t)D;
      for (int h = hk * group; h < (hk + 1) * group; ++h) {
        const int64_t bh = (int64_t)b * Hq + h;
        const uint16_t *qh = q + bh * Sq * (int64_t)D;
        const uint16_t *doh = dout + bh * Sq * (int64_t)D;
        double *dqh = dq + bh * Sq * (int64_t)D;
        for (int i = 0; i < Sq; ++i) {
          const int qb = i / block;
          const int8_t *mrow = blockmask +
                               (b * mask_stride_b + h * mask_stride_h) *
                                   (int64_t)nbq * nbk +
                               (int64_t)qb * nbk;
          for (int d = 0; d < D; ++d) {
            qrow[d] = bf16_to_double(qh[(int64_t)i * D + d]);
            drow[d] = bf16_to_double(doh[(int64_t)i * D + d]);
          }
          int64_t n_att = 0;
          for (int j = 0; j < Sk; ++j) {
            const int kb = j / block;
            const int valid = vbs ? vbs[kb] : block;
            if (mrow[kb] == 0 || (j % block) >= valid) continue;
            double dot = 0.0, dpd = 0.0;
            for (int d = 0; d < D; ++d) {
              dot += qrow[d] * bf16_to_double(kh[(int64_t)j * D + d]);
              dpd += drow[d] * bf16_to_double(vh[(int64_t)j * D + d]);
            }
            s_buf[n_att] = scale * dot;
            dp_buf[n_att] = dpd;
            j_buf[n_att] = j;
            ++n_att;
          }
          if (n_att == 0) continue;
          double m = s_buf[0];
          for (int64_t a = 1; a < n_att; ++a)
            if (s_buf[a] > m) m = s_buf[a];
          double l = 0.0;
          for (int64_t a = 0; a < n_att; ++a) l += exp(s_buf[a] - m);
          double Di = 0.0;
          for (int64_t a = 0; a < n_att; ++a) {
            s_buf[a] = exp(s_buf[a] - m) / l; /* now p_ij */
            Di += s_buf[a] * dp_buf[a];
          }
          for (int64_t a = 0; a < n_att; ++a) {
            const double p = s_buf[a];
            const double ds = p * (dp_buf[a] - Di);
            const int64_t j = j_buf[a];
            for (int d = 0; d < D; ++d) {
              const double kd = bf16_to_double(kh[j * D + d]);
              dqh[(int64_t)i * D + d] += scale * ds * kd;
              dkh[j * D + d] += scale * ds * qrow[d];
              dvh[j * D + d] += p * drow[d];
            }
          }
        }
      }
    }
    free(s_buf);
    free(dp_buf);
    free(j_buf);
    free(qrow);
    free(drow);
  }
}
