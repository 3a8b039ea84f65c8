/*
 * mxfa_oracle.c -- plain, slow, obviously-correct CPU oracle for MXFP8
 * block-scaled attention (forward and backward), the MX quantizer and the
 * fused RMSNorm+Quantize producer.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark may load this library.  It shares no code,
 * header, table or constant generator with the CUDA path.
 *
 * Arithmetic is fp64 throughout, except mxo_rmsnorm_quant, which follows the
 * fp32 operation order that the fused kernel documents (there the fp32 result
 * y decides every code, and the pages fix no other precision for it).  The
 * attention functions are the plain fp64 definitions of the method.
 *
 * Sources (each function cites the passage it follows):
 *  [MX]  "Low-Precision FlashAttention-4: End-to-End Block-Scaled Attention on
 *        Blackwell" (kongchang.com), section "Why MXFP8": OCP MX format,
 *        32-element blocks, one shared 8-bit power-of-two (E8M0) scale,
 *        E4M3 payload.
 *  [BITS] "MXFP8 FlashAttention-4 Hits 2.85 Petaflops in Meta's Production
 *        Training" (andresseo.expert), section "Inside the TMEM Bargain and
 *        Zero-Gather Jagged Pipeline": P converted online in 32-element blocks,
 *        scale by bit extraction (no logarithm, no division); row maximum
 *        reused for the scale; square 32x32 blocks for Q, K and dO in the
 *        backward pass; dS quantized once per square block.
 *  [KDIM] "Meta's MXFP8 FlashAttention-4 kernel, tackling TMEM scale-factor
 *        constraints, hits up to 1.6x over BF16" (theclarity.today), paragraph
 *        3: scales along the MMA K dimension (D for Q and K, N for V);
 *        paragraph 1: softmax in FP32, only then is P converted.
 *  [RMS] same andresseo.expert page, same section, and "Meta's FlashAttention-4
 *        Achieves 2.85 PF/s with MXFP8 on Blackwell GPUs" (brifing.si) item 7:
 *        fused RMSNorm+Quantize emitting FP8 with dual scale layouts.
 *  [BWD] kongchang.com page, section "Hardware Adaptation for Blackwell":
 *        backward recomputes the forward intermediates (P) instead of storing.
 *
 * Readings where the pages are silent (listed again in the design notes):
 *  - scale exponent = floor(log2(amax)) - 8 (E4M3 emax), clamped to the E8M0
 *    range [0, 254]; elements then round to nearest-even and saturate at 448;
 *  - a block holding a NaN or an Inf gets scale 0xFF and NaN payloads 0x7F;
 *  - P below 2^-126 is flushed to zero (fp32 flush-to-zero of the exponential);
 *  - fp32 row sum of the unquantized P;
 *  - backward P quantized in 1x32 blocks along queries (the dV contraction),
 *    dS in 32x32 blocks; tau applied after the contraction;
 *  - backward P = exp(min(S tau - lse, 0)): exact attention never exceeds 1,
 *    and the square-block scores can exceed the forward's lse.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define MXO_ROW 0 /* 1x32 along the last (column) dimension          */
#define MXO_COL 1 /* 32x1 along rows (tokens), anchored per segment  */
#define MXO_SQ 2  /* 32x32, anchored per segment in rows             */

/* ------------------------------------------------------------------ */
/* E4M3 and E8M0 codecs ([MX])                                         */
/* ------------------------------------------------------------------ */

/* Value of an E4M3 code: sign bit 7, exponent bits 6..3 (bias 7),
 * mantissa bits 2..0; exponent field 0 is subnormal (m * 2^-9);
 * 0x7F / 0xFF are NaN; there is no infinity. */
double mxo_e4m3_decode(uint8_t c) {
  int sign = (c >> 7) & 1;
  int e = (c >> 3) & 0xF;
  int m = c & 7;
  double v;
  if (e == 0xF && m == 7) return NAN;
  if (e == 0)
    v = ldexp((double)m, -9);
  else
    v = ldexp(1.0 + m / 8.0, e - 7);
  return sign ? -v : v;
}

/* Round a real value to E4M3: nearest, ties to even, saturating to +-448;
 * NaN -> 0x7F.  The sign of a zero result is kept. */
uint8_t mxo_e4m3_encode(double y) {
  if (isnan(y)) return 0x7F;
  uint8_t sign = signbit(y) ? 0x80 : 0x00;
  double a = fabs(y);
  if (a >= 448.0) return sign | 0x7E;
  if (a == 0.0) return sign;
  int ex;
  frexp(a, &ex);     /* a = f * 2^ex with f in [0.5, 1) */
  int E = ex - 1;    /* floor(log2 a) */
  if (E < -6) E = -6; /* subnormal binade shares the 2^-9 quantum */
  double quantum = ldexp(1.0, E - 3);
  double n = rint(a / quantum); /* default rounding mode: nearest-even */
  double v = n * quantum;
  if (v == 0.0) return sign;
  if (v > 448.0) v = 448.0; /* cannot happen for a < 448; kept for clarity */
  if (v < ldexp(1.0, -6)) return sign | (uint8_t)(int)(v / ldexp(1.0, -9));
  frexp(v, &ex);
  int E2 = ex - 1;
  int m3 = (int)((v / ldexp(1.0, E2) - 1.0) * 8.0);
  return sign | (uint8_t)(((E2 + 7) << 3) | m3);
}

/* Shared block scale from the block's absolute maximum: the exponent of
 * amax minus the largest E4M3 exponent (8), biased by 127 ([MX], [BITS]). */
uint8_t mxo_e8m0_from_amax(double amax) {
  if (isnan(amax) || isinf(amax)) return 0xFF;
  if (amax == 0.0) return 0;
  int ex;
  frexp(amax, &ex);
  int b = (ex - 1) - 8 + 127;
  if (b < 0) b = 0;
  if (b > 254) b = 254;
  return (uint8_t)b;
}

double mxo_e8m0_decode(uint8_t s) {
  if (s == 0xFF) return NAN;
  return ldexp(1.0, (int)s - 127);
}

/* Quantize one block of n values read with stride `vs`, writing n payload
 * codes with stride `qs` and returning the scale byte. */
static uint8_t quant_block(const double* v, int64_t n, int64_t vs, uint8_t* q,
                           int64_t qs) {
  double amax = 0.0;
  int bad = 0;
  for (int64_t i = 0; i < n; i++) {
    double a = fabs(v[i * vs]);
    if (isnan(a) || isinf(a)) bad = 1;
    else if (a > amax) amax = a;
  }
  if (bad) {
    for (int64_t i = 0; i < n; i++) q[i * qs] = 0x7F;
    return 0xFF;
  }
  uint8_t s = mxo_e8m0_from_amax(amax);
  int X = (int)s - 127;
  for (int64_t i = 0; i < n; i++) q[i * qs] = mxo_e4m3_encode(ldexp(v[i * vs], -X));
  return s;
}

/* Number of 32-row blocks before segment `g`, i.e. the compact row offset of
 * that segment's column/square scale rows. */
static int64_t seg_block_offset(const int32_t* cu, int g) {
  int64_t off = 0;
  for (int i = 0; i < g; i++) off += (cu[i + 1] - cu[i] + 31) / 32;
  return off;
}

/* Quantize x[rows][cols] (fp64 values) to E4M3 payload q[rows][cols] and
 * compact E8M0 scales ([MX], block orientation per [KDIM] and [BITS]):
 *   ROW: sf[rows][cols/32]                 1x32 along columns
 *   COL: sf[sum ceil(len/32)][cols]        32x1 along rows, per segment
 *   SQ : sf[sum ceil(len/32)][cols/32]     32x32, per segment
 * Segments are rows [cu[g], cu[g+1]); a trailing partial block takes its
 * maximum over the rows it holds.  cols must be a multiple of 32. */
void mxo_quantize(const double* x, int64_t rows, int64_t cols, int mode,
                  const int32_t* cu, int nseg, uint8_t* q, uint8_t* sf) {
  if (mode == MXO_ROW) {
    int64_t nb = cols / 32;
    for (int64_t r = 0; r < rows; r++)
      for (int64_t b = 0; b < nb; b++)
        sf[r * nb + b] = quant_block(x + r * cols + b * 32, 32, 1,
                                     q + r * cols + b * 32, 1);
    return;
  }
  for (int g = 0; g < nseg; g++) {
    int64_t r0 = cu[g], len = cu[g + 1] - cu[g];
    int64_t boff = seg_block_offset(cu, g);
    for (int64_t rb = 0; rb * 32 < len; rb++) {
      int64_t rs = r0 + rb * 32;
      int64_t nr = len - rb * 32 < 32 ? len - rb * 32 : 32;
      if (mode == MXO_COL) {
        for (int64_t c = 0; c < cols; c++)
          sf[(boff + rb) * cols + c] =
              quant_block(x + rs * cols + c, nr, cols, q + rs * cols + c, cols);
      } else { /* MXO_SQ: one scale for the nr x 32 block */
        int64_t nb = cols / 32;
        for (int64_t cb = 0; cb < nb; cb++) {
          double amax = 0.0;
          int bad = 0;
          for (int64_t i = 0; i < nr; i++)
            for (int64_t j = 0; j < 32; j++) {
              double a = fabs(x[(rs + i) * cols + cb * 32 + j]);
              if (isnan(a) || isinf(a)) bad = 1;
              else if (a > amax) amax = a;
            }
          uint8_t s = bad ? 0xFF : mxo_e8m0_from_amax(amax);
          int X = (int)s - 127;
          for (int64_t i = 0; i < nr; i++)
            for (int64_t j = 0; j < 32; j++) {
              int64_t idx = (rs + i) * cols + cb * 32 + j;
              q[idx] = bad ? 0x7F : mxo_e4m3_encode(ldexp(x[idx], -X));
            }
          sf[(boff + rb) * nb + cb] = s;
        }
      }
    }
  }
}

/* Dequantize: value = e4m3(q) * 2^(sf - 127), same layouts as mxo_quantize. */
void mxo_dequantize(const uint8_t* q, const uint8_t* sf, int64_t rows,
                    int64_t cols, int mode, const int32_t* cu, int nseg,
                    double* x) {
  if (mode == MXO_ROW) {
    int64_t nb = cols / 32;
    for (int64_t r = 0; r < rows; r++)
      for (int64_t c = 0; c < cols; c++)
        x[r * cols + c] = mxo_e4m3_decode(q[r * cols + c]) *
                          mxo_e8m0_decode(sf[r * nb + c / 32]);
    return;
  }
  for (int g = 0; g < nseg; g++) {
    int64_t r0 = cu[g], len = cu[g + 1] - cu[g];
    int64_t boff = seg_block_offset(cu, g);
    for (int64_t i = 0; i < len; i++) {
      int64_t r = r0 + i, rb = boff + i / 32;
      for (int64_t c = 0; c < cols; c++) {
        uint8_t s = mode == MXO_COL ? sf[rb * cols + c] : sf[rb * (cols / 32) + c / 32];
        x[r * cols + c] = mxo_e4m3_decode(q[r * cols + c]) * mxo_e8m0_decode(s);
      }
    }
  }
}

/* Quantize-dequantize one block of fp64 values in place (used for P and dS
 * inside the attention oracle).  Values below 2^-126 in magnitude have
 * already been flushed by the caller where the method says so. */
static void qdq_block(double* v, int64_t n, int64_t vs) {
  double amax = 0.0;
  for (int64_t i = 0; i < n; i++) {
    double a = fabs(v[i * vs]);
    if (a > amax) amax = a;
  }
  uint8_t s = mxo_e8m0_from_amax(amax);
  int X = (int)s - 127;
  for (int64_t i = 0; i < n; i++)
    v[i * vs] = mxo_e4m3_decode(mxo_e4m3_encode(ldexp(v[i * vs], -X))) * ldexp(1.0, X);
}

/* Quantize-dequantize a block with a given shared exponent X (the constant
 * scale mode of P: "Meta's FlashAttention-4 Achieves 2.85 PF/s with MXFP8
 * on Blackwell GPUs", item 4, constant scaling of softmax outputs). */
static void qdq_block_fixed(double* v, int64_t n, int64_t vs, int X) {
  for (int64_t i = 0; i < n; i++)
    v[i * vs] = mxo_e4m3_decode(mxo_e4m3_encode(ldexp(v[i * vs], -X))) * ldexp(1.0, X);
}

static double flush_fp32_subnormal(double p) {
  return p < ldexp(1.0, -126) ? 0.0 : p;
}

/* ------------------------------------------------------------------ */
/* Attention forward ([KDIM] paragraphs 1-2, [BITS])                   */
/* ------------------------------------------------------------------ */

/* Tensors are token-major: x[token][head][d].  Sequence g holds query tokens
 * [cu_q[g], cu_q[g+1]) and key tokens [cu_k[g], cu_k[g+1]).  q, k, v are the
 * dequantized MXFP8 operands.  For each query row the keys are visited in
 * tiles of tile_n (a multiple of 32), in ascending order, with an online
 * (running-max) softmax in base 2:
 *   s'  = (q.k) * scale * log2(e)        (-inf where masked)
 *   m_t = max over the tile; candidate m_n = max(m, m_t)
 *   the running max moves to m_n when m = -inf or m_n - m > lazy_thr
 *   (lazy_thr = 0: exact rescale at every increase)
 *   O, l *= 2^(m_old - m);  P~ = 2^(s' - m);  l += sum P~ (unquantized)
 *   P~ quantized per 32-key block of the tile (when quant_p), then O += P^ V.
 * p_scale = 1 replaces each block's own scale by one constant shared exponent
 * X = ceil(lazy_thr) - 8, so the largest possible P~ = 2^ceil(lazy_thr) maps
 * to 256 (constant scaling of softmax outputs, item 4 of the brifing.si page).
 * End: O /= l;  lse = (m + log2 l) * ln 2 (natural log); with no visible key
 * (an empty key sequence) O = 0 and lse = -inf.
 * causal masks key index > query index within a sequence (equal lengths).
 * lse layout: lse[head][query token]. */
void mxo_attn_fwd(const double* q, const double* k, const double* v,
                  const int32_t* cu_q, const int32_t* cu_k, int nseq, int H,
                  int D, double scale, int causal, int quant_p, int tile_n,
                  double lazy_thr, double* o, double* lse, int64_t total_q, int p_scale) {
  const int Xc = (int)ceil(lazy_thr) - 8;
  const double log2e = 1.4426950408889634074;
  const double ln2 = 0.69314718055994530942;
  /* rows (query token, head) are independent: one parallel loop over them */
  int32_t* seq_of = (int32_t*)malloc(sizeof(int32_t) * (size_t)(total_q > 0 ? total_q : 1));
  for (int g = 0; g < nseq; g++)
    for (int64_t t = cu_q[g]; t < cu_q[g + 1]; t++) seq_of[t] = g;
#pragma omp parallel
  {
    double* sp = (double*)malloc(sizeof(double) * (size_t)tile_n);
    double* acc = (double*)malloc(sizeof(double) * (size_t)D);
#pragma omp for schedule(dynamic, 16)
    for (int64_t w = 0; w < total_q * H; w++) {
      {
        const int64_t tok = w / H;
        const int h = (int)(w % H);
        const int g = seq_of[tok];
        int64_t q0 = cu_q[g];
        int64_t k0 = cu_k[g], lk = cu_k[g + 1] - cu_k[g];
        const int64_t i = tok - q0;
        const double* qi = q + ((q0 + i) * H + h) * D;
        double m = -INFINITY, l = 0.0;
        for (int d = 0; d < D; d++) acc[d] = 0.0;
        int64_t kend = causal ? (i + 1 < lk ? i + 1 : lk) : lk;
        for (int64_t t0 = 0; t0 < kend; t0 += tile_n) {
          int64_t nt = kend - t0 < tile_n ? kend - t0 : tile_n;
          double mt = -INFINITY;
          for (int64_t j = 0; j < tile_n; j++) {
            if (j < nt) {
              const double* kj = k + ((k0 + t0 + j) * H + h) * D;
              double s = 0.0;
              for (int d = 0; d < D; d++) s += qi[d] * kj[d];
              sp[j] = s * scale * log2e;
              if (sp[j] > mt) mt = sp[j];
            } else {
              sp[j] = -INFINITY;
            }
          }
          double mn = mt > m ? mt : m;
          double mu = (m == -INFINITY || mn - m > lazy_thr) ? mn : m;
          double alpha = (m == -INFINITY) ? 0.0 : exp2(m - mu);
          for (int d = 0; d < D; d++) acc[d] *= alpha;
          l *= alpha;
          m = mu;
          for (int64_t j = 0; j < tile_n; j++) {
            sp[j] = sp[j] == -INFINITY ? 0.0 : flush_fp32_subnormal(exp2(sp[j] - m));
            l += sp[j];
          }
          if (quant_p)
            for (int64_t b = 0; b < tile_n; b += 32) {
              if (p_scale)
                qdq_block_fixed(sp + b, 32, 1, Xc);
              else
                qdq_block(sp + b, 32, 1);
            }
          for (int64_t j = 0; j < nt; j++) {
            if (sp[j] == 0.0) continue;
            const double* vj = v + ((k0 + t0 + j) * H + h) * D;
            for (int d = 0; d < D; d++) acc[d] += sp[j] * vj[d];
          }
        }
        /* a query with no key to attend to (an empty key sequence): the
         * softmax sum is empty, so O = 0 and lse = log 0 = -inf */
        double* oi = o + ((q0 + i) * H + h) * D;
        for (int d = 0; d < D; d++) oi[d] = l > 0.0 ? acc[d] / l : 0.0;
        lse[(int64_t)h * total_q + q0 + i] = l > 0.0 ? (m + log2(l)) * ln2 : -INFINITY;
      }
    }
    free(sp);
    free(acc);
  }
  free(seq_of);
}

/* ------------------------------------------------------------------ */
/* Attention backward ([BITS], [BWD])                                  */
/* ------------------------------------------------------------------ */

/* q, k, dO are the dequantized square-block operands, v the dequantized
 * row-block operand; o_bf is the bf16 O and do_bf the dO that enters Delta
 * (the method passes the dequantized square-block dO, the one that also
 * enters dP; as fp64 values);
 * lse[head][query token] from the forward pass.  Per sequence and head:
 *   Delta_i = sum_d dO_bf[i,d] * O_bf[i,d]
 *   P_ij = exp(min(q_i.k_j * scale - lse_i, 0))   (0 where masked; < 2^-126 -> 0)
 *   The min keeps P <= 1, the bound exact attention obeys: the square-block
 *   operands recompute S differently from the forward's row-block operands,
 *   and with outliers S * scale can exceed the forward's lse by hundreds.
 *   dP_ij = dO_i.v_j;   dS_ij = P_ij (dP_ij - Delta_i)
 *   P^ : P quantized in 1x32 blocks along queries (per key), quant_p
 *   dS^: dS quantized in 32x32 blocks, quant_ds
 *   (blocks anchored at the sequence start in both dimensions)
 *   dV_j = sum_i P^_ij dO_i;  dK_j = scale sum_i dS^_ij q_i;
 *   dQ_i = scale sum_j dS^_ij k_j.
 * p_scale = 1: P^ takes the constant shared exponent -8 (P <= 1 maps to
 * <= 256) instead of each block's own. */
void mxo_attn_bwd(const double* q, const double* k, const double* v,
                  const double* dO, const double* o_bf, const double* do_bf,
                  const double* lse, const int32_t* cu_q, const int32_t* cu_k,
                  int nseq, int H, int D, double scale, int causal, int quant_p,
                  int quant_ds, double* dq, double* dk, double* dv,
                  int64_t total_q, int p_scale) {
  /* heads in turn; inside a head, independent rows / columns / blocks run in
   * parallel (every element keeps its own summation order) */
  for (int g = 0; g < nseq; g++) {
    for (int h = 0; h < H; h++) {
      int64_t q0 = cu_q[g], lq = cu_q[g + 1] - cu_q[g];
      int64_t k0 = cu_k[g], lk = cu_k[g + 1] - cu_k[g];
      double* P = (double*)calloc((size_t)(lq * lk > 0 ? lq * lk : 1), sizeof(double));
      double* dS = (double*)calloc((size_t)(lq * lk > 0 ? lq * lk : 1), sizeof(double));
#pragma omp parallel for schedule(dynamic, 8)
      for (int64_t i = 0; i < lq; i++) {
        const double* qi = q + ((q0 + i) * H + h) * D;
        const double* doi = dO + ((q0 + i) * H + h) * D;
        double delta = 0.0;
        for (int d = 0; d < D; d++)
          delta += do_bf[((q0 + i) * H + h) * D + d] * o_bf[((q0 + i) * H + h) * D + d];
        double li = lse[(int64_t)h * total_q + q0 + i];
        for (int64_t j = 0; j < lk; j++) {
          if (causal && j > i) continue;
          const double* kj = k + ((k0 + j) * H + h) * D;
          const double* vj = v + ((k0 + j) * H + h) * D;
          double s = 0.0, dp = 0.0;
          for (int d = 0; d < D; d++) {
            s += qi[d] * kj[d];
            dp += doi[d] * vj[d];
          }
          double p = flush_fp32_subnormal(exp(fmin(s * scale - li, 0.0)));
          P[i * lk + j] = p;
          dS[i * lk + j] = p * (dp - delta);
        }
      }
      if (quant_p) { /* 1x32 along queries, for every key column */
#pragma omp parallel for schedule(static)
        for (int64_t j = 0; j < lk; j++)
          for (int64_t ib = 0; ib < lq; ib += 32) {
            if (p_scale)
              qdq_block_fixed(P + ib * lk + j, lq - ib < 32 ? lq - ib : 32, lk, -8);
            else
              qdq_block(P + ib * lk + j, lq - ib < 32 ? lq - ib : 32, lk);
          }
      }
      if (quant_ds) /* 32x32 square blocks */
#pragma omp parallel for schedule(static)
        for (int64_t ib = 0; ib < lq; ib += 32)
          for (int64_t jb = 0; jb < lk; jb += 32) {
            int64_t ni = lq - ib < 32 ? lq - ib : 32, nj = lk - jb < 32 ? lk - jb : 32;
            double amax = 0.0;
            for (int64_t i = 0; i < ni; i++)
              for (int64_t j = 0; j < nj; j++) {
                double a = fabs(dS[(ib + i) * lk + jb + j]);
                if (a > amax) amax = a;
              }
            int X = (int)mxo_e8m0_from_amax(amax) - 127;
            for (int64_t i = 0; i < ni; i++)
              for (int64_t j = 0; j < nj; j++) {
                double* e = &dS[(ib + i) * lk + jb + j];
                *e = mxo_e4m3_decode(mxo_e4m3_encode(ldexp(*e, -X))) * ldexp(1.0, X);
              }
          }
#pragma omp parallel for schedule(dynamic, 8)
      for (int64_t j = 0; j < lk; j++) {
        double* dvj = dv + ((k0 + j) * H + h) * D;
        double* dkj = dk + ((k0 + j) * H + h) * D;
        for (int d = 0; d < D; d++) dvj[d] = dkj[d] = 0.0;
        for (int64_t i = 0; i < lq; i++) {
          double p = P[i * lk + j], ds = dS[i * lk + j];
          const double* doi = dO + ((q0 + i) * H + h) * D;
          const double* qi = q + ((q0 + i) * H + h) * D;
          for (int d = 0; d < D; d++) {
            dvj[d] += p * doi[d];
            dkj[d] += ds * qi[d];
          }
        }
        for (int d = 0; d < D; d++) dkj[d] *= scale;
      }
#pragma omp parallel for schedule(dynamic, 8)
      for (int64_t i = 0; i < lq; i++) {
        double* dqi = dq + ((q0 + i) * H + h) * D;
        for (int d = 0; d < D; d++) dqi[d] = 0.0;
        for (int64_t j = 0; j < lk; j++) {
          double ds = dS[i * lk + j];
          if (ds == 0.0) continue;
          const double* kj = k + ((k0 + j) * H + h) * D;
          for (int d = 0; d < D; d++) dqi[d] += ds * kj[d];
        }
        for (int d = 0; d < D; d++) dqi[d] *= scale;
      }
      free(P);
      free(dS);
    }
  }
}

/* ------------------------------------------------------------------ */
/* Fused RMSNorm + Quantize ([RMS])                                    */
/* ------------------------------------------------------------------ */

/* Sum of squares of one row in the fused kernel's documented fp32 order:
 * lane l (0..31) owns columns 8l + 256k + j (j = 0..7, k = 0..C/256-1) and
 * adds their squares sequentially, k outer and j inner; lanes then combine
 * by the butterfly s_l <- s_l + s_(l xor w) for w = 16, 8, 4, 2, 1.  Every
 * operation rounds to nearest (no fused multiply-add). */
static float rms_row_sumsq(const float* x, int64_t C) {
  float lane[32];
  for (int l = 0; l < 32; l++) {
    float s = 0.0f;
    for (int64_t kk = 0; kk < C / 256; kk++)
      for (int j = 0; j < 8; j++) {
        volatile float xv = x[8 * l + 256 * kk + j];
        volatile float sq = xv * xv;
        s = s + sq;
      }
    lane[l] = s;
  }
  for (int w = 16; w >= 1; w >>= 1) {
    float nxt[32];
    for (int l = 0; l < 32; l++) {
      volatile float t = lane[l] + lane[l ^ w];
      nxt[l] = t;
    }
    memcpy(lane, nxt, sizeof lane);
  }
  return lane[0];
}

/* y[t][c] = (x[t][c] * r_t) * gamma[c] with r_t = 1 / sqrt(mean_t + eps),
 * mean_t = sumsq_t / C, each step one correctly rounded fp32 operation; then
 * y is quantized ROW (1x32 along C), COL (32x1 along T) and/or SQ (32x32),
 * with row blocks anchored at every multiple of seg_len (out_mask bit 0 =
 * ROW, bit 1 = COL, bit 2 = SQ; outputs for unset bits may be NULL).
 * x holds the bf16 inputs as fp32 values.  y_out (nullable) receives y. */
void mxo_rmsnorm_quant(const float* x, const float* gamma, int64_t T, int64_t C,
                       float eps, int out_mask, int32_t seg_len, uint8_t* q_row,
                       uint8_t* sf_row, uint8_t* q_col, uint8_t* sf_col,
                       uint8_t* q_sq, uint8_t* sf_sq, float* y_out) {
  double* y = (double*)malloc(sizeof(double) * (size_t)(T * C));
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < T; t++) {
    const float* xr = x + t * C;
    float ss = rms_row_sumsq(xr, C);
    volatile float mean = ss / (float)C;
    volatile float me = mean + eps;
    volatile float sd = sqrtf(me);
    volatile float r = 1.0f / sd;
    for (int64_t c = 0; c < C; c++) {
      volatile float a = xr[c] * r;
      volatile float b = a * gamma[c];
      y[t * C + c] = (double)b;
      if (y_out) y_out[t * C + c] = b;
    }
  }
  int nseg = (int)((T + seg_len - 1) / seg_len);
  int32_t* cu = (int32_t*)malloc(sizeof(int32_t) * (size_t)(nseg + 1));
  for (int g = 0; g <= nseg; g++) cu[g] = (int32_t)((int64_t)g * seg_len < T ? (int64_t)g * seg_len : T);
  if (out_mask & 1) mxo_quantize(y, T, C, MXO_ROW, cu, nseg, q_row, sf_row);
  if (out_mask & 2) mxo_quantize(y, T, C, MXO_COL, cu, nseg, q_col, sf_col);
  if (out_mask & 4) mxo_quantize(y, T, C, MXO_SQ, cu, nseg, q_sq, sf_sq);
  free(cu);
  free(y);
}

/* ------------------------------------------------------------------ */
/* Lower-precision element formats (MXFP6, MXFP4, NVFP4): the formats the */
/* pages name as the next step ("Meta's FlashAttention-4 Achieves 2.85   */
/* PF/s with MXFP8 on Blackwell GPUs", item 12; "Meta's MXFP8             */
/* FlashAttention-4 kernel ...", paragraph 1: Blackwell's block-scaled   */
/* MMA runs MXFP8, MXFP6, MXFP4 and NVFP4).  The element formats follow  */
/* the OCP MX definitions: E2M1 (bias 1, max 6), E2M3 (bias 1, max 7.5), */
/* E3M2 (bias 3, max 28); no Inf or NaN codes, subnormals at exponent 0. */
/* ------------------------------------------------------------------ */

#define MXO_E2M1 0
#define MXO_E2M3 1
#define MXO_E3M2 2

static void fmt_params(int fmt, int* ebits, int* mbits, int* bias) {
  if (fmt == MXO_E2M1) { *ebits = 2; *mbits = 1; *bias = 1; }
  else if (fmt == MXO_E2M3) { *ebits = 2; *mbits = 3; *bias = 1; }
  else { *ebits = 3; *mbits = 2; *bias = 3; }
}

/* Value of a code of `fmt` (sign bit above the exponent and mantissa). */
double mxo_fp_decode(int fmt, uint8_t c) {
  int eb, mb, bias;
  fmt_params(fmt, &eb, &mb, &bias);
  int sign = (c >> (eb + mb)) & 1;
  int e = (c >> mb) & ((1 << eb) - 1);
  int m = c & ((1 << mb) - 1);
  double v = e == 0 ? ldexp((double)m, 1 - bias - mb) : ldexp(1.0 + (double)m / (1 << mb), e - bias);
  return sign ? -v : v;
}

/* Largest finite value of `fmt`. */
double mxo_fp_max(int fmt) {
  int eb, mb, bias;
  fmt_params(fmt, &eb, &mb, &bias);
  return ldexp(2.0 - ldexp(1.0, -mb), (1 << eb) - 1 - bias);
}

/* Round to `fmt`: nearest, ties to even code, saturating at the maximum
 * (OCP MX conversion with saturation); NaN -> the maximum (these formats
 * have no NaN; NaN blocks are marked by the scale instead). */
uint8_t mxo_fp_encode(int fmt, double y) {
  int eb, mb, bias;
  fmt_params(fmt, &eb, &mb, &bias);
  uint8_t sign = (!isnan(y) && signbit(y)) ? (uint8_t)(1 << (eb + mb)) : 0;
  double a = isnan(y) ? mxo_fp_max(fmt) : fabs(y);
  if (a >= mxo_fp_max(fmt)) a = mxo_fp_max(fmt);
  /* exhaustive search over the non-negative codes: the nearest value, ties
   * to the even code (codes are ordered by value) */
  int best = 0;
  double bd = INFINITY;
  for (int c = 0; c < (1 << (eb + mb)); c++) {
    double d = fabs(mxo_fp_decode(fmt, (uint8_t)c) - a);
    if (d < bd || (d == bd && (c & 1) == 0)) {
      bd = d;
      best = c;
    }
  }
  return sign | (uint8_t)best;
}

/* Largest exponent of `fmt` (emax): floor(log2 of its maximum). */
static int fp_emax(int fmt) {
  int eb, mb, bias;
  fmt_params(fmt, &eb, &mb, &bias);
  return (1 << eb) - 1 - bias;
}

/* MX quantization of x[rows][cols] in 1x32 blocks along the columns with
 * element format fmt: E8M0 scale from floor(log2 amax) - emax(fmt) clamped
 * to [0, 254] (the OCP rule, as for E4M3), elements rounded to fmt.  Codes
 * one per byte (unpacked); a block holding NaN or Inf gets scale 0xFF and
 * code 0. */
void mxo_quantize_mx(const double* x, int64_t rows, int64_t cols, int fmt, uint8_t* q, uint8_t* sf) {
  int64_t nb = cols / 32;
  for (int64_t r = 0; r < rows; r++)
    for (int64_t b = 0; b < nb; b++) {
      const double* v = x + r * cols + b * 32;
      double amax = 0.0;
      int bad = 0;
      for (int i = 0; i < 32; i++) {
        double a = fabs(v[i]);
        if (isnan(a) || isinf(a)) bad = 1;
        else if (a > amax) amax = a;
      }
      uint8_t* qq = q + r * cols + b * 32;
      if (bad) {
        sf[r * nb + b] = 0xFF;
        for (int i = 0; i < 32; i++) qq[i] = 0;
        continue;
      }
      int s = 0;
      if (amax > 0.0) {
        int ex;
        frexp(amax, &ex);
        s = (ex - 1) - fp_emax(fmt) + 127;
        if (s < 0) s = 0;
        if (s > 254) s = 254;
      }
      sf[r * nb + b] = (uint8_t)s;
      for (int i = 0; i < 32; i++) qq[i] = mxo_fp_encode(fmt, ldexp(v[i], 127 - s));
    }
}

/* NVFP4 quantization of x[rows][cols] (reading: the recipe the format is
 * published with): one fp32 tensor scale st = amax(|x|) / (448 * 6) (1 if
 * the tensor is all zero), per 16 columns an E4M3 block scale
 * sb = E4M3(amax_block / (6 st)) (nearest-even, saturating), and E2M1
 * elements x / (sb st) (0 where sb = 0).  Returns st. */
double mxo_quantize_nvfp4(const double* x, int64_t rows, int64_t cols, uint8_t* q, uint8_t* sf) {
  /* the scales are decided in fp32, each step one correctly rounded fp32
   * operation (x holds bf16 values, exact in fp32) */
  float amax = 0.0f;
  for (int64_t i = 0; i < rows * cols; i++)
    if ((float)fabs(x[i]) > amax) amax = (float)fabs(x[i]);
  volatile float st = 1.0f;
  if (amax > 0.0f) st = amax / 2688.0f; /* 448 * 6 */
  volatile float d6 = 6.0f * st;
  int64_t nb = cols / 16;
  for (int64_t r = 0; r < rows; r++)
    for (int64_t b = 0; b < nb; b++) {
      const double* v = x + r * cols + b * 16;
      float bm = 0.0f;
      for (int i = 0; i < 16; i++)
        if ((float)fabs(v[i]) > bm) bm = (float)fabs(v[i]);
      volatile float ratio = bm / d6;
      uint8_t code = mxo_e4m3_encode((double)ratio);
      sf[r * nb + b] = code;
      volatile float sbv = (float)mxo_e4m3_decode(code) * st;
      uint8_t* qq = q + r * cols + b * 16;
      for (int i = 0; i < 16; i++) {
        volatile float e = (float)v[i] / sbv;
        qq[i] = sbv > 0.0f ? mxo_fp_encode(MXO_E2M1, (double)e) : 0;
      }
    }
  return (double)st;
}

/* ------------------------------------------------------------------ */
/* Projection GEMM ([RMS]: GEMM+Quantize; the quantization of Y is      */
/* mxo_quantize, applied by the caller to the result)                   */
/* ------------------------------------------------------------------ */

/* y[m][n] = sum_k a[m][k] * b[n][k] in fp64 (a [M][K], b [N][K] row-major:
 * a weight stored [out][in], as a projection layer holds it). */
void mxo_gemm_nt(const double* a, const double* b, int64_t M, int64_t N, int64_t K, double* y) {
#pragma omp parallel for schedule(static)
  for (int64_t m = 0; m < M; m++)
    for (int64_t n = 0; n < N; n++) {
      double s = 0.0;
      for (int64_t k = 0; k < K; k++) s += a[m * K + k] * b[n * K + k];
      y[m * N + n] = s;
    }
}

int mxo_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Host threads the oracle uses from now on (timing runs; results do not
 * depend on it: every output element keeps its own summation order). */
void mxo_set_num_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}
