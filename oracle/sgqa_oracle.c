/*
 * sgqa_oracle.c -- plain, slow CPU reference of the Sparse GQA full-attention layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test-suite, the package smoke check and the
 * benchmark's CPU-baseline leg load this library.  The CUDA product path never
 * calls it, links it, or shares a header, helper or constant with it.
 *
 * What it follows (Step 5 Preview pages):
 *   [P1] ai4snews.wisdomeyes.cn news item "Step 5 Preview bets on depth over width",
 *        Interpretation, second paragraph: the indexer keys of adjacent historical
 *        positions are compressed into one representation per block of 8, and a
 *        top-k block selection follows; the selected tokens feed a sparse
 *        flash-attention operator.
 *   [P2] ai.info article "StepFun Details Step 5 Preview's 92-Block Agent Design",
 *        sections "Why StepFun chose 92 transformer blocks" (full attention is Gated
 *        GQA) and "Sparse GQA targets million-token context" (blocks of eight, top-k
 *        of 4,096 tokens = 512 blocks).
 *   [P5] phantomic12 catalog entry "Step 5 Preview": 64 heads in 4 KV groups,
 *        head_dim 192, sparse indexer with topk 512 and proxy_dim 256.
 *
 * Readings where the pages are silent (each is listed with its reason in the design notes):
 *   R1 block compression = element-wise mean of the block's token proxies; a block that
 *      is only partly filled averages the tokens present.
 *   R2 indexer score = plain dot product of the query proxy with the block proxy
 *      (no scale, no activation, one proxy per token per KV group).
 *   R3 the query's own block b_t = floor(t/B) is always kept and is never scored; the
 *      other k-1 slots go to the best strictly-earlier blocks.
 *   R4 order = score descending, ties to the larger block index; -0 equals +0.
 *   R5 causal mask at token level inside the own block (j <= t).
 *   R6 gate is element-wise: out[h,d] = o[h,d] * sigmoid(gate[h,d]) (or per head).
 *
 * Arithmetic: every bf16 input is widened exactly to double; sums and the softmax are
 * taken in double with a two-pass (max, then sum) softmax; the only rounding to bf16
 * is where the method stores a bf16 tensor (the block index), done once, to nearest,
 * ties to even.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct {
  int64_t G;            /* KV groups */
  int64_t Hg;           /* query heads per KV group */
  int64_t D;            /* head dim */
  int64_t P;            /* proxy dim */
  int64_t B;            /* block size (tokens per block) */
  int64_t k;            /* blocks kept per (token, group) */
  double scale;         /* softmax scale applied to q.k */
  int64_t gate_per_dim; /* 1: gate [.., Hg, D]; 0: gate [.., Hg] */
} orc_dims;

/* ---- bf16 <-> double ---------------------------------------------------------------- */

/* bf16 is the upper half of an IEEE binary32; widening is exact. */
double sgqa_oracle_bf16_to_f64(uint16_t h) {
  uint32_t u = ((uint32_t)h) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* Round a double to the nearest bf16 (8 significant bits, binary32 exponent range),
 * ties to even, in ONE rounding step: scale to an integer count of the bf16 quantum
 * at x's binade, round that count with nearbyint (round-half-even in the default
 * mode), scale back.  The result has at most 8 significant bits, so narrowing it to
 * float is exact (or overflows to inf exactly when the rounded value reaches 2^128). */
uint16_t sgqa_oracle_f64_to_bf16(double x) {
  if (isnan(x)) return (uint16_t)0x7fc0;
  if (x == 0.0) return signbit(x) ? (uint16_t)0x8000 : (uint16_t)0;
  int e;
  (void)frexp(fabs(x), &e);   /* |x| in [2^(e-1), 2^e) */
  int lead = e - 1;
  if (lead < -126) lead = -126; /* bf16 subnormals share the quantum 2^-133 */
  double quantum = ldexp(1.0, lead - 7);
  double r = nearbyint(x / quantum) * quantum;
  float f = (float)r;
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  return (uint16_t)(u >> 16);
}

void sgqa_oracle_round_bf16_array(const double* x, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = sgqa_oracle_f64_to_bf16(x[i]);
}

/* ---- O1: block index (R1) ----------------------------------------------------------- */

/* k_blk[g, b, :] = bf16( mean over tokens j in block b present before tok_end of
 * k_proxy[g, j, :] ), for every block b that holds a token of [tok_begin, tok_end). */
int sgqa_oracle_block_index(int64_t G, int64_t P, int64_t B, const uint16_t* k_proxy,
                            int64_t ctx_cap, int64_t tok_begin, int64_t tok_end,
                            uint16_t* k_blk, int64_t nb_cap) {
  if (G <= 0 || P <= 0 || B <= 0 || tok_begin < 0 || tok_end < tok_begin || tok_end > ctx_cap)
    return 1;
  if (tok_end == tok_begin) return 0;
  int64_t b0 = tok_begin / B;
  int64_t b1 = (tok_end + B - 1) / B;
  if (b1 > nb_cap) return 1;
  for (int64_t g = 0; g < G; ++g) {
#pragma omp parallel for schedule(static)
    for (int64_t b = b0; b < b1; ++b) {
      int64_t first = b * B;
      int64_t n = tok_end - first < B ? tok_end - first : B;
      for (int64_t p = 0; p < P; ++p) {
        double sum = 0.0;
        for (int64_t j = 0; j < n; ++j)
          sum += sgqa_oracle_bf16_to_f64(k_proxy[(g * ctx_cap + first + j) * P + p]);
        k_blk[(g * nb_cap + b) * P + p] = sgqa_oracle_f64_to_bf16(sum / (double)n);
      }
    }
  }
  return 0;
}

/* ---- FP8 block-proxy cache (decode variant) ----------------------------------------- */

/* The block proxies can be cached as FP8 E4M3 (1 sign bit, 4 exponent bits with bias 7,
 * 3 mantissa bits; no infinities, code 0x7f/0xff is NaN; largest finite 448 = 1.75 x 2^8,
 * smallest normal 2^-6, subnormals m x 2^-9 for m = 1..7).  The pages deploy the model in
 * FP8 (ai.info article, "Why StepFun chose 92 transformer blocks"); storing the block
 * index this way is a variant of R1, not a step the pages describe. */

/* Exact value of an E4M3 code. */
double sgqa_oracle_e4m3_to_f64(uint8_t c) {
  const int s = c >> 7, E = (c >> 3) & 15, M = c & 7;
  if (E == 15 && M == 7) return NAN;
  double v = E == 0 ? ldexp((double)M, -9) : ldexp(1.0 + M / 8.0, E - 7);
  return s ? -v : v;
}

/* One rounding step from double to E4M3: to nearest, ties to even, finite values beyond
 * the largest code saturating to +-448.  Same construction as the bf16 rounding above:
 * count quanta of x's binade (2^-9 below the normal range), round the count with
 * nearbyint (half to even), then encode the exactly representable result. */
uint8_t sgqa_oracle_f64_to_e4m3(double x) {
  if (isnan(x)) return (uint8_t)0x7f;
  const uint8_t sign = signbit(x) ? (uint8_t)0x80 : (uint8_t)0;
  const double a = fabs(x);
  if (a == 0.0) return sign;
  int e;
  (void)frexp(a, &e); /* a in [2^(e-1), 2^e) */
  int lead = e - 1;
  if (lead < -6) lead = -6;
  const double quantum = ldexp(1.0, lead - 3);
  double r = nearbyint(a / quantum) * quantum;
  if (r > 448.0) r = 448.0;
  if (r == 0.0) return sign;
  if (r < ldexp(1.0, -6)) return (uint8_t)(sign | (uint8_t)(r / ldexp(1.0, -9))); /* subnormal */
  int er;
  (void)frexp(r, &er); /* r in [2^(er-1), 2^er) */
  const int E = er - 1 + 7;
  const int M = (int)((r / ldexp(1.0, er - 1) - 1.0) * 8.0);
  return (uint8_t)(sign | (uint8_t)(E << 3) | (uint8_t)M);
}

void sgqa_oracle_round_e4m3_array(const double* x, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = sgqa_oracle_f64_to_e4m3(x[i]);
}

/* O1 with an E4M3 cache: the same fp64 block mean, rounded once to E4M3. */
int sgqa_oracle_block_index_e4m3(int64_t G, int64_t P, int64_t B, const uint16_t* k_proxy,
                                 int64_t ctx_cap, int64_t tok_begin, int64_t tok_end,
                                 uint8_t* k_blk, int64_t nb_cap) {
  if (G <= 0 || P <= 0 || B <= 0 || tok_begin < 0 || tok_end < tok_begin || tok_end > ctx_cap)
    return 1;
  if (tok_end == tok_begin) return 0;
  int64_t b0 = tok_begin / B;
  int64_t b1 = (tok_end + B - 1) / B;
  if (b1 > nb_cap) return 1;
  for (int64_t g = 0; g < G; ++g) {
#pragma omp parallel for schedule(static)
    for (int64_t b = b0; b < b1; ++b) {
      int64_t first = b * B;
      int64_t n = tok_end - first < B ? tok_end - first : B;
      for (int64_t p = 0; p < P; ++p) {
        double sum = 0.0;
        for (int64_t j = 0; j < n; ++j)
          sum += sgqa_oracle_bf16_to_f64(k_proxy[(g * ctx_cap + first + j) * P + p]);
        k_blk[(g * nb_cap + b) * P + p] = sgqa_oracle_f64_to_e4m3(sum / (double)n);
      }
    }
  }
  return 0;
}

/* ---- O2 + O3: indexer scores and top-k selection (R2, R3, R4) ----------------------- */

typedef struct {
  double score;
  int64_t idx;
} orc_cand;

/* score descending, then index descending.  -0 == +0 because the comparison is on
 * the real value. */
static int cand_cmp(const void* pa, const void* pb) {
  const orc_cand* a = (const orc_cand*)pa;
  const orc_cand* b = (const orc_cand*)pb;
  if (a->score > b->score) return -1;
  if (a->score < b->score) return 1;
  if (a->idx > b->idx) return -1;
  if (a->idx < b->idx) return 1;
  return 0;
}

static int int32_cmp(const void* pa, const void* pb) {
  int32_t a = *(const int32_t*)pa, b = *(const int32_t*)pb;
  return (a > b) - (a < b);
}

/* Score of one query proxy against one block proxy: plain dot product in double. */
static double proxy_dot(const uint16_t* qp, const uint16_t* kb, int64_t P) {
  double s = 0.0;
  for (int64_t p = 0; p < P; ++p) s += sgqa_oracle_bf16_to_f64(qp[p]) * sgqa_oracle_bf16_to_f64(kb[p]);
  return s;
}

/* For each requested row r = (token position pos[r], group grp[r]) with query proxy
 * qp_rows[r, :]:
 *   candidates = blocks 0 .. b_t-1 with b_t = pos / B (strictly earlier blocks)
 *   keep the first k-1 of them in (score desc, index desc) order, add b_t,
 *   return them sorted ascending in sel_idx[r, 0..cnt-1]; the rest of the row is -1.
 * scores_out (optional, [n_rows, max_cand]) receives the candidate scores by index. */
int sgqa_oracle_select(const orc_dims* d, int64_t n_rows, const int64_t* pos, const int32_t* grp,
                       const uint16_t* qp_rows, const uint16_t* k_blk, int64_t nb_cap,
                       int32_t* sel_idx, int32_t* sel_cnt, double* scores_out, int64_t max_cand) {
  if (!d || d->k < 1 || d->B < 1) return 1;
  int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
  for (int64_t r = 0; r < n_rows; ++r) {
    int64_t bt = pos[r] / d->B;
    int64_t g = grp[r];
    if (bt >= nb_cap || g < 0 || g >= d->G) {
      bad = 1;
      continue;
    }
    orc_cand* c = (orc_cand*)malloc(sizeof(orc_cand) * (size_t)(bt > 0 ? bt : 1));
    for (int64_t b = 0; b < bt; ++b) {
      c[b].score = proxy_dot(qp_rows + r * d->P, k_blk + (g * nb_cap + b) * d->P, d->P);
      c[b].idx = b;
      if (scores_out && b < max_cand) scores_out[r * max_cand + b] = c[b].score;
    }
    qsort(c, (size_t)bt, sizeof(orc_cand), cand_cmp);
    int64_t take = bt < d->k - 1 ? bt : d->k - 1;
    int32_t* out = sel_idx + r * d->k;
    for (int64_t i = 0; i < take; ++i) out[i] = (int32_t)c[i].idx;
    out[take] = (int32_t)bt;
    qsort(out, (size_t)(take + 1), sizeof(int32_t), int32_cmp);
    for (int64_t i = take + 1; i < d->k; ++i) out[i] = -1;
    sel_cnt[r] = (int32_t)(take + 1);
    free(c);
  }
  return bad;
}

/* ---- O4 + O5: gated attention over the selected tokens (R5, R6) --------------------- */

static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

/* For each row r = (pos[r], grp[r]) and each of its Hg heads h:
 *   tokens J = { j in blocks sel_idx[r, 0..cnt-1] : j <= pos }   (dense_mode: all j <= pos)
 *   s_j = scale * q[h] . K[g, kv_off + j]
 *   p_j = exp(s_j - max s) / sum exp(s - max s)             (two passes, double)
 *   o   = sum_j p_j V[g, kv_off + j]
 *   out[r, h, :] = o * sigmoid(gate)
 *   lse[r, h]    = max s + log sum exp(s - max s)
 *   coverage[r, h] (optional) = sum over j in J of the DENSE causal softmax weight of j,
 *                               computed from scratch over all j <= pos.
 * K, V are [G, ctx_cap, D]; kv_off (optional, per row) offsets a packed cache. */
int sgqa_oracle_attention(const orc_dims* d, int64_t n_rows, const int64_t* pos, const int32_t* grp,
                          const int64_t* kv_off, const uint16_t* q_rows, const uint16_t* gate_rows,
                          const uint16_t* K, const uint16_t* V, int64_t ctx_cap,
                          const int32_t* sel_idx, const int32_t* sel_cnt, int32_t dense_mode,
                          double* out, double* lse, double* coverage) {
  if (!d || d->D <= 0 || d->Hg <= 0) return 1;
  const int64_t D = d->D, Hg = d->Hg, B = d->B;
  int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
  for (int64_t r = 0; r < n_rows; ++r) {
    const int64_t t = pos[r];
    const int64_t g = grp[r];
    const int64_t off = kv_off ? kv_off[r] : 0;
    if (g < 0 || g >= d->G || t < 0 || off + t >= ctx_cap) {
      bad = 1;
      continue;
    }
    /* the attended token list */
    int64_t cap = dense_mode ? t + 1 : (int64_t)sel_cnt[r] * B;
    int64_t* J = (int64_t*)malloc(sizeof(int64_t) * (size_t)(cap > 0 ? cap : 1));
    int64_t nJ = 0;
    if (dense_mode) {
      for (int64_t j = 0; j <= t; ++j) J[nJ++] = j;
    } else {
      for (int64_t i = 0; i < sel_cnt[r]; ++i) {
        int64_t b = sel_idx[r * d->k + i];
        for (int64_t j = b * B; j < b * B + B; ++j)
          if (j <= t) J[nJ++] = j;
      }
    }
    double* s = (double*)malloc(sizeof(double) * (size_t)(t + 1));
    double* o = (double*)malloc(sizeof(double) * (size_t)D);
    for (int64_t h = 0; h < Hg; ++h) {
      const uint16_t* q = q_rows + (r * Hg + h) * D;
      /* scores over the attended tokens */
      double m = -INFINITY;
      for (int64_t i = 0; i < nJ; ++i) {
        const uint16_t* kr = K + (g * ctx_cap + off + J[i]) * D;
        double acc = 0.0;
        for (int64_t e = 0; e < D; ++e) acc += sgqa_oracle_bf16_to_f64(q[e]) * sgqa_oracle_bf16_to_f64(kr[e]);
        s[i] = d->scale * acc;
        if (s[i] > m) m = s[i];
      }
      double l = 0.0;
      for (int64_t i = 0; i < nJ; ++i) l += exp(s[i] - m);
      for (int64_t e = 0; e < D; ++e) o[e] = 0.0;
      for (int64_t i = 0; i < nJ; ++i) {
        double p = exp(s[i] - m) / l;
        const uint16_t* vr = V + (g * ctx_cap + off + J[i]) * D;
        for (int64_t e = 0; e < D; ++e) o[e] += p * sgqa_oracle_bf16_to_f64(vr[e]);
      }
      for (int64_t e = 0; e < D; ++e) {
        double gt = d->gate_per_dim ? sgqa_oracle_bf16_to_f64(gate_rows[(r * Hg + h) * D + e])
                                    : sgqa_oracle_bf16_to_f64(gate_rows[r * Hg + h]);
        out[(r * Hg + h) * D + e] = o[e] * sigmoid(gt);
      }
      if (lse) lse[r * Hg + h] = m + log(l);
      if (coverage) {
        /* dense causal softmax over all j <= t, from scratch */
        double md = -INFINITY;
        for (int64_t j = 0; j <= t; ++j) {
          const uint16_t* kr = K + (g * ctx_cap + off + j) * D;
          double acc = 0.0;
          for (int64_t e = 0; e < D; ++e) acc += sgqa_oracle_bf16_to_f64(q[e]) * sgqa_oracle_bf16_to_f64(kr[e]);
          s[j] = d->scale * acc;
          if (s[j] > md) md = s[j];
        }
        double ld = 0.0;
        for (int64_t j = 0; j <= t; ++j) ld += exp(s[j] - md);
        double mass = 0.0;
        for (int64_t i = 0; i < nJ; ++i) mass += exp(s[J[i]] - md) / ld;
        coverage[r * Hg + h] = mass;
      }
    }
    free(o);
    free(s);
    free(J);
  }
  return bad;
}

int sgqa_oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
