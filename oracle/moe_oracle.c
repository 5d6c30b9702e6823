/*
 * moe_oracle.c -- plain, slow, obviously-correct CPU oracle of the single-GPU
 * MoE layer path: group-limited top-k router, dispatch permutation, SwiGLU
 * expert FFN, weighted combine.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
 * baseline of the benchmark may load this library.  It shares no code,
 * header, table or constant with the CUDA path, and it never calls into it.
 *
 * Sources (web pages on the MoE dispatch/combine path):
 *   [ch15]   "第十五章：多节点大模型推理", section 4.1 (gating picks top-k
 *            logical experts), section 4.3 (assignment counts n_e, R_imbalance,
 *            capacity), section 3.4 (dispatch/combine volume T*k*H*b).
 *   [par02]  "推理INFRA方法论-02-parallelism", MoE-TP/EP comparison (gate_up
 *            fused expert GEMM, masked layout, M_e = B_local*P*k/E).
 *   [trace]  token trace through TP/CP/SP/EP/DP/PP, hop 4 "dispatch to two
 *            experts": y = p5*E5(x) + p27*E27(x).
 *   [ep]     "ep-deploy" handbook page, section "EPLB 与路由约束": 256 experts in
 *            8 groups, group score = sum of the group's two best scores, keep
 *            4 groups, pick 8 experts inside them.
 *
 * Readings where the pages are silent (each is also listed in the design
 * notes):
 *   R1  router logits are fp32 sums of exact bf16*bf16 products in a fixed
 *       order: "lane" l in [0,32) owns every i with (i/8) mod 32 == l and sums
 *       its products in increasing i from +0; the 32 lane sums are combined by
 *       the xor butterfly (offsets 16,8,4,2,1).
 *   R2  exp is a Cody-Waite reduction (ln2 split in a 16-bit head and a tail)
 *       followed by a degree-7 Taylor polynomial with coefficients 1/j!
 *       rounded to fp32, evaluated by fused multiply-add Horner steps, then an
 *       exact scaling by 2^n.  sigma(l) = 1 / (1 + exp(-l)), IEEE division.
 *   R3  selection score s' = sigma(l) + fl(bias_scale * b)   (sigmoid router)
 *       or s' = l                                          (softmax router;
 *       softmax is monotone so top-k over logits equals top-k over softmax).
 *   R4  group score = sum of the two largest s' of the group (fp32 sum in the
 *       fp32 router; fp64 for the fp64 routing simulation of [ep]).
 *   R5  keep the topk_group best groups, ties to the lower group index.
 *   R6  top-k experts among kept groups, ties to the lower expert index,
 *       output in descending score order.
 *   R7  sigmoid weights: sigma of the chosen experts (no bias) divided by
 *       their sequential fp32 sum; softmax weights: exp(l_j - l_0) divided by
 *       the sequential fp32 sum (the renormalised top-k of softmax).
 *   R8  dispatch is a stable counting sort of the flat assignments a = t*k+j.
 *   R9  expert FFN: h = silu(x.Wg) * (x.Wu), y = h.Wd, accumulated in fp64.
 *   R10 combine: y[t] = sum_j w[t,j] * y_perm[dest[t*k+j]], j ascending.
 *   R13 FP8: e4m3 codes with fp32 block scales, one per (row, 128 columns)
 *       of an activation and per 128 x 128 block of a weight; each scale is
 *       a power of two, s = 2^e with e the smallest integer >= -127 such
 *       that amax <= 448 * 2^e (1 for an all-zero block, 2^127 when amax is
 *       not finite), q = round-to-nearest-even e4m3 of x / s (exact: s is a
 *       power of two), saturating at 448.
 *   R11 capacity: the first C assignments of an expert in increasing
 *       a = t*k + j keep their place; later ones overflow.  Dropped ones add
 *       nothing (weights are not renormalised); second-round ones are
 *       computed like any other.
 *   R15 replicas: the r-th assignment (in increasing a) of logical expert e,
 *       which has n_rep copies, goes to copy r mod n_rep in the order the
 *       placement lists them (the least loaded copy, ties to the first,
 *       when copies fill in that order); rows are contiguous per physical
 *       copy in placement order, stable in a.
 *
 * Compile with -O2 -ffp-contract=off, no fast-math, so that every floating
 * point operation is exactly the one written.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------ */
/* bf16 helpers                                                              */
/* ------------------------------------------------------------------------ */

static float bf16_value(uint16_t h) {
  uint32_t u = ((uint32_t)h) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* round-to-nearest-even fp32 -> bf16 (finite inputs) */
static uint16_t bf16_round(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7FFFu + lsb;
  return (uint16_t)(u >> 16);
}

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

void oracle_set_num_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

/* ------------------------------------------------------------------------ */
/* R1: router logits, canonical fp32 order                                   */
/* ------------------------------------------------------------------------ */

/*
 * logits[t*E+e] = sum_i x[t,i] * w_r[i,e]  ([trace] hop 4: the router scores
 * every expert from the token's hidden state; [ch15] 4.1 gating).
 * x: [T,d] bf16, w_r: [d,E] bf16.  Order per reading R1.
 */
void oracle_router_logits(const uint16_t *x, const uint16_t *w_r, int T, int d,
                          int E, float *logits) {
  /* w_r widened to fp32 once (exact) */
  float *wf = (float *)malloc(sizeof(float) * (size_t)d * E);
  for (size_t q = 0; q < (size_t)d * E; ++q) wf[q] = bf16_value(w_r[q]);
#pragma omp parallel
  {
    /* lane[l*E + e]: partial sum of lane l for expert e */
    float *lane = (float *)malloc(sizeof(float) * 32 * (size_t)E);
#pragma omp for schedule(dynamic, 4)
    for (int t = 0; t < T; ++t) {
      for (int q = 0; q < 32 * E; ++q) lane[q] = 0.0f;
      for (int i = 0; i < d; ++i) {
        int l = (i / 8) % 32;
        float xi = bf16_value(x[(size_t)t * d + i]);
        const float *wrow = wf + (size_t)i * E;
        float *acc = lane + (size_t)l * E;
        for (int e = 0; e < E; ++e) {
          float prod = xi * wrow[e]; /* exact: 8-bit x 8-bit significands */
          acc[e] = acc[e] + prod;
        }
      }
      for (int e = 0; e < E; ++e) {
        float a[32], b[32];
        for (int l = 0; l < 32; ++l) a[l] = lane[(size_t)l * E + e];
        for (int off = 16; off >= 1; off /= 2) {
          for (int l = 0; l < 32; ++l) b[l] = a[l] + a[l ^ off];
          for (int l = 0; l < 32; ++l) a[l] = b[l];
        }
        logits[(size_t)t * E + e] = a[0];
      }
    }
    free(lane);
  }
  free(wf);
}

/* ------------------------------------------------------------------------ */
/* R2: exp and sigmoid                                                       */
/* ------------------------------------------------------------------------ */

/* ln 2 = LN2_HEAD + LN2_TAIL; the head keeps 16 significant bits of fl(ln 2)
 * (low 8 stored bits cleared) so that n * LN2_HEAD is exact for |n| < 256. */
static const float LN2_HEAD = 0x1.62e4p-1f;          /* 0.693145751953125 */
static const float LN2_TAIL = 0x1.7f7d1cp-20f;       /* fl(ln2 - head)    */
static const float LOG2_E = 0x1.715476p+0f;          /* fl(1/ln 2)        */
/* 1/j! rounded to fp32, j = 0..7 */
static const float INV_FACT[8] = {0x1p+0f,      0x1p+0f,      0x1p-1f,
                                  0x1.555556p-3f, 0x1.555556p-5f, 0x1.111112p-7f,
                                  0x1.6c16c2p-10f, 0x1.a01a02p-13f};

float oracle_exp(float y) {
  if (y > 80.0f) y = 80.0f;
  if (y < -80.0f) y = -80.0f;
  float n = rintf(y * LOG2_E);
  float r = fmaf(-n, LN2_HEAD, y);
  r = fmaf(-n, LN2_TAIL, r);
  float p = INV_FACT[7];
  for (int j = 6; j >= 0; --j) p = fmaf(p, r, INV_FACT[j]);
  return ldexpf(p, (int)n);
}

float oracle_sigmoid(float l) {
  float den = 1.0f + oracle_exp(-l);
  return 1.0f / den;
}

void oracle_exp_array(const float *in, float *out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_exp(in[i]);
}

void oracle_sigmoid_array(const float *in, float *out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_sigmoid(in[i]);
}

/* ------------------------------------------------------------------------ */
/* R4-R6: group-limited top-k selection                                      */
/* ------------------------------------------------------------------------ */

/*
 * Group-limited routing of [ep] "EPLB 与路由约束": experts are split in G equal
 * groups; a group's score is the sum of its two best expert scores; the
 * topk_group best groups are kept; the k best experts inside the kept groups
 * are chosen.  Scores are given as doubles; when group_sum_f32 is set every
 * score is an fp32 value and the group sum is rounded to fp32 (the binary64
 * sum of two binary32 values rounded to binary32 is the correctly rounded
 * binary32 sum).  With G == 1 the group step is skipped (plain top-k).
 * ids: [T,k], descending score, ties to the lower index.
 */
void oracle_select(const double *s, int T, int E, int G, int topk_group, int k,
                   int group_sum_f32, int32_t *ids) {
#pragma omp parallel for schedule(static)
  for (int t = 0; t < T; ++t) {
    const double *st = s + (size_t)t * E;
    int gs = E / G;
    unsigned char *eligible = (unsigned char *)calloc((size_t)E, 1);
    unsigned char *chosen = (unsigned char *)calloc((size_t)E, 1);
    if (G > 1) {
      double *gscore = (double *)malloc(sizeof(double) * G);
      unsigned char *kept = (unsigned char *)calloc((size_t)G, 1);
      for (int g = 0; g < G; ++g) {
        double m1 = -INFINITY, m2 = -INFINITY;
        for (int e = g * gs; e < (g + 1) * gs; ++e) {
          if (st[e] > m1) {
            m2 = m1;
            m1 = st[e];
          } else if (st[e] > m2) {
            m2 = st[e];
          }
        }
        double sum = (gs >= 2) ? m1 + m2 : m1;
        if (group_sum_f32) sum = (double)(float)sum;
        gscore[g] = sum;
      }
      for (int r = 0; r < topk_group; ++r) {
        int best = -1;
        for (int g = 0; g < G; ++g)
          if (!kept[g] && (best < 0 || gscore[g] > gscore[best])) best = g;
        kept[best] = 1;
      }
      for (int e = 0; e < E; ++e) eligible[e] = kept[e / gs];
      free(kept);
      free(gscore);
    } else {
      for (int e = 0; e < E; ++e) eligible[e] = 1;
    }
    for (int j = 0; j < k; ++j) {
      int best = -1;
      for (int e = 0; e < E; ++e)
        if (eligible[e] && !chosen[e] && (best < 0 || st[e] > st[best])) best = e;
      chosen[best] = 1;
      ids[(size_t)t * k + j] = best;
    }
    free(chosen);
    free(eligible);
  }
}

/* ------------------------------------------------------------------------ */
/* Full router: logits -> scores -> selection -> weights                      */
/* ------------------------------------------------------------------------ */

/*
 * score_kind 0: sigmoid router with bias (R3, R7); 1: softmax router (R7').
 * bias: [E] fp32 (ignored for softmax).  Outputs ids [T,k], weights [T,k],
 * and optionally the selection scores s' [T,E] (sel may be NULL).
 */
void oracle_route_from_logits(const float *logits, const float *bias, int T, int E,
                              int G, int topk_group, int k, int score_kind,
                              float bias_scale, int32_t *ids, float *weights,
                              float *sel) {
  double *s = (double *)malloc(sizeof(double) * (size_t)T * E);
#pragma omp parallel for schedule(static)
  for (int t = 0; t < T; ++t) {
    for (int e = 0; e < E; ++e) {
      float l = logits[(size_t)t * E + e];
      float v;
      if (score_kind == 0) {
        float b = bias_scale * bias[e];
        v = oracle_sigmoid(l) + b;
      } else {
        v = l;
      }
      s[(size_t)t * E + e] = (double)v;
      if (sel) sel[(size_t)t * E + e] = v;
    }
  }
  oracle_select(s, T, E, G, topk_group, k, 1, ids);
  free(s);
#pragma omp parallel for schedule(static)
  for (int t = 0; t < T; ++t) {
    const int32_t *id = ids + (size_t)t * k;
    float *w = weights + (size_t)t * k;
    const float *lt = logits + (size_t)t * E;
    float num[64];
    float *nump = (k <= 64) ? num : (float *)malloc(sizeof(float) * k);
    float sum = 0.0f;
    for (int j = 0; j < k; ++j) {
      float v;
      if (score_kind == 0)
        v = oracle_sigmoid(lt[id[j]]);
      else
        v = oracle_exp(lt[id[j]] - lt[id[0]]);
      nump[j] = v;
      sum = (j == 0) ? v : sum + v;
    }
    for (int j = 0; j < k; ++j) w[j] = nump[j] / sum;
    if (nump != num) free(nump);
  }
}

void oracle_route(const uint16_t *x, const uint16_t *w_r, const float *bias, int T,
                  int d, int E, int G, int topk_group, int k, int score_kind,
                  float bias_scale, int32_t *ids, float *weights, float *logits_out) {
  float *logits = logits_out ? logits_out
                             : (float *)malloc(sizeof(float) * (size_t)T * E);
  oracle_router_logits(x, w_r, T, d, E, logits);
  oracle_route_from_logits(logits, bias, T, E, G, topk_group, k, score_kind,
                           bias_scale, ids, weights, NULL);
  if (!logits_out) free(logits);
}

/* ------------------------------------------------------------------------ */
/* R8: dispatch permutation                                                  */
/* ------------------------------------------------------------------------ */

/*
 * counts[e] = number of assignments to e ([ch15] 4.3 n_e; sum = T*k),
 * offsets = exclusive prefix sum (E+1 entries), dest[a] = row of assignment a
 * in the expert-contiguous buffer, src_token[dest[a]] = a / k.
 * Returns 0, or -1 if an id is out of range.
 */
int oracle_dispatch(const int32_t *ids, int T, int k, int E, int32_t *counts,
                    int32_t *offsets, int32_t *dest, int32_t *src_token) {
  int64_t n = (int64_t)T * k;
  for (int e = 0; e < E; ++e) counts[e] = 0;
  for (int64_t a = 0; a < n; ++a) {
    if (ids[a] < 0 || ids[a] >= E) return -1;
    counts[ids[a]] += 1;
  }
  offsets[0] = 0;
  for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
  int32_t *cursor = (int32_t *)malloc(sizeof(int32_t) * (size_t)E);
  for (int e = 0; e < E; ++e) cursor[e] = offsets[e];
  for (int64_t a = 0; a < n; ++a) {
    int32_t p = cursor[ids[a]]++;
    dest[a] = p;
    src_token[p] = (int32_t)(a / k);
  }
  free(cursor);
  return 0;
}

/*
 * Dispatch onto physical expert copies ([ep] "EPLB 与路由约束": hot experts get
 * copies; [ch15] section 4.3: the gating picks logical experts and the
 * system routes each assignment to one of the expert's equivalent copies,
 * the less loaded one).  Copies: phys_expert[p] is the logical expert of
 * physical slot p (the placement's slot order); copy i of e is the i-th
 * slot, in increasing p, holding e.  Reading R15: the r-th assignment of e
 * (increasing a) goes to copy r mod n_rep(e).  Outputs: counts_phys [P],
 * offsets_phys [P+1], dest [T*k] (row of assignment a), src_token [T*k].
 * Returns -1 for an out-of-range id or an expert without a copy.
 */
int oracle_dispatch_replicated(const int32_t *ids, int T, int k, int E, int P,
                               const int32_t *phys_expert, int32_t *counts_phys,
                               int32_t *offsets_phys, int32_t *dest, int32_t *src_token) {
  int64_t n = (int64_t)T * k;
  int32_t *n_rep = (int32_t *)calloc((size_t)E, sizeof(int32_t));
  int32_t *seen = (int32_t *)calloc((size_t)E, sizeof(int32_t));
  int32_t *slot = (int32_t *)malloc(sizeof(int32_t) * (size_t)(n > 0 ? n : 1));
  int32_t *cursor = (int32_t *)malloc(sizeof(int32_t) * (size_t)(P > 0 ? P : 1));
  int rc = 0;
  for (int p = 0; p < P; ++p) {
    if (phys_expert[p] < 0 || phys_expert[p] >= E) rc = -1;
    else n_rep[phys_expert[p]] += 1;
  }
  /* 1. the copy of every assignment: count e's assignments in increasing a */
  for (int64_t a = 0; a < n && rc == 0; ++a) {
    int e = ids[a];
    if (e < 0 || e >= E || n_rep[e] == 0) {
      rc = -1;
      break;
    }
    int r = seen[e]++;
    int want = r % n_rep[e];
    /* the want-th slot holding e, in increasing p */
    int found = -1, c = 0;
    for (int p = 0; p < P; ++p)
      if (phys_expert[p] == e) {
        if (c == want) {
          found = p;
          break;
        }
        ++c;
      }
    slot[a] = found;
  }
  if (rc == 0) {
    /* 2. a stable counting sort of the assignments by slot */
    for (int p = 0; p < P; ++p) counts_phys[p] = 0;
    for (int64_t a = 0; a < n; ++a) counts_phys[slot[a]] += 1;
    offsets_phys[0] = 0;
    for (int p = 0; p < P; ++p) offsets_phys[p + 1] = offsets_phys[p] + counts_phys[p];
    for (int p = 0; p < P; ++p) cursor[p] = offsets_phys[p];
    for (int64_t a = 0; a < n; ++a) {
      int32_t row = cursor[slot[a]]++;
      dest[a] = row;
      src_token[row] = (int32_t)(a / k);
    }
  }
  free(n_rep);
  free(seen);
  free(slot);
  free(cursor);
  return rc;
}

/* ------------------------------------------------------------------------ */
/* FP8 (e4m3) with block scales ([par02] "DeepGEMM masked, FP8"; [ep] "the    */
/* dispatch sends FP8 with scales", 7168 + 224 bytes per token)              */
/* ------------------------------------------------------------------------ */

/*
 * e4m3: 1 sign, 4 exponent bits (bias 7), 3 mantissa bits; exponent field 0
 * holds the subnormals m/8 * 2^-6; 0x7f / 0xff are NaN; the largest finite
 * value is 448.  No infinities.
 */
float oracle_e4m3_to_float(uint8_t c) {
  int s = c >> 7, e = (c >> 3) & 15, m = c & 7;
  float v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    v = ldexpf((float)m, -9); /* m/8 * 2^-6 */
  else
    v = ldexpf((float)(8 + m), e - 10); /* (1 + m/8) * 2^(e-7) */
  return s ? -v : v;
}

/*
 * Nearest e4m3 value to x, ties to the even mantissa code, magnitudes past
 * 448 saturating to 448 (R13).  |x| < 2^-6: the subnormal code is
 * |x| * 2^9 rounded to nearest even (8 meaning the smallest normal);
 * otherwise |x| = f * 2^p with f in [1, 2): mantissa (f - 1) * 8 rounded to
 * nearest even, carrying into the exponent.  (Both products are exact in
 * double, and nearbyint rounds half to even.)
 */
uint8_t oracle_float_to_e4m3(float x) {
  double a = fabs((double)x);
  int code;
  if (a >= 448.0) {
    code = 126;
  } else if (a < ldexp(1.0, -6)) {
    code = (int)nearbyint(a * 512.0); /* 0..8 */
  } else {
    int p;
    double f = frexp(a, &p) * 2.0; /* a = f * 2^(p-1), f in [1,2) */
    int e = p - 1;                 /* unbiased exponent, -6..8 */
    int m = (int)nearbyint((f - 1.0) * 8.0);
    if (m == 8) {
      m = 0;
      e += 1;
    }
    code = ((e + 7) << 3) | m;
    if (code > 126) code = 126; /* saturate */
  }
  return (uint8_t)(code | (signbit(x) ? 0x80 : 0));
}

/* scale of a block with largest magnitude amax (R13): the power of two
   2^e with e the smallest integer >= -127 such that amax <= 448 * 2^e,
   found by counting e up from -127 (each comparison is exact in double);
   1 when the block is all zeros, 2^127 when amax is not finite */
static float fp8_scale(float amax) {
  if (!(amax > 0.0f)) return 1.0f;
  if (!isfinite(amax)) return ldexpf(1.0f, 127);
  int e = -127;
  while ((double)amax > 448.0 * ldexp(1.0, e)) ++e;
  return ldexpf(1.0f, e);
}

/*
 * Activations, per row and 128-column block (R13): s the power-of-two scale
 * above, q = e4m3(x / s) (the fp32 division by a power of two is exact).
 * x: [rows, cols] bf16, cols a multiple of 128; q: [rows, cols] codes;
 * scales: [rows, cols/128] fp32.
 */
void oracle_quantize_rows_fp8(const uint16_t *x, int64_t rows, int cols, uint8_t *q,
                              float *scales) {
  int nb = cols / 128;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r)
    for (int b = 0; b < nb; ++b) {
      const uint16_t *xb = x + (size_t)r * cols + (size_t)b * 128;
      float amax = 0.0f;
      for (int i = 0; i < 128; ++i) {
        float v = fabsf(bf16_value(xb[i]));
        if (v > amax) amax = v;
      }
      float s = fp8_scale(amax);
      scales[(size_t)r * nb + b] = s;
      for (int i = 0; i < 128; ++i)
        q[(size_t)r * cols + (size_t)b * 128 + i] = oracle_float_to_e4m3(bf16_value(xb[i]) / s);
    }
}

/*
 * Weights [mats, rows, cols] bf16, per 128 x 128 block (R13): one scale per
 * block, scales [mats, rows/128, cols/128].
 */
void oracle_quantize_blocks_fp8(const uint16_t *w, int mats, int rows, int cols, uint8_t *q,
                                float *scales) {
  int rb = rows / 128, cb = cols / 128;
#pragma omp parallel for schedule(static)
  for (int64_t blk = 0; blk < (int64_t)mats * rb * cb; ++blk) {
    int64_t m = blk / ((int64_t)rb * cb);
    int i = (int)((blk / cb) % rb), j = (int)(blk % cb);
    const uint16_t *base = w + (size_t)m * rows * cols;
    float amax = 0.0f;
    for (int r = 0; r < 128; ++r)
      for (int c = 0; c < 128; ++c) {
        float v = fabsf(bf16_value(base[(size_t)(i * 128 + r) * cols + j * 128 + c]));
        if (v > amax) amax = v;
      }
    float s = fp8_scale(amax);
    scales[blk] = s;
    for (int r = 0; r < 128; ++r)
      for (int c = 0; c < 128; ++c) {
        size_t o = (size_t)m * rows * cols + (size_t)(i * 128 + r) * cols + j * 128 + c;
        q[o] = oracle_float_to_e4m3(bf16_value(w[o]) / s);
      }
  }
}

/*
 * FP8 SwiGLU FFN of each row (R13): with x~ = q_x * s_x (per 128 block) and
 * W~ = q_W * s_W (per 128 x 128 block), g, u = x~ . W~gu, h = silu(g) * u in
 * fp64; h is rounded to bf16 (its storage format) and quantized per 128
 * block like an activation; y = h~ . W~d^T in fp64.
 */
void oracle_expert_ffn_rows_fp8(const uint8_t *xq, const float *xs, const int32_t *row_expert,
                                int n, int d, int inter, const uint8_t *wgu_q,
                                const float *wgu_s, const uint8_t *wd_q, const float *wd_s,
                                float *h_out, float *y_out) {
  int db = d / 128, ib = inter / 128;
#pragma omp parallel
  {
    double *xv = (double *)malloc(sizeof(double) * (size_t)d);
    uint16_t *hb = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)inter);
    uint8_t *hq = (uint8_t *)malloc((size_t)inter);
    float *hs = (float *)malloc(sizeof(float) * (size_t)ib);
    double *hv = (double *)malloc(sizeof(double) * (size_t)inter);
#pragma omp for schedule(dynamic, 1)
    for (int r = 0; r < n; ++r) {
      int e = row_expert[r];
      for (int i = 0; i < d; ++i)
        xv[i] = (double)oracle_e4m3_to_float(xq[(size_t)r * d + i]) * (double)xs[(size_t)r * db + i / 128];
      const uint8_t *wg = wgu_q + (size_t)e * 2 * inter * d;
      const float *sg = wgu_s + (size_t)e * (2 * inter / 128) * db;
      for (int j = 0; j < inter; ++j) {
        double g = 0.0, u = 0.0;
        for (int i = 0; i < d; ++i) {
          double wgv = (double)oracle_e4m3_to_float(wg[(size_t)j * d + i]) *
                       (double)sg[(size_t)(j / 128) * db + i / 128];
          double wuv = (double)oracle_e4m3_to_float(wg[(size_t)(inter + j) * d + i]) *
                       (double)sg[(size_t)((inter + j) / 128) * db + i / 128];
          g += xv[i] * wgv;
          u += xv[i] * wuv;
        }
        double h = g / (1.0 + exp(-g)) * u;
        hb[j] = bf16_round((float)h);
        if (h_out) h_out[(size_t)r * inter + j] = bf16_value(hb[j]);
      }
      oracle_quantize_rows_fp8(hb, 1, inter, hq, hs);
      for (int j = 0; j < inter; ++j)
        hv[j] = (double)oracle_e4m3_to_float(hq[j]) * (double)hs[j / 128];
      const uint8_t *wd = wd_q + (size_t)e * d * inter;
      const float *sd = wd_s + (size_t)e * db * ib;
      for (int c = 0; c < d; ++c) {
        double y = 0.0;
        for (int j = 0; j < inter; ++j)
          y += hv[j] * (double)oracle_e4m3_to_float(wd[(size_t)c * inter + j]) *
               (double)sd[(size_t)(c / 128) * ib + j / 128];
        y_out[(size_t)r * d + c] = (float)y;
      }
    }
    free(hv);
    free(hs);
    free(hq);
    free(hb);
    free(xv);
  }
}

/* ------------------------------------------------------------------------ */
/* Capacity ([ch15] 4.3 "Capacity Factor" and its overflow table)            */
/* ------------------------------------------------------------------------ */

/*
 * C = ceil(c * T * k / E), the page's per-expert capacity for capacity factor
 * c, evaluated in double.  (Its example: T = 5600, k = 16, E = 896, c = 1.2
 * gives 120 with a mean of 100.)
 */
int oracle_expert_capacity(int T, int k, int E, double c) {
  double mean = (double)T * (double)k / (double)E;
  return (int)ceil(c * mean);
}

/*
 * Dispatch with a capacity of C rows per expert.  The assignments a = t*k+j
 * are taken in increasing a (R11: first come, first served); the first C
 * assignments of expert e get the padded row e*C + r (r = their rank at e).
 * A later one overflows: with policy 1 ("second round": the overflow is run
 * after the first round, same expert) it gets row E*C + ovf_offsets[e] +
 * (r - C); with policy 0 ("drop") it gets no row, dest = -1.
 * counts[e] = n_e, kept[e] = min(n_e, C), ovf_offsets = exclusive prefix sum
 * of n_e - kept[e] (E+1 entries).  src_row has E*C + T*k entries: the token
 * of every used row, -1 for the others.  Returns 0, or -1 for a bad id.
 */
int oracle_dispatch_capacity(const int32_t *ids, int T, int k, int E, int C, int policy,
                             int32_t *counts, int32_t *kept, int32_t *ovf_offsets,
                             int32_t *dest, int32_t *src_row) {
  if (E <= 0 || C < 0) return -1;
  int64_t n = (int64_t)T * k;
  int64_t rows = (int64_t)E * C + n;
  for (int e = 0; e < E; ++e) counts[e] = 0;
  for (int64_t a = 0; a < n; ++a) {
    if (ids[a] < 0 || ids[a] >= E) return -1;
    counts[ids[a]] += 1;
  }
  ovf_offsets[0] = 0;
  for (int e = 0; e < E; ++e) {
    kept[e] = counts[e] < C ? counts[e] : C;
    ovf_offsets[e + 1] = ovf_offsets[e] + (counts[e] - kept[e]);
  }
  for (int64_t r = 0; r < rows; ++r) src_row[r] = -1;
  int32_t *rank = (int32_t *)calloc((size_t)E, sizeof(int32_t));
  for (int64_t a = 0; a < n; ++a) {
    int e = ids[a];
    int32_t r = rank[e]++;
    int64_t row;
    if (r < C)
      row = (int64_t)e * C + r;
    else if (policy == 1)
      row = (int64_t)E * C + ovf_offsets[e] + (r - C);
    else
      row = -1;
    dest[a] = (int32_t)row;
    if (row >= 0) src_row[row] = (int32_t)(a / k);
  }
  free(rank);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* Expert placement ([ep] "EPLB 与路由约束"): the three greedy steps         */
/* ------------------------------------------------------------------------ */

/*
 * Balanced packing of n items with weights w into n_packs packs of n/n_packs
 * items each: items in order of decreasing weight (equal weights: lower
 * index first); each goes to the pack with the smallest running sum among
 * the packs that are not full (equal sums: lower pack index).
 * packs[p * per + q] = q-th item put in pack p.
 */
static void eplb_pack(const double *w, int n, int n_packs, int32_t *packs) {
  int per = n / n_packs;
  int32_t *order = (int32_t *)malloc(sizeof(int32_t) * (size_t)n);
  int32_t *fill = (int32_t *)calloc((size_t)n_packs, sizeof(int32_t));
  double *sum = (double *)calloc((size_t)n_packs, sizeof(double));
  for (int i = 0; i < n; ++i) order[i] = i;
  /* insertion sort: decreasing weight, stable */
  for (int i = 1; i < n; ++i) {
    int32_t v = order[i];
    int j = i - 1;
    while (j >= 0 && w[order[j]] < w[v]) {
      order[j + 1] = order[j];
      --j;
    }
    order[j + 1] = v;
  }
  for (int q = 0; q < n; ++q) {
    int it = order[q], best = -1;
    for (int p = 0; p < n_packs; ++p)
      if (fill[p] < per && (best < 0 || sum[p] < sum[best])) best = p;
    packs[best * per + fill[best]] = it;
    fill[best] += 1;
    sum[best] += w[it];
  }
  free(sum);
  free(fill);
  free(order);
}

/*
 * Place E logical experts with per-expert loads on `gpus` GPUs as `phys`
 * physical experts.
 *   hierarchical (nodes > 0): (1) pack the expert groups (E/groups
 *   consecutive experts each) onto the nodes by group load, the same number
 *   of groups per node; (2) inside each node, add replicas one at a time to
 *   the expert with the largest load per replica (equal: first in the node's
 *   order) until the node has phys * (its experts) / E physical experts;
 *   (3) pack the node's physical experts, weight load / replicas, onto its
 *   gpus * (its experts) / E GPUs.
 *   global (nodes == 0): the whole cluster is one node.
 * A node's experts are its groups' experts, groups in the order they were
 * packed.  gpu_slots[g * (phys/gpus) + q] = logical expert of the q-th
 * physical expert of GPU g; replicas[e] = number of physical copies of e.
 * Returns 0, or -1 when the sizes do not divide as required.
 */
int oracle_eplb_place(const double *load, int E, int groups, int nodes, int gpus, int phys,
                      int32_t *gpu_slots, int32_t *replicas) {
  int n_nodes = nodes > 0 ? nodes : 1;
  if (E <= 0 || groups <= 0 || E % groups || groups % n_nodes || gpus % n_nodes ||
      phys % gpus || phys < E)
    return -1;
  int gsize = E / groups;
  int per_node_e = E / n_nodes;
  int node_phys = phys / n_nodes, node_gpus = gpus / n_nodes;
  int per_gpu = phys / gpus;
  if (node_phys * n_nodes != phys || node_gpus * per_gpu != node_phys) return -1;
  int32_t *node_experts = (int32_t *)malloc(sizeof(int32_t) * (size_t)E);
  if (nodes > 0) {
    double *gload = (double *)calloc((size_t)groups, sizeof(double));
    for (int g = 0; g < groups; ++g)
      for (int i = 0; i < gsize; ++i) gload[g] += load[g * gsize + i];
    int32_t *gpack = (int32_t *)malloc(sizeof(int32_t) * (size_t)groups);
    eplb_pack(gload, groups, nodes, gpack);
    int per_node_g = groups / nodes;
    for (int nd = 0; nd < nodes; ++nd)
      for (int q = 0; q < per_node_g; ++q) {
        int g = gpack[nd * per_node_g + q];
        for (int i = 0; i < gsize; ++i)
          node_experts[nd * per_node_e + q * gsize + i] = g * gsize + i;
      }
    free(gpack);
    free(gload);
  } else {
    for (int e = 0; e < E; ++e) node_experts[e] = e;
  }
  int32_t *cnt = (int32_t *)malloc(sizeof(int32_t) * (size_t)E);
  int32_t *pl = (int32_t *)malloc(sizeof(int32_t) * (size_t)node_phys);
  double *pw = (double *)malloc(sizeof(double) * (size_t)node_phys);
  int32_t *packs = (int32_t *)malloc(sizeof(int32_t) * (size_t)node_phys);
  for (int nd = 0; nd < n_nodes; ++nd) {
    const int32_t *ids = node_experts + nd * per_node_e;
    for (int i = 0; i < per_node_e; ++i) cnt[ids[i]] = 1;
    for (int r = per_node_e; r < node_phys; ++r) {
      int best = 0;
      for (int i = 1; i < per_node_e; ++i)
        if (load[ids[i]] / cnt[ids[i]] > load[ids[best]] / cnt[ids[best]]) best = i;
      cnt[ids[best]] += 1;
    }
    int m = 0;
    for (int i = 0; i < per_node_e; ++i)
      for (int c = 0; c < cnt[ids[i]]; ++c) {
        pl[m] = ids[i];
        pw[m] = load[ids[i]] / cnt[ids[i]];
        ++m;
      }
    eplb_pack(pw, node_phys, node_gpus, packs);
    for (int q = 0; q < node_phys; ++q)
      gpu_slots[nd * node_phys + q] = pl[packs[q]];
    for (int i = 0; i < per_node_e; ++i) replicas[ids[i]] = cnt[ids[i]];
  }
  free(packs);
  free(pw);
  free(pl);
  free(cnt);
  free(node_experts);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* R9: SwiGLU expert FFN, row by row                                         */
/* ------------------------------------------------------------------------ */

/*
 * For each of n rows r: expert e = row_expert[r], x = x_rows[r, :d] (bf16),
 *   g_j = sum_i x_i Wgu[e, j, i],  u_j = sum_i x_i Wgu[e, inter + j, i]
 *   h_j = silu(g_j) * u_j,          silu(g) = g / (1 + exp(-g))
 *   y_c = sum_j h_j Wd[e, c, j]
 * w_gu: [E, 2*inter, d] (rows 0..inter-1 gate, inter..2*inter-1 up),
 * w_down: [E, d, inter]; both bf16, out x in ([par02]: gate_up fused weight).
 * All sums in fp64.  round_h_bf16 != 0 rounds h to bf16 before the down
 * projection (diagnostic variant only).  h_out ([n, inter]) may be NULL.
 */
void oracle_expert_ffn_rows(const uint16_t *x_rows, const int32_t *row_expert,
                            int n, int d, int inter, const uint16_t *w_gu,
                            const uint16_t *w_down, int round_h_bf16,
                            float *h_out, float *y_out) {
#pragma omp parallel
  {
    double *xv = (double *)malloc(sizeof(double) * (size_t)d);
    double *h = (double *)malloc(sizeof(double) * (size_t)inter);
#pragma omp for schedule(dynamic, 1)
    for (int r = 0; r < n; ++r) {
      int e = row_expert[r];
      const uint16_t *xr = x_rows + (size_t)r * d;
      for (int i = 0; i < d; ++i) xv[i] = (double)bf16_value(xr[i]);
      const uint16_t *wg = w_gu + (size_t)e * 2 * inter * d;
      for (int j = 0; j < inter; ++j) {
        const uint16_t *gr = wg + (size_t)j * d;
        const uint16_t *ur = wg + (size_t)(inter + j) * d;
        double g = 0.0, u = 0.0;
        for (int i = 0; i < d; ++i) {
          g += xv[i] * (double)bf16_value(gr[i]);
          u += xv[i] * (double)bf16_value(ur[i]);
        }
        double hv = g / (1.0 + exp(-g)) * u;
        if (round_h_bf16) hv = (double)bf16_value(bf16_round((float)hv));
        h[j] = hv;
        if (h_out) h_out[(size_t)r * inter + j] = (float)hv;
      }
      const uint16_t *wd = w_down + (size_t)e * d * inter;
      for (int c = 0; c < d; ++c) {
        const uint16_t *dr = wd + (size_t)c * inter;
        double y = 0.0;
        for (int j = 0; j < inter; ++j) y += h[j] * (double)bf16_value(dr[j]);
        y_out[(size_t)r * d + c] = (float)y;
      }
    }
    free(h);
    free(xv);
  }
}

/* ------------------------------------------------------------------------ */
/* R10: combine                                                              */
/* ------------------------------------------------------------------------ */

/*
 * y[t, c] = sum_{j<k} w[t,j] * y_perm[dest[t*k+j], c]  ([trace] hop 4:
 * y = p5 E5(x) + p27 E27(x)), fp64 sum in ascending j.
 */
void oracle_combine(const float *y_perm, const int32_t *dest, const float *w, int T,
                    int k, int d, double *y) {
#pragma omp parallel for schedule(static)
  for (int t = 0; t < T; ++t) {
    for (int c = 0; c < d; ++c) {
      double acc = 0.0;
      for (int j = 0; j < k; ++j) {
        int32_t p = dest[(size_t)t * k + j];
        acc += (double)w[(size_t)t * k + j] * (double)y_perm[(size_t)p * d + c];
      }
      y[(size_t)t * d + c] = acc;
    }
  }
}

/* ------------------------------------------------------------------------ */
/* Whole layer for a subset of tokens                                        */
/* ------------------------------------------------------------------------ */

/*
 * For each listed token t: route it (R1-R7), run its k experts (R9) on its own
 * row and combine (R10).  Tokens are independent, so any subset can be
 * checked one by one.  y: [n_tok, d] fp64.  ids/weights: [n_tok, k].
 */
void oracle_layer_tokens_keep(const uint16_t *x, const uint16_t *w_r, const float *bias,
                              const uint16_t *w_gu, const uint16_t *w_down, int T, int d,
                              int E, int G, int topk_group, int k, int inter,
                              int score_kind, float bias_scale, const int32_t *tokens,
                              int n_tok, const uint8_t *keep, int32_t *ids, float *weights,
                              double *y);

void oracle_layer_tokens(const uint16_t *x, const uint16_t *w_r, const float *bias,
                         const uint16_t *w_gu, const uint16_t *w_down, int T, int d,
                         int E, int G, int topk_group, int k, int inter,
                         int score_kind, float bias_scale, const int32_t *tokens,
                         int n_tok, int32_t *ids, float *weights, double *y) {
  oracle_layer_tokens_keep(x, w_r, bias, w_gu, w_down, T, d, E, G, topk_group, k, inter,
                           score_kind, bias_scale, tokens, n_tok, NULL, ids, weights, y);
}

/*
 * As oracle_layer_tokens, but assignment (q, j) of listed token q only adds
 * its term when keep[q*k + j] != 0 (keep == NULL: every assignment) -- the
 * layer output under the "drop" overflow policy, where a dropped assignment
 * contributes nothing ([ch15] 4.3 overflow table: drop / residual path).
 */
void oracle_layer_tokens_keep(const uint16_t *x, const uint16_t *w_r, const float *bias,
                              const uint16_t *w_gu, const uint16_t *w_down, int T, int d,
                              int E, int G, int topk_group, int k, int inter,
                              int score_kind, float bias_scale, const int32_t *tokens,
                              int n_tok, const uint8_t *keep, int32_t *ids, float *weights,
                              double *y) {
  if (n_tok <= 0) return;
  uint16_t *xs = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)n_tok * d);
  for (int q = 0; q < n_tok; ++q)
    memcpy(xs + (size_t)q * d, x + (size_t)tokens[q] * d, sizeof(uint16_t) * d);
  (void)T;
  oracle_route(xs, w_r, bias, n_tok, d, E, G, topk_group, k, score_kind, bias_scale,
               ids, weights, NULL);
  int nrows = n_tok * k;
  uint16_t *xr = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)nrows * d);
  int32_t *re = (int32_t *)malloc(sizeof(int32_t) * (size_t)nrows);
  float *yr = (float *)malloc(sizeof(float) * (size_t)nrows * d);
  for (int q = 0; q < n_tok; ++q)
    for (int j = 0; j < k; ++j) {
      memcpy(xr + (size_t)(q * k + j) * d, xs + (size_t)q * d, sizeof(uint16_t) * d);
      re[q * k + j] = ids[q * k + j];
    }
  oracle_expert_ffn_rows(xr, re, nrows, d, inter, w_gu, w_down, 0, NULL, yr);
  for (int q = 0; q < n_tok; ++q)
    for (int c = 0; c < d; ++c) {
      double acc = 0.0;
      for (int j = 0; j < k; ++j)
        if (!keep || keep[q * k + j])
          acc += (double)weights[q * k + j] * (double)yr[(size_t)(q * k + j) * d + c];
      y[(size_t)q * d + c] = acc;
    }
  free(yr);
  free(re);
  free(xr);
  free(xs);
}
