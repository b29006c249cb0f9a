/*
 * kv_oracle.c -- plain fp64 CPU oracle for decode attention over a paged KV
 * cache with Quest-style page selection.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the package smoke check and
 * the benchmark's CPU-baseline leg load this file's library.  It shares no
 * code, header or constant with the CUDA path, and the CUDA path never calls
 * it.  Every loop below is written for a reader checking it against the
 * definitions, not for speed.
 *
 * Sources (page title, section):
 *  - KVDrive: A Holistic Multi-Tier KV Cache Management System for
 *    Long-Context LLM Inference, section 2.2 "Sparse attention": keys are split
 *    into blocks; a block's importance is estimated by multiplying the query
 *    with the channel-wise minimum and maximum of its keys; only the Top-K
 *    blocks per query are retrieved.
 *  - same page, section 2.3 "KV cache offloading": each decode token (1)
 *    selects critical entries through an index held in GPU memory, (2) fetches
 *    them, (3) computes sparse attention over them.
 *  - Dual-Blade: Dual-Path NVMe-Direct KV-Cache Offloading for Edge LLM
 *    Inference, "Background and key observations": every decode step loads all
 *    previous KV pairs of the cache (dense decode attention).
 *  - DirectKV (No Buffer, No Bottleneck), core method 2-3: decode keeps the
 *    single query and the output resident and scans every K/V once with a
 *    streaming softmax.  The streaming form is an evaluation order; the value
 *    it computes is plain softmax attention, which is what this file writes.
 *
 * Readings where the pages are silent (each listed in the design notes):
 *  - score = sum over channels of max(q_c * min_c, q_c * max_c), no 1/sqrt(d);
 *  - min/max order is IEEE totalOrder on non-NaN values, so -0.0 < +0.0;
 *  - top-K ties go to the lower page index; output pages ascending, padded
 *    with -1 when fewer than K pages exist;
 *  - query head h reads kv head h / (Hq / Hkv);
 *  - only the valid tokens of the last, partial page take part.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define OKV_F32 0
#define OKV_F16 1
#define OKV_BF16 2

/* ------------------------------------------------------------------------- */
/* element decode: exact value of a stored element                            */
/* ------------------------------------------------------------------------- */

/* IEEE binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
static double dec_f16(uint16_t h) {
  int sign = h >> 15;
  int e = (h >> 10) & 31;
  int m = h & 1023;
  double v;
  if (e == 0)
    v = ldexp((double)m, -24); /* subnormal: m * 2^(1-15-10) */
  else if (e == 31)
    v = m ? NAN : INFINITY;
  else
    v = ldexp((double)(1024 + m), e - 25); /* (1 + m/2^10) * 2^(e-15) */
  return sign ? -v : v;
}

/* bfloat16: the upper half of an IEEE binary32. */
static double dec_bf16(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

double okv_decode(int dtype, const void *base, int64_t i) {
  if (dtype == OKV_F32) return (double)((const float *)base)[i];
  if (dtype == OKV_F16) return dec_f16(((const uint16_t *)base)[i]);
  return dec_bf16(((const uint16_t *)base)[i]);
}

/* ------------------------------------------------------------------------- */
/* index build: channel-wise key min / max of one page                        */
/* ------------------------------------------------------------------------- */

/* a < b in IEEE totalOrder restricted to non-NaN values (-0.0 < +0.0). */
static int total_less(double a, double b) {
  if (a < b) return 1;
  if (a > b) return 0;
  return signbit(a) && !signbit(b);
}

/* Page of n valid tokens starting at element `off` of `k` ([n][d] row-major).
 * mn[c] = min over t < n of k[t][c]; mx[c] = max.  (KVDrive, section 2.2.) */
void okv_page_minmax(int dtype, int d, int n, const void *k, int64_t off, double *mn,
                     double *mx) {
  for (int c = 0; c < d; ++c) {
    double lo = okv_decode(dtype, k, off + c);
    double hi = lo;
    for (int t = 1; t < n; ++t) {
      double x = okv_decode(dtype, k, off + (int64_t)t * d + c);
      if (total_less(x, lo)) lo = x;
      if (total_less(hi, x)) hi = x;
    }
    mn[c] = lo;
    mx[c] = hi;
  }
}

/* Walk every (sequence, valid logical page, kv head) and write the page's
 * min/max at its physical page: mn/mx are [num_phys][Hkv][d].  Entries of
 * physical pages no row references are left untouched. */
void okv_minmax_build(int dtype, int B, int Hkv, int d, int ps, int max_pages,
                      const void *k_cache, const int32_t *block_table,
                      const int32_t *context_lens, double *mn, double *mx) {
  for (int b = 0; b < B; ++b) {
    int len = context_lens[b];
    int P = (len + ps - 1) / ps;
    for (int p = 0; p < P; ++p) {
      int n = len - p * ps < ps ? len - p * ps : ps;
      int64_t phys = block_table[(int64_t)b * max_pages + p];
      for (int kvh = 0; kvh < Hkv; ++kvh) {
        int64_t off = ((phys * Hkv + kvh) * ps) * (int64_t)d;
        int64_t o = (phys * Hkv + kvh) * (int64_t)d;
        okv_page_minmax(dtype, d, n, k_cache, off, mn + o, mx + o);
      }
    }
  }
}

/* ------------------------------------------------------------------------- */
/* mean-key index: one representative key per page                            */
/* ------------------------------------------------------------------------- */

/* Nearest storage-type value to x, ties to the even significand (IEEE
 * round-to-nearest-even), returned as its exact fp64 value.  f32: 24
 * significant bits, f16: 11, bf16: 8.  The spacing of representable values
 * near x is 2^(e - bits) for x = m * 2^e (0.5 <= |m| < 1); below the smallest
 * normal 2^emin (f16: -14; f32, bf16: -126) it stays at the subnormal
 * spacing 2^(emin - bits + 1).  Overflow is not needed here. */
double okv_round_to_dtype(int dtype, double x) {
  if (x == 0.0 || !isfinite(x)) return x;
  int bits = dtype == OKV_F32 ? 24 : dtype == OKV_F16 ? 11 : 8;
  int emin = dtype == OKV_F16 ? -14 : -126;
  int e;
  frexp(x, &e);
  int qexp = e - bits > emin - bits + 1 ? e - bits : emin - bits + 1;
  double r = nearbyint(ldexp(x, -qexp));       /* default mode: ties to even */
  return ldexp(r, qexp);
}

/* Exact sums of stored keys.  Every finite fp32, f16 and bf16 value is an
 * integer multiple of 2^-160 (the smallest subnormals are 2^-149, 2^-24 and
 * 2^-133) and below 2^128 in magnitude, so a sum of at most 128 of them is
 * an integer multiple of 2^-160 below 2^135: 295 bits.  It is held in ten
 * base-2^32 digits; a digit (an int64) takes at most 3 * 128 additions of
 * values below 2^32 before its carries are propagated, so it cannot
 * overflow. */
#define OKV_DIGITS 10
#define OKV_UNIT 160 /* the fixed point: value = sum_i digit[i] 2^(32 i - 160) */

static void fix_add(int64_t *dig, double x) {
  if (x == 0.0) return;
  int e;
  double f = frexp(fabs(x), &e);           /* |x| = f 2^e, f in [0.5, 1) */
  uint64_t m = (uint64_t)ldexp(f, 53);     /* |x| = m 2^(e - 53), m < 2^53 */
  int k = e - 53 + OKV_UNIT;               /* |x| = m 2^k units */
  while (k < 0) {                          /* only zero bits fall off (see above) */
    m >>= 1;
    ++k;
  }
  const int i = k / 32, r = k % 32;
  const int64_t sgn = x < 0 ? -1 : 1;
  const uint64_t lo = m & 0xFFFFFFFFull, hi = m >> 32; /* hi < 2^21 */
  const uint64_t a = lo << r, b = hi << r;             /* a < 2^63, b < 2^52 */
  dig[i] += sgn * (int64_t)(a & 0xFFFFFFFFull);
  dig[i + 1] += sgn * (int64_t)(a >> 32);
  dig[i + 1] += sgn * (int64_t)(b & 0xFFFFFFFFull);
  dig[i + 2] += sgn * (int64_t)(b >> 32);
}

/* Correctly rounded (to nearest, ties to even) mean sum / n of the exact
 * sum in dig, in the storage type: the magnitude by long division, then one
 * rounding to the type's significand at the exponent of the quotient (not
 * below the type's smallest subnormal spacing).  An exact zero sum gives
 * +0.0, or -0.0 when every summed key was -0.0 (IEEE addition's rule). */
static double fix_mean(int64_t *dig, int n, int dtype, int all_neg_zero) {
  /* carries: digits 0..8 into [0, 2^32), digit 9 signed */
  for (int i = 0; i < OKV_DIGITS - 1; ++i) {
    const int64_t low = dig[i] & 0xFFFFFFFFll;
    const int64_t carry = (dig[i] - low) / 4294967296ll;
    dig[i] = low;
    dig[i + 1] += carry;
  }
  const int neg = dig[OKV_DIGITS - 1] < 0;
  uint64_t mag[OKV_DIGITS];
  if (neg) { /* magnitude = two's complement of the digits */
    uint64_t carry = 1;
    for (int i = 0; i < OKV_DIGITS; ++i) {
      const uint64_t v = (~(uint64_t)dig[i] & 0xFFFFFFFFull) + carry;
      mag[i] = v & 0xFFFFFFFFull;
      carry = v >> 32;
    }
  } else {
    for (int i = 0; i < OKV_DIGITS; ++i) mag[i] = (uint64_t)dig[i];
  }
  /* quotient and remainder of the magnitude by n */
  uint64_t q[OKV_DIGITS], rem = 0;
  for (int i = OKV_DIGITS - 1; i >= 0; --i) {
    const uint64_t cur = (rem << 32) | mag[i];
    q[i] = cur / (uint64_t)n;
    rem = cur % (uint64_t)n;
  }
  int bits = 0; /* bit length of q */
  for (int i = OKV_DIGITS - 1; i >= 0 && bits == 0; --i)
    for (int j = 31; j >= 0; --j)
      if ((q[i] >> j) & 1u) {
        bits = 32 * i + j + 1;
        break;
      }
  if (bits == 0 && rem == 0) return (all_neg_zero) ? -0.0 : 0.0;
  /* significand bits p and the smallest spacing 2^(emin - p + 1) */
  const int p = dtype == OKV_F32 ? 24 : dtype == OKV_F16 ? 11 : 8;
  const int emin = dtype == OKV_F16 ? -14 : -126;
  int t = emin - p + 1 + OKV_UNIT; /* spacing of the result, in units: 2^t */
  if (bits - p > t) t = bits - p;
#define QBIT(b) ((int)((q[(b) / 32] >> ((b) % 32)) & 1u))
  uint64_t keep = 0;
  for (int b = bits - 1; b >= t; --b) keep = (keep << 1) | (uint64_t)QBIT(b);
  const int round = QBIT(t - 1);
  int sticky = rem != 0;
  for (int b = t - 2; b >= 0 && !sticky; --b) sticky = QBIT(b);
#undef QBIT
  if (round && (sticky || (keep & 1u))) keep += 1;
  const double v = ldexp((double)keep, t - OKV_UNIT);
  return neg ? -v : v;
}

/* Mean of the page's n valid keys, channel by channel: the exact sum of the
 * stored elements, divided by n and rounded once to the storage type.
 * ShadowKV-style spatial chunking (KVDrive, sections 2.3 and 3, and the
 * design overview: each page's mean key is its representative, half the
 * index bytes of the min/max pair). */
void okv_page_mean(int dtype, int d, int n, const void *k, int64_t off, double *mean) {
  for (int c = 0; c < d; ++c) {
    int64_t dig[OKV_DIGITS] = {0};
    int all_neg_zero = 1;
    for (int t = 0; t < n; ++t) {
      const double x = okv_decode(dtype, k, off + (int64_t)t * d + c);
      if (!(x == 0.0 && signbit(x))) all_neg_zero = 0;
      fix_add(dig, x);
    }
    mean[c] = fix_mean(dig, n, dtype, all_neg_zero);
  }
}

/* Every (sequence, valid logical page, kv head): mean[phys][kvh][:] of
 * [num_phys][Hkv][d]; entries of unreferenced pages are left untouched. */
void okv_mean_build(int dtype, int B, int Hkv, int d, int ps, int max_pages, const void *k_cache,
                    const int32_t *block_table, const int32_t *context_lens, double *mean) {
  for (int b = 0; b < B; ++b) {
    int len = context_lens[b];
    int P = (len + ps - 1) / ps;
    for (int p = 0; p < P; ++p) {
      int n = len - p * ps < ps ? len - p * ps : ps;
      int64_t phys = block_table[(int64_t)b * max_pages + p];
      for (int kvh = 0; kvh < Hkv; ++kvh) {
        int64_t off = ((phys * Hkv + kvh) * ps) * (int64_t)d;
        okv_page_mean(dtype, d, n, k_cache, off, mean + (phys * Hkv + kvh) * (int64_t)d);
      }
    }
  }
}

/* Mean-key page score: q . mean of the page (an estimate of q . k, not a
 * bound), -inf for p >= P_b. */
void okv_mean_scores(int dtype, int B, int Hq, int Hkv, int d, int ps, int max_pages,
                     const void *q, const double *mean, const int32_t *block_table,
                     const int32_t *context_lens, double *scores) {
  int G = Hq / Hkv;
  for (int b = 0; b < B; ++b) {
    int P = (context_lens[b] + ps - 1) / ps;
    for (int h = 0; h < Hq; ++h) {
      double *row = scores + ((int64_t)b * Hq + h) * max_pages;
      for (int p = 0; p < max_pages; ++p) {
        if (p >= P) {
          row[p] = -INFINITY;
          continue;
        }
        int64_t phys = block_table[(int64_t)b * max_pages + p];
        const double *m = mean + (phys * Hkv + h / G) * (int64_t)d;
        double s = 0.0;
        for (int c = 0; c < d; ++c) s += okv_decode(dtype, q, ((int64_t)b * Hq + h) * d + c) * m[c];
        row[p] = s;
      }
    }
  }
}

/* ------------------------------------------------------------------------- */
/* decode append: one new token per sequence                                   */
/* ------------------------------------------------------------------------- */

/* Each decode step appends the new key and value vectors to the cache
 * (KVDrive, section 2.1), and with the cache in pinned host memory the
 * manager appends the new token there (DirectKV, core method 4).  Token
 * position of sequence b is len_b = context_lens[b], its length before the
 * append: logical page p = len_b / ps, slot t = len_b % ps, physical page
 * block_table[b][p].  k_new / v_new are [B][Hkv][d] stored elements, copied
 * bit for bit to [phys][kvh][t][:].  The page's index entry is then the
 * channel-wise min/max of its t + 1 valid tokens, by the definition above
 * (mn/mx are [num_phys][Hkv][d]; NULL skips the index).  Rows with
 * len_b < 0 or len_b >= max_pages * ps are left alone. */
void okv_append(int dtype, int B, int Hkv, int d, int ps, int max_pages, const void *k_new,
                const void *v_new, void *k_cache, void *v_cache, const int32_t *block_table,
                const int32_t *context_lens, double *mn, double *mx) {
  size_t es = dtype == OKV_F32 ? 4 : 2;
  for (int b = 0; b < B; ++b) {
    int len = context_lens[b];
    if (len < 0 || len >= max_pages * ps) continue;
    int p = len / ps, t = len % ps;
    int64_t phys = block_table[(int64_t)b * max_pages + p];
    for (int kvh = 0; kvh < Hkv; ++kvh) {
      int64_t src = ((int64_t)b * Hkv + kvh) * d;
      int64_t page = (phys * Hkv + kvh) * ps * (int64_t)d;
      int64_t dst = page + (int64_t)t * d;
      memcpy((char *)k_cache + dst * es, (const char *)k_new + src * es, d * es);
      memcpy((char *)v_cache + dst * es, (const char *)v_new + src * es, d * es);
      if (mn && mx) {
        int64_t o = (phys * Hkv + kvh) * (int64_t)d;
        okv_page_minmax(dtype, d, t + 1, k_cache, page, mn + o, mx + o);
      }
    }
  }
}

/* ------------------------------------------------------------------------- */
/* page score: upper bound of q . k over the page                              */
/* ------------------------------------------------------------------------- */

/* sum_c max(q_c * mn_c, q_c * mx_c): for every key k in the page,
 * q_c * k_c <= max(q_c * mn_c, q_c * mx_c) channel by channel, so the sum
 * bounds q . k from above.  (KVDrive, section 2.2.) */
double okv_page_score(int d, const double *q, const double *mn, const double *mx) {
  double s = 0.0;
  for (int c = 0; c < d; ++c) {
    double a = q[c] * mn[c];
    double b = q[c] * mx[c];
    s += a > b ? a : b;
  }
  return s;
}

/* scores[b][h][p] for p < P_b, -inf for p >= P_b.  q is stored ([B][Hq][d]),
 * mn/mx are the fp64 tables of okv_minmax_build. */
void okv_scores(int dtype, int B, int Hq, int Hkv, int d, int ps, int max_pages, const void *q,
                const double *mn, const double *mx, const int32_t *block_table,
                const int32_t *context_lens, double *scores) {
  int G = Hq / Hkv;
  double *qd = (double *)malloc(sizeof(double) * d);
  for (int b = 0; b < B; ++b) {
    int P = (context_lens[b] + ps - 1) / ps;
    for (int h = 0; h < Hq; ++h) {
      int kvh = h / G;
      for (int c = 0; c < d; ++c) qd[c] = okv_decode(dtype, q, ((int64_t)b * Hq + h) * d + c);
      double *row = scores + ((int64_t)b * Hq + h) * max_pages;
      for (int p = 0; p < max_pages; ++p) {
        if (p >= P) {
          row[p] = -INFINITY;
          continue;
        }
        int64_t phys = block_table[(int64_t)b * max_pages + p];
        int64_t o = (phys * Hkv + kvh) * (int64_t)d;
        row[p] = okv_page_score(d, qd, mn + o, mx + o);
      }
    }
  }
  free(qd);
}

/* ------------------------------------------------------------------------- */
/* top-K page selection                                                        */
/* ------------------------------------------------------------------------- */

static const double *g_sort_scores; /* comparator context (single-threaded use) */

/* order: higher score first; equal scores -> lower page index first */
static int by_score_desc(const void *pa, const void *pb) {
  int a = *(const int *)pa, b = *(const int *)pb;
  double sa = g_sort_scores[a], sb = g_sort_scores[b];
  if (sa > sb) return -1;
  if (sa < sb) return 1;
  return (a > b) - (a < b);
}

static int by_index_asc(const void *pa, const void *pb) {
  int a = *(const int *)pa, b = *(const int *)pb;
  return (a > b) - (a < b);
}

/* The K pages with the largest scores among pages 0..P-1, returned in
 * ascending page order; slots past min(K, P) hold -1.  (KVDrive, section 2.2:
 * only the Top-K blocks per query are retrieved.) */
void okv_topk_row(int P, const double *scores, int K, int32_t *out) {
  int *order = (int *)malloc(sizeof(int) * (P > 0 ? P : 1));
  for (int p = 0; p < P; ++p) order[p] = p;
  g_sort_scores = scores;
  qsort(order, P, sizeof(int), by_score_desc);
  int keff = K < P ? K : P;
  qsort(order, keff, sizeof(int), by_index_asc);
  for (int i = 0; i < K; ++i) out[i] = i < keff ? order[i] : -1;
  free(order);
}

void okv_topk(int B, int Hq, int ps, int max_pages, const int32_t *context_lens,
              const double *scores, int K, int32_t *out) {
  for (int b = 0; b < B; ++b) {
    int P = (context_lens[b] + ps - 1) / ps;
    for (int h = 0; h < Hq; ++h)
      okv_topk_row(P, scores + ((int64_t)b * Hq + h) * max_pages, K,
                   out + ((int64_t)b * Hq + h) * K);
  }
}

/* Selection with forced pages.  Sparse-attention systems always keep the
 * sink tokens (the first few) and the most recent local tokens (KVDrive,
 * section 9.1, experimental setup: the first 4 and the last 64).  At page
 * granularity a page is forced when the tokens it holds, [p*ps, min(len,
 * (p+1)*ps)), meet [0, sink) or [len - local, len).  Forced pages come first,
 * in index order; then the other pages by score (higher first, ties to the
 * lower index); the first min(K, P) are returned ascending, -1 padded. */
static int page_is_forced(int p, int len, int ps, int sink, int local) {
  int lo = p * ps;
  int hi = (p + 1) * ps < len ? (p + 1) * ps : len; /* tokens [lo, hi) */
  if (sink > 0 && lo < sink) return 1;
  if (local > 0 && hi > len - local) return 1;
  return 0;
}

void okv_topk_forced_row(int P, int len, int ps, const double *scores, int K, int sink,
                         int local, int32_t *out) {
  int *order = (int *)malloc(sizeof(int) * (P > 0 ? P : 1));
  int nf = 0;
  for (int p = 0; p < P; ++p)
    if (page_is_forced(p, len, ps, sink, local)) order[nf++] = p;
  int n = nf;
  for (int p = 0; p < P; ++p)
    if (!page_is_forced(p, len, ps, sink, local)) order[n++] = p;
  g_sort_scores = scores;
  qsort(order + nf, P - nf, sizeof(int), by_score_desc);
  int keff = K < P ? K : P;
  qsort(order, keff, sizeof(int), by_index_asc);
  for (int i = 0; i < K; ++i) out[i] = i < keff ? order[i] : -1;
  free(order);
}

void okv_topk_forced(int B, int Hq, int ps, int max_pages, const int32_t *context_lens,
                     const double *scores, int K, int sink, int local, int32_t *out) {
  for (int b = 0; b < B; ++b) {
    int len = context_lens[b];
    int P = (len + ps - 1) / ps;
    for (int h = 0; h < Hq; ++h)
      okv_topk_forced_row(P, len, ps, scores + ((int64_t)b * Hq + h) * max_pages, K, sink, local,
                          out + ((int64_t)b * Hq + h) * K);
  }
}

/* ------------------------------------------------------------------------- */
/* GPU-resident window of critical pages                                       */
/* ------------------------------------------------------------------------- */

/* KVDrive, section 5.1 "Sliding window with lookahead eviction": the GPU keeps
 * a window of recently critical KV entries; each decode step fetches from host
 * memory only the critical entries the window lacks and evicts the entries
 * with the lowest attention score of the current step, the least likely to be
 * reused.  Section 3, Finding 1 sizes it in multiples (x N) of the per-step
 * budget.
 *
 * Unit: one (sequence b, kv head) group with C slots, each holding one page of
 * that kv head.  State: slot_page[g][C] (logical page or -1) and
 * page_slot[g][max_pages] (slot or -1).  One step, given the selection
 * indices[b][h][K] of the group's G query heads and this step's page scores:
 *   need    = the pages any of the G heads selected (p < P_b);
 *   hits    = needed pages already in a slot; misses = the others;
 *   a cached page at or past P_b scores -inf (stale); a cached page that is
 *   not needed scores max over the G heads of scores[b][h][page];
 *   evict   = the (misses - free slots) non-needed cached pages with the
 *             lowest score, ties to the lower slot;
 *   assign  = misses in ascending page order take the free and evicted slots
 *             in ascending slot order;
 *   fetch   = the misses, plus the row's last page when it is a hit (the
 *             cached copy may lack tokens appended since), each with its
 *             slot, in ascending page order.
 * Requires C >= |need|.  stats[g] = {needed, hits, fetched, evicted}. */
static const double *g_evict_score;
static int by_evict_order(const void *pa, const void *pb) {
  int a = *(const int *)pa, b = *(const int *)pb; /* slots */
  double sa = g_evict_score[a], sb = g_evict_score[b];
  if (sa < sb) return -1;
  if (sa > sb) return 1;
  return (a > b) - (a < b);
}

int okv_window_step(int B, int Hq, int Hkv, int ps, int max_pages, int C,
                    const int32_t *context_lens, const int32_t *indices, int K,
                    const double *scores, int32_t *slot_page, int32_t *page_slot,
                    int32_t *fetch_page, int32_t *fetch_slot, int32_t *fetch_count,
                    int32_t *stats) {
  int G = Hq / Hkv;
  char *need = (char *)malloc(max_pages > 0 ? max_pages : 1);
  double *escore = (double *)malloc(sizeof(double) * C);
  int *cand = (int *)malloc(sizeof(int) * C);
  int *freed = (int *)malloc(sizeof(int) * C);
  int *is_freed = (int *)malloc(sizeof(int) * C);
  int rc = 0;
  for (int b = 0; b < B; ++b) {
    int len = context_lens[b];
    int P = (len + ps - 1) / ps;
    for (int kvh = 0; kvh < Hkv; ++kvh) {
      int64_t g = (int64_t)b * Hkv + kvh;
      int32_t *sp = slot_page + g * C;
      int32_t *ps_map = page_slot + g * max_pages;
      memset(need, 0, max_pages);
      int n_need = 0;
      for (int h = kvh * G; h < (kvh + 1) * G; ++h)
        for (int i = 0; i < K; ++i) {
          int p = indices[((int64_t)b * Hq + h) * K + i];
          if (p >= 0 && p < P && !need[p]) {
            need[p] = 1;
            ++n_need;
          }
        }
      if (n_need > C) {
        rc = -1;
        continue;
      }
      int n_hit = 0, n_free = 0, n_cand = 0;
      for (int s = 0; s < C; ++s) {
        is_freed[s] = 0;
        int p = sp[s];
        if (p < 0) {
          is_freed[s] = 1;
          ++n_free;
        } else if (p < P && need[p]) {
          ++n_hit;
        } else {
          double sc = -INFINITY;
          if (p < P)
            for (int h = kvh * G; h < (kvh + 1) * G; ++h) {
              double v = scores[((int64_t)b * Hq + h) * max_pages + p];
              if (v > sc) sc = v;
            }
          escore[s] = sc;
          cand[n_cand++] = s;
        }
      }
      int n_miss = n_need - n_hit;
      int n_evict = n_miss > n_free ? n_miss - n_free : 0;
      g_evict_score = escore;
      qsort(cand, n_cand, sizeof(int), by_evict_order);
      for (int i = 0; i < n_evict; ++i) {
        int s = cand[i];
        ps_map[sp[s]] = -1;
        sp[s] = -1;
        is_freed[s] = 1;
      }
      int nf = 0;
      for (int s = 0; s < C; ++s)
        if (is_freed[s]) freed[nf++] = s;
      int r = 0, nfetch = 0;
      int32_t *fp = fetch_page + g * C;
      int32_t *fs = fetch_slot + g * C;
      for (int p = 0; p < P; ++p) {
        if (!need[p]) continue;
        if (ps_map[p] < 0) { /* a miss: next free slot */
          int s = freed[r++];
          sp[s] = p;
          ps_map[p] = s;
          fp[nfetch] = p;
          fs[nfetch++] = s;
        } else if (p == P - 1) { /* a hit on the growing last page: refresh */
          fp[nfetch] = p;
          fs[nfetch++] = ps_map[p];
        }
      }
      fetch_count[g] = nfetch;
      stats[g * 4 + 0] = n_need;
      stats[g * 4 + 1] = n_hit;
      stats[g * 4 + 2] = nfetch;
      stats[g * 4 + 3] = n_evict;
    }
  }
  free(need);
  free(escore);
  free(cand);
  free(freed);
  free(is_freed);
  return rc;
}

/* ------------------------------------------------------------------------- */
/* attention of one query head over a set of pages                             */
/* ------------------------------------------------------------------------- */

/* out[c] = sum_t e^{z_t - m} v_t[c] / sum_t e^{z_t - m},  z_t = scale * q . k_t,
 * m = max_t z_t, over the valid tokens of the listed logical pages (all pages
 * 0..P-1 when pages == NULL; entries < 0 are skipped).  Two passes in fp64. */
void okv_attention_row(int dtype, int Hkv, int d, int ps, int max_pages, double scale,
                       const void *q, int64_t q_off, const void *k_cache, const void *v_cache,
                       int kvh, const int32_t *bt_row, int len, const int32_t *pages,
                       int npages, double *out) {
  int P = (len + ps - 1) / ps;
  if (pages == NULL) npages = P;
  double *qd = (double *)malloc(sizeof(double) * d);
  double *z = (double *)malloc(sizeof(double) * ((int64_t)npages * ps + 1));
  for (int c = 0; c < d; ++c) qd[c] = okv_decode(dtype, q, q_off + c);

  /* pass 1: logits of every taking-part token, and their maximum */
  int64_t nt = 0;
  double m = -INFINITY;
  for (int i = 0; i < npages; ++i) {
    int p = pages ? pages[i] : i;
    if (p < 0 || p >= P) continue;
    int n = len - p * ps < ps ? len - p * ps : ps;
    int64_t phys = bt_row[p];
    for (int t = 0; t < n; ++t) {
      int64_t off = (((phys * Hkv + kvh) * ps) + t) * (int64_t)d;
      double dot = 0.0;
      for (int c = 0; c < d; ++c) dot += qd[c] * okv_decode(dtype, k_cache, off + c);
      z[nt] = scale * dot;
      if (z[nt] > m) m = z[nt];
      ++nt;
    }
  }

  /* pass 2: normalised weighted sum of values */
  for (int c = 0; c < d; ++c) out[c] = 0.0;
  double den = 0.0;
  nt = 0;
  for (int i = 0; i < npages; ++i) {
    int p = pages ? pages[i] : i;
    if (p < 0 || p >= P) continue;
    int n = len - p * ps < ps ? len - p * ps : ps;
    int64_t phys = bt_row[p];
    for (int t = 0; t < n; ++t) {
      int64_t off = (((phys * Hkv + kvh) * ps) + t) * (int64_t)d;
      double w = exp(z[nt] - m);
      den += w;
      for (int c = 0; c < d; ++c) out[c] += w * okv_decode(dtype, v_cache, off + c);
      ++nt;
    }
  }
  for (int c = 0; c < d; ++c) out[c] = den > 0.0 ? out[c] / den : 0.0;
  free(z);
  free(qd);
}

/* Attention for a list of rows r = b * Hq + h (all B*Hq rows when rows ==
 * NULL).  indices == NULL: dense over all pages; else indices is [B][Hq][K]
 * (logical pages, -1 padded).  out is [B][Hq][d]; only listed rows are
 * written.  nthreads > 0 sets the OpenMP thread count (ignored without it). */
void okv_attention(int dtype, int B, int Hq, int Hkv, int d, int ps, int max_pages,
                   double scale, const void *q, const void *k_cache, const void *v_cache,
                   const int32_t *block_table, const int32_t *context_lens,
                   const int32_t *indices, int K, const int32_t *rows, int nrows,
                   int nthreads, double *out) {
  int G = Hq / Hkv;
  if (rows == NULL) nrows = B * Hq;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
  for (int i = 0; i < nrows; ++i) {
    int r = rows ? rows[i] : i;
    int b = r / Hq, h = r % Hq;
    const int32_t *sel = indices ? indices + (int64_t)r * K : NULL;
    okv_attention_row(dtype, Hkv, d, ps, max_pages, scale, q, (int64_t)r * d, k_cache, v_cache,
                      h / G, block_table + (int64_t)b * max_pages, context_lens[b], sel,
                      indices ? K : 0, out + (int64_t)r * d);
  }
}

int okv_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
