/*
 * sv_oracle.c -- TEST INFRASTRUCTURE, not part of the product.
 *
 * A plain, slow, single-threaded CPU reference ("oracle") of the batched
 * speculative-decoding verifier (rejection sampler).  Only the test suite, the
 * smoke check and the benchmark's CPU-baseline leg load it.  It shares no code,
 * header, table or constant with the CUDA library: everything here is written
 * out from the pages' definitions, one request at a time, one row at a time,
 * in the order the pages state the steps.
 *
 * Sources (page title, section):
 *  [P1] "vLLM source walk-through (10): speculative decoding -- draft models,
 *       batched verification and the token-acceptance pipeline":
 *       section "SpecDecodeMetadata" (flattened drafts, cu_num_draft_tokens),
 *       section "Rejection sampling: the two branches of RejectionSampler"
 *       (bonus token, identical sampling transforms on p and q, output buffer
 *       filled with -1), section "Greedy kernel" (compare with the target argmax,
 *       stop at the first mismatch, bonus when all match), section "Random
 *       kernel" (exponential race: argmax of weight / exponential draw).
 *  [P2] "Speculative Decoding: propose, verify, accept": section 02 (shapes),
 *       section 03 (greedy), section 04 (alpha = min(1, p/q); residual
 *       max(0, p-q) renormalised), section 05 (two-token worked example),
 *       section 06 (per-round algorithm), section 13 (test guidance).
 *  [P3] "How speculative decoding interacts with the KV cache: placeholders,
 *       rollback and draft KV": section 3.1 (num_computed_tokens -= K - A when
 *       it is > 0), section 3.2 (block-granular example).
 *
 * Readings taken where the pages are silent or disagree (all listed in the
 * design notes as well):
 *  - accept iff fl32(u * q(y)) < p(y): strict, so equality rejects; this is
 *    u < min(1, p/q) without a division [P2 s04/s06];
 *  - residual = max(p - q, 0) computed as fl32(p - q) when that is > 0, else 0
 *    [P2 s04];
 *  - categorical draws use the exponential race of [P1 "Random kernel"]:
 *    key(x) = fl32(w(x) / E(x)) (IEEE division), token = lowest x of the
 *    largest key; weights w(x) <= 0 (or NaN) have key 0 and their E is not read;
 *  - one E vector per request serves its single draw (replacement or bonus);
 *  - if every residual key is 0 the replacement is drawn by the same race over
 *    p; if that is all 0 as well the token is 0 (the lowest index) and the
 *    EMPTY_DISTRIBUTION status bit is raised;
 *  - temperature 0 selects the greedy path; argmax keeps the lowest index;
 *    negative, NaN, infinite and subnormal (0 < T < FLT_MIN) temperatures are
 *    invalid;
 *  - logits entry: value/T, top-k keeps every x with l(x) >= the k-th largest
 *    value (ties kept), softmax over the kept set (double), top-p keeps the
 *    shortest descending prefix whose cumulative probability reaches top_p
 *    plus every entry tied with its last element, then the logits processors
 *    (banned ids, repetition penalty) act on the kept logits, renormalised,
 *    rounded to fp32;
 *  - the rows a request reads are the rows a sequential verifier reads: rows
 *    after the first rejection are never examined, so their contents can not
 *    raise a status bit;
 *  - a request whose own data is invalid (bad cu range, draft id outside
 *    [0, V) at an examined position, bad temperature/top-p, NaN values on the
 *    greedy path, NaN/+inf/no finite logit on the random logits path, missing
 *    draft rows) emits nothing: its output row stays -1, num_accepted = 0 and
 *    its KV bookkeeping is untouched;
 *  - synthetic acceptance (page 1, "About synthetic / block verification":
 *    preset per-position rates, non-increasing, "uniform < rate" accepts
 *    without the target probabilities): only the test changes -- accept iff
 *    u_j < rate_j; rows before the stopping position are not read (their
 *    probabilities are never formed) and the replacement or bonus draw there
 *    is the ordinary one; rates outside [0, 1] or increasing over the
 *    request's positions are a bad parameter;
 *  - rejected KV slots are the verify tokens j in (A, gamma_i] of the request
 *    (the KV of the rejected drafts), so their count gamma_i - A equals the
 *    num_computed_tokens decrement [P3 s3.1, s3.2].
 *
 * Production mode draws u and E from Philox4x32-10 (Salmon, Moraes, Dror,
 * Shaw, "Parallel random numbers: as easy as 1, 2, 3", SC'11), written here
 * from that paper's definition:
 *   u_j  : counter (j/4, 2*r+1, offset_lo, offset_hi), word j%4,
 *          u = (word >> 8) * 2^-24                       in [0, 1)
 *   E(x) : counter (x/4, 2*r,   offset_lo, offset_hi), word x%4,
 *          U = (2*(word >> 9) + 1) * 2^-24               in (0, 1)
 *          E = fl32(-ln U), ln evaluated in double
 *   key (seed_lo, seed_hi); r = rng_request_base + request index.
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* status bits (same numeric meaning as the library documents) */
#define ORC_BAD_CU 1
#define ORC_BAD_DRAFT_ID 2
#define ORC_BAD_EXPONENTIAL 4
#define ORC_EMPTY_DISTRIBUTION 8
#define ORC_BAD_VALUES 16
#define ORC_BAD_PARAM 32
#define ORC_MISSING_DRAFT 64

#define ORC_ENTRY_PROBS 0
#define ORC_ENTRY_LOGITS 1
#define ORC_F32 0
#define ORC_BF16 1

/* per-request diagnostics written when diag != NULL (tests use them to name
 * the decisions that sit within the stated tolerance of a flip).  A "flip
 * index" is max(needed_abs / 1e-6, needed_rel / 1e-5): the perturbation of p
 * and q needed to change the decision, in units of the tolerance -- 1e-6
 * absolute (the contract on probabilities) and 1e-5 relative.  An index < 1
 * means a perturbation inside both bounds could flip the decision. */
#define ORC_BAD_LIST 256 /* a processor or stop list range of the request is invalid */
#define ORC_NDIAG 6
#define DIAG_ACCEPT_MARGIN 0 /* min over examined positions of the flip index of the test */
#define DIAG_RACE_FLIP 1     /* min over supported x != x1 of the flip index of the race */
#define DIAG_RACE_RELGAP 2   /* min (k1 - k_x) / k1 over supported x != x1             */
#define DIAG_TOPP_EDGE 3     /* 1 if a cumulative sum at a top-p cut is within 1e-6   */
#define DIAG_FALLBACK 4      /* 1 if the residual race had no positive key            */
#define DIAG_PATH 5          /* 0 random, 1 greedy, -1 invalid                        */

typedef struct {
  int32_t num_reqs, max_spec_len, vocab_size, entry, dtype, pad0;
  int64_t num_draft_tokens_total;
  const int32_t *draft_ids;
  const int32_t *cu_num_draft_tokens;
  const void *target;
  int64_t target_row_stride;
  const void *draft;
  int64_t draft_row_stride;
  const float *temperature;
  const int32_t *top_k;
  const float *top_p;
  const float *uniforms;
  const float *exponentials;
  int64_t exponentials_row_stride;
  uint64_t seed, offset;
  uint32_t rng_request_base, pad1;
  int32_t *out_tokens;
  int32_t *num_accepted;
  int32_t *num_computed_tokens;
  int64_t *slot_mapping;
  float *dbg_py;
  float *dbg_qy;
  int32_t *status;
  double *diag;
  const float *synthetic_rates; /* [max_spec_len] or NULL */
  /* logits processors and stop tokens (per-request lists: request i owns
   * entries [cu[i-1], cu[i]) of the ids array) */
  const float *repetition_penalty; /* [N] theta, or NULL */
  const int64_t *penalty_cu;
  const int32_t *penalty_ids;
  int64_t penalty_total;
  const int64_t *banned_cu;
  const int32_t *banned_ids;
  int64_t banned_total;
  const int64_t *stop_cu;
  const int32_t *stop_ids;
  int64_t stop_total;
} oracle_args;

/* ------------------------------------------------------------------------ */
/* Philox4x32-10                                                             */
/* ------------------------------------------------------------------------ */
void oracle_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
  uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
  uint32_t k0 = key[0], k1 = key[1];
  for (int round = 0; round < 10; ++round) {
    if (round > 0) { /* Weyl-sequence key schedule */
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    uint64_t prod0 = (uint64_t)0xD2511F53u * (uint64_t)c0;
    uint64_t prod1 = (uint64_t)0xCD9E8D57u * (uint64_t)c2;
    uint32_t hi0 = (uint32_t)(prod0 >> 32), lo0 = (uint32_t)prod0;
    uint32_t hi1 = (uint32_t)(prod1 >> 32), lo1 = (uint32_t)prod1;
    uint32_t n0 = hi1 ^ c1 ^ k0;
    uint32_t n1 = lo1;
    uint32_t n2 = hi0 ^ c3 ^ k1;
    uint32_t n3 = lo0;
    c0 = n0; c1 = n1; c2 = n2; c3 = n3;
  }
  out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

static uint32_t philox_word(uint64_t seed, uint64_t offset, uint32_t c0, uint32_t c1, int lane) {
  uint32_t ctr[4] = {c0, c1, (uint32_t)offset, (uint32_t)(offset >> 32)};
  uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
  uint32_t w[4];
  oracle_philox4x32_10(ctr, key, w);
  return w[lane];
}

float oracle_uniform(uint64_t seed, uint64_t offset, uint32_t req, uint32_t j) {
  uint32_t w = philox_word(seed, offset, j / 4u, 2u * req + 1u, (int)(j % 4u));
  return (float)(w >> 8) * 0x1p-24f;
}

float oracle_exponential(uint64_t seed, uint64_t offset, uint32_t req, uint32_t x) {
  uint32_t w = philox_word(seed, offset, x / 4u, 2u * req, (int)(x % 4u));
  float U = (float)(2u * (w >> 9) + 1u) * 0x1p-24f;
  return (float)(-log((double)U));
}

/* ------------------------------------------------------------------------ */
/* rows                                                                      */
/* ------------------------------------------------------------------------ */
static float bf16_to_float(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

static void load_row(const void *base, int dtype, int64_t row, int64_t stride, int V, float *dst) {
  if (dtype == ORC_BF16) {
    const uint16_t *r = (const uint16_t *)base + row * stride;
    for (int x = 0; x < V; ++x) dst[x] = bf16_to_float(r[x]);
  } else {
    const float *r = (const float *)base + row * stride;
    for (int x = 0; x < V; ++x) dst[x] = r[x];
  }
}

/* argmax, lowest index on equal values (-0 and +0 are equal). Returns -1 if a
 * NaN is present (the caller raises BAD_VALUES). */
static int argmax_row(const float *v, int V) {
  for (int x = 0; x < V; ++x)
    if (isnan(v[x])) return -1;
  int best = 0;
  for (int x = 1; x < V; ++x)
    if (v[x] > v[best]) best = x;
  return best;
}

/* ------------------------------------------------------------------------ */
/* logits -> probabilities (temperature, top-k, softmax, top-p), one row      */
/* ------------------------------------------------------------------------ */
static int cmp_desc_double(const void *a, const void *b) {
  double x = *(const double *)a, y = *(const double *)b;
  return (x < y) - (x > y);
}

/* The transform of one logits row, in the order of "vLLM source walk-through
 * (10)", section "Rejection sampling: the two branches of RejectionSampler",
 * step 2 (sampling constraints -- temperature, top-k, top-p -- first, then the
 * logits processors such as penalties) and of "Speculative Decoding: propose,
 * verify, accept", section 06 (temperature, top-k, top-p, banned tokens,
 * repetition penalty):
 *   1. value / T;
 *   2. top-k on the raw row: keep x with l(x) >= tau, tau the k-th largest
 *      logit counted with multiplicity;
 *   3. softmax over the top-k set (double);
 *   4. top-p: keep the shortest descending prefix whose cumulative
 *      probability reaches top_p, plus every entry tied with its last one;
 *   5. the logits processors act on the surviving logits: lp[x] replaces l(x)
 *      for every kept x (a banned id's lp is -inf, a penalised id's lp is its
 *      rewritten logit); lp == NULL means the request has no processors;
 *   6. renormalise exp(v/T) over the kept x whose value v is finite, and round
 *      to fp32.
 * Returns 0 on success, ORC_BAD_VALUES for NaN / +inf / no finite logit in the
 * raw row, NaN / +inf among the kept processed values, or a kept set whose
 * every entry is banned (no distribution is left).  *edge is set to 1 if the
 * cumulative probability of the values above the top-p cut value, or of the
 * values through it, lies within 1e-6 of top_p (a perturbation of that size
 * could move the cut to another value). */
int oracle_transform_row(const float *l, const float *lp, int V, float temperature, int top_k, float top_p,
                         float *out, int *edge) {
  int n_finite = 0;
  for (int x = 0; x < V; ++x) {
    if (isnan(l[x]) || (isinf(l[x]) && l[x] > 0)) return ORC_BAD_VALUES;
    if (isfinite(l[x])) ++n_finite;
  }
  if (n_finite == 0) return ORC_BAD_VALUES;
  if (edge) *edge = 0;

  /* top-k: tau = k-th largest logit, counted with multiplicity */
  double tau = -INFINITY;
  if (top_k > 0 && top_k < V) {
    double *sorted = (double *)malloc(sizeof(double) * (size_t)V);
    for (int x = 0; x < V; ++x) sorted[x] = (double)l[x];
    qsort(sorted, (size_t)V, sizeof(double), cmp_desc_double);
    tau = sorted[top_k - 1];
    free(sorted);
  }
  /* softmax of l/T over the top-k set, in double (it only places the top-p cut) */
  double T = (double)temperature;
  double m = -INFINITY;
  for (int x = 0; x < V; ++x)
    if ((double)l[x] >= tau && (double)l[x] / T > m) m = (double)l[x] / T;
  double Z = 0.0;
  for (int x = 0; x < V; ++x)
    if ((double)l[x] >= tau) Z += exp((double)l[x] / T - m);
  /* top-p over the top-k set: walk the kept logits in descending order */
  double cut = tau;
  if (top_p < 1.0f) {
    int nk = 0;
    for (int x = 0; x < V; ++x)
      if ((double)l[x] >= tau) ++nk;
    double *kept = (double *)malloc(sizeof(double) * (size_t)nk);
    int t = 0;
    for (int x = 0; x < V; ++x)
      if ((double)l[x] >= tau) kept[t++] = (double)l[x];
    qsort(kept, (size_t)nk, sizeof(double), cmp_desc_double);
    double cum = 0.0;
    int found = 0;
    for (int r = 0; r < nk; ++r) {
      cum += exp(kept[r] / T - m) / Z;
      if (cum >= (double)top_p) {
        cut = kept[r];
        found = 1;
        break;
      }
    }
    if (edge) {
      /* Entries tied with the cut value are all kept, so the kept set changes
       * only when a value-group boundary moves across top_p: the cumulative
       * mass of the values above the cut value, and of those through it. */
      double above = 0.0, through = 0.0;
      for (int r = 0; r < nk; ++r) {
        double e = exp(kept[r] / T - m) / Z;
        if (kept[r] > cut) above += e;
        if (kept[r] >= cut) through += e;
      }
      if (!found || fabs(above - (double)top_p) < 1e-6 || fabs(through - (double)top_p) < 1e-6) *edge = 1;
    }
    free(kept);
  }
  /* the processors' values on the kept set, then the renormalisation */
  const float *v = lp ? lp : l;
  double m2 = -INFINITY;
  for (int x = 0; x < V; ++x) {
    if (!((double)l[x] >= tau && (double)l[x] >= cut)) continue;
    if (isnan(v[x]) || (isinf(v[x]) && v[x] > 0)) return ORC_BAD_VALUES;
    if (isfinite(v[x]) && (double)v[x] / T > m2) m2 = (double)v[x] / T;
  }
  if (m2 == -INFINITY) return ORC_BAD_VALUES; /* every kept logit was banned */
  double Z2 = 0.0;
  for (int x = 0; x < V; ++x)
    if ((double)l[x] >= tau && (double)l[x] >= cut && isfinite(v[x])) Z2 += exp((double)v[x] / T - m2);
  for (int x = 0; x < V; ++x)
    out[x] = ((double)l[x] >= tau && (double)l[x] >= cut && isfinite(v[x])) ? (float)(exp((double)v[x] / T - m2) / Z2)
                                                                            : 0.0f;
  return 0;
}

/* The transform without logits processors. */
int oracle_logits_to_probs(const float *l, int V, float temperature, int top_k, float top_p, float *out,
                           int *edge) {
  return oracle_transform_row(l, NULL, V, temperature, top_k, top_p, out, edge);
}

/* ------------------------------------------------------------------------ */
/* the verifier                                                              */
/* ------------------------------------------------------------------------ */
typedef struct {
  const oracle_args *a;
  int32_t *status;
  uint32_t rng_req;
  int test_mode;
  int V;
  const float *E_row; /* test mode */
  float *E_cache;     /* production mode: E computed lazily */
  unsigned char *E_have;
} race_ctx;

static float E_at(race_ctx *c, int x) {
  if (c->test_mode) return c->E_row[x];
  if (!c->E_have[x]) {
    c->E_cache[x] = oracle_exponential(c->a->seed, c->a->offset, c->rng_req, (uint32_t)x);
    c->E_have[x] = 1;
  }
  return c->E_cache[x];
}

/* Exponential race over weights w: key(x) = fl32(w(x)/E(x)) where w(x) > 0,
 * else 0. Returns the lowest x with the largest key; *kmax receives it. */
static int race(race_ctx *c, const float *w, float *kmax) {
  int best = -1;
  float bk = 0.0f;
  for (int x = 0; x < c->V; ++x) {
    float key = 0.0f;
    if (w[x] > 0.0f) {
      float E = E_at(c, x);
      if (E > 0.0f) {
        key = w[x] / E;
      } else { /* E <= 0 or NaN: invalid draw, key stays 0 */
        *c->status |= ORC_BAD_EXPONENTIAL;
      }
    }
    if (best < 0 || key > bk) {
      bk = key;
      best = x;
    }
  }
  *kmax = bk;
  return best;
}

/* diagnostics of a finished race: how far the winner is from a flip */
static double flip_index(double needed_abs, double needed_rel) {
  double a = needed_abs / 1e-6, r = needed_rel / 1e-5;
  return a > r ? a : r;
}

/* how far a finished race is from a flip: the winner x1 against every x in the
 * support of p or q.  A weight w = max(p - q, 0) (or p) moves by at most
 * delta absolute or eps*(p+q) relative, so keys k = w/E can swap when
 * k1 - k_x <= delta*(1/E1 + 1/E_x) and k1 - k_x <= eps*((p1+q1)/E1 + (p_x+q_x)/E_x). */
static void race_diag(race_ctx *c, const float *w, const float *pa, const float *qa, int win, double *flip,
                      double *relgap) {
  double k1 = 0, e1 = 1;
  if (w[win] > 0.0f) {
    e1 = (double)E_at(c, win);
    k1 = (double)(w[win] / (float)e1);
  }
  double m1 = (double)pa[win] + (qa ? (double)qa[win] : 0.0);
  double fmin = INFINITY, rmin = INFINITY;
  for (int x = 0; x < c->V; ++x) {
    if (x == win) continue;
    int supported = (pa[x] > 0.0f) || (qa && qa[x] > 0.0f);
    if (!supported) continue;
    double ex = (double)E_at(c, x);
    double kx = (w[x] > 0.0f && ex > 0) ? (double)(w[x] / (float)ex) : 0.0;
    double d = k1 - kx;
    double mx = (double)pa[x] + (qa ? (double)qa[x] : 0.0);
    double den_rel = m1 / e1 + mx / ex;
    double f = flip_index(d / (1.0 / e1 + 1.0 / ex), den_rel > 0 ? d / den_rel : INFINITY);
    if (f < fmin) fmin = f;
    double r = k1 > 0 ? d / k1 : 0.0;
    if (r < rmin) rmin = r;
  }
  *flip = fmin;
  *relgap = rmin;
}

/* ------------------------------------------------------------------------
 * Logits processors ("Speculative Decoding: propose, verify, accept", section
 * 06: the same banned tokens and repetition penalty on p and q at a position,
 * listed after temperature, top-k and top-p; "vLLM source walk-through (10)",
 * section "Rejection sampling: the two branches of RejectionSampler", step 2:
 * the sampling constraints first, then the logits processors such as
 * penalties).  Readings: a banned token's logit becomes -inf; the repetition
 * penalty (Keskar et al., CTRL, 2019) divides a positive logit by theta and
 * multiplies a non-positive one by it, once per distinct token of the
 * request's context list plus the drafts y_0 .. y_{j-1} already committed when
 * position j is verified; the result is rounded to the input type (bf16
 * round-to-nearest-even).  Ids outside [0, V) are ignored; a banned token is
 * not penalised.  On a random row the processed values replace the logits of
 * the entries that temperature, top-k and top-p kept (oracle_transform_row);
 * a greedy row (temperature 0) draws nothing, so no sampling constraint
 * applies to it: the processors act on the whole row and its argmax is taken.
 * ------------------------------------------------------------------------ */
static int list_range(const int64_t *cu, int64_t total, int i, int64_t *b, int64_t *e) {
  *b = i ? cu[i - 1] : 0;
  *e = cu[i];
  return *b >= 0 && *e >= *b && *e <= total;
}

static float round_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) {
    u |= 0x00400000u; /* NaN stays NaN */
  } else {
    u += 0x7FFFu + ((u >> 16) & 1u); /* round half to even on the dropped 16 bits */
  }
  u &= 0xFFFF0000u;
  memcpy(&f, &u, sizeof f);
  return f;
}

static int has_processors(const oracle_args *a) {
  return a->entry == ORC_ENTRY_LOGITS && (a->banned_cu || a->repetition_penalty);
}

/* The processors on one row, from explicit lists: banned ids ban[bb..be),
 * penalised ids pen[pb..pe) plus extra[0..nextra) when theta is given. */
static void process_lists(float *row, int V, int dtype, const float *theta, const int32_t *ban, int64_t bb,
                          int64_t be, const int32_t *pen, int64_t pb, int64_t pe, const int32_t *extra,
                          int nextra) {
  unsigned char *mark = calloc((size_t)V, 1); /* 1 banned, 2 penalised */
  for (int64_t k = bb; k < be; ++k) {
    int32_t x = ban[k];
    if (x >= 0 && x < V) mark[x] = 1;
  }
  if (theta) {
    for (int64_t k = pb; k < pe; ++k) {
      int32_t x = pen[k];
      if (x >= 0 && x < V && !mark[x]) mark[x] = 2;
    }
    for (int k = 0; k < nextra; ++k) {
      int32_t x = extra[k];
      if (x >= 0 && x < V && !mark[x]) mark[x] = 2;
    }
  }
  for (int x = 0; x < V; ++x) {
    if (mark[x] == 1) {
      row[x] = -INFINITY;
    } else if (mark[x] == 2) {
      float v = row[x] > 0.0f ? row[x] / *theta : row[x] * *theta;
      row[x] = dtype == ORC_BF16 ? round_to_bf16(v) : v;
    }
  }
  free(mark);
}

/* Position j of request i: its context list plus the drafts y_0 .. y_{j-1}. */
static void process_row(const oracle_args *a, int i, int64_t s, int j, float *row) {
  if (!has_processors(a)) return;
  int64_t bb = 0, be = 0, pb = 0, pe = 0;
  if (a->banned_cu) list_range(a->banned_cu, a->banned_total, i, &bb, &be);
  if (a->penalty_cu) list_range(a->penalty_cu, a->penalty_total, i, &pb, &pe);
  process_lists(row, a->vocab_size, a->dtype, a->repetition_penalty ? &a->repetition_penalty[i] : NULL,
                a->banned_ids, bb, be, a->penalty_ids, pb, pe, a->draft_ids + s, j);
}

/* A usable temperature: 0 (greedy) or a finite value of at least FLT_MIN.
 * Reading: negative, NaN and infinite temperatures are invalid, and so are the
 * subnormal ones in (0, FLT_MIN), whose reciprocal exceeds the fp32 range. */
static int temperature_ok(float t) { return t == 0.0f || (t >= FLT_MIN && !isinf(t)); }

static void emit_invalid(const oracle_args *a, int i) {
  int G = a->max_spec_len;
  for (int k = 0; k <= G; ++k) a->out_tokens[(int64_t)i * (G + 1) + k] = -1;
  a->num_accepted[i] = 0;
  if (a->diag) a->diag[(int64_t)i * ORC_NDIAG + DIAG_PATH] = -1;
}

static void emit(const oracle_args *a, int i, int64_t s, int64_t tb, int g, int A, const int32_t *toks) {
  int G = a->max_spec_len;
  /* stop tokens are checked on the committed prefix only, token by token
   * ("Speculative Decoding: propose, verify, accept", sections 13-14): the
   * commit ends at the first one, and the KV rollback follows the shorter
   * commit (reading: A becomes that token's index) */
  int64_t b, e;
  if (a->stop_cu && list_range(a->stop_cu, a->stop_total, i, &b, &e)) {
    for (int m = 0; m <= A; ++m) {
      int hit = 0;
      for (int64_t k = b; k < e && !hit; ++k) hit = toks[m] == a->stop_ids[k];
      if (hit) {
        A = m;
        break;
      }
    }
  }
  for (int k = 0; k <= G; ++k) a->out_tokens[(int64_t)i * (G + 1) + k] = (k <= A) ? toks[k] : -1;
  a->num_accepted[i] = A;
  /* KV rollback [P3 s3.1]: num_computed_tokens -= gamma_i - A when > 0 */
  if (a->num_computed_tokens && a->num_computed_tokens[i] > 0) a->num_computed_tokens[i] -= (g - A);
  /* rejected drafts' KV slots -> PADDING_SLOT_ID (-1): verify tokens A+1..g */
  if (a->slot_mapping)
    for (int j = A + 1; j <= g; ++j) a->slot_mapping[tb + j] = -1;
  (void)s;
}

/* fetch probability row j of the target (is_target) or draft side */
static int prob_row(const oracle_args *a, int is_target, int64_t row, float T, int top_k, float top_p,
                    float *tmp, float *proc, float *out, int *edge, int i, int64_t s, int j) {
  const void *base = is_target ? a->target : a->draft;
  int64_t stride = is_target ? a->target_row_stride : a->draft_row_stride;
  if (a->entry == ORC_ENTRY_PROBS) {
    load_row(base, ORC_F32, row, stride, a->vocab_size, out);
    return 0;
  }
  load_row(base, a->dtype, row, stride, a->vocab_size, tmp);
  const float *lp = NULL; /* the processed row, when the request has processors */
  if (has_processors(a)) {
    memcpy(proc, tmp, sizeof(float) * (size_t)a->vocab_size);
    process_row(a, i, s, j, proc);
    lp = proc;
  }
  int e = 0;
  int rc = oracle_transform_row(tmp, lp, a->vocab_size, T, top_k, top_p, out, &e);
  if (edge && e) *edge = 1;
  return rc;
}

static void verify_request(const oracle_args *a, int i, float *bufA, float *bufB, float *bufC, float *bufD,
                           float *bufE, int32_t *toks, race_ctx *rc) {
  const int G = a->max_spec_len, V = a->vocab_size;
  double *dg = a->diag ? a->diag + (int64_t)i * ORC_NDIAG : NULL;
  if (dg) {
    dg[DIAG_ACCEPT_MARGIN] = INFINITY;
    dg[DIAG_RACE_FLIP] = INFINITY;
    dg[DIAG_RACE_RELGAP] = INFINITY;
    dg[DIAG_TOPP_EDGE] = 0;
    dg[DIAG_FALLBACK] = 0;
    dg[DIAG_PATH] = 0;
  }
  /* ragged decode [P1 "SpecDecodeMetadata"] */
  int64_t s, e;
  if (a->cu_num_draft_tokens) {
    s = i ? a->cu_num_draft_tokens[i - 1] : 0;
    e = a->cu_num_draft_tokens[i];
  } else {
    s = (int64_t)i * G;
    e = s + G;
  }
  if (s < 0 || e < s || e > a->num_draft_tokens_total || e - s > G) {
    *a->status |= ORC_BAD_CU;
    emit_invalid(a, i);
    return;
  }
  const int g = (int)(e - s);
  const int64_t tb = s + i; /* first target row of request i */

  float temp = a->temperature ? a->temperature[i] : 1.0f;
  if (!temperature_ok(temp)) {
    *a->status |= ORC_BAD_PARAM;
    emit_invalid(a, i);
    return;
  }

  {
    int64_t b, e;
    if ((a->penalty_cu && !list_range(a->penalty_cu, a->penalty_total, i, &b, &e)) ||
        (a->banned_cu && !list_range(a->banned_cu, a->banned_total, i, &b, &e)) ||
        (a->stop_cu && !list_range(a->stop_cu, a->stop_total, i, &b, &e))) {
      *a->status |= ORC_BAD_LIST;
      emit_invalid(a, i);
      return;
    }
    if (a->repetition_penalty && a->entry == ORC_ENTRY_LOGITS &&
        !(a->repetition_penalty[i] > 0.0f && !isinf(a->repetition_penalty[i]))) {
      *a->status |= ORC_BAD_PARAM;
      emit_invalid(a, i);
      return;
    }
  }

  /* ---- greedy path (temperature 0) [P1 "Greedy kernel"; P2 s03] ---- */
  if (temp == 0.0f) {
    if (dg) dg[DIAG_PATH] = 1;
    for (int j = 0; j <= g; ++j) {
      load_row(a->target, a->entry == ORC_ENTRY_PROBS ? ORC_F32 : a->dtype, tb + j, a->target_row_stride, V,
               bufA);
      process_row(a, i, s, j, bufA);
      int gj = argmax_row(bufA, V);
      if (gj < 0) {
        *a->status |= ORC_BAD_VALUES;
        emit_invalid(a, i);
        return;
      }
      toks[j] = gj;
      if (j == g) { /* all matched: bonus = argmax of the last row */
        emit(a, i, s, tb, g, g, toks);
        return;
      }
      int32_t y = a->draft_ids[s + j];
      if (y < 0 || y >= V) {
        *a->status |= ORC_BAD_DRAFT_ID;
        emit_invalid(a, i);
        return;
      }
      if (y != gj) { /* first mismatch: commit the target's choice, stop */
        emit(a, i, s, tb, g, j, toks);
        return;
      }
    }
    return; /* not reached */
  }

  /* ---- random path [P2 s04, s06; P1 "Random kernel"] ---- */
  int top_k = 0;
  float top_p = 1.0f;
  if (a->entry == ORC_ENTRY_LOGITS) {
    top_k = a->top_k ? a->top_k[i] : 0;
    top_p = a->top_p ? a->top_p[i] : 1.0f;
    if (!(top_p > 0.0f)) {
      *a->status |= ORC_BAD_PARAM;
      emit_invalid(a, i);
      return;
    }
  }
  rc->rng_req = a->rng_request_base + (uint32_t)i;
  rc->E_row = a->exponentials ? a->exponentials + (int64_t)i * a->exponentials_row_stride : NULL;
  if (!rc->test_mode) memset(rc->E_have, 0, (size_t)V);

  int j0 = 0; /* first position whose rows are read */
  if (a->synthetic_rates) {
    for (int j = 0; j < g; ++j) {
      float rj = a->synthetic_rates[j];
      if (!(rj >= 0.0f && rj <= 1.0f) || (j > 0 && rj > a->synthetic_rates[j - 1])) {
        *a->status |= ORC_BAD_PARAM;
        emit_invalid(a, i);
        return;
      }
    }
    for (; j0 < g; ++j0) {
      int32_t y = a->draft_ids[s + j0];
      if (y < 0 || y >= V) {
        *a->status |= ORC_BAD_DRAFT_ID;
        emit_invalid(a, i);
        return;
      }
      float u = rc->test_mode ? a->uniforms[s + j0]
                              : oracle_uniform(a->seed, a->offset, rc->rng_req, (uint32_t)j0);
      if (!(u < a->synthetic_rates[j0])) break; /* first synthetic rejection */
      toks[j0] = y;
    }
  }
  int edge = 0;
  for (int j = j0; j < g; ++j) {
    if (!a->draft) {
      *a->status |= ORC_MISSING_DRAFT;
      emit_invalid(a, i);
      return;
    }
    float *p = bufA, *q = bufB;
    int bad = prob_row(a, 1, tb + j, temp, top_k, top_p, bufC, bufE, p, &edge, i, s, j);
    bad |= prob_row(a, 0, s + j, temp, top_k, top_p, bufD, bufE, q, &edge, i, s, j);
    if (bad) {
      *a->status |= ORC_BAD_VALUES;
      emit_invalid(a, i);
      return;
    }
    if (dg && edge) dg[DIAG_TOPP_EDGE] = 1;
    int32_t y = a->draft_ids[s + j];
    if (y < 0 || y >= V) {
      *a->status |= ORC_BAD_DRAFT_ID;
      emit_invalid(a, i);
      return;
    }
    float py = p[y], qy = q[y];
    if (a->dbg_py && !a->synthetic_rates) a->dbg_py[s + j] = py;
    if (a->dbg_qy && !a->synthetic_rates) a->dbg_qy[s + j] = qy;
    float u = rc->test_mode ? a->uniforms[s + j] : oracle_uniform(a->seed, a->offset, rc->rng_req, (uint32_t)j);
    if (dg && !a->synthetic_rates) { /* flip index of the test u*q < p (exact zeros on both sides cannot flip) */
      double uq = (double)u * (double)qy, gap = fabs(uq - (double)py), scale = uq + (double)py;
      double mg = scale > 0 ? flip_index(gap, gap / scale) : INFINITY;
      if (mg < dg[DIAG_ACCEPT_MARGIN]) dg[DIAG_ACCEPT_MARGIN] = mg;
    }
    float uq = u * qy; /* fp32 product, then a strict fp32 comparison */
    /* synthetic mode reaches the rows only at its first rejection */
    if (!a->synthetic_rates && uq < py) { /* accept y_j */
      toks[j] = y;
      continue;
    }
    /* first rejection: replacement from max(p - q, 0) [P2 s04] */
    float *w = bufC; /* reuse: the logits row is no longer needed */
    for (int x = 0; x < V; ++x) {
      float d = p[x] - q[x];
      w[x] = (d > 0.0f) ? d : 0.0f;
    }
    float kmax;
    int tok = race(rc, w, &kmax);
    if (kmax == 0.0f) { /* no positive residual key: draw from p instead */
      if (dg) dg[DIAG_FALLBACK] = 1;
      for (int x = 0; x < V; ++x) w[x] = (p[x] > 0.0f) ? p[x] : 0.0f;
      tok = race(rc, w, &kmax);
      if (kmax == 0.0f) *a->status |= ORC_EMPTY_DISTRIBUTION;
      if (dg) race_diag(rc, w, p, NULL, tok, &dg[DIAG_RACE_FLIP], &dg[DIAG_RACE_RELGAP]);
    } else if (dg) {
      race_diag(rc, w, p, q, tok, &dg[DIAG_RACE_FLIP], &dg[DIAG_RACE_RELGAP]);
    }
    toks[j] = tok;
    emit(a, i, s, tb, g, j, toks);
    return;
  }
  /* every draft accepted: bonus token from the last target row [P1; P2 s06] */
  float *p = bufA;
  if (prob_row(a, 1, tb + g, temp, top_k, top_p, bufC, bufE, p, &edge, i, s, g)) {
    *a->status |= ORC_BAD_VALUES;
    emit_invalid(a, i);
    return;
  }
  if (dg && edge) dg[DIAG_TOPP_EDGE] = 1;
  float *w = bufB;
  for (int x = 0; x < V; ++x) w[x] = (p[x] > 0.0f) ? p[x] : 0.0f;
  float kmax;
  int tok = race(rc, w, &kmax);
  if (kmax == 0.0f) *a->status |= ORC_EMPTY_DISTRIBUTION;
  if (dg) race_diag(rc, w, p, NULL, tok, &dg[DIAG_RACE_FLIP], &dg[DIAG_RACE_RELGAP]);
  toks[g] = tok;
  emit(a, i, s, tb, g, g, toks);
}

/* Verify requests [req_begin, req_end) of the batch described by *a. */
int oracle_verify_range(const oracle_args *a, int req_begin, int req_end) {
  const int V = a->vocab_size;
  if (V <= 0 || a->max_spec_len < 0) return -1;
  float *buf = (float *)malloc(sizeof(float) * (size_t)V * 5);
  int32_t *toks = (int32_t *)malloc(sizeof(int32_t) * (size_t)(a->max_spec_len + 1));
  float *E_cache = (float *)malloc(sizeof(float) * (size_t)V);
  unsigned char *E_have = (unsigned char *)malloc((size_t)V);
  if (!buf || !toks || !E_cache || !E_have) {
    free(buf); free(toks); free(E_cache); free(E_have);
    return -2;
  }
  race_ctx rc;
  memset(&rc, 0, sizeof rc);
  rc.a = a;
  rc.status = a->status;
  rc.V = V;
  rc.test_mode = (a->exponentials != NULL);
  rc.E_cache = E_cache;
  rc.E_have = E_have;
  for (int i = req_begin; i < req_end; ++i)
    verify_request(a, i, buf, buf + V, buf + 2 * (size_t)V, buf + 3 * (size_t)V, buf + 4 * (size_t)V, toks, &rc);
  free(buf);
  free(toks);
  free(E_cache);
  free(E_have);
  return 0;
}

int oracle_verify(const oracle_args *a) { return oracle_verify_range(a, 0, a->num_reqs); }

int oracle_sizeof_args(void) { return (int)sizeof(oracle_args); }

/* ------------------------------------------------------------------------ */
/* draft-side sampler: one token per logits row from the transformed row     */
/* ("vLLM source walk-through (10)", section "propose() multi-step loop":    */
/* _sample_draft_tokens draws each draft token from the draft distribution;  */
/* "Speculative Decoding: propose, verify, accept", section 02: the draft    */
/* keeps every step's distribution q_i).  Same transform as the verifier's    */
/* rows, same exponential race; temperature 0 takes the argmax.  Production  */
/* draws use the verifier's E counter under the key (seed_lo, seed_hi ^      */
/* 0x53414D50) so the sampler and the verifier never share a stream.          */
/* ------------------------------------------------------------------------ */
int oracle_sample_rows(int32_t rows, int32_t V, int32_t dtype, const void *logits, int64_t row_stride,
                       const float *temperature, const int32_t *top_k, const float *top_p,
                       const float *exponentials, int64_t exp_stride, uint64_t seed, uint64_t offset,
                       uint32_t rng_row_base, int32_t *tokens, float *probs_out, int32_t *status,
                       double *diag /* [rows, 2]: race flip index, top-p edge */,
                       /* logits processors per row (lists as in oracle_args, row r = request r) */
                       const float *repetition_penalty, const int64_t *penalty_cu, const int32_t *penalty_ids,
                       int64_t penalty_total, const int64_t *banned_cu, const int32_t *banned_ids,
                       int64_t banned_total) {
  float *l = (float *)malloc(sizeof(float) * (size_t)V);
  float *lp = (float *)malloc(sizeof(float) * (size_t)V);
  float *p = (float *)malloc(sizeof(float) * (size_t)V);
  float *E = (float *)malloc(sizeof(float) * (size_t)V);
  if (!l || !lp || !p || !E) {
    free(l); free(lp); free(p); free(E);
    return -2;
  }
  const uint64_t skey = seed ^ ((uint64_t)0x53414D50u << 32);
  for (int r = 0; r < rows; ++r) {
    load_row(logits, dtype, r, row_stride, V, l);
    float temp = temperature ? temperature[r] : 1.0f;
    if (diag) {
      diag[2 * r] = INFINITY;
      diag[2 * r + 1] = 0;
    }
    if (!temperature_ok(temp)) {
      *status |= ORC_BAD_PARAM;
      tokens[r] = -1;
      continue;
    }
    {
      int64_t pb = 0, pe = 0, bb = 0, be = 0;
      if ((penalty_cu && !list_range(penalty_cu, penalty_total, r, &pb, &pe)) ||
          (banned_cu && !list_range(banned_cu, banned_total, r, &bb, &be))) {
        *status |= ORC_BAD_LIST;
        tokens[r] = -1;
        continue;
      }
      if (repetition_penalty && !(repetition_penalty[r] > 0.0f && !isinf(repetition_penalty[r]))) {
        *status |= ORC_BAD_PARAM;
        tokens[r] = -1;
        continue;
      }
      /* the processed copy of the row (the raw row still places the cuts) */
      memcpy(lp, l, sizeof(float) * (size_t)V);
      if (banned_cu || repetition_penalty)
        process_lists(lp, V, dtype, repetition_penalty ? &repetition_penalty[r] : NULL, banned_ids, bb, be,
                      penalty_ids, pb, pe, NULL, 0);
    }
    if (temp == 0.0f) { /* greedy drafting: argmax of the processed logits */
      int g = argmax_row(lp, V);
      if (g < 0) *status |= ORC_BAD_VALUES;
      tokens[r] = g;
      continue;
    }
    int k = top_k ? top_k[r] : 0;
    float tp = top_p ? top_p[r] : 1.0f;
    if (!(tp > 0.0f)) {
      *status |= ORC_BAD_PARAM;
      tokens[r] = -1;
      continue;
    }
    int edge = 0;
    if (oracle_transform_row(l, (banned_cu || repetition_penalty) ? lp : NULL, V, temp, k, tp, p, &edge)) {
      *status |= ORC_BAD_VALUES;
      tokens[r] = -1;
      continue;
    }
    for (int x = 0; x < V; ++x) {
      if (exponentials) {
        E[x] = exponentials[(int64_t)r * exp_stride + x];
      } else {
        uint32_t w = philox_word(skey, offset, (uint32_t)x / 4u, 2u * (rng_row_base + (uint32_t)r), (int)(x % 4u));
        E[x] = (float)(-log((double)((float)(2u * (w >> 9) + 1u) * 0x1p-24f)));
      }
    }
    int best = -1;
    float bk = 0.0f;
    for (int x = 0; x < V; ++x) {
      float key = 0.0f;
      if (p[x] > 0.0f) {
        if (E[x] > 0.0f) key = p[x] / E[x];
        else *status |= ORC_BAD_EXPONENTIAL;
      }
      if (best < 0 || key > bk) {
        bk = key;
        best = x;
      }
    }
    if (bk == 0.0f) *status |= ORC_EMPTY_DISTRIBUTION;
    tokens[r] = best;
    if (probs_out)
      for (int x = 0; x < V; ++x) probs_out[(int64_t)r * V + x] = p[x];
    if (diag) {
      double k1 = (double)bk, e1 = (double)E[best], m1 = (double)p[best], fmin = INFINITY;
      for (int x = 0; x < V; ++x) {
        if (x == best || !(p[x] > 0.0f)) continue;
        double kx = (E[x] > 0) ? (double)(p[x] / E[x]) : 0.0, d = k1 - kx;
        double f = flip_index(d / (1.0 / e1 + 1.0 / (double)E[x]), d / (m1 / e1 + (double)p[x] / (double)E[x]));
        if (f < fmin) fmin = f;
      }
      diag[2 * r] = fmin;
      diag[2 * r + 1] = edge;
    }
  }
  free(l);
  free(lp);
  free(p);
  free(E);
  return 0;
}

/* ------------------------------------------------------------------------
 * N-gram proposer ("vLLM source walk-through (10)", section "NgramProposer":
 * no draft model; the history is read backwards so that "the current tail
 * seen earlier" becomes a prefix match, KMP-style, with match lengths capped
 * at max_ngram; the longest match with length in [min_ngram, max_ngram]
 * proposes the k tokens that followed it).
 *
 * Written out as its definition: r[j] = t[L-1-j] is the history read
 * backwards.  For each end index i in [1, L), m(i) is the largest
 * m <= min(max_ngram, i) with r[i-m+1 .. i] == r[0 .. m-1], i.e. the
 * occurrence t[L-1-i .. L-1-i+m) equals the last m tokens and is followed by
 * at least one token.  m* = max_i m(i); nothing is proposed if m* < min_ngram.
 * Otherwise i* is the smallest i with m(i) = m* -- the first match a scan of
 * r meets, the most recent occurrence in t -- and the proposal is
 * t[start .. start + k'), start = L - 1 - i* + m*, k' = min(k, max_model_len - L,
 * L - start).  Requests use the verifier's ragged layout: request q owns
 * tokens [cu[q-1], cu[q]) (cu[-1] = 0).  Output rows are [R, k], -1 after the
 * proposal; num[q] = k'.  Returns the status bits (1: bad cu range).
 * ------------------------------------------------------------------------ */
int oracle_ngram_propose(int32_t R, const int32_t *tokens, const int64_t *cu, int64_t total, int32_t min_ngram,
                         int32_t max_ngram, int32_t k, int64_t max_model_len, int32_t *out, int32_t *num) {
  int status = 0;
  for (int32_t q = 0; q < R; ++q) {
    int32_t *row = out + (int64_t)q * k;
    for (int32_t c = 0; c < k; ++c) row[c] = -1;
    num[q] = 0;
    const int64_t s = q ? cu[q - 1] : 0, e = cu[q];
    if (s < 0 || e < s || e > total) {
      status |= ORC_BAD_CU;
      continue;
    }
    const int32_t *t = tokens + s;
    const int64_t L = e - s;
    if (L < min_ngram) continue;
    int64_t kk = k;
    if (max_model_len - L < kk) kk = max_model_len - L;
    if (kk <= 0) continue;
    int64_t best_m = 0, best_i = -1;
    for (int64_t i = 1; i < L; ++i) {
      int64_t cap = i < max_ngram ? i : max_ngram;
      int64_t m = 0;
      for (int64_t len = cap; len >= 1; --len) { /* largest len whose windows agree */
        int same = 1;
        for (int64_t j = 0; j < len && same; ++j)
          if (t[L - 1 - (i - len + 1 + j)] != t[L - 1 - j]) same = 0;
        if (same) {
          m = len;
          break;
        }
      }
      if (m > best_m) { /* strictly longer only: the earliest i keeps a tie */
        best_m = m;
        best_i = i;
      }
    }
    if (best_m < min_ngram) continue;
    const int64_t start = L - 1 - best_i + best_m;
    if (L - start < kk) kk = L - start;
    for (int64_t c = 0; c < kk; ++c) row[c] = t[start + c];
    num[q] = (int32_t)kk;
  }
  return status;
}
