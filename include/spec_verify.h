/*
 * spec_verify.h -- C ABI of the batched speculative-decoding verifier
 * (rejection sampler) for NVIDIA GB300 (sm_103a).
 *
 * What it computes (page titles and sections of the sources it follows):
 *  - "Speculative Decoding: propose, verify, accept", section 02: per request
 *    draft ids [gamma], draft distributions q [gamma, V] and target
 *    distributions p [gamma+1, V]; section 04: draft y is accepted iff
 *    u < min(1, p(y)/q(y)), evaluated here as fl32(u * q(y)) < p(y); the first
 *    rejection is replaced by a draw from max(0, p - q) renormalised;
 *    section 06: keep the accepted prefix, stop at the first rejection, draw a
 *    bonus token from p[gamma] when every draft is accepted; section 03:
 *    temperature 0 compares the draft with the target argmax.
 *  - "vLLM source walk-through (10): speculative decoding", section
 *    "SpecDecodeMetadata": flattened drafts with cu_num_draft_tokens (inclusive
 *    prefix sums) and max_spec_len; section "Rejection sampling: the two
 *    branches of RejectionSampler": identical temperature/top-k/top-p on the
 *    target and draft sides, output [batch, max_spec_len + 1] filled with
 *    PLACEHOLDER_TOKEN_ID = -1; section "Random kernel": categorical draws by
 *    an exponential race (argmax of weight / exponential draw); section
 *    "Scheduler and KV": rejected draft KV slots become PADDING_SLOT_ID = -1.
 *  - "How speculative decoding interacts with the KV cache", section 3.1:
 *    num_computed_tokens -= gamma - A when it is > 0.
 *
 * Memory and execution model: every pointer in spec_verify_args is a DEVICE
 * pointer on the handle's device, owned by the caller (the library allocates
 * nothing per call).  For the probability entry, target/draft/exponentials may
 * also point into pinned host memory mapped into the device address space
 * (unified addressing): the kernel then reads only the rows a call needs over
 * the host link (NVLink-C2C on GB300).  The logits entry needs device rows.  spec_verify_run only validates on the host and enqueues
 * kernels on the caller's stream; it never synchronises.  Errors visible on
 * the host are returned before anything is enqueued.  Errors in the data are
 * reported through the optional device word `status` (bitwise OR of
 * SV_DATA_* bits; the caller zeroes it) and never trap: a request with invalid
 * data emits nothing (its output row stays -1, num_accepted 0, KV bookkeeping
 * untouched).  One handle may be used from one host thread at a time; calls on
 * different streams must not share output buffers.
 */
#ifndef SPEC_VERIFY_H_
#define SPEC_VERIFY_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SPEC_VERIFY_ABI_VERSION 8u
#define SV_PLACEHOLDER_TOKEN_ID (-1)
#define SV_PADDING_SLOT_ID (-1)
#define SV_MAX_SPEC_LEN 256 /* largest max_spec_len a handle accepts */
#define SV_MAX_NGRAM 64     /* largest max_ngram of the n-gram proposer */

/* Host-visible result codes. */
typedef enum sv_status {
  SV_OK = 0,
  SV_ERR_INVALID_ARG = 1, /* a null, negative, out-of-range or inconsistent argument */
  SV_ERR_UNSUPPORTED = 2, /* a combination this build does not implement (e.g. probs + bf16) */
  SV_ERR_CUDA = 3,        /* a CUDA runtime call failed; see spec_verify_last_error() */
  SV_ERR_CAPACITY = 4     /* the call exceeds the limits the handle was created with */
} sv_status;

/* Input kinds. */
enum sv_entry {
  SV_ENTRY_PROBS = 0, /* target/draft rows are fp32 probabilities, already transformed */
  SV_ENTRY_LOGITS = 1 /* target/draft rows are logits; temperature/top-k/top-p applied here */
};
enum sv_dtype { SV_F32 = 0, SV_BF16 = 1 };

/* Device status bits (bitwise OR into *status). */
enum sv_data_status {
  SV_DATA_BAD_CU = 1,             /* cu_num_draft_tokens not a valid range for this request */
  SV_DATA_BAD_DRAFT_ID = 2,       /* draft id outside [0, V) at an examined position */
  SV_DATA_BAD_EXPONENTIAL = 4,    /* test-mode E <= 0 or NaN where a key needed it (key taken as 0) */
  SV_DATA_EMPTY_DISTRIBUTION = 8, /* a draw found no positive key; token 0 emitted */
  SV_DATA_BAD_VALUES = 16,        /* NaN (greedy) or NaN/+inf/no finite logit (random logits) in a read row,
                                     or a kept set left empty by banned tokens */
  SV_DATA_BAD_PARAM = 32,         /* temperature < 0/NaN/inf/subnormal, or top_p <= 0/NaN */
  SV_DATA_MISSING_DRAFT = 64,     /* draft == NULL but a random request needs draft rows */
  SV_DATA_COPY_TIMEOUT = 128,     /* a bulk row copy did not complete within its wait limit (request
                                     emits nothing); never expected on a healthy GPU */
  SV_DATA_BAD_LIST = 256          /* a penalty, banned or stop list range of the request is invalid */
};

/* Handle flags.  SV_FLAG_RESIDENT_ROWS: the logits entry copies both the
 * target and the draft row chunk of a position into shared memory (two CTAs
 * per SM), and the sampler its row chunk.  By default aligned rows are read
 * in place after an L2 prefetch (four CTAs per SM); unaligned rows are always
 * copied.  Results are identical. */
#define SV_FLAG_RESIDENT_ROWS 1u
/* SV_FLAG_ONE_CTA_PER_REQUEST: logits-entry and sampler calls with aligned
 * rows (with or without logits processors), in a handle without
 * SV_FLAG_RESIDENT_ROWS, always take the
 * one-CTA-per-request (per-row) form (see SV_HINT_SMALL_TOP_K); by default
 * the library takes it only for hinted calls with at least two requests
 * (rows) per SM.  Without processors the two forms' results are identical;
 * with processors both stay within the tolerance of the exact definition
 * (the one-CTA form sums the processed kept set afresh, the cluster form
 * corrects the raw sum). */
#define SV_FLAG_ONE_CTA_PER_REQUEST 2u
/* SV_FLAG_SERIAL_LAUNCH: launch the handle's kernels in plain stream order.
 * By default every kernel is launched with programmatic stream serialization
 * (CUDA's programmatic dependent launch): it may be scheduled onto the SMs
 * while the previous kernel in the stream is still running, and its first
 * instruction waits until that kernel has completed and all of its memory
 * writes are visible.  Nothing is read or written earlier than in plain stream
 * order, so results are identical; only the gap between back-to-back kernels
 * shrinks.  Work that is not a kernel (copies, event records, host callbacks)
 * orders the stream as usual. */
#define SV_FLAG_SERIAL_LAUNCH 4u

/* Call hints (the hints field of spec_verify_args and spec_verify_sample_args;
 * they never change a result).  SV_HINT_SMALL_TOP_K: the caller states that
 * every random request (row) of the call has 1 <= top_k <= SV_SMALL_TOP_K_MAX.
 * For such a batch, large enough to give every request its own CTA at once,
 * the sampler samples each row with one CTA the same way, and the logits entry verifies
 * each request with one CTA that reads a position's two rows once (keeping
 * the largest key of every 128-byte block), reads again the few blocks that
 * can hold the top-k set, and derives the threshold, the top-p cut, the
 * normaliser and the race from those candidates; a request outside the
 * statement is still verified exactly, by a slower multi-pass path. */
#define SV_HINT_SMALL_TOP_K 1u
#define SV_SMALL_TOP_K_MAX 256

/* Call flags for tests (the test_flags field of the argument structs; 0 in
 * normal use).  SV_TEST_EXPIRE_COPY_WAIT: the first wait for every bulk row
 * copy into shared memory gives up at once, as if the copy had not completed
 * within its limit; the copy still gets the ordinary second wait, so it lands
 * before the CTA moves on.  The requests that copied rows then report
 * SV_DATA_COPY_TIMEOUT and emit nothing.  Only calls whose rows are copied
 * (SV_FLAG_RESIDENT_ROWS, or unaligned rows) are affected. */
#define SV_TEST_EXPIRE_COPY_WAIT 1u

typedef struct spec_verify_ctx *spec_verify_t;

/* Limits fixed at creation. */
typedef struct spec_verify_config {
  int32_t max_num_reqs; /* largest num_reqs of any call (>= 1) */
  int32_t max_spec_len; /* largest max_spec_len of any call (0 .. SV_MAX_SPEC_LEN) */
  int32_t vocab_size;   /* largest vocab_size of any call (>= 1) */
  int32_t device;       /* CUDA device ordinal the handle's calls run on */
  int32_t cluster_ctas; /* CTAs cooperating on one request: 0 = automatic, else 1, 2, 4, 8 or 16 */
  uint32_t flags;       /* 0, or SV_FLAG_* bits */
} spec_verify_config;

/* One verification call.  N = num_reqs, G = max_spec_len, V = vocab_size,
 * T = num_draft_tokens_total.  Request i owns draft rows [s_i, s_i + gamma_i)
 * and target rows [s_i + i, s_i + i + gamma_i] (its last target row is the
 * bonus row), where s_i = cu[i-1] (0 for i = 0) and gamma_i = cu[i] - s_i. */
typedef struct spec_verify_args {
  int32_t num_reqs;     /* N >= 0 (N = 0 is a no-op) */
  int32_t max_spec_len; /* G: output row length is G + 1; every gamma_i <= G */
  int32_t vocab_size;   /* V >= 1 */
  int32_t entry;        /* SV_ENTRY_PROBS or SV_ENTRY_LOGITS */
  int32_t dtype;        /* SV_F32 (both entries) or SV_BF16 (logits entry only) */
  uint32_t hints;       /* 0, or SV_HINT_* bits */
  int64_t num_draft_tokens_total; /* T = cu[N-1]; must equal N*G when cu == NULL */

  const int32_t *draft_ids;           /* [T] draft token ids, request-major */
  const int32_t *cu_num_draft_tokens; /* [N] inclusive prefix sums, or NULL: every gamma_i = G */
  const void *target;                 /* [T+N rows, target_row_stride] p rows or target logits */
  int64_t target_row_stride;          /* elements between target rows (>= V) */
  const void *draft;                  /* [T rows, draft_row_stride] q rows or draft logits; may be NULL
                                         when no random request has drafts */
  int64_t draft_row_stride;           /* elements between draft rows (>= V) */

  const float *temperature; /* [N]; 0 selects the greedy path; NULL = 1 for every request */
  const int32_t *top_k;     /* [N] or NULL; <= 0 or >= V disables (logits entry only) */
  const float *top_p;       /* [N] or NULL; >= 1 disables; must be > 0 (logits entry only) */

  /* Randomness.  Test mode: exponentials set (and uniforms, unless T = 0);
   * u [T] in [0, 1) and E [N rows, exponentials_row_stride] > 0 are read as
   * given.  Production mode: both NULL; u and E come from Philox4x32-10 (Salmon et al., SC'11) with key
   * (seed) and counters (j/4, 2r+1, offset) for u_j and (x/4, 2r, offset) for
   * E(x), r = rng_request_base + i; u = (w >> 8) 2^-24, E = -ln((2(w >> 9)+1) 2^-24). */
  const float *uniforms;
  const float *exponentials;
  int64_t exponentials_row_stride;
  uint64_t seed;
  uint64_t offset;
  uint32_t rng_request_base;
  uint32_t test_flags; /* 0, or SV_TEST_EXPIRE_COPY_WAIT (tests only) */

  /* Outputs. */
  int32_t *out_tokens;          /* [N, G+1] committed tokens, -1 after the last one */
  int32_t *num_accepted;        /* [N] accepted draft count A */
  int32_t *num_computed_tokens; /* [N] in/out or NULL: -= gamma_i - A when > 0 */
  int64_t *slot_mapping;        /* [T+N] in/out or NULL: verify tokens j in (A, gamma_i] -> -1 */
  float *dbg_py;                /* [T] or NULL: p_j(y_j) at examined positions j <= min(A, gamma_i - 1) */
  float *dbg_qy;                /* [T] or NULL: q_j(y_j) at the same positions */
  int32_t *status;              /* [1] or NULL: SV_DATA_* bits OR-ed in */

  /* Synthetic acceptance ("vLLM source walk-through (10)", section "About
   * synthetic / block verification": preset per-position rates, non-increasing,
   * accept with "uniform < rate" instead of the probability test).  [G] device
   * array in [0, 1], or NULL for the ordinary test.  Only the decision changes:
   * rows before the stopping position are never read, the replacement or bonus
   * draw there is the ordinary one, and dbg_py/dbg_qy are not written.  Rates
   * outside [0, 1] or increasing over a request's positions: SV_DATA_BAD_PARAM. */
  const float *synthetic_acceptance_rates;

  /* Logits processors, logits entry only ("Speculative Decoding: propose,
   * verify, accept", section 06: the same banned tokens and repetition penalty
   * on p and q at a position, after temperature, top-k and top-p; "vLLM
   * source walk-through (10)", section "Rejection sampling: the two branches
   * of RejectionSampler", step 2: the sampling constraints first, then the
   * processors).  Lists are per request, like cu_num_draft_tokens: request i
   * owns entries [cu[i-1], cu[i]) (cu[-1] = 0) of the id array; ids outside
   * [0, V) are ignored and repeats count once.  A banned token's logit
   * becomes -inf.  With repetition_penalty, every distinct token of the
   * request's penalty list, plus the drafts y_0 .. y_{j-1} when position j is
   * verified, has its logit l replaced by l / theta if l > 0, else l * theta
   * (fp32 arithmetic, rounded to the logits' type), on the target and the
   * draft row alike; banned tokens are not penalised.  On a random row the
   * kept set is placed on the raw logits (temperature, top-k, top-p); the
   * processed values then replace the kept logits and the kept set is
   * renormalised (an entry the cuts dropped stays dropped; a kept set whose
   * every entry is banned is SV_DATA_BAD_VALUES).  A greedy row takes the
   * argmax of the whole processed row.  Theta must be > 0 and finite (else
   * SV_DATA_BAD_PARAM).  The probability entry rejects these fields (its rows
   * are already transformed). */
  const float *repetition_penalty;    /* [N] theta, or NULL: no penalty */
  const int64_t *penalty_cu;          /* [N] or NULL */
  const int32_t *penalty_token_ids;   /* [penalty_total] */
  int64_t penalty_total;
  const int64_t *banned_cu;           /* [N] or NULL */
  const int32_t *banned_token_ids;    /* [banned_total] */
  int64_t banned_total;

  /* Stop tokens, both entries ("Speculative Decoding: propose, verify,
   * accept", sections 13-14: stop rules are checked on the committed prefix
   * only, token by token).  If a committed token c_m (m <= A) is in the
   * request's stop list, the commit ends at the first such m: out row
   * c_0 .. c_m, num_accepted = m, and the KV rollback follows (gamma_i - m
   * tokens, slots of verify tokens m+1 .. gamma_i). */
  const int64_t *stop_cu;             /* [N] or NULL */
  const int32_t *stop_token_ids;      /* [stop_total] */
  int64_t stop_total;
} spec_verify_args;

/* Draft-side sampler ("vLLM source walk-through (10)", section "propose()
 * multi-step loop": each draft step samples its token from the draft model's
 * distribution and keeps that distribution for the rejection sampler).  One
 * token per logits row: the row goes through the verifier's own transform
 * (temperature, top-k, softmax, top-p) and the token is drawn by the same
 * exponential race; temperature 0 takes the argmax (lowest index).  The
 * transformed fp32 row can be written out, ready to be the q input of the
 * probability entry.  R = num_rows, V = vocab_size.  Production draws use the
 * verifier's E counters under the key (seed_lo, seed_hi ^ 0x53414D50), so a
 * sampler call and a verifier call with the same seed never share a stream. */
typedef struct spec_verify_sample_args {
  int32_t num_rows;   /* R >= 0 (0 is a no-op); at most the handle's max_num_reqs */
  int32_t vocab_size; /* V, at most the handle's vocab_size */
  int32_t dtype;      /* SV_F32 or SV_BF16 logits */
  uint32_t hints;     /* 0, or SV_HINT_* bits */
  const void *logits; /* [R rows, row_stride] */
  int64_t row_stride; /* elements between rows (>= V) */
  const float *temperature; /* [R] or NULL (= 1) */
  const int32_t *top_k;     /* [R] or NULL */
  const float *top_p;       /* [R] or NULL */
  const float *exponentials; /* test mode: [R rows, exponentials_row_stride] E > 0; NULL = Philox */
  int64_t exponentials_row_stride;
  uint64_t seed;
  uint64_t offset;
  uint32_t rng_row_base; /* stream of row r: rng_row_base + r */
  uint32_t test_flags;   /* 0, or SV_TEST_EXPIRE_COPY_WAIT (tests only) */
  int32_t *tokens;       /* [R] out: sampled token, -1 for an invalid row */
  float *probs;          /* [R rows, probs_row_stride] out or NULL: the transformed row (random rows only) */
  int64_t probs_row_stride;
  int32_t *status;       /* [1] or NULL: SV_DATA_* bits OR-ed in */

  /* Logits processors per row, as in spec_verify_args (row r = request r;
   * no drafts are added implicitly: a row's penalty list holds its whole
   * context, drafts sampled before it included), so that the sampled q is the
   * q the verifier rebuilds. */
  const float *repetition_penalty;    /* [R] theta, or NULL */
  const int64_t *penalty_cu;          /* [R] or NULL */
  const int32_t *penalty_token_ids;
  int64_t penalty_total;
  const int64_t *banned_cu;           /* [R] or NULL */
  const int32_t *banned_token_ids;
  int64_t banned_total;
} spec_verify_sample_args;

sv_status spec_verify_sample(spec_verify_t handle, const spec_verify_sample_args *args, void *stream);

/* Host-only validation of sampler arguments against `config`. */
sv_status spec_verify_check_sample_args(const spec_verify_config *config, const spec_verify_sample_args *args);

/* Batched n-gram proposer ("vLLM source walk-through (10)", section
 * "NgramProposer": no draft model; the tail of a request's token history is
 * looked up earlier in the history -- the history read backwards, match
 * lengths capped at max_ngram -- and the longest match with a length in
 * [min_ngram, max_ngram] proposes the tokens that followed it).  Exactly: for
 * every end position E <= L - 2 of a request's history t[0 .. L), l(E) is the
 * number of j = 0, 1, ... with t[E - j] == t[L - 1 - j], capped at max_ngram
 * and at E + 1.  The proposal follows the E with the largest l(E), the latest
 * such E on ties (the most recent occurrence), if that l is at least
 * min_ngram: draft = t[E + 1 .. E + 1 + k'), k' = min(k, max_model_len - L,
 * L - 1 - E).  Otherwise nothing is proposed.  R = num_reqs; one CTA per
 * request reads its history once from HBM. */
typedef struct spec_verify_ngram_args {
  int32_t num_reqs;        /* R >= 0 (0 is a no-op); at most the handle's max_num_reqs */
  int32_t min_ngram;       /* 1 <= min_ngram <= max_ngram */
  int32_t max_ngram;       /* max_ngram <= SV_MAX_NGRAM */
  int32_t num_spec_tokens; /* k: 0 .. the handle's max_spec_len */
  int64_t max_model_len;   /* >= 1: a history of L tokens gets at most max_model_len - L */
  int64_t num_tokens_total;              /* length of token_ids (>= 0) */
  const int32_t *token_ids;              /* [num_tokens_total] histories, request after request */
  const int64_t *cu_num_tokens;          /* [R] inclusive prefix sums: request q owns [cu[q-1], cu[q]), cu[-1] = 0 */
  int32_t *draft_token_ids;              /* [R, k] out: the proposal, then -1 (may be NULL when k == 0) */
  int32_t *num_draft_tokens;             /* [R] out: k' (0 when nothing is proposed or the range is bad) */
  int32_t *status;                       /* [1] or NULL: SV_DATA_BAD_CU OR-ed in for a bad range */
} spec_verify_ngram_args;

sv_status spec_verify_ngram_propose(spec_verify_t handle, const spec_verify_ngram_args *args, void *stream);

/* Host-only validation of n-gram proposer arguments against `config`. */
sv_status spec_verify_check_ngram_args(const spec_verify_config *config, const spec_verify_ngram_args *args);

/* Create a handle.  Queries the device and sets kernel attributes on it
 * (temporarily making `device` current).  *out is set only on SV_OK. */
sv_status spec_verify_create(const spec_verify_config *config, spec_verify_t *out);

/* Enqueue one verification on `stream` (a cudaStream_t, NULL = legacy default
 * stream of the current device, which must be the handle's device). */
sv_status spec_verify_run(spec_verify_t handle, const spec_verify_args *args, void *stream);

/* Release a handle (no device memory is held).  NULL is accepted. */
sv_status spec_verify_destroy(spec_verify_t handle);

/* Host-only validation of `args` against `config`: the checks spec_verify_run
 * performs before enqueueing anything.  Touches no device and no pointer target. */
sv_status spec_verify_check_args(const spec_verify_config *config, const spec_verify_args *args);

/* Static name of a status code. */
const char *spec_verify_status_string(sv_status status);

/* Message of the last error raised on the calling thread ("" if none). */
const char *spec_verify_last_error(void);

/* ABI self-description, for bindings that mirror the structs. */
uint32_t spec_verify_abi_version(void);
size_t spec_verify_sizeof_config(void);
size_t spec_verify_sizeof_args(void);
size_t spec_verify_sizeof_sample_args(void);
size_t spec_verify_sizeof_ngram_args(void);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_VERIFY_H_ */
