// sv_api.cu -- the C ABI declared in include/spec_verify.h: handle lifetime,
// host-side validation and kernel dispatch.  No allocation, no host sync.
#include <climits>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <new>

#include "sv_internal.h"

namespace sv {

namespace {
thread_local char g_last_error[512] = "";

sv_status fail(sv_status s, const char *fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
  va_end(ap);
  return s;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
}  // namespace

void set_last_error(const char *fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
  va_end(ap);
}

int choose_cluster(const spec_verify_ctx *ctx, int N, int V) {
  if (ctx->cfg.cluster_ctas > 0) return ctx->cfg.cluster_ctas;
  // Split a request over more CTAs only while the batch alone gives fewer than
  // two CTAs per SM, and keep chunks of at least 4096 elements: every extra CTA
  // repeats the request's scan and adds a reduction (measured on GB300 at
  // N=512, V=151936: one CTA per request streams at 0.99 of the copy
  // bandwidth, four per request at 0.89).
  const long long target = 2LL * ctx->num_sms;
  int c = 1;
  while (c < ctx->max_cluster && static_cast<long long>(N) * c < target && V / (2 * c) >= 4096) c *= 2;
  return c;
}

bool choose_logits_layout(const spec_verify_ctx *ctx, int N, int V, int elem_bytes, int *cluster, int *chunk,
                          bool bitmaps, bool resident, bool chained) {
  // Resident rows live in the cluster's shared memory: start from the CTA
  // count of the probability entry and grow it until a CTA is small enough
  // for two to share an SM.  Rows read in place need no shared memory for
  // themselves (four CTAs share an SM).  The verifier walks a request's
  // positions one after another, so the latency of each position counts:
  // grow the cluster, up to the portable 8, until a CTA's chunk is small
  // enough for its group maxima to stay in registers.  The sampler's rows are
  // independent: grow only as far as the 16-bit window counts require
  // (measured on GB300 for 512 rows of V=151936: 4 CTAs per row 0.089 ms,
  // 8 CTAs 0.110 ms).
  auto chunk_for = [&](int c) { return ((V + c - 1) / c + 7) & ~7; };
  auto bytes_for = [&](int c) {
    return static_cast<long long>(logits_dyn_bytes(c, chunk_for(c), elem_bytes, resident, bitmaps));
  };
  int c = ctx->cfg.cluster_ctas > 0 ? ctx->cfg.cluster_ctas : choose_cluster(ctx, N, V);
  if (ctx->cfg.cluster_ctas == 0) {
    if (resident) {
      const long long per_cta = ctx->smem_per_sm / 2 - 1024 - static_cast<long long>(logits_static_smem());
      while (c < ctx->max_cluster && bytes_for(c) > per_cta) c *= 2;
    } else {
      const int cap = ctx->max_cluster < 8 ? ctx->max_cluster : 8;
      const int limit = chained ? logits_reg_group_chunk() : 65535;
      while (c < cap && chunk_for(c) > limit) c *= 2;
    }
  }
  // (window bins are 16-bit counts of one CTA's chunk)
  if (bytes_for(c) > ctx->max_dyn_smem || chunk_for(c) > 65535) return false;
  *cluster = c;
  *chunk = chunk_for(c);
  return true;
}

}  // namespace sv

using sv::fail;

extern "C" {

const char *spec_verify_status_string(sv_status s) {
  switch (s) {
    case SV_OK: return "SV_OK";
    case SV_ERR_INVALID_ARG: return "SV_ERR_INVALID_ARG";
    case SV_ERR_UNSUPPORTED: return "SV_ERR_UNSUPPORTED";
    case SV_ERR_CUDA: return "SV_ERR_CUDA";
    case SV_ERR_CAPACITY: return "SV_ERR_CAPACITY";
  }
  return "SV_UNKNOWN_STATUS";
}

const char *spec_verify_last_error(void) { return sv::g_last_error; }

uint32_t spec_verify_abi_version(void) { return SPEC_VERIFY_ABI_VERSION; }
size_t spec_verify_sizeof_config(void) { return sizeof(spec_verify_config); }
size_t spec_verify_sizeof_args(void) { return sizeof(spec_verify_args); }
size_t spec_verify_sizeof_sample_args(void) { return sizeof(spec_verify_sample_args); }
size_t spec_verify_sizeof_ngram_args(void) { return sizeof(spec_verify_ngram_args); }

static sv_status check_config(const spec_verify_config *c) {
  if (!c) return fail(SV_ERR_INVALID_ARG, "config is NULL");
  if (c->max_num_reqs < 1) return fail(SV_ERR_INVALID_ARG, "max_num_reqs must be >= 1");
  if (c->max_spec_len < 0 || c->max_spec_len > SV_MAX_SPEC_LEN)
    return fail(SV_ERR_INVALID_ARG, "max_spec_len must be in [0, %d]", SV_MAX_SPEC_LEN);
  if (c->vocab_size < 1) return fail(SV_ERR_INVALID_ARG, "vocab_size must be >= 1");
  if (c->device < 0) return fail(SV_ERR_INVALID_ARG, "device must be >= 0");
  const int cc = c->cluster_ctas;
  if (!(cc == 0 || cc == 1 || cc == 2 || cc == 4 || cc == 8 || cc == 16))
    return fail(SV_ERR_INVALID_ARG, "cluster_ctas must be 0, 1, 2, 4, 8 or 16");
  if (c->flags & ~(SV_FLAG_RESIDENT_ROWS | SV_FLAG_ONE_CTA_PER_REQUEST | SV_FLAG_SERIAL_LAUNCH))
    return fail(SV_ERR_INVALID_ARG, "unknown flags 0x%x", c->flags);
  if (static_cast<long long>(c->max_num_reqs) * (cc ? cc : 16) > INT_MAX)
    return fail(SV_ERR_INVALID_ARG, "max_num_reqs too large for one grid");
  return SV_OK;
}

sv_status spec_verify_check_args(const spec_verify_config *c, const spec_verify_args *a) {
  sv_status st = check_config(c);
  if (st != SV_OK) return st;
  if (!a) return fail(SV_ERR_INVALID_ARG, "args is NULL");
  if (a->num_reqs < 0) return fail(SV_ERR_INVALID_ARG, "num_reqs < 0");
  if (a->max_spec_len < 0) return fail(SV_ERR_INVALID_ARG, "max_spec_len < 0");
  if (a->vocab_size < 1) return fail(SV_ERR_INVALID_ARG, "vocab_size < 1");
  if (a->num_reqs > c->max_num_reqs) return fail(SV_ERR_CAPACITY, "num_reqs %d > handle max %d", a->num_reqs,
                                                 c->max_num_reqs);
  if (a->max_spec_len > c->max_spec_len)
    return fail(SV_ERR_CAPACITY, "max_spec_len %d > handle max %d", a->max_spec_len, c->max_spec_len);
  if (a->vocab_size > c->vocab_size)
    return fail(SV_ERR_CAPACITY, "vocab_size %d > handle max %d", a->vocab_size, c->vocab_size);
  if (a->entry != SV_ENTRY_PROBS && a->entry != SV_ENTRY_LOGITS) return fail(SV_ERR_INVALID_ARG, "bad entry");
  if (a->dtype != SV_F32 && a->dtype != SV_BF16) return fail(SV_ERR_INVALID_ARG, "bad dtype");
  if (a->entry == SV_ENTRY_PROBS && a->dtype != SV_F32)
    return fail(SV_ERR_UNSUPPORTED, "the probability entry takes fp32 rows");
  if (a->hints & ~SV_HINT_SMALL_TOP_K) return fail(SV_ERR_INVALID_ARG, "unknown hints 0x%x", a->hints);
  if (a->test_flags & ~SV_TEST_EXPIRE_COPY_WAIT) return fail(SV_ERR_INVALID_ARG, "unknown test_flags 0x%x", a->test_flags);
  if (a->num_draft_tokens_total < 0) return fail(SV_ERR_INVALID_ARG, "num_draft_tokens_total < 0");
  if (!a->cu_num_draft_tokens &&
      a->num_draft_tokens_total != static_cast<int64_t>(a->num_reqs) * a->max_spec_len)
    return fail(SV_ERR_INVALID_ARG, "without cu_num_draft_tokens, T must be num_reqs * max_spec_len");
  if (a->num_reqs == 0) return SV_OK;
  if (a->num_draft_tokens_total > static_cast<int64_t>(a->num_reqs) * a->max_spec_len)
    return fail(SV_ERR_INVALID_ARG, "T exceeds num_reqs * max_spec_len");
  if (a->num_draft_tokens_total > 0 && !a->draft_ids) return fail(SV_ERR_INVALID_ARG, "draft_ids is NULL");
  if (!a->target) return fail(SV_ERR_INVALID_ARG, "target is NULL");
  if (a->target_row_stride < a->vocab_size) return fail(SV_ERR_INVALID_ARG, "target_row_stride < vocab_size");
  if (a->draft && a->draft_row_stride < a->vocab_size)
    return fail(SV_ERR_INVALID_ARG, "draft_row_stride < vocab_size");
  if (a->uniforms && !a->exponentials)
    return fail(SV_ERR_INVALID_ARG, "uniforms without exponentials: test mode needs both");
  if (a->exponentials && !a->uniforms && a->num_draft_tokens_total > 0)
    return fail(SV_ERR_INVALID_ARG, "test mode with draft tokens needs uniforms");
  if (a->exponentials && a->exponentials_row_stride < a->vocab_size)
    return fail(SV_ERR_INVALID_ARG, "exponentials_row_stride < vocab_size");
  if (!a->out_tokens || !a->num_accepted) return fail(SV_ERR_INVALID_ARG, "out_tokens / num_accepted is NULL");
  if (a->entry == SV_ENTRY_PROBS && (a->repetition_penalty || a->penalty_cu || a->banned_cu))
    return fail(SV_ERR_INVALID_ARG, "logits processors apply to the logits entry (probability rows are transformed)");
  struct {
    const char *name;
    const int64_t *cu;
    const int32_t *ids;
    int64_t total;
  } lists[3] = {{"penalty", a->penalty_cu, a->penalty_token_ids, a->penalty_total},
                {"banned", a->banned_cu, a->banned_token_ids, a->banned_total},
                {"stop", a->stop_cu, a->stop_token_ids, a->stop_total}};
  for (const auto &l : lists) {
    if (!l.cu) continue;
    if (l.total < 0) return fail(SV_ERR_INVALID_ARG, "%s_total < 0", l.name);
    if (l.total > 0 && !l.ids) return fail(SV_ERR_INVALID_ARG, "%s_token_ids is NULL", l.name);
  }
  return SV_OK;
}

sv_status spec_verify_create(const spec_verify_config *config, spec_verify_t *out) {
  if (!out) return fail(SV_ERR_INVALID_ARG, "out is NULL");
  sv_status st = check_config(config);
  if (st != SV_OK) return st;
  int old = 0;
  cudaError_t e = cudaGetDevice(&old);
  if (e != cudaSuccess) return fail(SV_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if ((e = cudaSetDevice(config->device)) != cudaSuccess)
    return fail(SV_ERR_CUDA, "cudaSetDevice(%d): %s", config->device, cudaGetErrorString(e));
  int major = 0, minor = 0, sms = 0, smem_sm = 0;
  cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, config->device);
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, config->device);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, config->device);
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, config->device);
  sv_status result = SV_OK;
  int max_cluster = 16;
  int max_dyn = 0, optin_all = 0;
  if (e != cudaSuccess) {
    result = fail(SV_ERR_CUDA, "device query: %s", cudaGetErrorString(e));
  } else if (major != 10 || minor != 3) {
    result = fail(SV_ERR_UNSUPPORTED, "built for sm_103a only; device %d is sm_%d%d", config->device, major, minor);
  } else {
    int optin = 0;
    cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, config->device);
    max_dyn = optin - static_cast<int>(sv::logits_static_smem()) - 1024;
    optin_all = optin;
    if ((e = sv::enable_stream_kernels_bf16()) != cudaSuccess || (e = sv::enable_stream_kernels_f32()) != cudaSuccess ||
        (e = sv::enable_stream_kernels_bf16_proc(optin)) != cudaSuccess ||
        (e = sv::enable_stream_kernels_f32_proc(optin)) != cudaSuccess)
      result = fail(SV_ERR_CUDA, "kernel attributes: %s", cudaGetErrorString(e));
    if (sv::enable_probs_kernels(16) != cudaSuccess || sv::enable_logits_kernels(16, max_dyn) != cudaSuccess ||
        sv::enable_sample_kernels(16, max_dyn) != cudaSuccess) {
      cudaGetLastError();
      max_cluster = 8;
      if ((e = sv::enable_probs_kernels(8)) != cudaSuccess || (e = sv::enable_logits_kernels(8, max_dyn)) != cudaSuccess ||
          (e = sv::enable_sample_kernels(8, max_dyn)) != cudaSuccess)
        result = fail(SV_ERR_CUDA, "kernel attributes: %s", cudaGetErrorString(e));
    }
    if (config->cluster_ctas > max_cluster)
      result = fail(SV_ERR_UNSUPPORTED, "cluster_ctas %d > %d on this device", config->cluster_ctas, max_cluster);
  }
  cudaSetDevice(old);
  if (result != SV_OK) return result;
  spec_verify_ctx *h = new (std::nothrow) spec_verify_ctx;
  if (!h) return fail(SV_ERR_INVALID_ARG, "out of host memory");
  h->cfg = *config;
  h->num_sms = sms;
  h->max_cluster = max_cluster;
  h->max_dyn_smem = max_dyn;
  h->max_dyn_optin = optin_all;
  h->smem_per_sm = smem_sm;
  *out = h;
  return SV_OK;
}

sv_status spec_verify_destroy(spec_verify_t h) {
  delete h;
  return SV_OK;
}

sv_status spec_verify_run(spec_verify_t h, const spec_verify_args *a, void *stream) {
  if (!h) return fail(SV_ERR_INVALID_ARG, "handle is NULL");
  sv_status st = spec_verify_check_args(&h->cfg, a);
  if (st != SV_OK) return st;
  if (a->num_reqs == 0) return SV_OK;
  sv::VerifyParams p{};
  p.N = a->num_reqs;
  p.G = a->max_spec_len;
  p.V = a->vocab_size;
  p.T = a->num_draft_tokens_total;
  p.ids = a->draft_ids;
  p.cu = a->cu_num_draft_tokens;
  p.target = a->target;
  p.target_stride = a->target_row_stride;
  p.draft = a->draft;
  p.draft_stride = a->draft_row_stride;
  p.temperature = a->temperature;
  p.top_k = a->top_k;
  p.top_p = a->top_p;
  p.uniforms = a->uniforms;
  p.exponentials = a->exponentials;
  p.exp_stride = a->exponentials_row_stride;
  p.seed_lo = static_cast<uint32_t>(a->seed);
  p.seed_hi = static_cast<uint32_t>(a->seed >> 32);
  p.off_lo = static_cast<uint32_t>(a->offset);
  p.off_hi = static_cast<uint32_t>(a->offset >> 32);
  p.req_base = a->rng_request_base;
  p.out = a->out_tokens;
  p.nacc = a->num_accepted;
  p.ncomp = a->num_computed_tokens;
  p.slots = a->slot_mapping;
  p.dbg_py = a->dbg_py;
  p.dbg_qy = a->dbg_qy;
  p.status = a->status;
  p.rates = a->synthetic_acceptance_rates;
  p.rep_penalty = a->repetition_penalty;
  p.pen_cu = a->penalty_cu;
  p.pen_ids = a->penalty_token_ids;
  p.pen_total = a->penalty_total;
  p.ban_cu = a->banned_cu;
  p.ban_ids = a->banned_token_ids;
  p.ban_total = a->banned_total;
  p.stop_cu = a->stop_cu;
  p.stop_ids = a->stop_token_ids;
  p.stop_total = a->stop_total;
  p.first_wait = (a->test_flags & SV_TEST_EXPIRE_COPY_WAIT) ? 0u : sv::kCopyWaitPolls;
  p.pdl = !(h->cfg.flags & SV_FLAG_SERIAL_LAUNCH);
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (a->entry == SV_ENTRY_PROBS) {
    const int cluster = sv::choose_cluster(h, p.N, p.V);
    const bool vec = sv::aligned16(a->target) && (a->target_row_stride % 4 == 0) &&
                     (!a->draft || (sv::aligned16(a->draft) && a->draft_row_stride % 4 == 0));
    e = sv::launch_probs(p, cluster, vec, s);
  } else {
    const bool bf16 = a->dtype == SV_BF16;
    const int eb = bf16 ? 2 : 4;
    const int per16 = 16 / eb;  // elements per 16-byte vector
    int cluster = 0, chunk = 0;
    const bool procs = a->repetition_penalty || a->banned_cu;
    const bool vec = sv::aligned16(a->target) && (a->target_row_stride % per16 == 0) &&
                     (!a->draft || (sv::aligned16(a->draft) && a->draft_row_stride % per16 == 0));
    const bool resident = !vec || (h->cfg.flags & SV_FLAG_RESIDENT_ROWS);
    // one CTA per request: aligned rows read in place (with processors, the
    // row bitmaps within the shared memory a CTA may take), and either the
    // handle asks for it or the caller states small top-k values and the
    // batch gives every SM at least two requests
    const bool stream_form = vec && !(h->cfg.flags & SV_FLAG_RESIDENT_ROWS) &&
                             (!procs || sv::stream_dyn_smem(p.V, true) <= static_cast<size_t>(h->max_dyn_optin)) &&
                             ((h->cfg.flags & SV_FLAG_ONE_CTA_PER_REQUEST) ||
                              ((a->hints & SV_HINT_SMALL_TOP_K) && p.N >= 2 * h->num_sms));
    if (stream_form) {
      if (procs)
        e = bf16 ? sv::launch_stream_bf16_proc(p, s) : sv::launch_stream_f32_proc(p, s);
      else
        e = bf16 ? sv::launch_stream_bf16(p, s) : sv::launch_stream_f32(p, s);
      if (e != cudaSuccess) return fail(SV_ERR_CUDA, "verifier launch: %s", cudaGetErrorString(e));
      return SV_OK;
    }
    if (!sv::choose_logits_layout(h, p.N, p.V, eb, &cluster, &chunk, procs, resident, true))
      return fail(SV_ERR_UNSUPPORTED, "vocab_size %d too large for the rows to fit in the cluster's shared memory",
                  p.V);
    e = sv::launch_logits(p, bf16, cluster, chunk, vec, resident, s);
  }
  if (e != cudaSuccess) return fail(SV_ERR_CUDA, "verifier launch: %s", cudaGetErrorString(e));
  return SV_OK;
}

sv_status spec_verify_check_sample_args(const spec_verify_config *c, const spec_verify_sample_args *a) {
  sv_status st = check_config(c);
  if (st != SV_OK) return st;
  if (!a) return fail(SV_ERR_INVALID_ARG, "args is NULL");
  if (a->num_rows < 0) return fail(SV_ERR_INVALID_ARG, "num_rows < 0");
  if (a->vocab_size < 1) return fail(SV_ERR_INVALID_ARG, "vocab_size < 1");
  if (a->num_rows > c->max_num_reqs) return fail(SV_ERR_CAPACITY, "num_rows %d > handle max %d", a->num_rows,
                                                 c->max_num_reqs);
  if (a->vocab_size > c->vocab_size)
    return fail(SV_ERR_CAPACITY, "vocab_size %d > handle max %d", a->vocab_size, c->vocab_size);
  if (a->dtype != SV_F32 && a->dtype != SV_BF16) return fail(SV_ERR_INVALID_ARG, "bad dtype");
  if (a->hints & ~SV_HINT_SMALL_TOP_K) return fail(SV_ERR_INVALID_ARG, "unknown hints 0x%x", a->hints);
  if (a->test_flags & ~SV_TEST_EXPIRE_COPY_WAIT) return fail(SV_ERR_INVALID_ARG, "unknown test_flags 0x%x", a->test_flags);
  if (a->num_rows == 0) return SV_OK;
  if (!a->logits) return fail(SV_ERR_INVALID_ARG, "logits is NULL");
  if (a->row_stride < a->vocab_size) return fail(SV_ERR_INVALID_ARG, "row_stride < vocab_size");
  if (a->exponentials && a->exponentials_row_stride < a->vocab_size)
    return fail(SV_ERR_INVALID_ARG, "exponentials_row_stride < vocab_size");
  if (a->probs && a->probs_row_stride < a->vocab_size)
    return fail(SV_ERR_INVALID_ARG, "probs_row_stride < vocab_size");
  if (!a->tokens) return fail(SV_ERR_INVALID_ARG, "tokens is NULL");
  if (a->penalty_cu && (a->penalty_total < 0 || (a->penalty_total > 0 && !a->penalty_token_ids)))
    return fail(SV_ERR_INVALID_ARG, "bad penalty list");
  if (a->banned_cu && (a->banned_total < 0 || (a->banned_total > 0 && !a->banned_token_ids)))
    return fail(SV_ERR_INVALID_ARG, "bad banned list");
  return SV_OK;
}

sv_status spec_verify_sample(spec_verify_t h, const spec_verify_sample_args *a, void *stream) {
  if (!h) return fail(SV_ERR_INVALID_ARG, "handle is NULL");
  sv_status st = spec_verify_check_sample_args(&h->cfg, a);
  if (st != SV_OK) return st;
  if (a->num_rows == 0) return SV_OK;
  sv::SampleParams p{};
  p.R = a->num_rows;
  p.V = a->vocab_size;
  p.logits = a->logits;
  p.row_stride = a->row_stride;
  p.temperature = a->temperature;
  p.top_k = a->top_k;
  p.top_p = a->top_p;
  p.exponentials = a->exponentials;
  p.exp_stride = a->exponentials_row_stride;
  p.seed_lo = static_cast<uint32_t>(a->seed);
  p.seed_hi = static_cast<uint32_t>(a->seed >> 32);
  p.off_lo = static_cast<uint32_t>(a->offset);
  p.off_hi = static_cast<uint32_t>(a->offset >> 32);
  p.row_base = a->rng_row_base;
  p.tokens = a->tokens;
  p.probs = a->probs;
  p.probs_stride = a->probs_row_stride;
  p.status = a->status;
  p.rep_penalty = a->repetition_penalty;
  p.pen_cu = a->penalty_cu;
  p.pen_ids = a->penalty_token_ids;
  p.pen_total = a->penalty_total;
  p.ban_cu = a->banned_cu;
  p.ban_ids = a->banned_token_ids;
  p.ban_total = a->banned_total;
  p.first_wait = (a->test_flags & SV_TEST_EXPIRE_COPY_WAIT) ? 0u : sv::kCopyWaitPolls;
  p.pdl = !(h->cfg.flags & SV_FLAG_SERIAL_LAUNCH);
  const bool bf16 = a->dtype == SV_BF16;
  const int eb = bf16 ? 2 : 4;
  int cluster = 0, chunk = 0;
  const bool procs = p.rep_penalty || p.ban_cu;
  const bool vec = sv::aligned16(a->logits) && (a->row_stride % (16 / eb) == 0);
  // unaligned rows, or the handle flag, go through shared memory; other rows
  // are read where they lie
  const bool resident = !vec || (h->cfg.flags & SV_FLAG_RESIDENT_ROWS);
  // one CTA per row: the handle flag, or the small-top-k hint on a batch of at least two rows per SM
  // (with processors, when the row bitmaps fit a CTA's shared memory)
  if (vec && !(h->cfg.flags & SV_FLAG_RESIDENT_ROWS) &&
      (!procs || sv::stream_dyn_smem(p.V, true) <= static_cast<size_t>(h->max_dyn_optin)) &&
      ((h->cfg.flags & SV_FLAG_ONE_CTA_PER_REQUEST) || ((a->hints & SV_HINT_SMALL_TOP_K) && p.R >= 2 * h->num_sms))) {
    const cudaStream_t cs = static_cast<cudaStream_t>(stream);
    const cudaError_t e = procs ? (bf16 ? sv::launch_stream_sample_bf16_proc(p, cs) : sv::launch_stream_sample_f32_proc(p, cs))
                                : (bf16 ? sv::launch_stream_sample_bf16(p, cs) : sv::launch_stream_sample_f32(p, cs));
    if (e != cudaSuccess) return fail(SV_ERR_CUDA, "sampler launch: %s", cudaGetErrorString(e));
    return SV_OK;
  }
  if (!sv::choose_logits_layout(h, p.R, p.V, eb, &cluster, &chunk, procs, resident, false))
    return fail(SV_ERR_UNSUPPORTED, "vocab_size %d too large for a row to fit in the cluster's shared memory", p.V);
  const cudaError_t e = sv::launch_sample(p, bf16, cluster, chunk, vec, resident, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(SV_ERR_CUDA, "sampler launch: %s", cudaGetErrorString(e));
  return SV_OK;
}

sv_status spec_verify_check_ngram_args(const spec_verify_config *c, const spec_verify_ngram_args *a) {
  sv_status st = check_config(c);
  if (st != SV_OK) return st;
  if (!a) return fail(SV_ERR_INVALID_ARG, "args is NULL");
  if (a->num_reqs < 0) return fail(SV_ERR_INVALID_ARG, "num_reqs < 0");
  if (a->num_reqs > c->max_num_reqs)
    return fail(SV_ERR_CAPACITY, "num_reqs %d > handle max %d", a->num_reqs, c->max_num_reqs);
  if (a->num_spec_tokens < 0) return fail(SV_ERR_INVALID_ARG, "num_spec_tokens < 0");
  if (a->num_spec_tokens > c->max_spec_len)
    return fail(SV_ERR_CAPACITY, "num_spec_tokens %d > handle max_spec_len %d", a->num_spec_tokens, c->max_spec_len);
  if (a->min_ngram < 1 || a->max_ngram < a->min_ngram)
    return fail(SV_ERR_INVALID_ARG, "need 1 <= min_ngram <= max_ngram (got %d, %d)", a->min_ngram, a->max_ngram);
  if (a->max_ngram > SV_MAX_NGRAM) return fail(SV_ERR_UNSUPPORTED, "max_ngram %d > %d", a->max_ngram, SV_MAX_NGRAM);
  if (a->max_model_len < 1) return fail(SV_ERR_INVALID_ARG, "max_model_len < 1");
  if (a->num_tokens_total < 0) return fail(SV_ERR_INVALID_ARG, "num_tokens_total < 0");
  if (a->num_reqs == 0) return SV_OK;
  if (!a->cu_num_tokens) return fail(SV_ERR_INVALID_ARG, "cu_num_tokens is NULL");
  if (!a->token_ids && a->num_tokens_total > 0) return fail(SV_ERR_INVALID_ARG, "token_ids is NULL");
  if (!a->num_draft_tokens) return fail(SV_ERR_INVALID_ARG, "num_draft_tokens is NULL");
  if (!a->draft_token_ids && a->num_spec_tokens > 0) return fail(SV_ERR_INVALID_ARG, "draft_token_ids is NULL");
  return SV_OK;
}

sv_status spec_verify_ngram_propose(spec_verify_t h, const spec_verify_ngram_args *a, void *stream) {
  if (!h) return fail(SV_ERR_INVALID_ARG, "handle is NULL");
  sv_status st = spec_verify_check_ngram_args(&h->cfg, a);
  if (st != SV_OK) return st;
  if (a->num_reqs == 0) return SV_OK;
  sv::NgramParams p{};
  p.R = a->num_reqs;
  p.min_n = a->min_ngram;
  p.max_n = a->max_ngram;
  p.k = a->num_spec_tokens;
  p.max_model_len = a->max_model_len;
  p.total = a->num_tokens_total;
  p.tokens = a->token_ids;
  p.cu = a->cu_num_tokens;
  p.out = a->draft_token_ids;
  p.num = a->num_draft_tokens;
  p.status = a->status;
  p.pdl = !(h->cfg.flags & SV_FLAG_SERIAL_LAUNCH);
  const cudaError_t e = sv::launch_ngram(p, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(SV_ERR_CUDA, "n-gram proposer launch: %s", cudaGetErrorString(e));
  return SV_OK;
}

}  // extern "C"
