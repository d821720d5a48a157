// sv_ngram.cu -- batched n-gram proposer ("vLLM source walk-through (10)",
// section "NgramProposer": the tail of a request's history looked up earlier
// in the history, match lengths capped at max_ngram, the longest match with a
// length in [min_ngram, max_ngram] proposing the tokens that followed it).
//
// One CTA per request.  The CTA streams the request's history from HBM with
// 16-byte loads, up to kLoads per thread in flight (a longer history is first
// prefetched into L2 in one bulk request), and compares each token
// with the last one; only the rare equal tokens E (E <= L - 2, so a token
// follows) start the backward comparison t[E - j] == t[L - 1 - j] against the
// tail held in shared memory, on the thread's own group and the previous
// lane's (a warp shuffle) for the first four steps.  The CTA keeps the
// largest (length, E) -- the longest match, then the most recent occurrence --
// and copies the proposal.
#include <cstdint>

#include "sv_device.cuh"
#include "sv_internal.h"

namespace sv {
namespace {

constexpr int kLoads = 8;  // 16-byte loads in flight per thread

__global__ void __launch_bounds__(kThreads) ngram_kernel(const NgramParams P) {
  pdl_enter();
  __shared__ int32_t tail[SV_MAX_NGRAM];
  __shared__ unsigned long long warp_best[kWarps];
  const int q = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int32_t *row = P.out ? P.out + static_cast<int64_t>(q) * P.k : nullptr;
  const int64_t s = q ? P.cu[q - 1] : 0, e = P.cu[q];
  if (s < 0 || e < s || e > P.total || e - s > 0x7FFFFFFF) {
    for (int c = tid; c < P.k; c += kThreads) row[c] = -1;
    if (tid == 0) {
      P.num[q] = 0;
      if (P.status) atomicOr(P.status, static_cast<int>(SV_DATA_BAD_CU));
    }
    return;
  }
  const int64_t L = e - s;
  const int32_t *t = P.tokens + s;
  int64_t kk = P.k;
  if (P.max_model_len - L < kk) kk = P.max_model_len - L;
  unsigned long long best = 0ull;  // (length << 32) | E; 0 = no match
  if (L >= P.min_n && kk > 0) {
    // candidate ends occupy global positions [s, s + L - 2]; 16-byte groups
    // start at the aligned position at or below s
    const int64_t g0 = s & ~static_cast<int64_t>(3), g_end = s + L - 1;  // exclusive end
    const int64_t ngroups = (g_end - g0 + 3) >> 2;
    const bool vec = (reinterpret_cast<uintptr_t>(P.tokens) & 15u) == 0;
    int4 d[kLoads];
    auto load_round = [&](int64_t vb) {
#pragma unroll
      for (int u = 0; u < kLoads; ++u) {
        const int64_t v = vb + u * kThreads + tid;
        const int64_t g = g0 + 4 * v;
        if (v < ngroups && vec && g + 3 < P.total) {
          d[u] = __ldg(reinterpret_cast<const int4 *>(P.tokens + g));
        } else {
          int32_t w[4];
#pragma unroll
          for (int c = 0; c < 4; ++c) w[c] = (v < ngroups && g + c < P.total) ? P.tokens[g + c] : 0;
          d[u] = make_int4(w[0], w[1], w[2], w[3]);
        }
      }
    };
    // a history longer than one round warms L2 in one bulk prefetch, so the
    // later rounds find it there instead of waiting on HBM one after another
    if (vec && tid == 0 && ngroups > static_cast<int64_t>(kLoads) * kThreads) {
      const int64_t gend = min(g0 + 4 * ngroups, P.total & ~static_cast<int64_t>(3));
      if (gend > g0) prefetch_l2(P.tokens + g0, static_cast<uint32_t>((gend - g0) * 4));
    }
    load_round(0);  // in flight together with the tail
    const int span = static_cast<int>(min(static_cast<int64_t>(P.max_n), L));
    for (int j = tid; j < span; j += kThreads) tail[j] = t[L - 1 - j];
    __syncthreads();
    const int32_t last = tail[0];
    for (int64_t vb = 0; vb < ngroups; vb += static_cast<int64_t>(kLoads) * kThreads) {
      if (vb > 0) load_round(vb);
#pragma unroll
      for (int u = 0; u < kLoads; ++u) {
        const bool hit = d[u].x == last || d[u].y == last || d[u].z == last || d[u].w == last;
        if (!__any_sync(0xFFFFFFFFu, hit)) continue;  // (almost every group of the warp)
        // the group before this one is the previous lane's, so a match finds
        // its preceding tokens in registers; lane 0 reads its neighbour's again
        int4 pv;
        pv.x = __shfl_up_sync(0xFFFFFFFFu, d[u].x, 1);
        pv.y = __shfl_up_sync(0xFFFFFFFFu, d[u].y, 1);
        pv.z = __shfl_up_sync(0xFFFFFFFFu, d[u].z, 1);
        pv.w = __shfl_up_sync(0xFFFFFFFFu, d[u].w, 1);
        if (!hit) continue;
        const int64_t v = vb + u * kThreads + tid;
        const int64_t E0 = g0 + 4 * v - s;  // history index of the group's first token
        if (lane == 0) {
          // (unused for the first group, whose matches never reach back, and
          // for groups past the end, whose matches fail the range test)
          pv = make_int4(0, 0, 0, 0);
          if (v > 0 && v < ngroups) {
            const int64_t gp = g0 + 4 * (v - 1);  // below the current group's start, so inside the buffer
            if (vec) {
              pv = __ldg(reinterpret_cast<const int4 *>(P.tokens + gp));
            } else {
              pv = make_int4(P.tokens[gp], P.tokens[gp + 1], P.tokens[gp + 2], P.tokens[gp + 3]);
            }
          }
        }
        const int32_t win[8] = {pv.x, pv.y, pv.z, pv.w, d[u].x, d[u].y, d[u].z, d[u].w};
#pragma unroll
        for (int c = 0; c < 4; ++c) {  // a match at E = E0 + c: t[E - j] is win[4 + c - j]
          const int64_t E = E0 + c;
          if (win[4 + c] != last || E < 0 || E > L - 2) continue;  // (groups past the end fail the range test)
          const int cap = static_cast<int>(min(static_cast<int64_t>(P.max_n), E + 1));
          int len = 1;
          bool run = true;
#pragma unroll
          for (int j = 1; j <= 4 + c; ++j) {  // (len == j while the run lasts)
            if (run && len < cap && win[4 + c - j] == tail[j])
              ++len;
            else
              run = false;
          }
          if (run)  // longer n-grams than the registers hold
            while (len < cap && __ldg(t + E - len) == tail[len]) ++len;
          if (len >= P.min_n)
            best = umax64(best, (static_cast<unsigned long long>(len) << 32) | static_cast<uint64_t>(E));
        }
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) best = umax64(best, __shfl_xor_sync(0xFFFFFFFFu, best, o));
  if (lane == 0) warp_best[warp] = best;
  __syncthreads();
  if (warp == 0) {
    best = lane < kWarps ? warp_best[lane] : 0ull;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) best = umax64(best, __shfl_xor_sync(0xFFFFFFFFu, best, o));
    if (lane == 0) warp_best[0] = best;
  }
  __syncthreads();
  best = warp_best[0];
  int64_t start = 0, n = 0;
  if (best != 0ull) {
    start = static_cast<int64_t>(best & 0xFFFFFFFFull) + 1;
    n = min(kk, L - start);
  }
  for (int c = tid; c < P.k; c += kThreads) row[c] = c < n ? t[start + c] : -1;
  if (tid == 0) P.num[q] = static_cast<int32_t>(n);
}

}  // namespace

cudaError_t launch_ngram(const NgramParams &p, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p.R), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  cfg.attrs = attr;
  cfg.numAttrs = launch_attrs(attr, 0, p.pdl);
  return cudaLaunchKernelEx(&cfg, ngram_kernel, p);
}

}  // namespace sv
