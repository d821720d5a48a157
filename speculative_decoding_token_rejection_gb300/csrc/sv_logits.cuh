// sv_logits.cuh -- verifier kernel for the logits entry (bf16 or fp32 logits)
// and the draft-side sampler.  Kernel templates and their launchers; the
// translation units sv_logits_{bf16,f32}.cu and sv_sample_{bf16,f32}.cu
// instantiate them per kernel and element type (compiled in parallel), and
// sv_logits.cu dispatches.
//
// The target and draft logits go through the same transform before the test
// ("vLLM source walk-through (10)", section "Rejection sampling: the two
// branches of RejectionSampler": temperature, top-k, top-p on both sides;
// "Speculative Decoding: propose, verify, accept", section 06: identical
// transforms are required for exactness):
//   p(x) = exp((l(x) - l_max) / T) / Z'  for l(x) in the kept set, else 0,
// where the kept set is {x : key(x) >= tau_k} (tau_k = k-th largest logit,
// ties kept) cut further by top-p to the shortest descending prefix whose
// mass reaches top_p (ties at the cut kept), and Z' sums the kept terms.
//
// One thread-block cluster per request.  A random request walks its positions
// in order, as a sequential verifier reads them: position j brings each CTA's
// chunk of the target and draft rows from HBM once (into L2 by a bulk
// prefetch and read in place, or copied into shared memory where the logits
// processors rewrite them), computes the row statistics (max, the top-k
// threshold and top-p cut from exact per-key window counts, normaliser),
// tests fl32(u * q(y)) < p(y), and either moves on or runs the exponential
// race of the residual max(p - q, 0) over the same chunks.  When all drafts
// pass, the bonus row is raced over p.  Rows after the first rejection are
// never read.  Greedy requests stream target rows from HBM and take the
// cluster argmax of the raw logits, stopping at the first mismatch.
//
// All sums are deterministic: integer histograms and fixed-point (2^-40)
// masses use atomics whose order cannot change the result, and float sums
// use a fixed reduction tree and rank order across the cluster.
#pragma once

#include <cuda_bf16.h>

#include <cmath>
#include <type_traits>

#include "sv_device.cuh"
#include "sv_internal.h"

namespace sv {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kMassScale = 1099511627776.0f;  // 2^40: fixed-point scale of the top-p masses

// ---------------------------------------------------------------------------
// element types: raw bits in shared memory, order-preserving integer keys
// (-0 folded onto +0, so equal values have equal keys)
// ---------------------------------------------------------------------------
template <typename TIn>
struct Elem;

template <>
struct Elem<uint16_t> {  // bf16 bit patterns
  static constexpr int kBits = 16;
  __device__ static float val(uint32_t b) { return __uint_as_float(b << 16); }
  __device__ static uint32_t key(uint32_t b) {
    if (b == 0x8000u) b = 0u;
    return (b & 0x8000u) ? (~b & 0xFFFFu) : (b | 0x8000u);
  }
  __device__ static float val_of_key(uint32_t k) {
    const uint32_t b = (k & 0x8000u) ? (k & 0x7FFFu) : (~k & 0xFFFFu);
    return val(b);
  }
  __device__ static bool is_nan(uint32_t b) { return (b & 0x7F80u) == 0x7F80u && (b & 0x7Fu) != 0u; }
  __device__ static bool is_pinf(uint32_t b) { return b == 0x7F80u; }
  __device__ static bool finite(uint32_t b) { return (b & 0x7F80u) != 0x7F80u; }
};

template <>
struct Elem<float> {  // fp32 values (bits handled as uint32)
  static constexpr int kBits = 32;
  __device__ static float val(uint32_t b) { return __uint_as_float(b); }
  __device__ static uint32_t key(uint32_t b) {
    if (b == 0x80000000u) b = 0u;
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  }
  __device__ static float val_of_key(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
  }
  __device__ static bool is_nan(uint32_t b) { return (b & 0x7F800000u) == 0x7F800000u && (b & 0x7FFFFFu) != 0u; }
  __device__ static bool is_pinf(uint32_t b) { return b == 0x7F800000u; }
  __device__ static bool finite(uint32_t b) { return (b & 0x7F800000u) != 0x7F800000u; }
};

template <typename TIn>
__device__ __forceinline__ uint32_t bits_at(const TIn *row, int x) {
  return static_cast<uint32_t>(row[x]);
}
template <>
__device__ __forceinline__ uint32_t bits_at<float>(const float *row, int x) {
  return __float_as_uint(row[x]);
}

// Visit this thread's elements of a shared-memory row chunk through 16-byte
// reads (8 bf16 or 4 fp32 per read), then the tail; f(bits, x).
template <typename TIn, typename F>
__device__ __forceinline__ void for_each_elem(const TIn *s, int n, F f) {
  constexpr int kPer = 16 / sizeof(TIn);
  const int nv = n / kPer;
  const uint4 *s4 = reinterpret_cast<const uint4 *>(s);
  for (int v = threadIdx.x; v < nv; v += kThreads) {
    const uint4 d = s4[v];
    const uint32_t w[4] = {d.x, d.y, d.z, d.w};
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      if (sizeof(TIn) == 2) {
        f(w[t] & 0xFFFFu, v * kPer + 2 * t);
        f(w[t] >> 16, v * kPer + 2 * t + 1);
      } else {
        f(w[t], v * kPer + t);
      }
    }
  }
  for (int x = nv * kPer + threadIdx.x; x < n; x += kThreads) f(bits_at(s, x), x);
}

// bf16 pairs with native bf16x2 instructions.  max.NaN propagates NaN, so
// one running max per thread also reveals NaN and +inf in the chunk.
__device__ __forceinline__ uint32_t bf16x2_max_nan(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
// 0xFFFF in each half of w that is >= the bf16 value in both halves of t2
// (false for NaN halves).
__device__ __forceinline__ uint32_t bf16x2_ge_mask(uint32_t w, uint32_t t2) {
  return __hge2_mask(*reinterpret_cast<const __nv_bfloat162 *>(&w), *reinterpret_cast<const __nv_bfloat162 *>(&t2));
}
// bf16 bits of an order key (inverse of Elem<uint16_t>::key).
__device__ __forceinline__ uint32_t bf16_bits_of_key(uint32_t k) {
  return (k & 0x8000u) ? (k & 0x7FFFu) : (~k & 0xFFFFu);
}

// ---------------------------------------------------------------------------
// shared memory
// ---------------------------------------------------------------------------
constexpr uint32_t kFlagBad = 1u;      // NaN or +inf in a random row
constexpr uint32_t kFlagFinite = 2u;   // at least one finite logit
constexpr uint32_t kFlagTimeout = 4u;  // the row's bulk copy did not complete in time
constexpr int kNearBins = 128;         // near-max bins: distances 0..127 from the row's largest key
constexpr int kMaxCluster = 16;
constexpr int kWalkGroups = 8;  // 16-byte groups a lane tests per window-scan step
constexpr int kGroupWords = 5;  // registers of packed group maxima per row and thread (2 groups each)
// largest bf16 chunk whose 16-byte groups all have their maxima in registers
constexpr int kRegGroupChunk = 2 * kGroupWords * 8 * kThreads;

struct StatPart {  // one CTA's partials of one reduction round, for up to 2 rows
  uint32_t maxkey[2];
  uint32_t flags[2];
  uint32_t floor[2];  // lower bound of the row's top-k threshold (key), from the thread maxima
  uint32_t nbins[2];  // window bins that can be non-zero (the window's width)
  float z[2];
  unsigned long long tot[2];
  uint32_t cnt[2][256];
  float massf[2][256];  // masses (fast path: the window, relative to this CTA's max)
};
constexpr int kBinsShift = 8;  // an inbox header carries nbins in the flags word above this bit

struct StatSum {  // cluster totals of a reduction round (the same in every CTA)
  uint32_t maxkey[2];
  uint32_t flags[2];
  float z[2];
  unsigned long long tot[2];
  uint32_t cnt[2][256];
  unsigned long long mass[2][256];  // 2^-40 fixed point, from the peers' fp32 masses in rank order
};

struct RowStats {
  uint32_t cut;  // kept set: key >= cut
  float vmax;    // largest logit
  float c2;      // log2(e) / T
  float zp;      // normaliser over the kept set
};

struct Select {  // running state of a radix selection, per row
  uint32_t prefix[2];          // key bits fixed so far
  int known_lo[2];             // bits [kB-1, known_lo) of prefix are fixed
  unsigned long long need[2];  // rank (counts) or mass still to cover inside the prefix range
  unsigned long long above[2]; // count / mass of keys above the prefix range
  unsigned long long last[2];  // count / mass of the last selected bin
  int ok[2];
};

struct NearSum {  // cluster-wide near-max histograms on the global maximum, per row
  unsigned long long cnt[2][kNearBins];
  unsigned long long mass[2][kNearBins];  // 2^-40 fixed point
  float z[2];                             // dense normaliser
  unsigned long long tot[2];              // fixed-point mass of every element
  uint32_t gmax[2];
  uint32_t flags[2];
};

// One CTA's contribution to a fast-path reduction round, as stored into every
// peer's shared memory (slot [parity][sender rank]).  Window bins count the
// keys at distance d below the sender's largest key; a CTA's chunk never holds
// more than 65535 elements, so 16-bit counts suffice.
struct Inbox {
  uint32_t maxkey[2];
  uint32_t flags[2];
  float z[2];
  uint32_t pad[2];
  unsigned long long tot[2];
  uint16_t cnt[2][kNearBins];
};
static_assert(sizeof(Inbox) % 16 == 0, "inbox slots are written with 16-byte stores");

// Windows below the first: running totals and results per row.
struct Bands {
  unsigned long long cnt_above[2];   // keys above the current window
  unsigned long long mass_above[2];  // their fixed-point mass
  unsigned long long kept[2];        // mass of the kept set once resolved
  uint32_t cut[2];                   // resolved cut (16-bit key)
  int done[2];                       // resolved (or needs no further window)
  int fallback;                      // give the rows to the multi-pass selection
};

struct LogitsSmem {
  ReduceSmem red;
  Bands bands;
  StatPart part[2];
  StatSum sum;
  NearSum near;
  float wz[2][kWarps];
  unsigned long long wt[2][kWarps];
  Select sel;
  uint64_t bar;
  int stop_first;      // first committed stop token
  uint4 xw[kMaxCluster];  // every CTA's word of the last cluster exchange, by rank
  float pz[2];            // block totals of the processors' correction
  uint32_t pmark;         // marks of the draft token, from the CTA holding it
  uint32_t xmax[2];       // block maxima (ordered bits) of the processors' rescue pass
  int32_t tok[SV_MAX_SPEC_LEN + 1];
};

enum : uint32_t { kRMax = 1u, kRCnt = 2u, kRMass = 4u, kRZ = 8u, kRTot = 16u };

__device__ __forceinline__ void zero_part(StatPart &p, uint32_t what, int nr) {
  const int tid = threadIdx.x;
  if (what & kRMass)
    for (int t = tid; t < nr * 256; t += kThreads) p.massf[t >> 8][t & 255] = 0.0f;
  if (what & kRCnt)
    for (int t = tid; t < nr * 256; t += kThreads) p.cnt[t >> 8][t & 255] = 0u;
  if (tid < 2) {
    p.maxkey[tid] = 0u;
    p.flags[tid] = 0u;
    p.floor[tid] = 0xFFFFFFFFu;
    p.nbins[tid] = 0u;
    p.z[tid] = 0.0f;
    p.tot[tid] = 0ull;
  }
}

__device__ __forceinline__ unsigned long long to_fixed(float e) {
  return static_cast<unsigned long long>(__float2ull_rn(e * kMassScale));
}

// Combine every CTA's part[par] into sum (the same in every CTA of the cluster).
__device__ __forceinline__ void stat_reduce(LogitsSmem &sm, int par, uint32_t what, int nr, uint32_t ncta) {
  __syncthreads();
  cluster_sync();
  const int tid = threadIdx.x;
  StatPart &p = sm.part[par];
  if (what & kRCnt) {
    for (int t = tid; t < nr * 256; t += kThreads) {
      const uint32_t a = smem_addr(&p.cnt[t >> 8][t & 255]);
      uint32_t v[kMaxCluster];
#pragma unroll
      for (int c = 0; c < kMaxCluster; ++c) v[c] = c < static_cast<int>(ncta) ? ld_dsmem_u32(map_to_rank(a, c)) : 0u;
      uint32_t s = 0;
#pragma unroll
      for (int c = 0; c < kMaxCluster; ++c) s += v[c];
      sm.sum.cnt[t >> 8][t & 255] = s;
    }
  }
  if (what & kRMass) {
    for (int t = tid; t < nr * 256; t += kThreads) {
      const uint32_t a = smem_addr(&p.massf[t >> 8][t & 255]);
      uint32_t v[kMaxCluster];
#pragma unroll
      for (int c = 0; c < kMaxCluster; ++c) v[c] = c < static_cast<int>(ncta) ? ld_dsmem_u32(map_to_rank(a, c)) : 0u;
      unsigned long long s = 0;
#pragma unroll
      for (int c = 0; c < kMaxCluster; ++c) s += to_fixed(__uint_as_float(v[c]));  // exact integer sum
      sm.sum.mass[t >> 8][t & 255] = s;
    }
  }
  if (tid < nr) {  // every remote load is issued before any is consumed
    if (what & kRMax) {
      uint32_t mk[kMaxCluster], fl[kMaxCluster];
#pragma unroll
      for (int c = 0; c < kMaxCluster; ++c) {
        const bool in = c < static_cast<int>(ncta);
        mk[c] = in ? ld_dsmem_u32(map_to_rank(smem_addr(&p.maxkey[tid]), c)) : 0u;
        fl[c] = in ? ld_dsmem_u32(map_to_rank(smem_addr(&p.flags[tid]), c)) : 0u;
      }
      uint32_t m = 0, f = 0;
#pragma unroll
      for (int c = 0; c < kMaxCluster; ++c) {
        m = max(m, mk[c]);
        f |= fl[c];
      }
      sm.sum.maxkey[tid] = m;
      sm.sum.flags[tid] = f;
    }
    if (what & kRZ) {
      uint32_t zb[kMaxCluster];
#pragma unroll
      for (int c = 0; c < kMaxCluster; ++c)
        zb[c] = c < static_cast<int>(ncta) ? ld_dsmem_u32(map_to_rank(smem_addr(&p.z[tid]), c)) : 0u;
      float z = 0.0f;
#pragma unroll
      for (int c = 0; c < kMaxCluster; ++c) z += __uint_as_float(zb[c]);
      sm.sum.z[tid] = z;
    }
    if (what & kRTot) {
      unsigned long long tv[kMaxCluster];
#pragma unroll
      for (int c = 0; c < kMaxCluster; ++c)
        tv[c] = c < static_cast<int>(ncta) ? ld_dsmem_u64(map_to_rank(smem_addr(&p.tot[tid]), c)) : 0ull;
      unsigned long long t = 0;
#pragma unroll
      for (int c = 0; c < kMaxCluster; ++c) t += tv[c];
      sm.sum.tot[tid] = t;
    }
  }
  __syncthreads();
}

// Deterministic block sums (fixed shuffle tree, then warps in order) into part.
__device__ __forceinline__ void block_sum_z(LogitsSmem &sm, StatPart &p, const float v[2], int nr) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int r = 0; r < nr; ++r) {
    float s = v[r];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, o);
    if (lane == 0) sm.wz[r][warp] = s;
  }
  __syncthreads();
  if (threadIdx.x < nr) {
    float s = 0.0f;
    for (int w = 0; w < kWarps; ++w) s += sm.wz[threadIdx.x][w];
    p.z[threadIdx.x] = s;
  }
}
__device__ __forceinline__ void block_sum_tot(LogitsSmem &sm, StatPart &p, const unsigned long long v[2], int nr) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int r = 0; r < nr; ++r) {
    unsigned long long s = v[r];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, o);
    if (lane == 0) sm.wt[r][warp] = s;
  }
  __syncthreads();
  if (threadIdx.x < nr) {
    unsigned long long s = 0;
    for (int w = 0; w < kWarps; ++w) s += sm.wt[threadIdx.x][w];
    p.tot[threadIdx.x] = s;
  }
}

// One warp picks a bin of row r.  Bins are walked from the largest keys
// down: logical bin L is physical bin L for near-max histograms (distance from
// the largest key) and 255 - L for digit histograms.  The chosen bin is the
// first whose running total reaches `need`; records what lies above it.
template <bool kNear, typename H>
__device__ __forceinline__ void select_bin(LogitsSmem &sm, int r, const H *h, int lo, uint32_t near_base) {
  const int lane = threadIdx.x & 31;
  auto hv = [&](int L) -> unsigned long long { return static_cast<unsigned long long>(h[kNear ? L : 255 - L]); };
  unsigned long long own = 0;
#pragma unroll
  for (int t = 0; t < 8; ++t) own += hv(8 * lane + t);
  unsigned long long inc = own;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long v = __shfl_up_sync(0xFFFFFFFFu, inc, o);
    if (lane >= o) inc += v;
  }
  const unsigned long long before = inc - own;
  const unsigned long long need = sm.sel.need[r];
  int found = -1;
  unsigned long long above = 0, last = 0;
  if (before < need && inc >= need) {
    unsigned long long acc = before;
    for (int t = 0; t < 8; ++t) {
      const unsigned long long x = hv(8 * lane + t);
      if (acc + x >= need) {
        found = 8 * lane + t;
        above = acc;
        last = x;
        break;
      }
      acc += x;
    }
  }
  const unsigned ball = __ballot_sync(0xFFFFFFFFu, found >= 0);
  if (ball == 0) {
    if (lane == 0) sm.sel.ok[r] = 0;
    return;
  }
  const int src = __ffs(ball) - 1;
  const int L = __shfl_sync(0xFFFFFFFFu, found, src);
  above = __shfl_sync(0xFFFFFFFFu, above, src);
  last = __shfl_sync(0xFFFFFFFFu, last, src);
  if (lane == 0) {
    if (kNear) {
      sm.sel.prefix[r] = (near_base - static_cast<uint32_t>(L)) << lo;  // the top 16 key bits
    } else {
      sm.sel.prefix[r] |= static_cast<uint32_t>(255 - L) << lo;
    }
    sm.sel.known_lo[r] = lo;
    sm.sel.need[r] = need - above;
    sm.sel.above[r] += above;
    sm.sel.last[r] = last;
    sm.sel.ok[r] = 1;
  }
}

template <typename TIn>
__device__ __forceinline__ uint32_t key16_of(uint32_t k) {
  return Elem<TIn>::kBits == 16 ? k : (k >> 16);
}


// Refine the selection of every row whose prefix is not complete, one 8-bit
// digit per level (counts, or fixed-point masses of keys >= tau).
template <typename TIn, bool kMass>
__device__ void radix_refine(LogitsSmem &sm, TIn *const srow[2], int nr, int n, const uint32_t tau[2],
                             const RowStats st[2], int &step, uint32_t ncta) {
  using E = Elem<TIn>;
  constexpr int kB = E::kBits;
  const int tid = threadIdx.x;
  for (int lo = kB - 8; lo >= 0; lo -= 8) {
    bool any = false;
    for (int r = 0; r < nr; ++r) any |= sm.sel.known_lo[r] > lo;
    if (!any) continue;
    const int par = step & 1;
    zero_part(sm.part[par], kMass ? kRMass : kRCnt, nr);
    __syncthreads();
    for (int r = 0; r < nr; ++r) {
      if (sm.sel.known_lo[r] <= lo) continue;
      const int hi_shift = lo + 8;
      const uint32_t hi = hi_shift >= 32 ? 0u : (sm.sel.prefix[r] >> hi_shift);
      const TIn *s = srow[r];
      for (int x = tid; x < n; x += kThreads) {
        const uint32_t b = bits_at(s, x);
        const uint32_t k = E::key(b);
        if (hi_shift < 32 && (k >> hi_shift) != hi) continue;
        if (kMass) {
          if (k < tau[r]) continue;
          const float e = exp2f(__fmul_rn(__fsub_rn(E::val(b), st[r].vmax), st[r].c2));
          atomicAdd(&sm.part[par].massf[r][(k >> lo) & 255u], e);
        } else {
          atomicAdd(&sm.part[par].cnt[r][(k >> lo) & 255u], 1u);
        }
      }
    }
    stat_reduce(sm, par, kMass ? kRMass : kRCnt, nr, ncta);
    ++step;
    const int warp = tid >> 5;
    if (warp < nr && sm.sel.known_lo[warp] > lo) {
      if (kMass) select_bin<false>(sm, warp, sm.sum.mass[warp], lo, 0u);
      else select_bin<false>(sm, warp, sm.sum.cnt[warp], lo, 0u);
    }
    __syncthreads();
  }
}

// ---------------------------------------------------------------------------
// row statistics, multi-pass path: exact radix selections over the rows in
// shared memory, one cluster reduction per 8-bit digit.  Used when the
// threshold or cut lies beyond the near-max window, for fp32 logits, and for
// top-p without top-k over a wide nucleus.  st[r].vmax / c2 are already set.
// ---------------------------------------------------------------------------
template <typename TIn>
__device__ bool stats_slow(LogitsSmem &sm, TIn *const srow[2], int nr, int n, float c2, int topk, float topp,
                           const uint32_t maxk16[2], RowStats st[2], int &step, uint32_t ncta) {
  using E = Elem<TIn>;
  constexpr int kB = E::kBits;
  const int tid = threadIdx.x;
  const bool use_k = topk > 0;
  const bool use_p = topp < 1.0f;
  int par;

  // top-k: the k-th largest key (ties kept).  First count the keys within
  // kNearBins steps of the largest (where the threshold almost always lies),
  // then refine or fall back to a full radix selection.
  uint32_t tau[2] = {0u, 0u};
  if (use_k) {
    par = step & 1;
    zero_part(sm.part[par], kRCnt, nr);
    if (tid < 2) {
      sm.sel.prefix[tid] = 0u;
      sm.sel.known_lo[tid] = kB;
      sm.sel.need[tid] = static_cast<unsigned long long>(topk);
      sm.sel.above[tid] = 0ull;
    }
    __syncthreads();
    for (int r = 0; r < nr; ++r) {
      const TIn *s = srow[r];
      for (int x = tid; x < n; x += kThreads) {
        const uint32_t d = maxk16[r] - key16_of<TIn>(E::key(bits_at(s, x)));
        if (d < static_cast<uint32_t>(kNearBins)) atomicAdd(&sm.part[par].cnt[r][d], 1u);
      }
    }
    stat_reduce(sm, par, kRCnt, nr, ncta);
    ++step;
    if ((tid >> 5) < nr) select_bin<true>(sm, tid >> 5, sm.sum.cnt[tid >> 5], kB - 16, maxk16[tid >> 5]);
    __syncthreads();
    if (tid < nr && !sm.sel.ok[tid]) {  // threshold farther than the near bins: full selection
      sm.sel.prefix[tid] = 0u;
      sm.sel.known_lo[tid] = kB;
      sm.sel.need[tid] = static_cast<unsigned long long>(topk);
      sm.sel.above[tid] = 0ull;
    }
    __syncthreads();
    radix_refine<TIn, false>(sm, srow, nr, n, tau, st, step, ncta);
    for (int r = 0; r < nr; ++r) tau[r] = sm.sel.prefix[r];
  }

  if (!use_p) {  // normaliser over the top-k set
    par = step & 1;
    zero_part(sm.part[par], kRZ, nr);
    __syncthreads();
    float zt[2] = {0.0f, 0.0f};
    for (int r = 0; r < nr; ++r) {
      const TIn *s = srow[r];
      float sum = 0.0f, comp = 0.0f;
      for (int x = tid; x < n; x += kThreads) {
        const uint32_t b = bits_at(s, x);
        if (E::key(b) < tau[r]) continue;
        const float e = exp2f(__fmul_rn(__fsub_rn(E::val(b), st[r].vmax), c2));
        const float y = e - comp;  // Kahan
        const float t = sum + y;
        comp = (t - sum) - y;
        sum = t;
      }
      zt[r] = sum;
    }
    block_sum_z(sm, sm.part[par], zt, nr);
    stat_reduce(sm, par, kRZ, nr, ncta);
    ++step;
    for (int r = 0; r < nr; ++r) {
      st[r].cut = tau[r];
      st[r].zp = sm.sum.z[r];
    }
    return true;
  }

  // top-p: the largest key c with mass(key >= c) >= top_p * mass(top-k set),
  // masses in 2^-40 fixed point; near-max bins first, then refine / fall back.
  par = step & 1;
  zero_part(sm.part[par], kRMass | kRTot, nr);
  __syncthreads();
  {
    unsigned long long tt[2] = {0ull, 0ull};
    for (int r = 0; r < nr; ++r) {
      const TIn *s = srow[r];
      unsigned long long tot = 0;
      for (int x = tid; x < n; x += kThreads) {
        const uint32_t b = bits_at(s, x);
        const uint32_t k = E::key(b);
        if (k < tau[r]) continue;
        const float e = exp2f(__fmul_rn(__fsub_rn(E::val(b), st[r].vmax), c2));
        tot += to_fixed(e);
        const uint32_t d = maxk16[r] - key16_of<TIn>(k);
        if (d < static_cast<uint32_t>(kNearBins)) atomicAdd(&sm.part[par].massf[r][d], e);
      }
      tt[r] = tot;
    }
    block_sum_tot(sm, sm.part[par], tt, nr);
  }
  stat_reduce(sm, par, kRMass | kRTot, nr, ncta);
  ++step;
  if (tid < 2) {
    const unsigned long long tot = sm.sum.tot[tid < nr ? tid : 0];
    unsigned long long need = static_cast<unsigned long long>(static_cast<double>(topp) * static_cast<double>(tot));
    sm.sel.prefix[tid] = 0u;
    sm.sel.known_lo[tid] = kB;
    sm.sel.need[tid] = need > 0 ? need : 1ull;
    sm.sel.above[tid] = 0ull;
    sm.sel.last[tid] = 0ull;
  }
  __syncthreads();
  if ((tid >> 5) < nr) select_bin<true>(sm, tid >> 5, sm.sum.mass[tid >> 5], kB - 16, maxk16[tid >> 5]);
  __syncthreads();
  if (tid < nr && !sm.sel.ok[tid]) {
    const unsigned long long tot = sm.sum.tot[tid];
    const unsigned long long need = static_cast<unsigned long long>(static_cast<double>(topp) * static_cast<double>(tot));
    sm.sel.prefix[tid] = 0u;
    sm.sel.known_lo[tid] = kB;
    sm.sel.need[tid] = need > 0 ? need : 1ull;
    sm.sel.above[tid] = 0ull;
  }
  __syncthreads();
  radix_refine<TIn, true>(sm, srow, nr, n, tau, st, step, ncta);
  for (int r = 0; r < nr; ++r) {
    st[r].cut = max(tau[r], sm.sel.prefix[r]);
    const unsigned long long kept = sm.sel.above[r] + sm.sel.last[r];  // mass of keys >= cut
    st[r].zp = static_cast<float>(static_cast<double>(kept) * (1.0 / static_cast<double>(kMassScale)));
  }
  return true;
}

// ---------------------------------------------------------------------------
// row statistics of one position (target row, and draft row when nr == 2),
// the rows already in shared memory.
//
// Fast path, one cluster reduction: every CTA measures its chunk against its
// own largest key -- value checks, and for bf16 top-k/top-p rows the count of
// each key within kNearBins steps below that maximum (and not below a floor
// the k-th largest key cannot undercut); dense rows: the local normaliser.
// Each CTA stores these into every peer's inbox; after one cluster barrier
// every CTA shifts the peers' bins onto the global maximum, sums them as
// integers and weighs each bin (one bf16 value) by exp2((v - max) * c2) in
// 2^-40 fixed point.  That resolves the k-th largest key, the top-p cut and
// the normaliser whenever they lie in the window.
// ---------------------------------------------------------------------------
// One warp resolves a row's kept set from its near bins (walking from
// distance 0, the largest key): the top-k bin L (the first whose running
// count reaches k; all 128 bins when top-k is off) and, for top-p, the first
// bin at or above L whose running mass reaches top_p times the mass kept so
// far.  `total` is the mass of every key of the row (used when top-k is
// off).  Counts and masses share one prefix scan; all sums are integers, so
// every CTA of the cluster chooses alike.  Returns false when a bin lies
// outside the window.
constexpr int kBinsPerLane = kNearBins / 32;
struct NearChoice {
  int last;                 // last kept bin (distance from the largest key)
  unsigned long long kept;  // fixed-point mass of bins 0..last
};
__device__ __forceinline__ bool near_select(const unsigned long long *cnt, const unsigned long long *mass, int topk,
                                            bool use_p, float topp, unsigned long long total, NearChoice *out) {
  const int lane = threadIdx.x & 31;
  unsigned long long c[kBinsPerLane], m[kBinsPerLane], cs = 0, ms = 0;
#pragma unroll
  for (int t = 0; t < kBinsPerLane; ++t) {
    c[t] = cnt[kBinsPerLane * lane + t];
    m[t] = mass[kBinsPerLane * lane + t];
    cs += c[t];
    ms += m[t];
  }
  unsigned long long ci = cs, mi = ms;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long vc = __shfl_up_sync(0xFFFFFFFFu, ci, o);
    const unsigned long long vm = __shfl_up_sync(0xFFFFFFFFu, mi, o);
    if (lane >= o) {
      ci += vc;
      mi += vm;
    }
  }
  const unsigned long long cb = ci - cs, mb = mi - ms;  // totals before this lane's bins
  int last = kNearBins - 1;
  unsigned long long kept = total;
  if (topk > 0) {
    const unsigned long long k = static_cast<unsigned long long>(topk);
    int found = -1;
    unsigned long long kin = 0;
    if (cb < k && ci >= k) {
      unsigned long long acc = cb, macc = mb;
#pragma unroll
      for (int t = 0; t < kBinsPerLane; ++t) {
        acc += c[t];
        macc += m[t];
        if (found < 0 && acc >= k) {
          found = kBinsPerLane * lane + t;
          kin = macc;
        }
      }
    }
    const unsigned ball = __ballot_sync(0xFFFFFFFFu, found >= 0);
    if (!ball) return false;
    const int src = __ffs(ball) - 1;
    last = __shfl_sync(0xFFFFFFFFu, found, src);
    kept = __shfl_sync(0xFFFFFFFFu, kin, src);
  }
  if (use_p) {
    unsigned long long need = static_cast<unsigned long long>(static_cast<double>(topp) * static_cast<double>(kept));
    if (need == 0ull) need = 1ull;
    int found = -1;
    unsigned long long in = 0;
    if (mb < need && mi >= need) {
      unsigned long long acc = mb;
#pragma unroll
      for (int t = 0; t < kBinsPerLane; ++t) {
        acc += m[t];
        if (found < 0 && acc >= need) {
          found = kBinsPerLane * lane + t;
          in = acc;
        }
      }
    }
    const unsigned ball = __ballot_sync(0xFFFFFFFFu, found >= 0 && found <= last);
    if (!ball) return false;
    const int src = __ffs(ball) - 1;
    last = __shfl_sync(0xFFFFFFFFu, found, src);
    kept = __shfl_sync(0xFFFFFFFFu, in, src);
  }
  out->last = last;
  out->kept = kept;
  return true;
}

// One warp resolves a row in a window below the first one.  cnt_above and
// mass_above are the count and fixed-point mass of every key above the
// window; the choices are those of near_select continued across windows.
// Returns 1 when resolved (*out), 0 when the threshold or cut lies further
// down (*cnt_tot, *mass_tot: this window's totals), 2 when the top-p cut of a
// top-k row lies above this window (the multi-pass selection takes over).
__device__ __forceinline__ int band_select(const unsigned long long *cnt, const unsigned long long *mass, int topk,
                                           bool use_p, float topp, unsigned long long total,
                                           unsigned long long cnt_above, unsigned long long mass_above,
                                           NearChoice *out, unsigned long long *cnt_tot,
                                           unsigned long long *mass_tot) {
  const int lane = threadIdx.x & 31;
  unsigned long long c[kBinsPerLane], m[kBinsPerLane], cs = 0, ms = 0;
#pragma unroll
  for (int t = 0; t < kBinsPerLane; ++t) {
    c[t] = cnt[kBinsPerLane * lane + t];
    m[t] = mass[kBinsPerLane * lane + t];
    cs += c[t];
    ms += m[t];
  }
  unsigned long long ci = cs, mi = ms;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long vc = __shfl_up_sync(0xFFFFFFFFu, ci, o);
    const unsigned long long vm = __shfl_up_sync(0xFFFFFFFFu, mi, o);
    if (lane >= o) {
      ci += vc;
      mi += vm;
    }
  }
  *cnt_tot = __shfl_sync(0xFFFFFFFFu, ci, 31);
  *mass_tot = __shfl_sync(0xFFFFFFFFu, mi, 31);
  const unsigned long long cb = cnt_above + ci - cs, mb = mass_above + mi - ms;  // totals before this lane's bins
  int last = kNearBins - 1;
  unsigned long long kept = 0;
  if (topk > 0) {
    const unsigned long long k = static_cast<unsigned long long>(topk);
    int found = -1;
    unsigned long long kin = 0;
    if (cb < k && cnt_above + ci >= k) {
      unsigned long long acc = cb, macc = mb;
#pragma unroll
      for (int t = 0; t < kBinsPerLane; ++t) {
        acc += c[t];
        macc += m[t];
        if (found < 0 && acc >= k) {
          found = kBinsPerLane * lane + t;
          kin = macc;
        }
      }
    }
    const unsigned ball = __ballot_sync(0xFFFFFFFFu, found >= 0);
    if (!ball) return 0;
    const int src = __ffs(ball) - 1;
    last = __shfl_sync(0xFFFFFFFFu, found, src);
    kept = __shfl_sync(0xFFFFFFFFu, kin, src);
    if (!use_p) {
      out->last = last;
      out->kept = kept;
      return 1;
    }
  } else {
    kept = total;
  }
  unsigned long long need = static_cast<unsigned long long>(static_cast<double>(topp) * static_cast<double>(kept));
  if (need == 0ull) need = 1ull;
  if (topk > 0 && need <= mass_above) return 2;
  int found = -1;
  unsigned long long in = 0;
  if (mb < need && mass_above + mi >= need) {
    unsigned long long acc = mb;
#pragma unroll
    for (int t = 0; t < kBinsPerLane; ++t) {
      acc += m[t];
      if (found < 0 && acc >= need) {
        found = kBinsPerLane * lane + t;
        in = acc;
      }
    }
  }
  const unsigned ball = __ballot_sync(0xFFFFFFFFu, found >= 0 && found <= last);
  if (!ball) return 0;
  const int src = __ffs(ball) - 1;
  out->last = __shfl_sync(0xFFFFFFFFu, found, src);
  out->kept = __shfl_sync(0xFFFFFFFFu, in, src);
  return 1;
}

// Every 16-byte group of a bf16 chunk, kWalkGroups per lane with their loads
// in flight together: mask(group) gives 8 candidate bits (bit t: the low half
// of word t, bit 4 + t: its high half), the lanes' masks form one 64-bit word
// each, and the warp walks the set bits in step (one candidate per lane per
// trip), handing each candidate's bits to take.
template <typename TIn, typename MaskF, typename TakeF>
__device__ __forceinline__ void walk_groups(const TIn *row, int ng, MaskF mask, TakeF take) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint4 *s4 = reinterpret_cast<const uint4 *>(row);
  for (int vb = warp * 32; vb < ng; vb += kWalkGroups * kThreads) {
    unsigned long long M = 0ull;
#pragma unroll
    for (int h = 0; h < kWalkGroups; ++h) {
      const int v = vb + h * kThreads + lane;
      if (v < ng) M |= static_cast<unsigned long long>(mask(s4[v])) << (8 * h);
    }
    while (__any_sync(0xFFFFFFFFu, M != 0ull)) {
      if (M != 0ull) {
        const int pos = __ffsll(static_cast<long long>(M)) - 1;
        M &= M - 1ull;
        take(bits_at(row, 8 * (vb + (pos >> 3) * kThreads + lane) + 2 * (pos & 3) + ((pos >> 2) & 1)));
      }
    }
  }
}

constexpr int kMaxBands = 24;  // windows below the first before the multi-pass selection takes over

// Windows 1, 2, ... below the first: window b holds the keys
// [g - kNearBins (b + 1) + 1, g - kNearBins b] of the row's global maximum g.
// Rows the first window resolved keep its result.  Returns false when a row
// needs the multi-pass selection (the cut of a top-k row above its threshold's
// window, or more than kMaxBands windows).
template <typename TIn>
__device__ bool window_rounds(LogitsSmem &sm, Inbox *inbox, TIn *const srow[2], int nr, int n, float c2, int topk,
                              bool use_p, float topp, RowStats st[2], int &step, uint32_t ncta, uint32_t rank) {
  using E = Elem<TIn>;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  NearSum &ns = sm.near;
  Bands &bd = sm.bands;
  if (warp < nr) {  // the first window's totals (complete whenever it failed)
    const int r = warp;
    unsigned long long c = 0, m = 0;
#pragma unroll
    for (int t = 0; t < kBinsPerLane; ++t) {
      c += ns.cnt[r][kBinsPerLane * lane + t];
      m += ns.mass[r][kBinsPerLane * lane + t];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      c += __shfl_xor_sync(0xFFFFFFFFu, c, o);
      m += __shfl_xor_sync(0xFFFFFFFFu, m, o);
    }
    if (lane == 0) {
      bd.done[r] = sm.sel.ok[r];
      bd.cnt_above[r] = c;
      bd.mass_above[r] = m;
    }
  }
  if (tid == 0) bd.fallback = 0;
  __syncthreads();
  uint32_t g16[2] = {0u, 0u};
  float gv[2] = {0.0f, 0.0f};
  for (int r = 0; r < nr; ++r) {
    g16[r] = ns.gmax[r];
    gv[r] = E::val_of_key(ns.gmax[r]);
  }
  const int ng = n >> 3;
  for (int band = 1;; ++band) {
    bool active = false;
    for (int r = 0; r < nr; ++r) active |= !bd.done[r];
    if (!active || bd.fallback) break;
    const int par = step & 1;
    StatPart &bp = sm.part[par];
    zero_part(bp, kRCnt, nr);
    __syncthreads();
    for (int r = 0; r < nr; ++r) {
      if (bd.done[r]) continue;
      const int hi = static_cast<int>(g16[r]) - kNearBins * band;  // this window's largest key
      if (hi < 0x80) continue;  // below every finite key: nothing to count
      const int lo = max(hi - (kNearBins - 1), 0x80);
      const uint32_t lob = bf16_bits_of_key(static_cast<uint32_t>(lo)),
                     hib = bf16_bits_of_key(static_cast<uint32_t>(hi + 1));
      const uint32_t lo2 = lob | (lob << 16), hi2 = hib | (hib << 16);
      uint32_t *cnt = bp.cnt[r];
      const TIn *row = srow[r];
      auto band_mask = [&](const uint4 &dv) {  // bit t: low half of word t in the window, bit 4 + t: high half
        uint32_t g = ((bf16x2_ge_mask(dv.x, lo2) & ~bf16x2_ge_mask(dv.x, hi2)) & 0x00010001u) |
                     (((bf16x2_ge_mask(dv.y, lo2) & ~bf16x2_ge_mask(dv.y, hi2)) & 0x00010001u) << 1) |
                     (((bf16x2_ge_mask(dv.z, lo2) & ~bf16x2_ge_mask(dv.z, hi2)) & 0x00010001u) << 2) |
                     (((bf16x2_ge_mask(dv.w, lo2) & ~bf16x2_ge_mask(dv.w, hi2)) & 0x00010001u) << 3);
        return (g | (g >> 12)) & 0xFFu;
      };
      auto count = [&](uint32_t b) {
        const uint32_t d = static_cast<uint32_t>(hi) - E::key(b);
        if (E::finite(b) && d < static_cast<uint32_t>(kNearBins)) atomicAdd(&cnt[d], 1u);
      };
      // every group is read again (keeping the group maxima live through the
      // reduction would cost registers on the common path)
      walk_groups(row, ng, band_mask, count);
      for (int x = (ng << 3) + tid; x < n; x += kThreads) count(bits_at(row, x));
    }
    __syncthreads();
    // every CTA stores its window counts (16-bit) into its slot of every peer's
    // inbox; after the barrier the sums need no shift (one anchor for all)
    Inbox *const ibx = inbox + par * static_cast<int>(ncta);
    {
      const int words = kNearBins / 8;
      for (int t = tid; t < nr * words * static_cast<int>(ncta); t += kThreads) {
        const int c = t / (nr * words), k = t % (nr * words);
        const int r = k / words, d0 = (k % words) * 8;
        uint32_t h[4] = {0u, 0u, 0u, 0u};
        if (!bd.done[r]) {
#pragma unroll
          for (int q = 0; q < 4; ++q) h[q] = bp.cnt[r][d0 + 2 * q] | (bp.cnt[r][d0 + 2 * q + 1] << 16);
        }
        st_dsmem_v4(map_to_rank(smem_addr(reinterpret_cast<uint4 *>(&ibx[rank]) + 3 + r * words + d0 / 8),
                                static_cast<uint32_t>(c)),
                    make_uint4(h[0], h[1], h[2], h[3]));
      }
    }
    cluster_sync();
    ++step;
    if (tid < nr * kNearBins) {
      const int r = tid / kNearBins, d = tid % kNearBins;
      unsigned long long cs = 0;
      const int key = static_cast<int>(g16[r]) - kNearBins * band - d;
      if (!bd.done[r] && key >= 0x80) {
        for (int c = 0; c < static_cast<int>(ncta); ++c) cs += ibx[c].cnt[r][d];
      }
      ns.cnt[r][d] = cs;
      ns.mass[r][d] = cs ? cs * to_fixed(exp2f(__fmul_rn(__fsub_rn(E::val_of_key(static_cast<uint32_t>(key)), gv[r]),
                                                       c2)))
                         : 0ull;
    }
    __syncthreads();
    if (warp < nr && !bd.done[warp]) {
      const int r = warp;
      NearChoice ch;
      unsigned long long ct = 0, mt = 0;
      const int res = band_select(ns.cnt[r], ns.mass[r], topk, use_p, topp, ns.tot[r], bd.cnt_above[r],
                                  bd.mass_above[r], &ch, &ct, &mt);
      if (lane == 0) {
        const int hi = static_cast<int>(g16[r]) - kNearBins * band;
        if (res == 1) {
          bd.done[r] = 1;
          bd.cut[r] = static_cast<uint32_t>(hi - ch.last);
          bd.kept[r] = ch.kept;
        } else if (res == 2 || band >= kMaxBands || hi - (kNearBins - 1) <= 0x80) {
          bd.fallback = 1;  // (keys exhausted without a cut: rounding between the totals)
        } else {
          bd.cnt_above[r] += ct;
          bd.mass_above[r] += mt;
        }
      }
    }
    __syncthreads();
  }
  if (bd.fallback) {
    __syncthreads();
    return false;
  }
  for (int r = 0; r < nr; ++r) {
    if (sm.sel.ok[r]) {  // resolved by the first window
      st[r].cut = sm.sel.prefix[r];
      st[r].zp = ns.z[r];
    } else {
      st[r].cut = bd.cut[r];
      st[r].zp = static_cast<float>(static_cast<double>(bd.kept[r]) * (1.0 / static_cast<double>(kMassScale)));
    }
  }
  return true;
}

template <typename TIn>
__device__ bool position_stats(LogitsSmem &sm, Inbox *inbox, TIn *const srow[2], int nr, int n, float c2, int topk,
                               float topp, uint32_t load_flags, RowStats st[2], uint32_t *req_bits, int &step,
                               uint32_t ncta, uint32_t rank) {
  using E = Elem<TIn>;
  constexpr int kB = E::kBits;
  const int tid = threadIdx.x;
  const bool use_k = topk > 0;
  const bool use_p = topp < 1.0f;
  const bool near = use_k || use_p;
  // top-k rows with k <= 32 * kWarps: a per-CTA lower bound of the threshold
  // narrows the window scan (keys below it cannot be among the top k)
  const bool use_floor = kB == 16 && use_k && topk <= 32 * kWarps;
  const int par = step & 1;
  StatPart &lp = sm.part[par];

  // local pass A: largest key and value checks of this CTA's chunk
  zero_part(lp, (kB == 16 && near) ? kRCnt : 0u, nr);
  __syncthreads();
  uint32_t mk[2] = {0u, 0u}, fl[2] = {load_flags, load_flags};  // this thread's largest finite key, flags
  // bf16 rows whose chunk gives a thread at most 2 * kGroupWords 16-byte
  // groups keep each group's largest value in registers (two per word, NaN
  // for absent groups), so the window pass re-reads only groups that hold a
  // candidate
  const int ng_all = n >> 3;
  const bool reg_groups = kB == 16 && ng_all <= 2 * kGroupWords * kThreads;
  uint32_t gw[2][kGroupWords];
  // dense rows with register-held group maxima also sum their weights in this
  // pass: each thread keeps a compensated sum relative to its running maximum
  // and rescales it when the maximum rises (once per rising group)
  const bool fuse_z = reg_groups && (!near || (use_p && !use_k));  // dense rows, or top-p alone (its total)
  float omax[2] = {-INFINITY, -INFINITY}, osum[2] = {0.0f, 0.0f};
  // rows with register-held group maxima: both rows in one unrolled loop, so
  // their group loads are in flight together; one copy of the loop for
  // summing rows and one for top-k / top-p rows, which so keeps no branch
  // between its loads.  Wider bf16 chunks and fp32 rows take the per-row loop
  // after it.
  const bool both_rows = kB == 16 && reg_groups;
  auto both_rows_pass = [&](auto sums) {
    constexpr bool kSums = decltype(sums)::value;
    uint32_t acc[2] = {0xFF80FF80u, 0xFF80FF80u};  // (-inf, -inf)
    float om2[2] = {-INFINITY, -INFINITY}, oz2[2] = {0.0f, 0.0f}, oc2[2] = {0.0f, 0.0f};
    auto raise2 = [&](int r, float m) {  // a larger running maximum: rescale the sum
      if (m > om2[r]) {
        if (om2[r] != -INFINITY) {
          const float f = exp2f(__fmul_rn(__fsub_rn(om2[r], m), c2));
          oz2[r] = __fmul_rn(oz2[r], f);
          oc2[r] = __fmul_rn(oc2[r], f);
        }
        om2[r] = m;
      }
    };
    auto add2 = [&](int r, uint32_t b) {  // (-inf adds 0; NaN/+inf rows are rejected anyway)
      const float y = exp2f(__fmul_rn(__fsub_rn(E::val(b), om2[r]), c2)) - oc2[r];  // Kahan
      const float t = oz2[r] + y;
      oc2[r] = (t - oz2[r]) - y;
      oz2[r] = t;
    };
#pragma unroll
    for (int i = 0; i < kGroupWords; ++i) {
      uint32_t half[2][2] = {{0x7FFFu, 0x7FFFu}, {0x7FFFu, 0x7FFFu}};  // NaN: never a window candidate
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int v = tid + (2 * i + h) * kThreads;
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          if (r < nr && v < ng_all) {
            const uint4 d = reinterpret_cast<const uint4 *>(srow[r])[v];
            uint32_t p2 = bf16x2_max_nan(bf16x2_max_nan(d.x, d.y), bf16x2_max_nan(d.z, d.w));
            p2 = bf16x2_max_nan(p2, (p2 >> 16) | (p2 << 16));
            acc[r] = bf16x2_max_nan(acc[r], p2);
            half[r][h] = p2 & 0xFFFFu;
            if (kSums) {
              raise2(r, E::val(p2 & 0xFFFFu));
              if (om2[r] != -INFINITY) {
                const uint32_t w[4] = {d.x, d.y, d.z, d.w};
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                  add2(r, w[t] & 0xFFFFu);
                  add2(r, w[t] >> 16);
                }
              }
            }
          }
        }
      }
#pragma unroll
      for (int r = 0; r < 2; ++r) gw[r][i] = half[r][0] | (half[r][1] << 16);
    }
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      if (r >= nr) continue;
      for (int x = (ng_all << 3) + tid; x < n; x += kThreads) {
        const uint32_t b = bits_at(srow[r], x);
        acc[r] = bf16x2_max_nan(acc[r], b | 0xFF800000u);
        if (kSums) {
          raise2(r, E::val(b));
          if (om2[r] != -INFINITY) add2(r, b);
        }
      }
      omax[r] = om2[r];
      osum[r] = oz2[r];
      const uint32_t a2 = bf16x2_max_nan(acc[r], (acc[r] >> 16) | (acc[r] << 16));
      const uint32_t mb = a2 & 0xFFFFu;  // this thread's largest value, NaN if it saw one
      if (E::is_nan(mb) || E::is_pinf(mb)) fl[r] |= kFlagBad;
      if (E::finite(mb)) {
        fl[r] |= kFlagFinite;
        mk[r] = E::key(mb);
      }
    }
  };
  if (both_rows) {
    if (fuse_z) both_rows_pass(std::true_type{});
    else both_rows_pass(std::false_type{});
  }
  for (int r = 0; !both_rows && r < nr; ++r) {
    if (kB == 16) {
      // pairs of bf16 through one NaN-propagating bf16x2 max per pair
      const int nw = n >> 1;
      const uint4 *s4 = reinterpret_cast<const uint4 *>(srow[r]);
      uint32_t acc = 0xFF80FF80u, acc2 = 0xFF80FF80u;  // (-inf, -inf); two chains
      const int ng = nw >> 2;
      int v = tid;
      for (; v + 3 * kThreads < ng; v += 4 * kThreads) {  // four 16-byte loads in flight
        const uint4 d0 = s4[v], d1 = s4[v + kThreads], d2 = s4[v + 2 * kThreads], d3 = s4[v + 3 * kThreads];
        acc = bf16x2_max_nan(acc, bf16x2_max_nan(bf16x2_max_nan(d0.x, d0.y), bf16x2_max_nan(d0.z, d0.w)));
        acc2 = bf16x2_max_nan(acc2, bf16x2_max_nan(bf16x2_max_nan(d1.x, d1.y), bf16x2_max_nan(d1.z, d1.w)));
        acc = bf16x2_max_nan(acc, bf16x2_max_nan(bf16x2_max_nan(d2.x, d2.y), bf16x2_max_nan(d2.z, d2.w)));
        acc2 = bf16x2_max_nan(acc2, bf16x2_max_nan(bf16x2_max_nan(d3.x, d3.y), bf16x2_max_nan(d3.z, d3.w)));
      }
      for (; v < ng; v += kThreads) {
        const uint4 d = s4[v];
        acc = bf16x2_max_nan(acc, bf16x2_max_nan(bf16x2_max_nan(d.x, d.y), bf16x2_max_nan(d.z, d.w)));
      }
      acc = bf16x2_max_nan(acc, acc2);
      for (int x = ((nw >> 2) << 3) + tid; x < n; x += kThreads) acc = bf16x2_max_nan(acc, bits_at(srow[r], x) | 0xFF800000u);
      acc = bf16x2_max_nan(acc, (acc >> 16) | (acc << 16));
      const uint32_t mb = acc & 0xFFFFu;  // this thread's largest value, NaN if it saw one
      if (E::is_nan(mb) || E::is_pinf(mb)) fl[r] |= kFlagBad;
      if (E::finite(mb)) {
        fl[r] |= kFlagFinite;
        mk[r] = E::key(mb);
      }
    } else {
      for_each_elem(srow[r], n, [&](uint32_t b, int) {
        if (E::is_nan(b) || E::is_pinf(b)) fl[r] |= kFlagBad;
        if (E::finite(b)) {
          fl[r] |= kFlagFinite;
          mk[r] = max(mk[r], E::key(b));  // largest finite key
        }
      });
    }
  }
  // warp maxima and flags of both rows (the two shuffle chains interleave)
  uint32_t wk[2] = {mk[0], mk[1]}, wf[2] = {fl[0], fl[1]};
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      wk[r] = max(wk[r], __shfl_xor_sync(0xFFFFFFFFu, wk[r], o));
      wf[r] |= __shfl_xor_sync(0xFFFFFFFFu, wf[r], o);
    }
  }
  uint32_t wfloor[2] = {0u, 0u};
  if (use_floor) {
    // The thread maxima are distinct elements of disjoint subsets: if f is the
    // j-th largest of a warp's 32, that warp holds j elements >= f, so the
    // smallest f over the kWarps warps (j = ceil(k / kWarps)) has at least k
    // elements at or above it and cannot exceed the k-th largest key of the
    // chunk, nor therefore of the row.  The j-th largest is searched as the
    // j-th smallest distance below the warp's maximum, clamped to 255: a
    // clamped result lies more than kNearBins below the CTA's maximum, under
    // the window's own lower edge, so it never narrows the window.
    const int need = (topk + kWarps - 1) / kWarps;
    uint32_t near_key[2], f[2] = {0u, 0u};
#pragma unroll
    for (int r = 0; r < 2; ++r) near_key[r] = 255u - min(wk[r] - mk[r], 255u);  // larger = nearer the maximum
#pragma unroll
    for (int bit = 7; bit >= 0; --bit) {
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const uint32_t t = f[r] | (1u << bit);
        if (__popc(__ballot_sync(0xFFFFFFFFu, near_key[r] >= t)) >= need) f[r] = t;
      }
    }
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const uint32_t dist = 255u - f[r];
      wfloor[r] = wk[r] > dist ? wk[r] - dist : 0u;
    }
  }
  if ((tid & 31) == 0) {
    for (int r = 0; r < nr; ++r) {
      atomicMax(&lp.maxkey[r], wk[r]);
      atomicOr(&lp.flags[r], wf[r]);
      if (use_floor) atomicMin(&lp.floor[r], wfloor[r]);
    }
  }
  __syncthreads();

  // local pass B.  bf16 top-k/top-p rows: count the keys within the window
  // below this CTA's largest key (a bin is one bf16 value, so its mass is its
  // count times one weight, formed after the reduction); top-p without top-k
  // also sums every kept weight.  Dense rows: the local normaliser.  fp32
  // top-k/top-p rows are left to the multi-pass path.
  if (kB == 16 && near) {
    unsigned long long tt[2] = {0ull, 0ull};
    // each row's window: at most kNearBins - 1 keys below the CTA's largest,
    // and not below the threshold's floor; at or below key(-inf): every
    // finite key
    uint32_t lk16s[2] = {0u, 0u}, los[2] = {0u, 0u};
    for (int r = 0; r < nr; ++r) {
      if (!(lp.flags[r] & kFlagFinite)) continue;  // empty or no finite value: contributes nothing
      const uint32_t lk16 = key16_of<TIn>(lp.maxkey[r]);
      uint32_t lo = lk16 >= static_cast<uint32_t>(kNearBins - 1) ? lk16 - (kNearBins - 1) : 0u;
      if (use_floor) lo = max(lo, lp.floor[r]);
      if (tid == 0) lp.nbins[r] = min(static_cast<uint32_t>(kNearBins), lk16 - lo + 1u);
      lk16s[r] = lk16;
      los[r] = lo;
    }
    auto lo_pair = [&](int r) {
      const uint32_t lob = los[r] > 0x007Fu ? bf16_bits_of_key(los[r]) : 0xFF80u;
      return lob | (lob << 16);
    };
    // 8-bit candidate mask of one 16-byte group: bit t is the low half of
    // word t, bit 4 + t its high half
    auto group_mask = [](const uint4 &dv, uint32_t lo2) {
      uint32_t g = (bf16x2_ge_mask(dv.x, lo2) & 0x00010001u) | ((bf16x2_ge_mask(dv.y, lo2) & 0x00010001u) << 1) |
                   ((bf16x2_ge_mask(dv.z, lo2) & 0x00010001u) << 2) |
                   ((bf16x2_ge_mask(dv.w, lo2) & 0x00010001u) << 3);
      return (g | (g >> 12)) & 0xFFu;
    };
    if (reg_groups) {
      // groups whose largest value reaches the window, two per compare; only
      // those are read again.  Each trip a lane reloads its next candidate
      // group of both rows (the two loads in flight together), and the warp
      // walks the set bits of their candidate masks in step (one candidate
      // per lane per trip)
      uint32_t cg[2] = {0u, 0u}, lo2s[2];
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        lo2s[r] = lo_pair(r);
        if (r < nr && (lp.flags[r] & kFlagFinite)) {
#pragma unroll
          for (int i = 0; i < kGroupWords; ++i) {
            const uint32_t m = bf16x2_ge_mask(gw[r][i], lo2s[r]);
            cg[r] |= ((m & 1u) | ((m >> 15) & 2u)) << (2 * i);
          }
        }
      }
      while (__any_sync(0xFFFFFFFFu, (cg[0] | cg[1]) != 0u)) {
        uint4 dv[2] = {make_uint4(0u, 0u, 0u, 0u), make_uint4(0u, 0u, 0u, 0u)};
        uint32_t em[2] = {0u, 0u};
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          if (cg[r] != 0u) {
            const int pos = __ffs(cg[r]) - 1;
            cg[r] &= cg[r] - 1u;
            dv[r] = reinterpret_cast<const uint4 *>(srow[r])[tid + pos * kThreads];
            em[r] = 0x100u;  // loaded: the mask follows once both loads are issued
          }
        }
#pragma unroll
        for (int r = 0; r < 2; ++r)
          if (em[r]) em[r] = group_mask(dv[r], lo2s[r]);
        // the candidates come out of the groups already in registers
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          uint32_t *cnt = lp.cnt[r];
          while (__any_sync(0xFFFFFFFFu, em[r] != 0u)) {
            if (em[r] != 0u) {
              const int pos = __ffs(em[r]) - 1;
              em[r] &= em[r] - 1u;
              const uint32_t wv = (pos & 2) ? ((pos & 1) ? dv[r].w : dv[r].z) : ((pos & 1) ? dv[r].y : dv[r].x);
              const uint32_t b = (pos & 4) ? (wv >> 16) : (wv & 0xFFFFu);
              const uint32_t d = lk16s[r] - E::key(b);
              if (E::finite(b) && d < static_cast<uint32_t>(kNearBins)) atomicAdd(&cnt[d], 1u);
            }
          }
        }
      }
    }
    for (int r = 0; r < nr; ++r) {
      if (!(lp.flags[r] & kFlagFinite)) continue;  // empty or no finite value: contributes nothing
      const uint32_t lk16 = lk16s[r], lo = los[r], lo2 = lo_pair(r);
      uint32_t *cnt = lp.cnt[r];
      const TIn *row = srow[r];
      const int nw = n >> 1;
      const int ng = nw >> 2;  // 16-byte groups
      // Otherwise every group is tested, kWalkGroups per lane at once.
      if (!reg_groups)
        walk_groups(row, ng, [&](const uint4 &dv) { return group_mask(dv, lo2); }, [&](uint32_t b) {
          const uint32_t d = lk16 - E::key(b);
          if (E::finite(b) && d < static_cast<uint32_t>(kNearBins)) atomicAdd(&cnt[d], 1u);
        });
      for (int x = ((nw >> 2) << 3) + tid; x < n; x += kThreads) {
        const uint32_t b = bits_at(srow[r], x);
        const uint32_t d = lk16 - E::key(b);
        if (E::finite(b) && E::key(b) >= lo && d < static_cast<uint32_t>(kNearBins)) atomicAdd(&cnt[d], 1u);
      }
      if (use_p && !use_k && fuse_z) {  // top-p alone: the max pass summed the whole row already
        const float lv = E::val_of_key(lp.maxkey[r]);
        tt[r] = omax[r] != -INFINITY
                    ? to_fixed(__fmul_rn(osum[r], exp2f(__fmul_rn(__fsub_rn(omax[r], lv), c2))))
                    : 0ull;
      } else if (use_p && !use_k) {  // top-p alone: the whole row is kept before the cut
        // a compensated fp32 sum per thread, converted once to fixed point
        const float lv = E::val_of_key(lp.maxkey[r]);
        float sum = 0.0f, comp = 0.0f;
        for_each_elem(srow[r], n, [&](uint32_t b, int) {
          if (!E::finite(b)) return;
          const float y = exp2f(__fmul_rn(__fsub_rn(E::val(b), lv), c2)) - comp;  // Kahan
          const float t = sum + y;
          comp = (t - sum) - y;
          sum = t;
        });
        tt[r] = to_fixed(sum);
      }
    }
    if (use_p && !use_k) block_sum_tot(sm, lp, tt, nr);
  } else if (!near) {
    float zt[2] = {0.0f, 0.0f};
    for (int r = 0; r < nr; ++r) {
      if (!(lp.flags[r] & kFlagFinite)) continue;
      const float lv = E::val_of_key(lp.maxkey[r]);
      if (fuse_z) {  // the max pass summed already: rescale onto the CTA's maximum
        zt[r] = omax[r] != -INFINITY ? __fmul_rn(osum[r], exp2f(__fmul_rn(__fsub_rn(omax[r], lv), c2))) : 0.0f;
        continue;
      }
      float sum = 0.0f, comp = 0.0f;
      for_each_elem(srow[r], n, [&](uint32_t b, int) {
        if (!E::finite(b)) return;  // -inf adds nothing (NaN/+inf already flagged)
        const float y = exp2f(__fmul_rn(__fsub_rn(E::val(b), lv), c2)) - comp;  // Kahan
        const float t = sum + y;
        comp = (t - sum) - y;
        sum = t;
      });
      zt[r] = sum;
    }
    block_sum_z(sm, lp, zt, nr);
  }

  // The one cluster reduction.  Every CTA stores its header and window bins
  // into its slot of every peer's inbox, then one cluster barrier makes them
  // visible; the sums below read local shared memory only.
  __syncthreads();
  Inbox *const ibx = inbox + par * static_cast<int>(ncta);
  {
    // header, then only the words of bins that can be non-zero (eight per word)
    const int w0 = (kB == 16 && near) ? static_cast<int>((lp.nbins[0] + 7u) / 8u) : 0;
    const int w1 = (kB == 16 && near) ? static_cast<int>((lp.nbins[1] + 7u) / 8u) : 0;
    const int nwords = 3 + w0 + w1;
    for (int t = tid; t < nwords * static_cast<int>(ncta); t += kThreads) {
      const int c = t / nwords, k = t % nwords;
      const int wd = k < 3 + w0 ? k : k - w0 + kNearBins / 8;  // row 1's words start at 3 + kNearBins / 8
      uint4 v;
      if (wd == 0) {
        v = make_uint4(lp.maxkey[0], lp.maxkey[1], lp.flags[0] | (lp.nbins[0] << kBinsShift),
                       lp.flags[1] | (lp.nbins[1] << kBinsShift));
      } else if (wd == 1) {
        v = make_uint4(__float_as_uint(lp.z[0]), __float_as_uint(lp.z[1]), 0u, 0u);
      } else if (wd == 2) {
        v = make_uint4(static_cast<uint32_t>(lp.tot[0]), static_cast<uint32_t>(lp.tot[0] >> 32),
                       static_cast<uint32_t>(lp.tot[1]), static_cast<uint32_t>(lp.tot[1] >> 32));
      } else {  // eight 16-bit bins per word
        const int r = (wd - 3) / (kNearBins / 8), d0 = ((wd - 3) % (kNearBins / 8)) * 8;
        uint32_t h[4] = {0u, 0u, 0u, 0u};
        if (r < nr) {
#pragma unroll
          for (int k = 0; k < 4; ++k) h[k] = lp.cnt[r][d0 + 2 * k] | (lp.cnt[r][d0 + 2 * k + 1] << 16);
        }
        v = make_uint4(h[0], h[1], h[2], h[3]);
      }
      st_dsmem_v4(map_to_rank(smem_addr(reinterpret_cast<uint4 *>(&ibx[rank]) + wd), static_cast<uint32_t>(c)), v);
    }
  }
  cluster_sync();
  ++step;
  NearSum &ns = sm.near;
  if (tid < nr * kNearBins) {  // one thread per (row, bin) of the window
    const int r = tid / kNearBins, d = tid % kNearBins;
    uint32_t gk = 0, fl = 0;
    for (int c = 0; c < static_cast<int>(ncta); ++c) {
      const uint32_t pf = ibx[c].flags[r];
      fl |= pf & ((1u << kBinsShift) - 1u);
      if (pf & kFlagFinite) gk = max(gk, ibx[c].maxkey[r]);
    }
    const uint32_t g16 = key16_of<TIn>(gk);
    if (d == 0) {
      ns.gmax[r] = gk;
      ns.flags[r] = fl;
    }
    if (kB == 16 && near) {
      // peers' bins shifted onto the global maximum, summed as integers; the
      // bin's mass is its count times the weight of its one bf16 value
      uint32_t cs = 0;
      if (fl & kFlagFinite) {
        for (int c = 0; c < static_cast<int>(ncta); ++c) {
          const uint32_t pf = ibx[c].flags[r];
          if (!(pf & kFlagFinite)) continue;
          const int dl = d - static_cast<int>(g16 - key16_of<TIn>(ibx[c].maxkey[r]));
          if (dl >= 0 && dl < static_cast<int>(pf >> kBinsShift)) cs += ibx[c].cnt[r][dl];  // (others not sent)
        }
      }
      ns.cnt[r][d] = cs;
      ns.mass[r][d] = cs ? cs * to_fixed(exp2f(__fmul_rn(__fsub_rn(E::val_of_key(g16 - static_cast<uint32_t>(d)),
                                                                      E::val_of_key(gk)), c2)))
                         : 0ull;
    }
    if (d == 0) {  // rescale the peers' sums onto the global maximum, in rank order
      float z = 0.0f;
      unsigned long long tot = 0;
      if ((fl & kFlagFinite) && (!near || (use_p && !use_k))) {
        const float gv = E::val_of_key(gk);
        for (int c = 0; c < static_cast<int>(ncta); ++c) {
          if (!(ibx[c].flags[r] & kFlagFinite)) continue;
          const float scale = exp2f(__fmul_rn(__fsub_rn(E::val_of_key(ibx[c].maxkey[r]), gv), c2));
          if (!near) z += ibx[c].z[r] * scale;
          else if (ibx[c].tot[r]) tot += __float2ull_rn(__ull2float_rn(ibx[c].tot[r]) * scale);
        }
      }
      ns.z[r] = z;
      ns.tot[r] = tot;
    }
  }
  __syncthreads();

  for (int r = 0; r < nr; ++r) {
    const uint32_t f = ns.flags[r];
    if (f & kFlagTimeout) {
      *req_bits |= SV_DATA_COPY_TIMEOUT;
      return false;
    }
    if ((f & kFlagBad) || !(f & kFlagFinite)) {
      *req_bits |= SV_DATA_BAD_VALUES;
      return false;
    }
    st[r].vmax = E::val_of_key(ns.gmax[r]);
    st[r].c2 = c2;
    st[r].cut = 0u;
    st[r].zp = ns.z[r];
  }
  if (!near) return true;

  // resolve the threshold, the cut and the normaliser from the near bins
  const int warp = tid >> 5;
  if (warp < nr) {
    const int r = warp;
    NearChoice ch;
    const bool ok = near_select(ns.cnt[r], ns.mass[r], use_k ? topk : 0, use_p, topp, ns.tot[r], &ch);
    if ((tid & 31) == 0) {
      sm.sel.ok[r] = ok && (kB == 16);  // fp32 keys need the low 16 bits refined: multi-pass path
      sm.sel.prefix[r] = key16_of<TIn>(ns.gmax[r]) - static_cast<uint32_t>(ok ? ch.last : 0);
      ns.z[r] = static_cast<float>(static_cast<double>(ok ? ch.kept : 0ull) * (1.0 / static_cast<double>(kMassScale)));
    }
  }
  __syncthreads();
  bool all_ok = true;
  for (int r = 0; r < nr; ++r) all_ok &= sm.sel.ok[r] != 0;
  if (all_ok) {
    for (int r = 0; r < nr; ++r) {
      st[r].cut = sm.sel.prefix[r];
      st[r].zp = ns.z[r];
    }
    return true;
  }
  // bf16 rows whose top-k threshold or top-p cut lies below the first window:
  // count the next windows of kNearBins keys, anchored on the global maximum
  // (the first window's bins are complete when it fails: with top-p alone no
  // floor applies, and a top-k threshold below the window puts every CTA's
  // floor below it too), one reduction per window
  if (kB == 16 && window_rounds<TIn>(sm, inbox, srow, nr, n, c2, use_k ? topk : 0, use_p, topp, st, step, ncta,
                                     rank))
    return true;
  uint32_t maxk16[2] = {0u, 0u};
  for (int r = 0; r < nr; ++r) maxk16[r] = key16_of<TIn>(ns.gmax[r]);
  __syncthreads();
  return stats_slow<TIn>(sm, srow, nr, n, c2, topk, topp, maxk16, st, step, ncta);
}

// Probability of one logit under a row's statistics (0 outside the kept set).
template <typename TIn>
__device__ __forceinline__ float prob_of(uint32_t b, const RowStats &st) {
  using E = Elem<TIn>;
  if (E::key(b) < st.cut) return 0.0f;
  const float e = exp2f(__fmul_rn(__fsub_rn(E::val(b), st.vmax), st.c2));
  return __fdiv_rn(e, st.zp);
}

// ---------------------------------------------------------------------------
// logits processors ("Speculative Decoding: propose, verify, accept", section
// 06: the same banned tokens and repetition penalty on p and q at a position,
// listed after temperature, top-k and top-p; "vLLM source walk-through (10)",
// section "Rejection sampling: the two branches of RejectionSampler", step 2:
// the sampling constraints first, then the logits processors).  The kept set
// is placed on the raw rows by the ordinary statistics; the processors then
// change only the marked entries it contains: a banned one drops out, a
// penalised one takes the weight of l / theta (l > 0) or l * theta (fp32,
// rounded to the row's type; Keskar et al., CTRL, 2019).  Each CTA marks its
// chunk in two bitmaps (banned, penalised); the rows themselves are never
// rewritten.  A greedy row (temperature 0) draws nothing, so no sampling
// constraint applies to it: its argmax is taken over the processed row.
// ---------------------------------------------------------------------------
struct Procs {
  const uint32_t *pen;  // penalised keys of this CTA's chunk, one bit each
  const uint32_t *ban;  // banned keys (a banned key is never penalised)
  float theta;
};

// 0: unmarked, 1: banned, 2: penalised (chunk-relative index xl)
__device__ __forceinline__ uint32_t mark_at(const Procs &pr, int xl) {
  const int w = xl >> 5, b = xl & 31;
  if ((pr.ban[w] >> b) & 1u) return 1u;
  return (pr.pen[w] >> b) & 1u ? 2u : 0u;
}
// Bit t set if entry xl + t is marked, for kPer entries from xl (a multiple of kPer).
template <int kPer>
__device__ __forceinline__ uint32_t group_marks(const Procs &pr, int xl) {
  const int w = xl >> 5;
  return ((pr.pen[w] | pr.ban[w]) >> (xl & 31)) & ((1u << kPer) - 1u);
}

// The value an entry takes under the processors, as bits of the row's type.
template <typename TIn>
__device__ __forceinline__ uint32_t processed_bits(uint32_t b, uint32_t mark, float theta) {
  if (mark == 1u) return sizeof(TIn) == 2 ? 0xFF80u : 0xFF800000u;  // -inf
  if (mark != 2u) return b;
  const float v = Elem<TIn>::val(b);
  const float f = v > 0.0f ? __fdiv_rn(v, theta) : __fmul_rn(v, theta);
  if constexpr (sizeof(TIn) == 2) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(f));
  } else {
    return __float_as_uint(f);
  }
}

// Weight of value bits pb relative to the row's reference maximum (0 for -inf).
template <typename TIn>
__device__ __forceinline__ float kept_weight(uint32_t pb, const RowStats &st) {
  return exp2f(__fmul_rn(__fsub_rn(Elem<TIn>::val(pb), st.vmax), st.c2));
}

// Probability of raw logit bits b with marks `mark` (prob_of when unmarked).
template <typename TIn>
__device__ __forceinline__ float prob_of_m(uint32_t b, uint32_t mark, const RowStats &st, float theta) {
  if (Elem<TIn>::key(b) < st.cut) return 0.0f;  // kept sets are placed on the raw logits
  return __fdiv_rn(kept_weight<TIn>(processed_bits<TIn>(b, mark, theta), st), st.zp);
}

// ---------------------------------------------------------------------------
// race over the row chunks (in shared memory or read in place)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void consider_drawn_l(float w, uint32_t word, int x, float &bk, int &bx) {
  const float U = e_word_to_open_uniform(word);
  const float om = 1.0f - U;
  if (__fmaf_rn(bk, om, -w) > 0.0f) return;  // w / (1-U) < bk and E >= 1-U: cannot win
  const float E = -logf(U);
  const float key = __fdiv_rn(w, E);
  if (key > bk) {
    bk = key;
    bx = x;
  }
}

// Race candidates of one quad (4 consecutive entries starting at a multiple of
// 4): E from the test-mode row or from one Philox call.
template <bool kTest>
__device__ __forceinline__ void race_quad_l(const float w[4], int xg, const float *Erow, const RngKey &rk,
                                            uint32_t rs, float &bk, int &bx, uint32_t &flags) {
  if (!(w[0] > 0.0f || w[1] > 0.0f || w[2] > 0.0f || w[3] > 0.0f)) return;
  if (kTest) {
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      if (!(w[t] > 0.0f)) continue;
      const float E = Erow[xg + t];
      if (!(E > 0.0f)) {
        flags |= SV_DATA_BAD_EXPONENTIAL;
        continue;
      }
      const float key = __fdiv_rn(w[t], E);
      if (key > bk) {
        bk = key;
        bx = xg + t;
      }
    }
  } else {
    const uint4 wd = draw_e_words(rk, rs, static_cast<uint32_t>(xg) >> 2);
    if (w[0] > 0.0f) consider_drawn_l(w[0], wd.x, xg + 0, bk, bx);
    if (w[1] > 0.0f) consider_drawn_l(w[1], wd.y, xg + 1, bk, bx);
    if (w[2] > 0.0f) consider_drawn_l(w[2], wd.z, xg + 2, bk, bx);
    if (w[3] > 0.0f) consider_drawn_l(w[3], wd.w, xg + 3, bk, bx);
  }
}

// A race weight: the probability with the normaliser applied as a product
// with its reciprocal (within an ulp of the quotient prob_of gives; race keys
// that close are inside the tolerance band anyway), which spares a division
// per entry of a dense row.
template <typename TIn>
__device__ __forceinline__ float weight_of(uint32_t b, const RowStats &st, float rz) {
  using E = Elem<TIn>;
  if (E::key(b) < st.cut) return 0.0f;
  return __fmul_rn(exp2f(__fmul_rn(__fsub_rn(E::val(b), st.vmax), st.c2)), rz);
}

template <typename TIn, bool kResidual>
__device__ __forceinline__ float race_w(uint32_t bp, uint32_t bq, const RowStats &ps, const RowStats &qs, float rp,
                                        float rq) {
  const float p = weight_of<TIn>(bp, ps, rp);
  if (kResidual) {
    const float d = __fsub_rn(p, weight_of<TIn>(bq, qs, rq));
    return d > 0.0f ? d : 0.0f;
  }
  return p > 0.0f ? p : 0.0f;
}

// race_w for an entry with processor marks: the kept tests on the raw logits,
// the weights from the processed ones.
template <typename TIn, bool kResidual>
__device__ __forceinline__ float race_w_m(uint32_t bp, uint32_t bq, uint32_t mark, const RowStats &ps,
                                          const RowStats &qs, float rp, float rq, float theta) {
  using E = Elem<TIn>;
  const float p =
      E::key(bp) < ps.cut ? 0.0f : __fmul_rn(kept_weight<TIn>(processed_bits<TIn>(bp, mark, theta), ps), rp);
  if (kResidual) {
    const float q =
        E::key(bq) < qs.cut ? 0.0f : __fmul_rn(kept_weight<TIn>(processed_bits<TIn>(bq, mark, theta), qs), rq);
    const float d = __fsub_rn(p, q);
    return d > 0.0f ? d : 0.0f;
  }
  return p > 0.0f ? p : 0.0f;
}

// The race over this CTA's row chunks.  Each thread takes 16-byte groups in
// increasing order (then the tail quads), so its strict '>' keeps its lowest
// index on ties.  kProc: marked entries take their processed weights.
template <typename TIn, bool kTest, bool kResidual, bool kProc = false>
__device__ __forceinline__ void race_chunks(const TIn *sp, const TIn *sq, const RowStats &ps, const RowStats &qs,
                                          int x0, int n, const float *Erow, const RngKey &rk, uint32_t rs, float &bk,
                                          int &bx, uint32_t &flags, const Procs &pr = Procs{nullptr, nullptr, 1.0f}) {
  constexpr int kPer = 16 / sizeof(TIn);  // 8 bf16 or 4 fp32 = 2 or 1 quads
  const int nv = n / kPer;
  const uint4 *p4 = reinterpret_cast<const uint4 *>(sp);
  const uint4 *q4 = reinterpret_cast<const uint4 *>(kResidual ? sq : sp);
  // bf16 rows with a cut: pairs of keys are tested against the cuts first, so
  // entries outside both kept sets cost two SIMD compares per pair
  const uint32_t cpb = bf16_bits_of_key(ps.cut), cqb = bf16_bits_of_key(qs.cut);
  const uint32_t cp2 = cpb | (cpb << 16), cq2 = cqb | (cqb << 16);
  const bool packed_test = sizeof(TIn) == 2 && (ps.cut > 0x007Fu) && (!kResidual || qs.cut > 0x007Fu);
  const float rp = __frcp_rn(ps.zp), rq = __frcp_rn(qs.zp);
  for (int v = threadIdx.x; v < nv; v += kThreads) {
    const uint4 dp = p4[v];
    const uint4 dq = kResidual ? q4[v] : dp;
    const uint32_t wp[4] = {dp.x, dp.y, dp.z, dp.w}, wq[4] = {dq.x, dq.y, dq.z, dq.w};
    if (packed_test) {
      uint32_t any = 0u;
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        any |= bf16x2_ge_mask(wp[t], cp2);
        if (kResidual) any |= bf16x2_ge_mask(wq[t], cq2);
      }
      if (any == 0u) continue;  // no kept entry in these 8: every weight is 0
    }
    float w[kPer];
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      if (sizeof(TIn) == 2) {
        w[2 * t] = race_w<TIn, kResidual>(wp[t] & 0xFFFFu, wq[t] & 0xFFFFu, ps, qs, rp, rq);
        w[2 * t + 1] = race_w<TIn, kResidual>(wp[t] >> 16, wq[t] >> 16, ps, qs, rp, rq);
      } else {
        w[t] = race_w<TIn, kResidual>(wp[t], wq[t], ps, qs, rp, rq);
      }
    }
    if (kProc) {  // marked entries of the group: processed weights
      uint32_t mk = group_marks<kPer>(pr, v * kPer);
      while (mk) {
        const int t = __ffs(mk) - 1;
        mk &= mk - 1u;
        const int wi = sizeof(TIn) == 2 ? t >> 1 : t, sh = sizeof(TIn) == 2 ? 16 * (t & 1) : 0;
        const uint32_t msk = sizeof(TIn) == 2 ? 0xFFFFu : 0xFFFFFFFFu;
        w[t] = race_w_m<TIn, kResidual>((wp[wi] >> sh) & msk, (wq[wi] >> sh) & msk, mark_at(pr, v * kPer + t), ps,
                                        qs, rp, rq, pr.theta);
      }
    }
#pragma unroll
    for (int qd = 0; qd < kPer / 4; ++qd)
      race_quad_l<kTest>(&w[4 * qd], x0 + v * kPer + 4 * qd, Erow, rk, rs, bk, bx, flags);
  }
  for (int q = nv * (kPer / 4) + threadIdx.x; 4 * q < n; q += kThreads) {
    float w[4];
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const int x = 4 * q + t;
      if (x >= n) {
        w[t] = 0.0f;
      } else if (kProc) {
        w[t] = race_w_m<TIn, kResidual>(bits_at(sp, x), kResidual ? bits_at(sq, x) : 0u, mark_at(pr, x), ps, qs, rp,
                                        rq, pr.theta);
      } else {
        w[t] = race_w<TIn, kResidual>(bits_at(sp, x), kResidual ? bits_at(sq, x) : 0u, ps, qs, rp, rq);
      }
    }
    race_quad_l<kTest>(w, x0 + 4 * q, Erow, rk, rs, bk, bx, flags);
  }
}

// Load this CTA's chunk of nr rows into shared memory.  Aligned rows arrive
// through one bulk copy per row (TMA, completing on the CTA's mbarrier), with
// plain loads only for a last partial 16-byte group; other rows use plain
// loads.  With kRes false (aligned rows only) nothing is copied: the rows are
// read where they lie, and their chunks are only prefetched into L2 here.
// Returns kFlagTimeout if the copy did not complete within `first_limit`
// polls; the copies in flight then get one more wait of the ordinary limit
// (a test sets first_limit to 0 to take this path while every copy lands).
template <typename TIn, bool kVec, bool kRes = true>
__device__ uint32_t load_rows(LogitsSmem &sm, const TIn *const grow[2], TIn *const srow[2], int nr, int n,
                              uint32_t &phase, uint32_t first_limit) {
  const int tid = threadIdx.x;
  if (kVec && !kRes) {  // both chunks are read in place: warm L2 with them
    if (tid == 0) {
      const uint32_t body = (static_cast<uint32_t>(n) * sizeof(TIn)) & ~15u;
      if (body)
        for (int r = 0; r < nr; ++r) prefetch_l2(grow[r], body);
    }
    return 0u;
  }
  const int nc = kRes ? nr : 1;  // rows copied into shared memory
  fence_proxy_async_smem();  // earlier reads of the rows before the async overwrite
  __syncthreads();
  uint32_t flags = 0;
  if (kVec) {
    const uint32_t body = (static_cast<uint32_t>(n) * sizeof(TIn)) & ~15u;
    if (tid == 0) {
      if (!kRes && nr == 2 && body) prefetch_l2(grow[1], body);
      mbar_arrive_expect_tx(&sm.bar, body * static_cast<uint32_t>(nc));
      if (body)
        for (int r = 0; r < nc; ++r) bulk_g2s(srow[r], grow[r], body, &sm.bar);
    }
    const int nb = static_cast<int>(body / sizeof(TIn));
    for (int r = 0; r < nc; ++r)
      for (int x = nb + tid; x < n; x += kThreads) srow[r][x] = grow[r][x];
    __syncthreads();
    if (!mbar_wait_bounded(&sm.bar, phase, first_limit)) {
      flags = kFlagTimeout;
      mbar_wait_bounded(&sm.bar, phase, kCopyWaitPolls);  // give the copies in flight one more bound
    }
    phase ^= 1u;
  } else {
    for (int r = 0; r < nc; ++r)
      for (int x = tid; x < n; x += kThreads) srow[r][x] = grow[r][x];
    __syncthreads();
  }
  return flags;
}

// ---------------------------------------------------------------------------
// the processors' correction of a position's statistics
// ---------------------------------------------------------------------------
// One cluster exchange of a 16-byte word per CTA: threads 0 .. ncta-1 store
// `v` into this CTA's slot of every peer's inbox (the slots of the parity of
// `step`), one cluster barrier, then sm.xw[c] holds CTA c's word in every CTA.
__device__ __forceinline__ void cluster_exchange(LogitsSmem &sm, Inbox *inbox, const uint4 &v, int &step,
                                                 uint32_t ncta, uint32_t rank) {
  Inbox *const ibx = inbox + (step & 1) * static_cast<int>(ncta);
  if (threadIdx.x < ncta) st_dsmem_v4(map_to_rank(smem_addr(&ibx[rank]), threadIdx.x), v);
  cluster_sync();
  ++step;
  if (threadIdx.x < ncta) sm.xw[threadIdx.x] = *reinterpret_cast<const uint4 *>(&ibx[threadIdx.x]);
  __syncthreads();
}

// Fixed-tree block sums of two floats into sm.pz (valid after the barrier).
__device__ __forceinline__ void block_sum_pz(LogitsSmem &sm, const float v[2]) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int r = 0; r < 2; ++r) {
    float x = v[r];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xFFFFFFFFu, x, o);
    if (lane == 0) sm.wz[r][warp] = x;
  }
  __syncthreads();
  if (threadIdx.x < 2) {
    float x = 0.0f;
    for (int w = 0; w < kWarps; ++w) x += sm.wz[threadIdx.x][w];
    sm.pz[threadIdx.x] = x;
  }
  __syncthreads();
}

// Exact statistics of rows whose corrected normaliser cancelled (below half
// of the raw one) or overflowed: the reference maximum becomes the largest
// processed value among the kept, unbanned entries, and the normaliser is
// summed afresh against it.  Two cluster exchanges; every CTA takes this path
// alike (the condition is computed from cluster-wide totals).  Returns false
// if a row keeps no unbanned entry (no distribution is left).
template <typename TIn>
__device__ bool proc_rescue(LogitsSmem &sm, Inbox *inbox, TIn *const rows[2], int nr, int n, const Procs &pr,
                            RowStats st[2], const bool need[2], int &step, uint32_t ncta, uint32_t rank) {
  using E = Elem<TIn>;
  const int tid = threadIdx.x;
  if (tid < 2) sm.xmax[tid] = 0u;
  __syncthreads();
  auto visit = [&](int r, auto f) {  // f(processed bits) over the kept, unbanned entries of row r
    for_each_elem(rows[r], n, [&](uint32_t b, int x) {
      if (E::key(b) < st[r].cut) return;
      const uint32_t m = mark_at(pr, x);
      if (m == 1u) return;
      const uint32_t pb = processed_bits<TIn>(b, m, pr.theta);
      if (E::finite(pb)) f(pb);  // (-inf adds nothing; NaN and +inf were rejected before)
    });
  };
  for (int r = 0; r < nr; ++r) {
    if (!need[r]) continue;
    uint32_t mx = 0u;
    visit(r, [&](uint32_t pb) { mx = max(mx, ordered_bits(E::val(pb))); });
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
    if ((tid & 31) == 0 && mx) atomicMax(&sm.xmax[r], mx);
  }
  __syncthreads();
  cluster_exchange(sm, inbox, make_uint4(sm.xmax[0], sm.xmax[1], 0u, 0u), step, ncta, rank);
  float ref[2] = {0.0f, 0.0f};
  for (int r = 0; r < nr; ++r) {
    if (!need[r]) continue;
    uint32_t mx = 0u;
    for (int c = 0; c < static_cast<int>(ncta); ++c) mx = max(mx, r ? sm.xw[c].y : sm.xw[c].x);
    if (mx == 0u) return false;
    const uint32_t b = (mx & 0x80000000u) ? (mx & 0x7FFFFFFFu) : ~mx;  // inverse of ordered_bits
    ref[r] = __uint_as_float(b);
  }
  float z[2] = {0.0f, 0.0f};
  for (int r = 0; r < nr; ++r) {
    if (!need[r]) continue;
    float comp = 0.0f;
    visit(r, [&](uint32_t pb) {  // compensated sum against the new reference
      const float y = exp2f(__fmul_rn(__fsub_rn(E::val(pb), ref[r]), st[r].c2)) - comp;
      const float t = z[r] + y;
      comp = (t - z[r]) - y;
      z[r] = t;
    });
  }
  block_sum_pz(sm, z);
  cluster_exchange(sm, inbox, make_uint4(__float_as_uint(sm.pz[0]), __float_as_uint(sm.pz[1]), 0u, 0u), step, ncta,
                   rank);
  for (int r = 0; r < nr; ++r) {
    if (!need[r]) continue;
    float t = 0.0f;
    for (int c = 0; c < static_cast<int>(ncta); ++c) t += __uint_as_float(r ? sm.xw[c].y : sm.xw[c].x);
    st[r].vmax = ref[r];
    st[r].zp = t;
  }
  return true;
}

// After the raw statistics of a position: every marked entry of this CTA's
// chunk that the kept set holds trades its raw weight for its processed one
// (0 when banned), for the normaliser of each row.  Fixed summation order
// (bitmap words by thread, bits ascending, a fixed block tree, then ranks in
// order), so every CTA of the cluster gets the same totals.  The CTA holding
// the draft token (y_local >= 0) publishes its marks in the same exchange.
// Sets SV_DATA_BAD_VALUES and returns false if a kept processed value is NaN
// or +inf or no unbanned entry is kept.
template <typename TIn>
__device__ bool proc_correct(LogitsSmem &sm, Inbox *inbox, TIn *const rows[2], int nr, int n, int words,
                             const Procs &pr, RowStats st[2], int y_local, uint32_t &ymark, uint32_t *req_bits,
                             int &step, uint32_t ncta, uint32_t rank) {
  using E = Elem<TIn>;
  const int tid = threadIdx.x;
  float d[2] = {0.0f, 0.0f};
  uint32_t bad = 0u;
  for (int w = tid; w < words; w += kThreads) {
    uint32_t bits = pr.pen[w] | pr.ban[w];
    while (bits) {
      const int b = __ffs(bits) - 1;
      bits &= bits - 1u;
      const int xl = 32 * w + b;
      if (xl >= n) break;
      const uint32_t m = ((pr.ban[w] >> b) & 1u) ? 1u : 2u;
      for (int r = 0; r < nr; ++r) {
        const uint32_t rb = bits_at(rows[r], xl);
        if (E::key(rb) < st[r].cut) continue;  // outside the kept set: the processors cannot bring it in
        const uint32_t pb = processed_bits<TIn>(rb, m, pr.theta);
        if (E::is_nan(pb) || E::is_pinf(pb)) bad = 1u;
        d[r] += kept_weight<TIn>(pb, st[r]) - kept_weight<TIn>(rb, st[r]);
      }
    }
  }
  bad = __syncthreads_or(bad) ? 1u : 0u;
  if (tid == 0) sm.pmark = y_local >= 0 ? 0x100u | mark_at(pr, y_local) : 0u;
  block_sum_pz(sm, d);
  cluster_exchange(sm, inbox, make_uint4(__float_as_uint(sm.pz[0]), __float_as_uint(sm.pz[1]), sm.pmark, bad), step,
                   ncta, rank);
  float z[2] = {st[0].zp, st[1].zp};
  uint32_t ym = 0u, fb = 0u;
  for (int c = 0; c < static_cast<int>(ncta); ++c) {
    z[0] += __uint_as_float(sm.xw[c].x);
    z[1] += __uint_as_float(sm.xw[c].y);
    ym |= sm.xw[c].z;
    fb |= sm.xw[c].w;
  }
  ymark = ym & 3u;
  if (fb) {
    *req_bits |= SV_DATA_BAD_VALUES;
    return false;
  }
  bool need[2] = {false, false}, any = false;
  for (int r = 0; r < nr; ++r) {
    need[r] = !(z[r] >= 0.5f * st[r].zp && z[r] < INFINITY);
    if (!need[r]) st[r].zp = z[r];
    any |= need[r];
  }
  if (any && !proc_rescue<TIn>(sm, inbox, rows, nr, n, pr, st, need, step, ncta, rank)) {
    *req_bits |= SV_DATA_BAD_VALUES;
    return false;
  }
  return true;
}

// Greedy with processors: thread-local argmax of a row chunk (in shared memory
// or read in place), every marked entry taking its processed value (-inf when
// banned; a banned NaN is no longer a NaN).
template <typename TIn>
__device__ __forceinline__ void argmax_proc(const TIn *row, int x0, int n, const Procs &pr, unsigned long long &best,
                                            uint32_t &flags) {
  using E = Elem<TIn>;
  for_each_elem(row, n, [&](uint32_t b, int x) {
    const uint32_t m = mark_at(pr, x);
    if (m) b = processed_bits<TIn>(b, m, pr.theta);
    if (E::is_nan(b)) {
      flags |= SV_DATA_BAD_VALUES;
      return;
    }
    best = umax64(best, (static_cast<unsigned long long>(E::key(b)) << 32) |
                            static_cast<unsigned long long>(~static_cast<uint32_t>(x0 + x)));
  });
}

// Greedy: thread-local argmax of raw logits of a global row chunk.
template <typename TIn, bool kVec>
__device__ __forceinline__ void argmax_logits(const TIn *g, int x0, int n, unsigned long long &best, uint32_t &flags) {
  using E = Elem<TIn>;
  const int tid = threadIdx.x;
  auto take = [&](uint32_t b, int x) {
    if (E::is_nan(b)) {
      flags |= SV_DATA_BAD_VALUES;
      return;
    }
    const unsigned long long k =
        (static_cast<unsigned long long>(E::key(b)) << 32) | static_cast<unsigned long long>(~static_cast<uint32_t>(x0 + x));
    best = umax64(best, k);
  };
  int xs = 0;
  if (kVec) {
    constexpr int kPer = 16 / sizeof(TIn);
    const int nv = n / kPer;
    const uint4 *g4 = reinterpret_cast<const uint4 *>(g);
    for (int v = tid; v < nv; v += kThreads) {
      uint4 d;
      asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                   : "=r"(d.x), "=r"(d.y), "=r"(d.z), "=r"(d.w)
                   : "l"(g4 + v));
      const uint32_t w[4] = {d.x, d.y, d.z, d.w};
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        if (E::kBits == 16) {
          take(w[t] & 0xFFFFu, v * kPer + 2 * t);
          take(w[t] >> 16, v * kPer + 2 * t + 1);
        } else {
          take(w[t], v * kPer + t);
        }
      }
    }
    xs = nv * kPer;
  }
  for (int x = xs + tid; x < n; x += kThreads) take(bits_at(g, x), x);
}

// kRes: both row chunks of a position live in shared memory (two CTAs per
// SM).  Otherwise (aligned rows) both chunks are read where they lie after a
// bulk L2 prefetch: a CTA then holds only its statistics and inbox in shared
// memory, and four share an SM.  Logits processors work in either form (the
// rows are never rewritten).
template <typename TIn, bool kTest, bool kVec, bool kRes, bool kProc>
__global__ void __launch_bounds__(kThreads, kRes ? 2 : 4) logits_kernel(const VerifyParams P, int chunk) {
  pdl_enter();
  static_assert(kRes || kVec, "rows read in place must be 16-byte aligned");
  using E = Elem<TIn>;
  extern __shared__ __align__(16) unsigned char dyn_smem[];
  __shared__ LogitsSmem sm;
  TIn *const srow[2] = {reinterpret_cast<TIn *>(dyn_smem), reinterpret_cast<TIn *>(dyn_smem) + (kRes ? chunk : 0)};
  Inbox *const inbox = reinterpret_cast<Inbox *>(dyn_smem + (kRes ? 2 : 0) * static_cast<size_t>(chunk) * sizeof(TIn));

  const uint32_t ncta = cluster_nctarank(), rank = cluster_ctarank();
  const int i = static_cast<int>(blockIdx.x / ncta);
  // processor bitmaps (present only when the call has processors)
  const int words = (chunk + 31) / 32;
  uint32_t *const pen_bits = reinterpret_cast<uint32_t *>(inbox + 2 * ncta);
  uint32_t *const ban_bits = pen_bits + words;
  const int tid = threadIdx.x;
  const int G = P.G, V = P.V;
  const TIn *tgt = static_cast<const TIn *>(P.target);
  const TIn *drf = static_cast<const TIn *>(P.draft);
  const int64_t ts = P.target_stride, ds = P.draft_stride;
  const int x0 = min(V, static_cast<int>(rank) * chunk);
  const int n = min(V, x0 + chunk) - x0;

  // a0: ragged decode
  int64_t s, e;
  if (P.cu) {
    s = i ? P.cu[i - 1] : 0;
    e = P.cu[i];
  } else {
    s = static_cast<int64_t>(i) * G;
    e = s + G;
  }
  uint32_t req_bits = 0;
  bool valid = true;
  if (s < 0 || e < s || e > P.T || e - s > G) {
    req_bits |= SV_DATA_BAD_CU;
    valid = false;
  }
  const int g = valid ? static_cast<int>(e - s) : 0;
  const int64_t tb = s + i;
  const float temp = P.temperature ? P.temperature[i] : 1.0f;
  if (valid && !temperature_ok(temp)) {
    req_bits |= SV_DATA_BAD_PARAM;
    valid = false;
  }
  int64_t pen_b = 0, pen_e = 0, ban_b = 0, ban_e = 0, stop_b = 0, stop_e = 0;
  if (valid && ((P.pen_cu && !list_range(P.pen_cu, P.pen_total, i, pen_b, pen_e)) ||
                (P.ban_cu && !list_range(P.ban_cu, P.ban_total, i, ban_b, ban_e)) ||
                (P.stop_cu && !list_range(P.stop_cu, P.stop_total, i, stop_b, stop_e)))) {
    req_bits |= SV_DATA_BAD_LIST;
    valid = false;
  }
  float theta = 1.0f;
  if (valid && P.rep_penalty) {
    theta = P.rep_penalty[i];
    if (!(theta > 0.0f) || isinf(theta)) {
      req_bits |= SV_DATA_BAD_PARAM;
      valid = false;
    }
  }
  constexpr bool procs = kProc;  // the call has logits processors (P.rep_penalty or P.ban_cu)
  const Procs pr{pen_bits, ban_bits, theta};
  const bool greedy = valid && temp == 0.0f;
  int A = 0;
  int32_t last_tok = -1;
  int step = 0;
  uint32_t phase = 0;
  int added = 0;  // drafts already in the penalty bitmap
  if (tid == 0) {
    mbar_init(&sm.bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  // Peers' shared memory may be written only once every CTA of the cluster
  // runs: arrive now, wait before the first store into a peer (the first row
  // copy proceeds meanwhile).
  cluster_arrive_relaxed();
  bool joined = false;
  auto join = [&]() {
    if (!joined) cluster_wait_acquire();
    joined = true;
  };

  auto mark = [&](uint32_t *bm, int32_t x) {
    if (x >= x0 && x < x0 + n) atomicOr(&bm[(x - x0) >> 5], 1u << ((x - x0) & 31));
  };
  if (valid && procs) {  // this chunk's banned and penalised keys
    for (int w = tid; w < 2 * words; w += kThreads) pen_bits[w] = 0u;
    __syncthreads();
    if (P.ban_cu)
      for (int64_t k = ban_b + tid; k < ban_e; k += kThreads) mark(ban_bits, P.ban_ids[k]);
    if (P.rep_penalty && P.pen_cu)
      for (int64_t k = pen_b + tid; k < pen_e; k += kThreads) mark(pen_bits, P.pen_ids[k]);
    __syncthreads();
  }
  // position j penalises the drafts y_0 .. y_{j-1} too (they are committed by then)
  auto add_drafts = [&](int j) {
    if (P.rep_penalty)
      for (; added < j; ++added)
        if (tid == 0) mark(pen_bits, P.ids[s + added]);
  };

  if (greedy) {
    join();
    for (int j = 0;; ++j) {
      unsigned long long best = 0;
      uint32_t fl = 0;
      if (procs) {  // the argmax of the processed row
        add_drafts(j);
        const TIn *grow[2] = {tgt + (tb + j) * ts + x0, nullptr};
        const TIn *row = grow[0];
        if (kRes) {
          if (load_rows<TIn, kVec>(sm, grow, srow, 1, n, phase, P.first_wait) & kFlagTimeout)
            fl |= SV_DATA_COPY_TIMEOUT;
          row = srow[0];
        }
        __syncthreads();  // the drafts' marks
        argmax_proc<TIn>(row, x0, n, pr, best, fl);
      } else {
        argmax_logits<TIn, kVec>(tgt + (tb + j) * ts + x0, x0, n, best, fl);
      }
      const KeyFlags r = cluster_reduce(KeyFlags{best, fl}, sm.red, step++, ncta);
      if (r.flags & (SV_DATA_BAD_VALUES | SV_DATA_COPY_TIMEOUT)) {
        req_bits |= r.flags & (SV_DATA_BAD_VALUES | SV_DATA_COPY_TIMEOUT);
        valid = false;
        break;
      }
      const int gj = static_cast<int>(key_index(r.key));
      if (tid == 0) sm.tok[j] = gj;
      if (j == g) {
        A = g;
        break;
      }
      const int y = P.ids[s + j];
      if (y < 0 || y >= V) {
        req_bits |= SV_DATA_BAD_DRAFT_ID;
        valid = false;
        break;
      }
      if (y != gj) {
        A = j;
        break;
      }
    }
  } else if (valid) {
    int topk = P.top_k ? P.top_k[i] : 0;
    if (topk >= V) topk = 0;
    if (topk < 0) topk = 0;
    const float topp = P.top_p ? P.top_p[i] : 1.0f;
    if (!(topp > 0.0f)) {
      req_bits |= SV_DATA_BAD_PARAM;
      valid = false;
    } else {
      const float c2 = __fdiv_rn(kLog2e, temp);
      const RngKey rk{P.seed_lo, P.seed_hi, P.off_lo, P.off_hi};
      const uint32_t rs = P.req_base + static_cast<uint32_t>(i);
      const float *Erow = kTest ? P.exponentials + static_cast<int64_t>(i) * P.exp_stride : nullptr;
      RowStats st[2];
      // synthetic acceptance: the stopping position follows from u_j < rate_j
      // alone; the rows of the positions before it are never read
      int j_start = 0;
      if (P.rates) {
        bool bad_rates = false;
        for (int j = 0; j < g; ++j) {
          const float rj = P.rates[j];
          if (!(rj >= 0.0f && rj <= 1.0f) || (j > 0 && rj > P.rates[j - 1])) bad_rates = true;
        }
        if (bad_rates) {
          req_bits |= SV_DATA_BAD_PARAM;
          valid = false;
        }
        for (; valid && j_start < g; ++j_start) {
          const int y = P.ids[s + j_start];
          if (y < 0 || y >= V) {
            req_bits |= SV_DATA_BAD_DRAFT_ID;
            valid = false;
            break;
          }
          const float u = kTest ? P.uniforms[s + j_start] : draw_uniform(rk, rs, static_cast<uint32_t>(j_start));
          if (!(u < P.rates[j_start])) break;
          if (tid == 0) sm.tok[j_start] = y;
        }
      }
      for (int j = j_start; valid; ++j) {
        const int nr = (j < g) ? 2 : 1;
        if (nr == 2 && drf == nullptr) {
          req_bits |= SV_DATA_MISSING_DRAFT;
          valid = false;
          break;
        }
        // the draft id, its two logits and u are fetched now, so their latency
        // hides behind the row copy and the statistics
        int y = -1;
        uint32_t bty = 0u, bdy = 0u;
        float u = 0.0f;
        if (j < g) {
          y = P.ids[s + j];
          if (y >= 0 && y < V) {
            bty = bits_at(tgt + (tb + j) * ts, y);
            bdy = bits_at(drf + (s + j) * ds, y);
          }
          u = kTest ? P.uniforms[s + j] : draw_uniform(rk, rs, static_cast<uint32_t>(j));
        }
        const TIn *grow[2] = {tgt + (tb + j) * ts + x0, nr == 2 ? drf + (s + j) * ds + x0 : nullptr};
        if (procs) add_drafts(j);
        const uint32_t lf = load_rows<TIn, kVec, kRes>(sm, grow, srow, nr, n, phase, P.first_wait);
        // this position's rows: in shared memory, or where they lie
        TIn *const rows[2] = {kRes ? srow[0] : const_cast<TIn *>(grow[0]), kRes ? srow[1] : const_cast<TIn *>(grow[1])};
        join();
        if (!position_stats<TIn>(sm, inbox, rows, nr, n, c2, topk, topp, lf, st, &req_bits, step, ncta, rank)) {
          valid = false;
          break;
        }
        // the processors on the kept sets: corrected normalisers, the draft token's marks
        uint32_t ymark = 0u;
        if (procs) {
          const int y_local = (j < g && y >= x0 && y < x0 + n) ? y - x0 : -1;
          if (!proc_correct<TIn>(sm, inbox, rows, nr, n, words, pr, st, y_local, ymark, &req_bits, step, ncta,
                                 rank)) {
            valid = false;
            break;
          }
        }
        float bk = 0.0f;
        int bx = -1;
        uint32_t fl = 0;
        bool residual = false;
        if (j < g) {
          if (y < 0 || y >= V) {
            req_bits |= SV_DATA_BAD_DRAFT_ID;
            valid = false;
            break;
          }
          const float py = prob_of_m<TIn>(bty, ymark, st[0], theta);
          const float qy = prob_of_m<TIn>(bdy, ymark, st[1], theta);
          if (rank == 0 && tid == 0 && !P.rates) {
            if (P.dbg_py) P.dbg_py[s + j] = py;
            if (P.dbg_qy) P.dbg_qy[s + j] = qy;
          }
          if (!P.rates && __fmul_rn(u, qy) < py) {  // (synthetic mode reaches here only at its rejection)
            if (tid == 0) sm.tok[j] = y;
            continue;  // accepted: next position
          }
          residual = true;
          if (procs)
            race_chunks<TIn, kTest, true, true>(rows[0], rows[1], st[0], st[1], x0, n, Erow, rk, rs, bk, bx, fl, pr);
          else
            race_chunks<TIn, kTest, true>(rows[0], rows[1], st[0], st[1], x0, n, Erow, rk, rs, bk, bx, fl);
        } else if (procs) {
          race_chunks<TIn, kTest, false, true>(rows[0], rows[1], st[0], st[0], x0, n, Erow, rk, rs, bk, bx, fl, pr);
        } else {
          race_chunks<TIn, kTest, false>(rows[0], rows[1], st[0], st[0], x0, n, Erow, rk, rs, bk, bx, fl);
        }
        KeyFlags r = cluster_reduce(KeyFlags{bx >= 0 ? pack_key(bk, bx) : 0ull, fl}, sm.red, step++, ncta);
        if (r.key == 0ull && residual) {  // no positive residual key: race over p with the same E
          bk = 0.0f;
          bx = -1;
          fl = 0;
          if (procs)
            race_chunks<TIn, kTest, false, true>(rows[0], rows[1], st[0], st[0], x0, n, Erow, rk, rs, bk, bx, fl, pr);
          else
            race_chunks<TIn, kTest, false>(rows[0], rows[1], st[0], st[0], x0, n, Erow, rk, rs, bk, bx, fl);
          const KeyFlags r2 = cluster_reduce(KeyFlags{bx >= 0 ? pack_key(bk, bx) : 0ull, fl}, sm.red, step++, ncta);
          r.key = r2.key;
          r.flags |= r2.flags;
        }
        req_bits |= r.flags;
        if (r.key == 0ull) {
          req_bits |= SV_DATA_EMPTY_DISTRIBUTION;
          last_tok = 0;
        } else {
          last_tok = static_cast<int32_t>(key_index(r.key));
        }
        A = j;
        break;
      }
    }
  }
  join();
  __syncthreads();
  if (rank == 0) {
    const int A0 = A;
    auto tok = [&](int k) -> int32_t { return (k == A0 && !greedy) ? last_tok : sm.tok[k]; };
    if (valid && P.stop_cu) A = stop_commit(A0, tok, P.stop_ids, stop_b, stop_e, &sm.stop_first);
    emit_request(i, G, g, A, valid, tb, req_bits, tok, P.out, P.nacc, P.ncomp, P.slots, P.status);
  }
  cluster_sync();
}

// ---------------------------------------------------------------------------
// draft-side sampler: one token per logits row from the transformed row
// ("vLLM source walk-through (10)", section "propose() multi-step loop":
// each draft step samples its token from the draft distribution and keeps the
// distribution for the rejection sampler).  One cluster per row; the row is
// transformed exactly like a verifier row, the token is drawn by the same
// exponential race (argmax at temperature 0), and the fp32 probability row can
// be written out for the probability entry.
// ---------------------------------------------------------------------------
template <typename TIn, bool kTest, bool kVec, bool kRes, bool kProc>
__global__ void __launch_bounds__(kThreads, kRes ? 2 : 4) sample_kernel(const SampleParams P, int chunk) {
  pdl_enter();
  static_assert(kRes || kVec, "rows read in place must be 16-byte aligned");
  extern __shared__ __align__(16) unsigned char dyn_smem[];
  __shared__ LogitsSmem sm;
  const uint32_t ncta = cluster_nctarank(), rank = cluster_ctarank();
  const int r = static_cast<int>(blockIdx.x / ncta);
  const int tid = threadIdx.x;
  const int V = P.V;
  const TIn *row = static_cast<const TIn *>(P.logits) + static_cast<int64_t>(r) * P.row_stride;
  const int x0 = min(V, static_cast<int>(rank) * chunk);
  const int n = min(V, x0 + chunk) - x0;
  // the row chunk: in shared memory, or read where it lies
  TIn *const rc = kRes ? reinterpret_cast<TIn *>(dyn_smem) : const_cast<TIn *>(row + x0);
  TIn *const srow[2] = {rc, rc};
  Inbox *const inbox = reinterpret_cast<Inbox *>(dyn_smem + (kRes ? static_cast<size_t>(chunk) * sizeof(TIn) : 0));
  uint32_t bits = 0;
  int32_t token = -1;
  int step = 0;
  uint32_t phase = 0;
  // processor bitmaps (present only when the call has processors)
  constexpr bool procs = kProc;  // P.rep_penalty or P.ban_cu
  const int words = (chunk + 31) / 32;
  uint32_t *const pen_bits = reinterpret_cast<uint32_t *>(inbox + 2 * ncta);
  uint32_t *const ban_bits = pen_bits + words;
  if (tid == 0) {
    mbar_init(&sm.bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  cluster_sync();  // every CTA of the cluster runs before any store into a peer
  const float temp = P.temperature ? P.temperature[r] : 1.0f;
  bool ok = true;
  if (!temperature_ok(temp)) {
    bits |= SV_DATA_BAD_PARAM;
    ok = false;
  }
  int64_t pen_b = 0, pen_e = 0, ban_b = 0, ban_e = 0;
  if (ok && ((P.pen_cu && !list_range(P.pen_cu, P.pen_total, r, pen_b, pen_e)) ||
             (P.ban_cu && !list_range(P.ban_cu, P.ban_total, r, ban_b, ban_e)))) {
    bits |= SV_DATA_BAD_LIST;
    ok = false;
  }
  float theta = 1.0f;
  if (ok && P.rep_penalty) {
    theta = P.rep_penalty[r];
    if (!(theta > 0.0f) || isinf(theta)) {
      bits |= SV_DATA_BAD_PARAM;
      ok = false;
    }
  }
  if (ok && procs) {  // this chunk's banned and penalised keys
    auto mark = [&](uint32_t *bm, int32_t x) {
      if (x >= x0 && x < x0 + n) atomicOr(&bm[(x - x0) >> 5], 1u << ((x - x0) & 31));
    };
    for (int w = tid; w < 2 * words; w += kThreads) pen_bits[w] = 0u;
    __syncthreads();
    if (P.ban_cu)
      for (int64_t k = ban_b + tid; k < ban_e; k += kThreads) mark(ban_bits, P.ban_ids[k]);
    if (P.rep_penalty && P.pen_cu)
      for (int64_t k = pen_b + tid; k < pen_e; k += kThreads) mark(pen_bits, P.pen_ids[k]);
    __syncthreads();
  }
  const Procs pr{pen_bits, ban_bits, theta};
  if (!ok) {
    // nothing sampled
  } else if (temp == 0.0f) {
    unsigned long long best = 0;
    uint32_t fl = 0;
    if (procs) {  // the argmax of the processed row
      const TIn *grow[2] = {row + x0, nullptr};
      const TIn *src = grow[0];
      if (kRes) {
        if (load_rows<TIn, kVec>(sm, grow, srow, 1, n, phase, P.first_wait) & kFlagTimeout)
          fl |= SV_DATA_COPY_TIMEOUT;
        src = srow[0];
      }
      argmax_proc<TIn>(src, x0, n, pr, best, fl);
    } else {
      argmax_logits<TIn, kVec>(row + x0, x0, n, best, fl);
    }
    const KeyFlags kr = cluster_reduce(KeyFlags{best, fl}, sm.red, step++, ncta);
    if (kr.flags & (SV_DATA_BAD_VALUES | SV_DATA_COPY_TIMEOUT)) bits |= kr.flags & (SV_DATA_BAD_VALUES | SV_DATA_COPY_TIMEOUT);
    else token = static_cast<int32_t>(key_index(kr.key));
  } else {
    int topk = P.top_k ? P.top_k[r] : 0;
    if (topk >= V || topk < 0) topk = 0;
    const float topp = P.top_p ? P.top_p[r] : 1.0f;
    if (!(topp > 0.0f)) {
      bits |= SV_DATA_BAD_PARAM;
    } else {
      const TIn *grow[2] = {row + x0, nullptr};
      const uint32_t lf = load_rows<TIn, kVec, kRes>(sm, grow, srow, 1, n, phase, P.first_wait);
      RowStats st[2];
      uint32_t ymark = 0u;
      if (!position_stats<TIn>(sm, inbox, srow, 1, n, __fdiv_rn(kLog2e, temp), topk, topp, lf, st, &bits, step,
                               ncta, rank) ||
          (procs && !proc_correct<TIn>(sm, inbox, srow, 1, n, words, pr, st, -1, ymark, &bits, step, ncta, rank))) {
        // nothing sampled (the status bit is set)
      } else {
        const RngKey rk{P.seed_lo, P.seed_hi ^ 0x53414D50u, P.off_lo, P.off_hi};  // the sampler's own streams
        const float *Erow = kTest ? P.exponentials + static_cast<int64_t>(r) * P.exp_stride : nullptr;
        float bk = 0.0f;
        int bx = -1;
        uint32_t fl = 0;
        if (procs)
          race_chunks<TIn, kTest, false, true>(srow[0], srow[0], st[0], st[0], x0, n, Erow, rk,
                                               P.row_base + static_cast<uint32_t>(r), bk, bx, fl, pr);
        else
          race_chunks<TIn, kTest, false>(srow[0], srow[0], st[0], st[0], x0, n, Erow, rk,
                                         P.row_base + static_cast<uint32_t>(r), bk, bx, fl);
        const KeyFlags kr = cluster_reduce(KeyFlags{bx >= 0 ? pack_key(bk, bx) : 0ull, fl}, sm.red, step++, ncta);
        bits |= kr.flags;
        if (kr.key == 0ull) {
          bits |= SV_DATA_EMPTY_DISTRIBUTION;
          token = 0;
        } else {
          token = static_cast<int32_t>(key_index(kr.key));
        }
        if (P.probs) {  // this CTA's chunk of the transformed row
          float *prow = P.probs + static_cast<int64_t>(r) * P.probs_stride + x0;
          int xs = 0;
          if (kVec && sizeof(TIn) == 2 && (reinterpret_cast<uintptr_t>(prow) & 15u) == 0) {
            // eight bf16 logits in, two float4 probabilities out
            const uint4 *s4 = reinterpret_cast<const uint4 *>(srow[0]);
            float4 *p4 = reinterpret_cast<float4 *>(prow);
            const int ng = n >> 3;
            for (int v = tid; v < ng; v += kThreads) {
              const uint4 d = s4[v];
              const uint32_t w[4] = {d.x, d.y, d.z, d.w};
              float o[8];
#pragma unroll
              for (int t = 0; t < 4; ++t) {
                o[2 * t] = prob_of<TIn>(w[t] & 0xFFFFu, st[0]);
                o[2 * t + 1] = prob_of<TIn>(w[t] >> 16, st[0]);
              }
              if (procs) {  // marked entries: their processed probabilities
                uint32_t mk = group_marks<8>(pr, 8 * v);
                while (mk) {
                  const int t = __ffs(mk) - 1;
                  mk &= mk - 1u;
                  o[t] = prob_of_m<TIn>((w[t >> 1] >> (16 * (t & 1))) & 0xFFFFu, mark_at(pr, 8 * v + t), st[0], theta);
                }
              }
              p4[2 * v] = make_float4(o[0], o[1], o[2], o[3]);
              p4[2 * v + 1] = make_float4(o[4], o[5], o[6], o[7]);
            }
            xs = ng << 3;
          }
          for (int x = xs + tid; x < n; x += kThreads)
            prow[x] = prob_of_m<TIn>(bits_at(srow[0], x), procs ? mark_at(pr, x) : 0u, st[0], theta);
        }
      }
    }
  }
  if (rank == 0 && tid == 0) {
    P.tokens[r] = token;
    if (bits && P.status) atomicOr(P.status, static_cast<int>(bits));
  }
  cluster_sync();
}

template <typename TIn, bool kTest, bool kVec, bool kRes, bool kProc>
cudaError_t launch_sample_one(const SampleParams &p, int cluster, int chunk, size_t dyn, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p.R) * static_cast<unsigned>(cluster), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = dyn;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  cfg.attrs = attr;
  cfg.numAttrs = launch_attrs(attr, static_cast<unsigned>(cluster), p.pdl);
  return cudaLaunchKernelEx(&cfg, sample_kernel<TIn, kTest, kVec, kRes, kProc>, p, chunk);
}

template <typename TIn, bool kTest, bool kVec, bool kRes, bool kProc>
cudaError_t enable_sample_one(int max_cluster, int max_dyn) {
  cudaError_t e = cudaFuncSetAttribute(sample_kernel<TIn, kTest, kVec, kRes, kProc>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, max_dyn);
  if (e != cudaSuccess) return e;
  if (max_cluster > 8)
    return cudaFuncSetAttribute(sample_kernel<TIn, kTest, kVec, kRes, kProc>,
                                cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  return cudaSuccess;
}

// Sampler forms per element type, randomness and processors: unaligned rows
// (in shared memory), aligned rows in shared memory, aligned rows in place.
template <typename TIn, bool kTest, bool kProc>
cudaError_t enable_sample_forms(int max_cluster, int max_dyn) {
  cudaError_t e;
  if ((e = enable_sample_one<TIn, kTest, false, true, kProc>(max_cluster, max_dyn)) != cudaSuccess) return e;
  if ((e = enable_sample_one<TIn, kTest, true, true, kProc>(max_cluster, max_dyn)) != cudaSuccess) return e;
  return enable_sample_one<TIn, kTest, true, false, kProc>(max_cluster, max_dyn);
}

template <typename TIn, bool kTest, bool kProc>
cudaError_t launch_sample_form(const SampleParams &p, int cluster, int chunk, size_t dyn, bool vec, bool resident,
                               cudaStream_t stream) {
  if (!vec) return launch_sample_one<TIn, kTest, false, true, kProc>(p, cluster, chunk, dyn, stream);
  return resident ? launch_sample_one<TIn, kTest, true, true, kProc>(p, cluster, chunk, dyn, stream)
                  : launch_sample_one<TIn, kTest, true, false, kProc>(p, cluster, chunk, dyn, stream);
}

template <typename TIn, bool kTest, bool kVec, bool kRes, bool kProc>
cudaError_t launch_one(const VerifyParams &p, int cluster, int chunk, size_t dyn, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p.N) * static_cast<unsigned>(cluster), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = dyn;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  cfg.attrs = attr;
  cfg.numAttrs = launch_attrs(attr, static_cast<unsigned>(cluster), p.pdl);
  return cudaLaunchKernelEx(&cfg, logits_kernel<TIn, kTest, kVec, kRes, kProc>, p, chunk);
}

template <typename TIn, bool kTest, bool kVec, bool kRes, bool kProc>
cudaError_t enable_one(int max_cluster, int max_dyn) {
  cudaError_t e = cudaFuncSetAttribute(logits_kernel<TIn, kTest, kVec, kRes, kProc>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, max_dyn);
  if (e != cudaSuccess) return e;
  if (max_cluster > 8)
    return cudaFuncSetAttribute(logits_kernel<TIn, kTest, kVec, kRes, kProc>,
                                cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  return cudaSuccess;
}

// Forms built per element type, randomness and processors: unaligned rows
// (resident), aligned rows with both chunks resident, aligned rows read in
// place.
template <typename TIn, bool kTest, bool kProc>
cudaError_t enable_forms(int max_cluster, int max_dyn) {
  cudaError_t e;
  if ((e = enable_one<TIn, kTest, false, true, kProc>(max_cluster, max_dyn)) != cudaSuccess) return e;
  if ((e = enable_one<TIn, kTest, true, true, kProc>(max_cluster, max_dyn)) != cudaSuccess) return e;
  return enable_one<TIn, kTest, true, false, kProc>(max_cluster, max_dyn);
}

template <typename TIn, bool kTest, bool kProc>
cudaError_t launch_form(const VerifyParams &p, int cluster, int chunk, size_t dyn, bool vec, bool resident,
                        cudaStream_t stream) {
  if (!vec) return launch_one<TIn, kTest, false, true, kProc>(p, cluster, chunk, dyn, stream);
  return resident ? launch_one<TIn, kTest, true, true, kProc>(p, cluster, chunk, dyn, stream)
                  : launch_one<TIn, kTest, true, false, kProc>(p, cluster, chunk, dyn, stream);
}

// Every form of both kernels for one element type and processor setting
// (test and production randomness), and their launches; each translation unit
// turns these into its named entry points.
template <typename TIn, bool kProc>
cudaError_t enable_type_logits(int max_cluster, int max_dyn) {
  cudaError_t e;
  if ((e = enable_forms<TIn, true, kProc>(max_cluster, max_dyn)) != cudaSuccess) return e;
  return enable_forms<TIn, false, kProc>(max_cluster, max_dyn);
}

template <typename TIn, bool kProc>
cudaError_t enable_type_sample(int max_cluster, int max_dyn) {
  cudaError_t e;
  if ((e = enable_sample_forms<TIn, true, kProc>(max_cluster, max_dyn)) != cudaSuccess) return e;
  return enable_sample_forms<TIn, false, kProc>(max_cluster, max_dyn);
}

template <typename TIn, bool kProc>
cudaError_t launch_type_logits(const VerifyParams &p, int cluster, int chunk, size_t dyn, bool vec, bool resident,
                               cudaStream_t stream) {
  return p.exponentials != nullptr ? launch_form<TIn, true, kProc>(p, cluster, chunk, dyn, vec, resident, stream)
                                   : launch_form<TIn, false, kProc>(p, cluster, chunk, dyn, vec, resident, stream);
}

template <typename TIn, bool kProc>
cudaError_t launch_type_sample(const SampleParams &p, int cluster, int chunk, size_t dyn, bool vec, bool resident,
                               cudaStream_t stream) {
  return p.exponentials != nullptr
             ? launch_sample_form<TIn, true, kProc>(p, cluster, chunk, dyn, vec, resident, stream)
             : launch_sample_form<TIn, false, kProc>(p, cluster, chunk, dyn, vec, resident, stream);
}

}  // namespace
}  // namespace sv
