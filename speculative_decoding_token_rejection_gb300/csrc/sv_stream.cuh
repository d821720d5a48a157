// sv_stream.cuh -- the logits entry with one CTA per request ("streaming"
// form), for batches large enough that every request has its own CTA at once
// (up to four per SM).  The same verification as logits_kernel ("vLLM source
// walk-through (10)", section "Rejection sampling: the two branches of
// RejectionSampler": temperature, top-k, top-p on both sides; "Speculative
// Decoding: propose, verify, accept", sections 04 and 06), organised so that a
// position costs one read of its two rows and no cluster exchange:
//
//  * one pass over the target and draft rows (read in place; at later
//    positions, when fewer requests are left, the next steps are prefetched
//    into L2) takes each row's largest value (NaN-propagating, so it also
//    reveals NaN and +inf) and, for rows with 1 <= top_k <= kStreamTopK, the
//    largest key of every block (one thread's groups over kBlockSteps steps,
//    128 bytes) into shared memory; the loop has no barrier and no branch
//    between its loads;
//  * the top_k-th largest block maximum is a floor: top_k distinct elements
//    reach it, so it never exceeds the row's top_k-th largest key.  The
//    blocks whose maximum reaches it (about top_k of them) are read again,
//    from L2, and their elements at or above it become candidates: the whole
//    top-k set, ties included;
//  * the exact top_k-th largest key, the top-p cut and the normaliser then
//    come from the candidates alone, with the masses in 2^-40 fixed point
//    summed as integers (the same masses, cut and normaliser as
//    logits_kernel's window path), and the residual or bonus race runs over
//    the kept candidates only (a residual is positive only where p is);
//  * rows outside that case (top-k off or above kStreamTopK, rows longer
//    than kMaxBlocks blocks, or candidates overflowing their room) take the
//    exact multi-pass statistics and the race over the whole rows, as a
//    cluster of one.
#pragma once

#include "sv_logits.cuh"

namespace sv {
namespace {

constexpr int kCand = 1024;         // candidate slots per row
constexpr int kStreamTopK = 256;    // largest top-k the candidate path serves
constexpr int kStreamU = 4;         // 16-byte groups per row and thread in one step
constexpr int kStep = kThreads * kStreamU;  // groups per row in one step
constexpr int kBlockSteps = 2;      // steps per block: a block is one thread's 8 groups of two consecutive steps
constexpr int kMaxBlocks = 4096;    // blocks per row (rows up to 32 steps: 262144 bf16 or 131072 fp32 logits)
constexpr int kWarpHits = kMaxBlocks / kWarps;  // blocks a warp reads again (its share of the block maxima's room, as 32-bit entries)
constexpr int kHitPass = 4;         // groups per lane in flight while reading them

struct StreamSmem {
  ReduceSmem red;                      // block / cluster-of-one reductions of the races and argmaxes
  int32_t tok[SV_MAX_SPEC_LEN + 1];    // committed tokens
  int stop_first;
  unsigned long long zk[2];    // fixed-point mass of the top-k set
  unsigned long long kept[2];  // fixed-point mass of the final kept set
  uint32_t maxkey[2];      // largest finite key of each row
  uint32_t flags[2];       // kFlagBad / kFlagFinite
  uint32_t prefix[2];      // selection state: digits fixed so far
  uint32_t need[2];        // selection state: rank still to cover inside the prefix range
  uint32_t cut[2];         // top-p cut (key)
  int cnt[2];              // candidates per row
  int overflow;            // candidates or blocks beyond their room
  union {
    struct {  // the candidate path
      uint32_t key[2][kCand];  // candidate keys (order-preserving) of the target and draft rows
      int32_t idx[2][kCand];   // their vocabulary indices
      uint32_t hist[2][256];   // digit histograms of the selections
      union {
        uint16_t bm[2][kMaxBlocks];         // until the candidates are gathered: 16 high bits of each block's largest key
        unsigned long long mass[2][kCand];  // afterwards: fixed-point masses of the kept candidates
      };
    };
    LogitsSmem fb;  // the multi-pass statistics of the other rows (never alongside the candidates)
  };
};

// The k-th largest (with multiplicity) of the kB-bit keys get(r, 0 .. n[r]-1)
// of each row r with sel[r] set, one 8-bit digit per round (warp-aggregated
// histograms); out[r] receives it.  Requires n[r] >= k.
template <int kB, typename Get>
__device__ void radix_kth(StreamSmem &ss, const bool sel[2], const int n[2], int k, Get get, uint32_t out[2]) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid < 2) {
    ss.prefix[tid] = 0u;
    ss.need[tid] = static_cast<uint32_t>(k);
  }
  for (int lo = kB - 8; lo >= 0; lo -= 8) {
    for (int t = tid; t < 512; t += kThreads) ss.hist[t >> 8][t & 255] = 0u;
    __syncthreads();
    for (int r = 0; r < 2; ++r) {
      if (!sel[r]) continue;
      const int hs = lo + 8;
      const uint32_t hp = hs >= kB ? 0u : (ss.prefix[r] >> hs);
      const int c = n[r];
      for (int base = tid & ~31; base < c; base += kThreads) {  // whole warps: lanes with equal bins add once
        const int i = base + lane;
        const uint32_t key = i < c ? get(r, i) : 0u;
        const bool in = i < c && (hs >= kB || (key >> hs) == hp);
        const uint32_t bin = in ? ((key >> lo) & 255u) : 256u;
        const unsigned peers = __match_any_sync(0xFFFFFFFFu, bin);
        if (in && lane == __ffs(peers) - 1) atomicAdd(&ss.hist[r][bin], static_cast<uint32_t>(__popc(peers)));
      }
    }
    __syncthreads();
    if (warp < 2 && sel[warp]) {  // one warp per row walks the bins from the top
      const int r = warp;
      uint32_t c[8], s = 0;
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        c[t] = ss.hist[r][255 - (8 * lane + t)];
        s += c[t];
      }
      uint32_t inc = s;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, inc, o);
        if (lane >= o) inc += v;
      }
      const uint32_t before = inc - s, need = ss.need[r];
      int found = -1;
      uint32_t above = 0;
      if (before < need && inc >= need) {
        uint32_t acc = before;
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          if (found < 0 && acc + c[t] >= need) {
            found = 8 * lane + t;
            above = acc;
          }
          acc += c[t];
        }
      }
      const unsigned ball = __ballot_sync(0xFFFFFFFFu, found >= 0);
      const int src = ball ? __ffs(ball) - 1 : 0;
      const int bin = __shfl_sync(0xFFFFFFFFu, found, src);
      const uint32_t ab = __shfl_sync(0xFFFFFFFFu, above, src);
      if (lane == 0 && ball) {
        ss.prefix[r] |= static_cast<uint32_t>(255 - bin) << lo;
        ss.need[r] = need - ab;
      }
    }
    __syncthreads();
  }
  for (int r = 0; r < 2; ++r) out[r] = ss.prefix[r];
}

// Keep the candidates of each row r with sel[r] whose key is >= thr[r]
// (order not kept: every later use is order-free).  Each thread holds its
// kCand / kThreads slots in registers (fixed indices), then every warp claims
// room for its kept entries with one atomic per slot column.
__device__ void cand_compact(StreamSmem &ss, const bool sel[2], const uint32_t thr[2]) {
  const int tid = threadIdx.x, lane = tid & 31;
  constexpr int kPerThread = kCand / kThreads;
  for (int r = 0; r < 2; ++r) {
    if (!sel[r]) continue;
    const int c = min(ss.cnt[r], kCand);
    uint32_t k[kPerThread];
    int32_t x[kPerThread];
    bool keep[kPerThread];
#pragma unroll
    for (int t = 0; t < kPerThread; ++t) {
      const int i = tid + t * kThreads;
      k[t] = i < c ? ss.key[r][i] : 0u;
      x[t] = i < c ? ss.idx[r][i] : 0;
      keep[t] = i < c && k[t] >= thr[r];
    }
    __syncthreads();
    if (tid == 0) ss.cnt[r] = 0;
    __syncthreads();
#pragma unroll
    for (int t = 0; t < kPerThread; ++t) {
      const unsigned ball = __ballot_sync(0xFFFFFFFFu, keep[t]);
      int base = 0;
      if (lane == 0 && ball) base = atomicAdd(&ss.cnt[r], __popc(ball));
      base = __shfl_sync(0xFFFFFFFFu, base, 0);
      if (keep[t]) {
        const int pos = base + __popc(ball & ((1u << lane) - 1u));
        ss.key[r][pos] = k[t];
        ss.idx[r][pos] = x[t];
      }
    }
    __syncthreads();
  }
}

template <typename TIn>
__device__ __forceinline__ void cand_push(StreamSmem &ss, int r, uint32_t key, int x) {
  const int p = atomicAdd(&ss.cnt[r], 1);
  if (p < kCand) {
    ss.key[r][p] = key;
    ss.idx[r][p] = x;
  } else {
    ss.overflow = 1;
  }
}

// NaN-propagating maximum of two value words (bf16: both halves; fp32: the value).
template <typename TIn>
__device__ __forceinline__ uint32_t max_word(uint32_t a, uint32_t b) {
  if constexpr (sizeof(TIn) == 2) {
    return bf16x2_max_nan(a, b);
  } else {
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(__uint_as_float(a)), "f"(__uint_as_float(b)));
    return __float_as_uint(r);
  }
}
// The largest value of a word (bf16: of its two halves) as value bits.
template <typename TIn>
__device__ __forceinline__ uint32_t word_top(uint32_t w) {
  if constexpr (sizeof(TIn) == 2) return bf16x2_max_nan(w, (w >> 16) | (w << 16)) & 0xFFFFu;
  else return w;
}
// The 16 high bits of an element's key.
template <typename TIn>
__device__ __forceinline__ uint32_t key16_of_bits(uint32_t b) {
  return Elem<TIn>::key(b) >> (Elem<TIn>::kBits - 16);
}

// One pass over this position's rows, the only read of their bytes from HBM:
// each row's largest value and value checks (ss.maxkey, ss.flags) and, with
// kBlocks, the 16 high bits of every block's largest key (ss.bm).  Block b of
// a row holds groups (2s + h) * kStep + u * kThreads + t for h < 2, u <
// kStreamU, where s = b / kThreads and t = b % kThreads: a thread's loads of
// two consecutive steps.  The loop keeps only its loads and two running
// maxima per row in registers and has no barrier.
template <typename TIn, bool kBlocks>
__device__ __noinline__ void stream_pass(StreamSmem &ss, const TIn *const rows[2], int nr, int n, int ahead) {
  using E = Elem<TIn>;
  constexpr int kPer = 16 / sizeof(TIn);
  const int tid = threadIdx.x;
  const int ng = n / kPer;
  const int nsteps = (ng + kStep - 1) / kStep;
  const uint4 *const r0 = reinterpret_cast<const uint4 *>(rows[0]);
  const uint4 *const r1 = reinterpret_cast<const uint4 *>(nr > 1 ? rows[1] : rows[0]);
  // With fewer requests left (later positions), one thread keeps `ahead`
  // steps of both rows in flight as bulk L2 prefetches.
  auto prefetch_step = [&](int st) {
    const int g0 = st * kStep, g1 = min(ng, g0 + kStep);
    prefetch_l2(r0 + g0, static_cast<uint32_t>(g1 - g0) * 16u);
    if (nr > 1) prefetch_l2(r1 + g0, static_cast<uint32_t>(g1 - g0) * 16u);
  };
  if (tid == 0)
    for (int st = 0; st < ahead && st < nsteps; ++st) prefetch_step(st);
  if (tid < 2) {
    ss.cnt[tid] = 0;
    ss.maxkey[tid] = 0u;
    ss.flags[tid] = 0u;
  }
  if (tid == 0) ss.overflow = 0;
  constexpr uint32_t kNoneW = sizeof(TIn) == 2 ? 0xFF80FF80u : 0xFF800000u;  // -inf
  const uint4 kNone = make_uint4(kNoneW, kNoneW, kNoneW, kNoneW);
  uint32_t bm0 = kNoneW, bm1 = kNoneW;  // running block maxima
  uint32_t rm0 = kNoneW, rm1 = kNoneW;  // running row maxima
  for (int st = 0; st < nsteps; ++st) {
    if (tid == 0 && ahead && st + ahead < nsteps) prefetch_step(st + ahead);
    const int g = st * kStep + tid;
    uint4 a[kStreamU], b[kStreamU];
#pragma unroll
    for (int u = 0; u < kStreamU; ++u) {
      const bool in = g + u * kThreads < ng;
      a[u] = in ? ld_stream_u4(r0 + g + u * kThreads) : kNone;
      b[u] = (in && nr > 1) ? ld_stream_u4(r1 + g + u * kThreads) : kNone;
    }
#pragma unroll
    for (int u = 0; u < kStreamU; ++u) {
      bm0 = max_word<TIn>(bm0, max_word<TIn>(max_word<TIn>(a[u].x, a[u].y), max_word<TIn>(a[u].z, a[u].w)));
      bm1 = max_word<TIn>(bm1, max_word<TIn>(max_word<TIn>(b[u].x, b[u].y), max_word<TIn>(b[u].z, b[u].w)));
    }
    if (st % kBlockSteps == kBlockSteps - 1 || st == nsteps - 1) {  // the end of a block
      if (kBlocks) {
        const int blk = (st / kBlockSteps) * kThreads + tid;
        const bool any = (st - st % kBlockSteps) * kStep + tid < ng;  // the block holds at least one group of the row
        ss.bm[0][blk] = static_cast<uint16_t>(any ? key16_of_bits<TIn>(word_top<TIn>(bm0)) : 0u);
        if (nr > 1) ss.bm[1][blk] = static_cast<uint16_t>(any ? key16_of_bits<TIn>(word_top<TIn>(bm1)) : 0u);
      }
      rm0 = max_word<TIn>(rm0, bm0);
      rm1 = max_word<TIn>(rm1, bm1);
      bm0 = kNoneW;
      bm1 = kNoneW;
    }
  }
  // the last elements (fewer than a 16-byte group)
  for (int x = ng * kPer + tid; x < n; x += kThreads) {
    const uint32_t b0 = bits_at(rows[0], x);
    rm0 = max_word<TIn>(rm0, sizeof(TIn) == 2 ? (b0 | (b0 << 16)) : b0);
    if (nr > 1) {
      const uint32_t b1 = bits_at(rows[1], x);
      rm1 = max_word<TIn>(rm1, sizeof(TIn) == 2 ? (b1 | (b1 << 16)) : b1);
    }
  }
  uint32_t mk[2], fl[2];
  const uint32_t rms[2] = {word_top<TIn>(rm0), word_top<TIn>(rm1)};
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const uint32_t bb = rms[r];
    fl[r] = (E::is_nan(bb) || E::is_pinf(bb)) ? kFlagBad : 0u;
    if (E::finite(bb)) fl[r] |= kFlagFinite;
    mk[r] = E::finite(bb) ? E::key(bb) : 0u;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      mk[r] = max(mk[r], __shfl_xor_sync(0xFFFFFFFFu, mk[r], o));
      fl[r] |= __shfl_xor_sync(0xFFFFFFFFu, fl[r], o);
    }
  __syncthreads();  // (the counters' reset above)
  if ((tid & 31) == 0)
    for (int r = 0; r < nr; ++r) {
      atomicMax(&ss.maxkey[r], mk[r]);
      atomicOr(&ss.flags[r], fl[r]);
    }
  __syncthreads();
}

// The candidates of this position's rows (after stream_pass with kBlocks).
// The floor of each row is the topk-th largest block maximum (16 high key
// bits): a histogram of the block maxima's distances below the row's largest
// key (one 256-bin round), or, if fewer than topk of them lie within 255
// steps, the radix selection.  Each thread then reads again those of its own
// blocks whose maximum reaches the floor; their elements whose key's high
// bits reach it become candidates, as do such elements among the last few
// (fewer than a group).  Sets ss.overflow if the candidates exceed their room.
template <typename TIn>
__device__ __forceinline__ void gather_candidates(StreamSmem &ss, const TIn *const rows[2], int nr, int n, int topk) {
  using E = Elem<TIn>;
  constexpr int kPer = 16 / sizeof(TIn);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int ng = n / kPer;
  const int nsteps = (ng + kStep - 1) / kStep;
  const int nb = ((nsteps + kBlockSteps - 1) / kBlockSteps) * kThreads;
  const uint32_t m16[2] = {ss.maxkey[0] >> (E::kBits - 16), ss.maxkey[1] >> (E::kBits - 16)};
  for (int t = tid; t < 512; t += kThreads) ss.hist[t >> 8][t & 255] = 0u;
  __syncthreads();
  for (int r = 0; r < nr; ++r) {
    const uint32_t *const bm2 = reinterpret_cast<const uint32_t *>(ss.bm[r]);  // two block maxima per word
    for (int b = tid; b < nb / 2; b += kThreads) {
      const uint32_t two = bm2[b];
      const uint32_t d0 = m16[r] - (two & 0xFFFFu), d1 = m16[r] - (two >> 16);  // (no block maximum exceeds the row's)
      if (d0 < 256u) atomicAdd(&ss.hist[r][d0], 1u);
      if (d1 < 256u) atomicAdd(&ss.hist[r][d1], 1u);
    }
  }
  __syncthreads();
  if (warp < nr) {  // one warp per row walks the distances from 0
    const int r = warp;
    uint32_t c[8], sum = 0;
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      c[t] = ss.hist[r][8 * lane + t];
      sum += c[t];
    }
    uint32_t inc = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, inc, o);
      if (lane >= o) inc += v;
    }
    const uint32_t need = static_cast<uint32_t>(topk);
    int found = -1;
    if (inc - sum < need && inc >= need) {
      uint32_t acc = inc - sum;
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        if (found < 0 && acc + c[t] >= need) found = 8 * lane + t;
        acc += c[t];
      }
    }
    const unsigned ball = __ballot_sync(0xFFFFFFFFu, found >= 0);
    const int dist = ball ? __shfl_sync(0xFFFFFFFFu, found, __ffs(ball) - 1) : -1;
    if (lane == 0) ss.prefix[r] = dist >= 0 ? m16[r] - static_cast<uint32_t>(dist) : 0xFFFFFFFFu;
  }
  __syncthreads();
  uint32_t f16[2] = {ss.prefix[0], ss.prefix[1]};
  if (f16[0] == 0xFFFFFFFFu || (nr > 1 && f16[1] == 0xFFFFFFFFu)) {  // a row's floor lies farther down
    const bool sel[2] = {true, nr > 1};
    const int nbs[2] = {nb, nb};
    radix_kth<16>(ss, sel, nbs, topk, [&](int r, int i) -> uint32_t { return ss.bm[r][i]; }, f16);
  }
  // this thread's blocks s * kThreads + tid (s < 16) that reach the floor, as bits r * 16 + s
  const int nsb = nb / kThreads;
  uint32_t lim[2], hm = 0u;
#pragma unroll
  for (int r = 0; r < 2; ++r)  // a +0.0 maximum may come out of the NaN-propagating max as -0.0 (one key below)
    lim[r] = f16[r] == 0x8000u ? 0x7FFFu : f16[r];
  for (int r = 0; r < nr; ++r)
    for (int sb = 0; sb < nsb; ++sb)
      if (ss.bm[r][sb * kThreads + tid] >= lim[r]) hm |= 1u << (16 * r + sb);
  // Each warp lists its lanes' blocks (bit << 8 | owner thread) in its part
  // of the block maxima's room, then reads their groups one per lane, all in
  // flight together (kHitPass per lane at a time).
  __syncthreads();  // (every thread has read the block maxima)
  uint32_t *const hl = reinterpret_cast<uint32_t *>(&ss.bm[0][0]) + warp * kWarpHits;
  const int pc = __popc(hm);
  int incl = pc;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += v;
  }
  const int H = __shfl_sync(0xFFFFFFFFu, incl, 31);
  int slot = incl - pc;
  for (uint32_t m = hm; m; m &= m - 1u, ++slot)
    if (slot < kWarpHits) hl[slot] = (static_cast<uint32_t>(__ffs(m) - 1) << 8) | static_cast<uint32_t>(tid);
  if (H > kWarpHits && lane == 0) ss.overflow = 1;
  __syncwarp();
  const int items = min(H, kWarpHits) * kBlockSteps * kStreamU;  // one 16-byte group each
  for (int base = 0; base < items; base += 32 * kHitPass) {
    uint4 d[kHitPass];
    int gg[kHitPass], rr[kHitPass];
#pragma unroll
    for (int k = 0; k < kHitPass; ++k) {
      const int it = base + 32 * k + lane;
      gg[k] = -1;
      rr[k] = 0;
      d[k] = make_uint4(0u, 0u, 0u, 0u);
      if (it < items) {
        const uint32_t e = hl[it >> 3];
        const int q = it & 7, bit = static_cast<int>(e >> 8), t = static_cast<int>(e & 255u);
        const int r = bit >> 4, sb = bit & 15;
        const int g = (kBlockSteps * sb + q / kStreamU) * kStep + (q % kStreamU) * kThreads + t;
        if (g < ng) {
          d[k] = ld_stream_u4(reinterpret_cast<const uint4 *>(r ? rows[1] : rows[0]) + g);
          gg[k] = g;
          rr[k] = r;
        }
      }
    }
    // the elements at or above the floor, of the groups whose maximum reaches it
    // (a NaN maximum does; its NaNs do not)
    uint32_t em[kHitPass];
    uint32_t cnt = 0u;  // this lane's elements: row 0 in the low 16 bits, row 1 in the high 16
#pragma unroll
    for (int k = 0; k < kHitPass; ++k) {
      em[k] = 0u;
      if (gg[k] < 0) continue;
      const int r = rr[k];
      const uint32_t tk = (r ? f16[1] : f16[0]) << (E::kBits - 16);
      if constexpr (sizeof(TIn) == 2) {
        // two elements per packed compare against the floor's value (NaN fails;
        // a -0.0 may pass a +0.0 floor: an extra candidate below the floor,
        // which the exact selection that follows ignores)
        uint32_t t2 = bf16_bits_of_key(tk);
        t2 |= t2 << 16;
        const uint32_t m0 = bf16x2_ge_mask(d[k].x, t2), m1 = bf16x2_ge_mask(d[k].y, t2);
        const uint32_t m2 = bf16x2_ge_mask(d[k].z, t2), m3 = bf16x2_ge_mask(d[k].w, t2);
        em[k] = (m0 & 1u) | ((m0 >> 15) & 2u) | ((m1 & 1u) << 2) | ((m1 >> 13) & 8u) | ((m2 & 1u) << 4) |
                ((m2 >> 11) & 32u) | ((m3 & 1u) << 6) | ((m3 >> 9) & 128u);
      } else {
        const uint32_t gm = word_top<TIn>(max_word<TIn>(max_word<TIn>(d[k].x, d[k].y), max_word<TIn>(d[k].z, d[k].w)));
        if (key16_of_bits<TIn>(gm) < (r ? lim[1] : lim[0])) continue;
#pragma unroll
        for (int t = 0; t < kPer; ++t) {
          const uint32_t bb = t == 0 ? d[k].x : t == 1 ? d[k].y : t == 2 ? d[k].z : d[k].w;
          if (!E::is_nan(bb) && E::key(bb) >= tk) em[k] |= 1u << t;
        }
      }
      cnt += static_cast<uint32_t>(__popc(em[k])) << (16 * r);
    }
    // one shared atomic per warp and row claims the room (pushes from every
    // warp at once on one counter serialise)
    uint32_t incl2 = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl2, o);
      if (lane >= o) incl2 += v;
    }
    const uint32_t tot = __shfl_sync(0xFFFFFFFFu, incl2, 31);
    if (tot == 0u) continue;
    int b0 = 0, b1 = 0;
    if (lane == 31) {
      if (tot & 0xFFFFu) b0 = atomicAdd(&ss.cnt[0], static_cast<int>(tot & 0xFFFFu));
      if (tot >> 16) b1 = atomicAdd(&ss.cnt[1], static_cast<int>(tot >> 16));
    }
    const uint32_t excl = incl2 - cnt;
    int pos0 = __shfl_sync(0xFFFFFFFFu, b0, 31) + static_cast<int>(excl & 0xFFFFu);
    int pos1 = __shfl_sync(0xFFFFFFFFu, b1, 31) + static_cast<int>(excl >> 16);
#pragma unroll
    for (int k = 0; k < kHitPass; ++k) {
      const int r = rr[k];
      for (uint32_t m = em[k]; m; m &= m - 1u) {
        const int t = __ffs(m) - 1;
        const int wi = sizeof(TIn) == 2 ? t >> 1 : t;
        const uint32_t wv = wi == 0 ? d[k].x : wi == 1 ? d[k].y : wi == 2 ? d[k].z : d[k].w;
        const uint32_t bb = sizeof(TIn) == 2 ? ((t & 1) ? (wv >> 16) : (wv & 0xFFFFu)) : wv;
        const int pos = r ? pos1++ : pos0++;
        if (pos < kCand) {
          ss.key[r][pos] = E::key(bb);
          ss.idx[r][pos] = gg[k] * kPer + t;
        } else {
          ss.overflow = 1;
        }
      }
    }
  }
  for (int r = 0; r < nr; ++r) {
    const uint32_t tk = f16[r] << (E::kBits - 16);
    for (int x = ng * kPer + tid; x < n; x += kThreads) {
      const uint32_t bb = bits_at(rows[r], x);
      if (!E::is_nan(bb) && E::key(bb) >= tk) cand_push<TIn>(ss, r, E::key(bb), x);
    }
  }
  __syncthreads();
}

// Sum of a per-thread u64 over the block into *dst (one shared atomic per warp;
// integer sums, so the order does not matter).
__device__ __forceinline__ void block_add_u64(unsigned long long v, unsigned long long *dst) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  if ((threadIdx.x & 31) == 0 && v) atomicAdd(dst, v);
}

// Statistics of the candidate rows: the exact k-th largest key, the top-p cut
// and the normaliser, from the candidates alone (masses in 2^-40 fixed point
// relative to the row maximum, summed as integers).
// Sorts 64 keys held two per lane (element lane + 32 h in k[h]) into
// descending order along that numbering (bitonic network).
__device__ __forceinline__ void warp_sort64_desc(uint32_t k[2]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int size = 2; size <= 64; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      uint32_t nk[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int e = lane + 32 * h;
        const uint32_t pk = stride == 32 ? k[h ^ 1] : __shfl_xor_sync(0xFFFFFFFFu, k[h], stride);
        const bool take_max = ((e & stride) == 0) == ((e & size) == 0);
        nk[h] = take_max ? max(k[h], pk) : min(k[h], pk);
      }
      k[0] = nk[0];
      k[1] = nk[1];
    }
  }
}

__device__ __forceinline__ unsigned long long warp_sum_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

// cand_stats for rows of at most 64 candidates: one warp per row sorts the
// keys and takes the k-th largest, the masses, the top-p cut (the key at the
// first sorted position whose running mass reaches the target: the largest
// key whose mass at or above it does) and the kept mass, without a block
// barrier; the same results as the block-wide selection below.
template <typename TIn>
__device__ __forceinline__ void warp_stats(StreamSmem &ss, int nr, int topk, float topp, const RowStats st[2]) {
  using E = Elem<TIn>;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (warp >= nr) return;
  const int r = warp;
  const float vmax = r ? st[1].vmax : st[0].vmax, c2 = r ? st[1].c2 : st[0].c2;
  const int c = ss.cnt[r];
  uint32_t k[2];
  k[0] = lane < c ? ss.key[r][lane] : 0u;  // 0: no candidate (a NaN key is never one)
  k[1] = lane + 32 < c ? ss.key[r][lane + 32] : 0u;
  warp_sort64_desc(k);
  const int kk = topk - 1;  // (topk <= c)
  const uint32_t tk = __shfl_sync(0xFFFFFFFFu, (kk >> 5) ? k[1] : k[0], kk & 31);
  unsigned long long m[2];
#pragma unroll
  for (int h = 0; h < 2; ++h)
    m[h] = k[h] >= tk ? to_fixed(exp2f(__fmul_rn(__fsub_rn(E::val_of_key(k[h]), vmax), c2))) : 0ull;
  const unsigned long long zk = warp_sum_u64(m[0] + m[1]);
  uint32_t cut = tk;
  unsigned long long kept = zk;
  if (topp < 1.0f) {
    unsigned long long need = static_cast<unsigned long long>(static_cast<double>(topp) * static_cast<double>(zk));
    if (need == 0ull) need = 1ull;
    unsigned long long p0 = m[0], p1 = m[1];  // inclusive running masses in sorted order
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long v0 = __shfl_up_sync(0xFFFFFFFFu, p0, o), v1 = __shfl_up_sync(0xFFFFFFFFu, p1, o);
      if (lane >= o) {
        p0 += v0;
        p1 += v1;
      }
    }
    p1 += __shfl_sync(0xFFFFFFFFu, p0, 31);
    const unsigned b0 = __ballot_sync(0xFFFFFFFFu, p0 >= need), b1 = __ballot_sync(0xFFFFFFFFu, p1 >= need);
    const uint32_t c0 = __shfl_sync(0xFFFFFFFFu, k[0], b0 ? __ffs(b0) - 1 : 0);
    const uint32_t c1 = __shfl_sync(0xFFFFFFFFu, k[1], b1 ? __ffs(b1) - 1 : 0);
    if (b0) cut = c0;
    else if (b1) cut = c1;
    kept = warp_sum_u64((k[0] >= cut ? m[0] : 0ull) + (k[1] >= cut ? m[1] : 0ull));
  }
  if (lane == 0) {
    ss.cut[r] = cut;
    ss.zk[r] = zk;
    ss.kept[r] = kept;
  }
}

template <typename TIn>
__device__ __noinline__ void cand_stats(StreamSmem &ss, int nr, int topk, float topp, RowStats st[2]) {
  using E = Elem<TIn>;
  const int tid = threadIdx.x;
  if (ss.cnt[0] <= 64 && (nr < 2 || ss.cnt[1] <= 64)) {
    warp_stats<TIn>(ss, nr, topk, topp, st);
    __syncthreads();
    for (int r = 0; r < nr; ++r) {
      st[r].cut = ss.cut[r];
      st[r].zp = static_cast<float>(static_cast<double>(ss.kept[r]) * (1.0 / static_cast<double>(kMassScale)));
    }
    __syncthreads();
    return;
  }
  const bool sel[2] = {true, nr > 1};
  uint32_t tk[2];
  const int cn[2] = {ss.cnt[0], ss.cnt[1]};
  radix_kth<E::kBits>(ss, sel, cn, topk, [&](int r, int i) -> uint32_t { return ss.key[r][i]; }, tk);
  cand_compact(ss, sel, tk);  // the top-k set (ties included) alone
  if (tid < 2) {
    ss.zk[tid] = 0ull;
    ss.kept[tid] = 0ull;
    ss.cut[tid] = tk[tid];
  }
  for (int r = 0; r < nr; ++r) {
    unsigned long long z = 0;
    for (int i = tid; i < ss.cnt[r]; i += kThreads) {
      const unsigned long long m =
          to_fixed(exp2f(__fmul_rn(__fsub_rn(E::val_of_key(ss.key[r][i]), st[r].vmax), st[r].c2)));
      ss.mass[r][i] = m;
      z += m;
    }
    block_add_u64(z, &ss.zk[r]);
  }
  __syncthreads();
  if (topp < 1.0f) {
    // the cut: the largest kept key c with mass(key >= c) >= need
    for (int r = 0; r < nr; ++r) {
      unsigned long long need =
          static_cast<unsigned long long>(static_cast<double>(topp) * static_cast<double>(ss.zk[r]));
      if (need == 0ull) need = 1ull;
      const int c = ss.cnt[r];
      for (int i = tid; i < c; i += kThreads) {
        const uint32_t ki = ss.key[r][i];
        unsigned long long m = 0;
        for (int j = 0; j < c; ++j)
          if (ss.key[r][j] >= ki) m += ss.mass[r][j];
        if (m >= need) atomicMax(&ss.cut[r], ki);
      }
    }
    __syncthreads();
    for (int r = 0; r < nr; ++r) {
      unsigned long long z = 0;
      for (int i = tid; i < ss.cnt[r]; i += kThreads)
        if (ss.key[r][i] >= ss.cut[r]) z += ss.mass[r][i];
      block_add_u64(z, &ss.kept[r]);
    }
    __syncthreads();
  }
  for (int r = 0; r < nr; ++r) {
    st[r].cut = ss.cut[r];
    const unsigned long long kept = topp < 1.0f ? ss.kept[r] : ss.zk[r];
    st[r].zp = static_cast<float>(static_cast<double>(kept) * (1.0 / static_cast<double>(kMassScale)));
  }
  __syncthreads();
}

// The race over the kept candidates of the target row (kResidual: of
// max(p - q, 0), with q looked up among the draft row's candidates).
// The value bits of an order key (the inverse of Elem<TIn>::key).
template <typename TIn>
__device__ __forceinline__ uint32_t bits_of_key(uint32_t k) {
  const uint32_t f = __float_as_uint(Elem<TIn>::val_of_key(k));
  return sizeof(TIn) == 2 ? (f >> 16) : f;  // (bf16 to fp32 is exact)
}

// Weight of a kept candidate (raw key k, index x) under a row's statistics;
// with kProc, its processed value (0 when banned).
template <typename TIn, bool kProc>
__device__ __forceinline__ float cand_weight(uint32_t k, int x, const RowStats &st, const Procs &pr) {
  if (kProc) return kept_weight<TIn>(processed_bits<TIn>(bits_of_key<TIn>(k), mark_at(pr, x), pr.theta), st);
  return exp2f(__fmul_rn(__fsub_rn(Elem<TIn>::val_of_key(k), st.vmax), st.c2));
}

template <typename TIn, bool kTest, bool kResidual, bool kProc = false>
__device__ __noinline__ void cand_race(const StreamSmem &ss, const RowStats &ps, const RowStats &qs, const float *Erow,
                          const RngKey &rk, uint32_t rs, float &bk, int &bx, uint32_t &flags, const Procs &pr) {
  const float rp = __frcp_rn(ps.zp), rq = __frcp_rn(qs.zp);
  for (int i = threadIdx.x; i < ss.cnt[0]; i += kThreads) {
    const uint32_t key = ss.key[0][i];
    if (key < ps.cut) continue;
    const int x = ss.idx[0][i];
    float w = __fmul_rn(cand_weight<TIn, kProc>(key, x, ps, pr), rp);
    if (kResidual) {
      float q = 0.0f;
      for (int j = 0; j < ss.cnt[1]; ++j) {
        if (ss.idx[1][j] != x) continue;
        const uint32_t kq = ss.key[1][j];
        if (kq >= qs.cut) q = __fmul_rn(cand_weight<TIn, kProc>(kq, x, qs, pr), rq);
        break;
      }
      w = __fsub_rn(w, q);
    }
    if (!(w > 0.0f)) continue;
    if (kTest) {
      const float Ex = Erow[x];
      if (!(Ex > 0.0f)) {
        flags |= SV_DATA_BAD_EXPONENTIAL;
        continue;
      }
      const float k = __fdiv_rn(w, Ex);
      if (k > bk || (k == bk && x < bx)) {
        bk = k;
        bx = x;
      }
    } else {
      const uint4 wd = draw_e_words(rk, rs, static_cast<uint32_t>(x) >> 2);
      const uint32_t word = (x & 3) == 0 ? wd.x : (x & 3) == 1 ? wd.y : (x & 3) == 2 ? wd.z : wd.w;
      const float U = e_word_to_open_uniform(word);
      const float k = __fdiv_rn(w, -logf(U));
      if (k > bk || (k == bk && x < bx)) {
        bk = k;
        bx = x;
      }
    }
  }
}

// The logits processors on the kept candidates ("vLLM source walk-through
// (10)", section "Rejection sampling: the two branches of RejectionSampler",
// step 2; "Speculative Decoding: propose, verify, accept", section 06): the
// kept set stays the one the raw statistics placed; each kept candidate takes
// its processed value (a banned one drops out), and the normaliser is summed
// afresh over them against the largest processed kept value, in 2^-40 fixed
// point as integers.  st[r].vmax / zp are replaced.  Returns false (a status
// bit is set) if a kept processed value is NaN or +inf, or no unbanned entry
// is kept.
template <typename TIn>
__device__ __noinline__ bool cand_process(StreamSmem &ss, int nr, const Procs &pr, RowStats st[2], uint32_t *req_bits) {
  using E = Elem<TIn>;
  const int tid = threadIdx.x;
  if (tid < 2) {
    ss.maxkey[tid] = 0u;
    ss.flags[tid] = 0u;
    ss.kept[tid] = 0ull;
  }
  __syncthreads();
  for (int r = 0; r < nr; ++r) {
    uint32_t mk = 0u, fl = 0u;
    for (int i = tid; i < ss.cnt[r]; i += kThreads) {
      const uint32_t key = ss.key[r][i];
      if (key < st[r].cut) continue;
      const uint32_t m = mark_at(pr, ss.idx[r][i]);
      if (m == 1u) continue;  // banned
      const uint32_t pb = processed_bits<TIn>(bits_of_key<TIn>(key), m, pr.theta);
      if (!E::finite(pb)) fl |= kFlagBad;  // (finite raw values only reach here)
      else mk = max(mk, E::key(pb) + 1u);  // +1: 0 means none
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      mk = max(mk, __shfl_xor_sync(0xFFFFFFFFu, mk, o));
      fl |= __shfl_xor_sync(0xFFFFFFFFu, fl, o);
    }
    if ((tid & 31) == 0) {
      atomicMax(&ss.maxkey[r], mk);
      atomicOr(&ss.flags[r], fl);
    }
  }
  __syncthreads();
  for (int r = 0; r < nr; ++r)
    if ((ss.flags[r] & kFlagBad) || ss.maxkey[r] == 0u) {
      *req_bits |= SV_DATA_BAD_VALUES;
      return false;
    }
  for (int r = 0; r < nr; ++r) {
    st[r].vmax = E::val_of_key(ss.maxkey[r] - 1u);
    unsigned long long z = 0;
    for (int i = tid; i < ss.cnt[r]; i += kThreads) {
      const uint32_t key = ss.key[r][i];
      if (key < st[r].cut) continue;
      const uint32_t m = mark_at(pr, ss.idx[r][i]);
      if (m == 1u) continue;
      z += to_fixed(kept_weight<TIn>(processed_bits<TIn>(bits_of_key<TIn>(key), m, pr.theta), st[r]));
    }
    block_add_u64(z, &ss.kept[r]);
  }
  __syncthreads();
  for (int r = 0; r < nr; ++r)
    st[r].zp = static_cast<float>(static_cast<double>(ss.kept[r]) * (1.0 / static_cast<double>(kMassScale)));
  __syncthreads();
  return true;
}

// Dynamic shared memory of the logits-entry form: the state, then with
// processors the banned and penalised bitmaps of the whole row and the
// inboxes the exact statistics' processor correction exchanges through.
__host__ __device__ constexpr size_t stream_bitmap_words(int V) { return (static_cast<size_t>(V) + 31) / 32; }
__host__ __device__ constexpr size_t stream_dyn_bytes(int V, bool procs) {
  return sizeof(StreamSmem) + (procs ? ((2 * stream_bitmap_words(V) * 4 + 15) & ~size_t{15}) + 2 * sizeof(Inbox) : 0);
}

// CTAs per SM of the logits-entry form: three (85 registers) measure faster
// than four on the fused batch (0.269 against 0.291 ms); the requests beyond
// the first wave start as the shortest walks finish.
constexpr int kStreamCtasPerSm = 3;

template <typename TIn, bool kTest, bool kProc>
__global__ void __launch_bounds__(kThreads, kStreamCtasPerSm) stream_kernel(const VerifyParams P) {
  pdl_enter();
  using E = Elem<TIn>;
  extern __shared__ __align__(16) unsigned char dyn_smem[];
  StreamSmem &ss = *reinterpret_cast<StreamSmem *>(dyn_smem);
  const int words = static_cast<int>(stream_bitmap_words(P.V));
  uint32_t *const pen_bits = reinterpret_cast<uint32_t *>(dyn_smem + sizeof(StreamSmem));  // (kProc only)
  uint32_t *const ban_bits = pen_bits + words;
  Inbox *const inbox = reinterpret_cast<Inbox *>(dyn_smem + sizeof(StreamSmem) +
                                                 ((2 * static_cast<size_t>(words) * 4 + 15) & ~size_t{15}));
  const int i = static_cast<int>(blockIdx.x);
  const int tid = threadIdx.x;
  const int G = P.G, V = P.V;
  const TIn *tgt = static_cast<const TIn *>(P.target);
  const TIn *drf = static_cast<const TIn *>(P.draft);
  const int64_t ts = P.target_stride, ds = P.draft_stride;

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
  int64_t stop_b = 0, stop_e = 0, pen_b = 0, pen_e = 0, ban_b = 0, ban_e = 0;
  if (valid && ((P.stop_cu && !list_range(P.stop_cu, P.stop_total, i, stop_b, stop_e)) ||
                (kProc && P.pen_cu && !list_range(P.pen_cu, P.pen_total, i, pen_b, pen_e)) ||
                (kProc && P.ban_cu && !list_range(P.ban_cu, P.ban_total, i, ban_b, ban_e)))) {
    req_bits |= SV_DATA_BAD_LIST;
    valid = false;
  }
  float theta = 1.0f;
  if (kProc && valid && P.rep_penalty) {
    theta = P.rep_penalty[i];
    if (!(theta > 0.0f) || isinf(theta)) {
      req_bits |= SV_DATA_BAD_PARAM;
      valid = false;
    }
  }
  const Procs pr{pen_bits, ban_bits, theta};
  auto mark = [&](uint32_t *bm, int32_t x) {
    if (x >= 0 && x < V) atomicOr(&bm[x >> 5], 1u << (x & 31));
  };
  int added = 0;  // drafts already in the penalty bitmap
  // position j penalises the drafts y_0 .. y_{j-1} too (they are committed by then)
  auto add_drafts = [&](int j) {
    if (kProc && P.rep_penalty) {
      for (; added < j; ++added)
        if (tid == 0) mark(pen_bits, P.ids[s + added]);
      __syncthreads();
    }
  };
  if (kProc && valid) {  // the whole row's banned and penalised keys
    for (int w = tid; w < 2 * words; w += kThreads) pen_bits[w] = 0u;
    __syncthreads();
    if (P.ban_cu)
      for (int64_t k = ban_b + tid; k < ban_e; k += kThreads) mark(ban_bits, P.ban_ids[k]);
    if (P.rep_penalty && P.pen_cu)
      for (int64_t k = pen_b + tid; k < pen_e; k += kThreads) mark(pen_bits, P.pen_ids[k]);
    __syncthreads();
  }
  const bool greedy = valid && temp == 0.0f;
  int A = 0;
  int32_t last_tok = -1;
  int step = 0;

  if (greedy) {
    for (int j = 0;; ++j) {
      unsigned long long best = 0;
      uint32_t fl = 0;
      if (kProc) {  // the argmax of the processed row
        add_drafts(j);
        argmax_proc<TIn>(tgt + (tb + j) * ts, 0, V, pr, best, fl);
      } else {
        argmax_logits<TIn, true>(tgt + (tb + j) * ts, 0, V, best, fl);
      }
      const KeyFlags r = cluster_reduce(KeyFlags{best, fl}, ss.red, step++, 1);
      if (r.flags & SV_DATA_BAD_VALUES) {
        req_bits |= SV_DATA_BAD_VALUES;
        valid = false;
        break;
      }
      const int gj = static_cast<int>(key_index(r.key));
      if (tid == 0) ss.tok[j] = gj;
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
    if (topk >= V || topk < 0) topk = 0;
    const float topp = P.top_p ? P.top_p[i] : 1.0f;
    if (!(topp > 0.0f)) {
      req_bits |= SV_DATA_BAD_PARAM;
      valid = false;
    } else {
      const float c2 = __fdiv_rn(kLog2e, temp);
      const RngKey rk{P.seed_lo, P.seed_hi, P.off_lo, P.off_hi};
      const uint32_t rs = P.req_base + static_cast<uint32_t>(i);
      const float *Erow = kTest ? P.exponentials + static_cast<int64_t>(i) * P.exp_stride : nullptr;
      const bool cand = topk > 0 && topk <= kStreamTopK && (V / (16 / static_cast<int>(sizeof(TIn))) + kStep - 1) / kStep <= kBlockSteps * (kMaxBlocks / kThreads);
      RowStats st[2];
      int j_start = 0;
      if (P.rates) {  // synthetic acceptance: the stopping position follows from u_j < rate_j alone
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
          if (tid == 0) ss.tok[j_start] = y;
        }
      }
      for (int j = j_start; valid; ++j) {
        const int nr = (j < g) ? 2 : 1;
        if (nr == 2 && drf == nullptr) {
          req_bits |= SV_DATA_MISSING_DRAFT;
          valid = false;
          break;
        }
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
        TIn *const rows[2] = {const_cast<TIn *>(tgt + (tb + j) * ts),
                              nr == 2 ? const_cast<TIn *>(drf + (s + j) * ds) : nullptr};
        add_drafts(j);
        if (cand)
          stream_pass<TIn, true>(ss, rows, nr, V, j >= 1 ? 4 : 0);
        else
          stream_pass<TIn, false>(ss, rows, nr, V, j >= 1 ? 4 : 0);
        for (int r = 0; r < nr; ++r) {
          const uint32_t f = ss.flags[r];
          if ((f & kFlagBad) || !(f & kFlagFinite)) {
            req_bits |= SV_DATA_BAD_VALUES;
            valid = false;
          }
          st[r].vmax = E::val_of_key(ss.maxkey[r]);
          st[r].c2 = c2;
          st[r].cut = 0u;
          st[r].zp = 0.0f;
        }
        if (!valid) break;
        if (cand) gather_candidates<TIn>(ss, rows, nr, V, topk);
        const bool fast = cand && !ss.overflow;
        if (fast) {
          cand_stats<TIn>(ss, nr, topk, topp, st);
        } else {  // every other setting: exact multi-pass statistics over the whole rows
          const uint32_t maxk16[2] = {key16_of<TIn>(ss.maxkey[0]), key16_of<TIn>(ss.maxkey[1])};
          stats_slow<TIn>(ss.fb, rows, nr, V, c2, topk, topp, maxk16, st, step, 1);
        }
        // the processors on the kept sets: their weights and normalisers, the draft token's marks
        uint32_t ymark = 0u;
        if (kProc) {
          if (fast) {
            if (!cand_process<TIn>(ss, nr, pr, st, &req_bits)) {
              valid = false;
              break;
            }
          } else if (!proc_correct<TIn>(ss.fb, inbox, rows, nr, V, words, pr, st,
                                        (j < g && y >= 0 && y < V) ? y : -1, ymark, &req_bits, step, 1, 0)) {
            valid = false;
            break;
          }
          ymark = (j < g && y >= 0 && y < V) ? mark_at(pr, y) : 0u;
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
          const float py = kProc ? prob_of_m<TIn>(bty, ymark, st[0], theta) : prob_of<TIn>(bty, st[0]);
          const float qy = kProc ? prob_of_m<TIn>(bdy, ymark, st[1], theta) : prob_of<TIn>(bdy, st[1]);
          if (tid == 0 && !P.rates) {
            if (P.dbg_py) P.dbg_py[s + j] = py;
            if (P.dbg_qy) P.dbg_qy[s + j] = qy;
          }
          if (!P.rates && __fmul_rn(u, qy) < py) {
            if (tid == 0) ss.tok[j] = y;
            continue;  // accepted: next position
          }
          residual = true;
          if (fast)
            cand_race<TIn, kTest, true, kProc>(ss, st[0], st[1], Erow, rk, rs, bk, bx, fl, pr);
          else
            race_chunks<TIn, kTest, true, kProc>(rows[0], rows[1], st[0], st[1], 0, V, Erow, rk, rs, bk, bx, fl, pr);
        } else if (fast) {
          cand_race<TIn, kTest, false, kProc>(ss, st[0], st[0], Erow, rk, rs, bk, bx, fl, pr);
        } else {
          race_chunks<TIn, kTest, false, kProc>(rows[0], rows[1], st[0], st[0], 0, V, Erow, rk, rs, bk, bx, fl, pr);
        }
        KeyFlags r = cluster_reduce(KeyFlags{bx >= 0 ? pack_key(bk, bx) : 0ull, fl}, ss.red, step++, 1);
        if (r.key == 0ull && residual) {  // no positive residual key: race over p with the same E
          bk = 0.0f;
          bx = -1;
          fl = 0;
          if (fast)
            cand_race<TIn, kTest, false, kProc>(ss, st[0], st[0], Erow, rk, rs, bk, bx, fl, pr);
          else
            race_chunks<TIn, kTest, false, kProc>(rows[0], rows[1], st[0], st[0], 0, V, Erow, rk, rs, bk, bx, fl, pr);
          const KeyFlags r2 = cluster_reduce(KeyFlags{bx >= 0 ? pack_key(bk, bx) : 0ull, fl}, ss.red, step++, 1);
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
  __syncthreads();
  const int A0 = A;
  auto tok = [&](int k) -> int32_t { return (k == A0 && !greedy) ? last_tok : ss.tok[k]; };
  if (valid && P.stop_cu) A = stop_commit(A0, tok, P.stop_ids, stop_b, stop_e, &ss.stop_first);
  emit_request(i, G, g, A, valid, tb, req_bits, tok, P.out, P.nacc, P.ncomp, P.slots, P.status);
}

template <typename TIn, bool kTest, bool kProc>
cudaError_t launch_stream_one(const VerifyParams &p, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p.N), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = stream_dyn_bytes(p.V, kProc);
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];  // a cluster of one (the fallback paths use cluster barriers)
  cfg.attrs = attr;
  cfg.numAttrs = launch_attrs(attr, 1, p.pdl);
  return cudaLaunchKernelEx(&cfg, stream_kernel<TIn, kTest, kProc>, p);
}

// The draft-side sampler in the same form: one CTA per row ("vLLM source
// walk-through (10)", section "propose() multi-step loop": each draft step
// samples its token from the transformed draft row).  The row is read once
// with its block maxima, the candidates give the threshold, cut and
// normaliser, and the bonus-style race runs over the kept candidates; the
// transformed fp32 row, if asked for, is written from a second read of the
// row (from L2).  Rows outside the candidate path take the exact statistics
// and the race over the whole row.  The same results as sample_kernel.
template <typename TIn, bool kTest, bool kProc>
__global__ void __launch_bounds__(kThreads, 4) stream_sample_kernel(const SampleParams P) {
  pdl_enter();
  using E = Elem<TIn>;
  extern __shared__ __align__(16) unsigned char dyn_smem[];
  StreamSmem &ss = *reinterpret_cast<StreamSmem *>(dyn_smem);
  const int r = static_cast<int>(blockIdx.x);
  const int tid = threadIdx.x;
  const int V = P.V;
  TIn *const row = const_cast<TIn *>(static_cast<const TIn *>(P.logits) + static_cast<int64_t>(r) * P.row_stride);
  TIn *const rows[2] = {row, row};
  // with processors: the row's banned and penalised bitmaps, then the inboxes (as the logits entry)
  const int words = static_cast<int>(stream_bitmap_words(V));
  uint32_t *const pen_bits = reinterpret_cast<uint32_t *>(dyn_smem + sizeof(StreamSmem));
  uint32_t *const ban_bits = pen_bits + words;
  Inbox *const inbox = reinterpret_cast<Inbox *>(dyn_smem + sizeof(StreamSmem) +
                                                 ((2 * static_cast<size_t>(words) * 4 + 15) & ~size_t{15}));
  uint32_t bits = 0;
  int32_t token = -1;
  int step = 0;
  const float temp = P.temperature ? P.temperature[r] : 1.0f;
  bool ok = temperature_ok(temp);
  if (!ok) bits |= SV_DATA_BAD_PARAM;
  int64_t pen_b = 0, pen_e = 0, ban_b = 0, ban_e = 0;
  if (kProc && ok && ((P.pen_cu && !list_range(P.pen_cu, P.pen_total, r, pen_b, pen_e)) ||
                      (P.ban_cu && !list_range(P.ban_cu, P.ban_total, r, ban_b, ban_e)))) {
    bits |= SV_DATA_BAD_LIST;
    ok = false;
  }
  float theta = 1.0f;
  if (kProc && ok && P.rep_penalty) {
    theta = P.rep_penalty[r];
    if (!(theta > 0.0f) || isinf(theta)) {
      bits |= SV_DATA_BAD_PARAM;
      ok = false;
    }
  }
  const Procs pr{pen_bits, ban_bits, theta};
  if (kProc && ok) {  // the row's banned and penalised keys
    auto mark = [&](uint32_t *bm, int32_t x) {
      if (x >= 0 && x < V) atomicOr(&bm[x >> 5], 1u << (x & 31));
    };
    for (int w = tid; w < 2 * words; w += kThreads) pen_bits[w] = 0u;
    __syncthreads();
    if (P.ban_cu)
      for (int64_t k = ban_b + tid; k < ban_e; k += kThreads) mark(ban_bits, P.ban_ids[k]);
    if (P.rep_penalty && P.pen_cu)
      for (int64_t k = pen_b + tid; k < pen_e; k += kThreads) mark(pen_bits, P.pen_ids[k]);
    __syncthreads();
  }
  if (!ok) {
    // nothing sampled
  } else if (temp == 0.0f) {
    unsigned long long best = 0;
    uint32_t fl = 0;
    if (kProc)  // the argmax of the processed row
      argmax_proc<TIn>(row, 0, V, pr, best, fl);
    else
      argmax_logits<TIn, true>(row, 0, V, best, fl);
    const KeyFlags kr = cluster_reduce(KeyFlags{best, fl}, ss.red, step++, 1);
    if (kr.flags & SV_DATA_BAD_VALUES) bits |= SV_DATA_BAD_VALUES;
    else token = static_cast<int32_t>(key_index(kr.key));
  } else {
    int topk = P.top_k ? P.top_k[r] : 0;
    if (topk >= V || topk < 0) topk = 0;
    const float topp = P.top_p ? P.top_p[r] : 1.0f;
    if (!(topp > 0.0f)) {
      bits |= SV_DATA_BAD_PARAM;
    } else {
      const bool cand = topk > 0 && topk <= kStreamTopK &&
                        (V / (16 / static_cast<int>(sizeof(TIn))) + kStep - 1) / kStep <=
                            kBlockSteps * (kMaxBlocks / kThreads);
      if (cand)
        stream_pass<TIn, true>(ss, rows, 1, V, 0);
      else
        stream_pass<TIn, false>(ss, rows, 1, V, 0);
      const uint32_t f = ss.flags[0];
      if ((f & kFlagBad) || !(f & kFlagFinite)) {
        bits |= SV_DATA_BAD_VALUES;
      } else {
        RowStats st[2];
        for (int q = 0; q < 2; ++q) {
          st[q].vmax = E::val_of_key(ss.maxkey[0]);
          st[q].c2 = __fdiv_rn(kLog2e, temp);
          st[q].cut = 0u;
          st[q].zp = 0.0f;
        }
        if (cand) gather_candidates<TIn>(ss, rows, 1, V, topk);
        const bool fast = cand && !ss.overflow;
        if (fast) {
          cand_stats<TIn>(ss, 1, topk, topp, st);
        } else {
          const uint32_t maxk16[2] = {key16_of<TIn>(ss.maxkey[0]), key16_of<TIn>(ss.maxkey[0])};
          stats_slow<TIn>(ss.fb, rows, 1, V, st[0].c2, topk, topp, maxk16, st, step, 1);
        }
        bool live = true;  // (false: the processors left no distribution; the status bit is set)
        if (kProc) {
          uint32_t ymark = 0u;
          live = fast ? cand_process<TIn>(ss, 1, pr, st, &bits)
                      : proc_correct<TIn>(ss.fb, inbox, rows, 1, V, words, pr, st, -1, ymark, &bits, step, 1, 0);
        }
        if (live) {
          const RngKey rk{P.seed_lo, P.seed_hi ^ 0x53414D50u, P.off_lo, P.off_hi};  // the sampler's own streams
          const uint32_t rs = P.row_base + static_cast<uint32_t>(r);
          const float *Erow = kTest ? P.exponentials + static_cast<int64_t>(r) * P.exp_stride : nullptr;
          float bk = 0.0f;
          int bx = -1;
          uint32_t fl = 0;
          if (fast)
            cand_race<TIn, kTest, false, kProc>(ss, st[0], st[0], Erow, rk, rs, bk, bx, fl, pr);
          else
            race_chunks<TIn, kTest, false, kProc>(row, row, st[0], st[0], 0, V, Erow, rk, rs, bk, bx, fl, pr);
          const KeyFlags kr = cluster_reduce(KeyFlags{bx >= 0 ? pack_key(bk, bx) : 0ull, fl}, ss.red, step++, 1);
          bits |= kr.flags;
          if (kr.key == 0ull) {
            bits |= SV_DATA_EMPTY_DISTRIBUTION;
            token = 0;
          } else {
            token = static_cast<int32_t>(key_index(kr.key));
          }
          if (P.probs) {  // the transformed row
            float *prow = P.probs + static_cast<int64_t>(r) * P.probs_stride;
            int xs = 0;
            if (sizeof(TIn) == 2 && (reinterpret_cast<uintptr_t>(prow) & 15u) == 0) {
              // eight bf16 logits in, two float4 probabilities out
              const uint4 *s4 = reinterpret_cast<const uint4 *>(row);
              float4 *p4 = reinterpret_cast<float4 *>(prow);
              const int ng = V >> 3;
              for (int v = tid; v < ng; v += kThreads) {
                const uint4 d = ld_stream_u4(s4 + v);
                const uint32_t w[4] = {d.x, d.y, d.z, d.w};
                float o[8];
  #pragma unroll
                for (int t = 0; t < 4; ++t) {
                  o[2 * t] = prob_of<TIn>(w[t] & 0xFFFFu, st[0]);
                  o[2 * t + 1] = prob_of<TIn>(w[t] >> 16, st[0]);
                }
                if (kProc) {  // marked entries: their processed probabilities
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
            for (int x = xs + tid; x < V; x += kThreads)
              prow[x] = kProc ? prob_of_m<TIn>(bits_at(row, x), mark_at(pr, x), st[0], theta)
                              : prob_of<TIn>(bits_at(row, x), st[0]);
          }
        }
      }
    }
  }
  if (tid == 0) {
    P.tokens[r] = token;
    if (bits && P.status) atomicOr(P.status, static_cast<int>(bits));
  }
}

template <typename TIn, bool kTest, bool kProc>
cudaError_t launch_stream_sample_one(const SampleParams &p, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p.R), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = stream_dyn_bytes(p.V, kProc);
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];  // a cluster of one (the exact statistics use cluster barriers)
  cfg.attrs = attr;
  cfg.numAttrs = launch_attrs(attr, 1, p.pdl);
  return cudaLaunchKernelEx(&cfg, stream_sample_kernel<TIn, kTest, kProc>, p);
}

// max_dyn: the dynamic shared memory the processor form may request (its row bitmaps grow with V)
template <typename TIn, bool kProc>
cudaError_t enable_type_stream(int max_dyn) {
  const int dyn = kProc ? max_dyn : static_cast<int>(sizeof(StreamSmem));
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(stream_kernel<TIn, true, kProc>, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn)) !=
      cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(stream_kernel<TIn, false, kProc>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                dyn)) != cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(stream_sample_kernel<TIn, true, kProc>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                dyn)) != cudaSuccess)
    return e;
  return cudaFuncSetAttribute(stream_sample_kernel<TIn, false, kProc>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              dyn);
}

template <typename TIn, bool kProc>
cudaError_t launch_type_stream(const VerifyParams &p, cudaStream_t stream) {
  return p.exponentials != nullptr ? launch_stream_one<TIn, true, kProc>(p, stream)
                                   : launch_stream_one<TIn, false, kProc>(p, stream);
}

template <typename TIn, bool kProc>
cudaError_t launch_type_stream_sample(const SampleParams &p, cudaStream_t stream) {
  return p.exponentials != nullptr ? launch_stream_sample_one<TIn, true, kProc>(p, stream)
                                   : launch_stream_sample_one<TIn, false, kProc>(p, stream);
}

}  // namespace
}  // namespace sv
