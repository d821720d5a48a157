// sv_device.cuh -- device building blocks shared by the verifier kernels:
// thread-block-cluster primitives (inline PTX), streaming loads, the
// Philox4x32-10 counter generator, packed argmax keys and the warp / block /
// cluster max-reductions over them.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace sv {

constexpr int kThreads = 256;  // threads per CTA of every verifier kernel
constexpr int kWarps = kThreads / 32;

// ---------------------------------------------------------------------------
// cluster primitives (sm_90+ PTX; the kernels here are always launched with a
// cluster dimension, a cluster of one CTA included)
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_nctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
// Full cluster barrier: release our shared-memory writes, acquire the peers'.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
               "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Programmatic dependent launch (sm_90+): the kernels are launched so that
// they may be scheduled while the previous kernel in the stream is still
// running.  The first statement of every kernel waits until that grid has
// completed and its memory operations are visible (at once when the launch
// carried no such attribute), so nothing is read or written earlier than
// under plain stream order; it then lets the next kernel in the stream be
// scheduled in the same way.
__device__ __forceinline__ void pdl_enter() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
// Split form: arrive early (nothing to publish), wait later.
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
// Address of the same shared-memory variable in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
  return r;
}
__device__ __forceinline__ unsigned long long ld_dsmem_u64(uint32_t addr) {
  unsigned long long v;
  asm volatile("ld.shared::cluster.u64 %0, [%1];" : "=l"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ void st_dsmem_v4(uint32_t addr, uint4 v) {
  asm volatile("st.shared::cluster.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}
__device__ __forceinline__ uint32_t ld_dsmem_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}

// ---------------------------------------------------------------------------
// streaming loads: read-once rows bypass L1 allocation
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint4 ld_stream_u4(const uint4 *p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ float4 ld_stream_f4(const float4 *p) {
  float4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ float ld_stream_f1(const float *p) {
  float v;
  asm volatile("ld.global.nc.L1::no_allocate.f32 %0, [%1];" : "=f"(v) : "l"(p));
  return v;
}

// ---------------------------------------------------------------------------
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11): ten rounds of two 32x32
// multiplies with the round keys bumped by the Weyl constants in between.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r > 0) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    const uint32_t lo0 = 0xD2511F53u * c.x, hi0 = __umulhi(0xD2511F53u, c.x);
    const uint32_t lo1 = 0xCD9E8D57u * c.z, hi1 = __umulhi(0xCD9E8D57u, c.z);
    c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
  }
  return c;
}

struct RngKey {
  uint32_t k0, k1, off_lo, off_hi;
};

// u_j of request stream r: [0, 1) on the 2^-24 grid.
__device__ __forceinline__ float draw_uniform(const RngKey &k, uint32_t r, uint32_t j) {
  const uint4 w = philox4x32_10(make_uint4(j >> 2, 2u * r + 1u, k.off_lo, k.off_hi), k.k0, k.k1);
  const uint32_t word = (j & 3u) == 0 ? w.x : (j & 3u) == 1 ? w.y : (j & 3u) == 2 ? w.z : w.w;
  return static_cast<float>(word >> 8) * 0x1p-24f;
}
// Four E-stream words for vocabulary entries 4*quad .. 4*quad+3 of stream r.
__device__ __forceinline__ uint4 draw_e_words(const RngKey &k, uint32_t r, uint32_t quad) {
  return philox4x32_10(make_uint4(quad, 2u * r, k.off_lo, k.off_hi), k.k0, k.k1);
}
// U in (0, 1), odd multiples of 2^-24 (exact in fp32), so 1 - U is exact too.
__device__ __forceinline__ float e_word_to_open_uniform(uint32_t w) {
  return static_cast<float>(2u * (w >> 9) + 1u) * 0x1p-24f;
}

// ---------------------------------------------------------------------------
// packed argmax keys: high word = order-preserving image of the value
// (-0 and +0 equal), low word = ~index, so a u64 max picks the largest value
// and, among equal values, the lowest index.  0 means "no candidate".
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t ordered_bits(float v) {
  const uint32_t b = __float_as_uint(v == 0.0f ? 0.0f : v);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ unsigned long long pack_key(float v, uint32_t idx) {
  return (static_cast<unsigned long long>(ordered_bits(v)) << 32) | static_cast<unsigned long long>(~idx);
}
__device__ __forceinline__ uint32_t key_index(unsigned long long k) {
  return ~static_cast<uint32_t>(k & 0xFFFFFFFFull);
}
__device__ __forceinline__ unsigned long long umax64(unsigned long long a, unsigned long long b) {
  return a > b ? a : b;
}

struct KeyFlags {
  unsigned long long key;
  uint32_t flags;
};

__device__ __forceinline__ KeyFlags warp_reduce(KeyFlags v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    v.key = umax64(v.key, __shfl_xor_sync(0xFFFFFFFFu, v.key, o));
    v.flags |= __shfl_xor_sync(0xFFFFFFFFu, v.flags, o);
  }
  return v;
}

// Shared-memory staging for block and cluster reductions.  `slot` is the value
// this CTA publishes to its cluster peers; it is double-buffered by step
// parity so that one cluster barrier per step suffices.
struct ReduceSmem {
  unsigned long long warp_key[kWarps];
  uint32_t warp_flags[kWarps];
  unsigned long long slot_key[2];
  uint32_t slot_flags[2];
  unsigned long long result_key;
  uint32_t result_flags;
};

// Reduce `v` over the CTA, then over the cluster.  Every thread of every CTA
// of the cluster returns the same value.  Must be called by all threads of all
// CTAs of the cluster the same number of times (it contains one cluster barrier).
__device__ __forceinline__ KeyFlags cluster_reduce(KeyFlags v, ReduceSmem &sm, int step, uint32_t ncta) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int par = step & 1;
  v = warp_reduce(v);
  if (lane == 0) {
    sm.warp_key[warp] = v.key;
    sm.warp_flags[warp] = v.flags;
  }
  __syncthreads();
  if (warp == 0) {
    KeyFlags w{lane < kWarps ? sm.warp_key[lane] : 0ull, lane < kWarps ? sm.warp_flags[lane] : 0u};
    w = warp_reduce(w);
    if (lane == 0) {
      sm.slot_key[par] = w.key;
      sm.slot_flags[par] = w.flags;
    }
  }
  cluster_sync();
  if (warp == 0) {
    KeyFlags w{0ull, 0u};
    if (lane < static_cast<int>(ncta)) {
      w.key = ld_dsmem_u64(map_to_rank(smem_addr(&sm.slot_key[par]), lane));
      w.flags = ld_dsmem_u32(map_to_rank(smem_addr(&sm.slot_flags[par]), lane));
    }
    w = warp_reduce(w);
    if (lane == 0) {
      sm.result_key = w.key;
      sm.result_flags = w.flags;
    }
  }
  __syncthreads();
  return KeyFlags{sm.result_key, sm.result_flags};
}

// Chunk [x0, x1) of a V-long row handled by CTA `rank` of `ncta`; chunk starts
// are multiples of 4 elements so aligned rows stay 16-byte aligned per chunk.
__device__ __forceinline__ void chunk_of(int V, uint32_t rank, uint32_t ncta, int &x0, int &x1) {
  const int per = ((V + static_cast<int>(ncta) - 1) / static_cast<int>(ncta) + 3) & ~3;
  x0 = min(V, static_cast<int>(rank) * per);
  x1 = min(V, x0 + per);
}

}  // namespace sv

namespace sv {

// Committed tokens, num_accepted and the KV rollback of request i, written by
// the whole CTA that calls it (the cluster's first CTA).  tok(k) yields the
// k-th committed token for k <= A.  ("Rejection sampling ... RejectionSampler":
// output [batch, max_spec_len + 1] padded with -1; "How speculative decoding
// interacts with the KV cache" 3.1: num_computed_tokens -= gamma - A when > 0;
// rejected drafts' slots -> PADDING_SLOT_ID.)
// Stop tokens checked on the committed prefix only ("Speculative Decoding:
// propose, verify, accept", sections 13-14): the commit c_0 .. c_A ends at
// the first c_m in the request's stop list [b, e).  Called by every thread of
// the emitting CTA; returns the new A.  *first is one shared-memory word.
template <typename TokFn>
__device__ __forceinline__ int stop_commit(int A, TokFn tok, const int32_t *ids, int64_t b, int64_t e, int *first) {
  if (threadIdx.x == 0) *first = A;
  __syncthreads();
  for (int m = threadIdx.x; m <= A; m += kThreads) {
    const int32_t t = tok(m);
    for (int64_t k = b; k < e; ++k)
      if (ids[k] == t) {
        atomicMin(first, m);
        break;
      }
  }
  __syncthreads();
  return *first;
}

// A usable temperature: 0 (the greedy path) or a finite value of at least
// FLT_MIN; negative, NaN, infinite and subnormal ones are bad parameters (the
// reciprocal of a subnormal temperature leaves the fp32 range).
__device__ __forceinline__ bool temperature_ok(float t) {
  return t == 0.0f || (t >= __uint_as_float(0x00800000u) && !isinf(t));
}

// A per-request list range [b, e) (inclusive prefix sums, like
// cu_num_draft_tokens); false if it is not inside [0, total].
__device__ __forceinline__ bool list_range(const int64_t *cu, int64_t total, int i, int64_t &b, int64_t &e) {
  b = i ? cu[i - 1] : 0;
  e = cu[i];
  return b >= 0 && e >= b && e <= total;
}

template <typename TokFn>
__device__ __forceinline__ void emit_request(int i, int G, int g, int A, bool valid, int64_t tb, uint32_t req_bits,
                                             TokFn tok, int32_t *out, int32_t *nacc, int32_t *ncomp,
                                             int64_t *slots, int32_t *status) {
  const int tid = threadIdx.x;
  const int row_len = G + 1;
  int32_t *orow = out + static_cast<int64_t>(i) * row_len;
  for (int k = tid; k < row_len; k += kThreads) orow[k] = (valid && k <= A) ? tok(k) : -1;
  if (valid && slots)
    for (int j = A + 1 + tid; j <= g; j += kThreads) slots[tb + j] = -1;
  if (tid == 0) {
    nacc[i] = valid ? A : 0;
    if (valid && ncomp && ncomp[i] > 0) ncomp[i] -= (g - A);
    if (req_bits && status) atomicOr(status, static_cast<int>(req_bits));
  }
}

}  // namespace sv

namespace sv {

// ---------------------------------------------------------------------------
// 1-D bulk copies (TMA) global -> shared, completing on an mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
// Order this thread's earlier generic-proxy shared-memory accesses before
// later async-proxy (bulk copy) writes to the same memory.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}
// Bulk prefetch of `bytes` (a multiple of 16, 16-byte aligned) into L2.
__device__ __forceinline__ void prefetch_l2(const void *src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.b32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Wait for phase `parity` of the barrier, giving up after `limit` polls
// (each poll may itself suspend for a while).  Returns false on give-up.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity, uint32_t limit) {
  for (uint32_t it = 0; it < limit; ++it)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

}  // namespace sv
