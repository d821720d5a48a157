// sv_probs.cu -- verifier kernel for the probability entry (fp32 p and q rows).
//
// One thread-block cluster per request ("one program per request" of the
// greedy/random kernels in "vLLM source walk-through (10)", section "Greedy
// kernel"), with the V-long row split into equal chunks across the cluster's
// CTAs so that a batch of a few hundred requests fills all SMs.
//
// Random requests (temperature != 0):
//   a2  every CTA gathers p_j(y_j), q_j(y_j) for all j < gamma_i in parallel
//       (one thread per position) and finds the first j whose test
//       fl32(u_j * q) < p fails ("Speculative Decoding: propose, verify,
//       accept", sections 04 and 06);
//   a3  at a rejection, each CTA streams its chunk of the row pair
//       (p[A], q[A]) once with 128-bit loads and keeps the best race key
//       w(x)/E(x), w = max(p - q, 0) (section 04's residual, unnormalised, and
//       the exponential race of the walk-through's "Random kernel" section);
//   a4  when all are accepted the same race runs over p[gamma_i] (bonus);
//   the per-CTA keys meet in a DSMEM max-reduction; if no residual key is
//   positive the race is rerun over p with the same E.
// Greedy requests (temperature 0): row by row, cluster-wide argmax of p_j
// (lowest index on ties), stop at the first mismatch with y_j (section 03).
// Rank 0 of the cluster writes the committed tokens, num_accepted and the KV
// rollback ("How speculative decoding interacts with the KV cache", 3.1).
//
// Production-mode E(x) = -ln U(x) comes from Philox only where w(x) > 0, and
// only when the cheap bound w/(1-U) >= w/E could beat the thread's current
// best key (a skipped entry can never win, so the result is unchanged).
#include <cmath>

#include "sv_device.cuh"
#include "sv_internal.h"

namespace sv {
namespace {

constexpr int kUnroll = 4;  // float4 loads in flight per row per thread

struct ProbsSmem {
  ReduceSmem red;
  int stop;       // first position whose test stops the scan (gamma_i if none)
  int stop_bad;   // that position has an invalid draft id
  int bad_rates;  // synthetic rates outside [0, 1] or increasing
  int stop_first; // first committed stop token
  int32_t tok[SV_MAX_SPEC_LEN + 1];
};

template <bool kResidual>
__device__ __forceinline__ float race_weight(float p, float q) {
  if (kResidual) {
    const float d = __fsub_rn(p, q);
    return d > 0.0f ? d : 0.0f;
  }
  return p > 0.0f ? p : 0.0f;
}

// Production-mode candidate: E from the Philox word, with the bound test first.
__device__ __forceinline__ void consider_drawn(float w, uint32_t word, int x, float &bk, int &bx) {
  const float U = e_word_to_open_uniform(word);
  const float om = 1.0f - U;  // exact: U is an odd multiple of 2^-24
  if (__fmaf_rn(bk, om, -w) > 0.0f) return;  // w / (1-U) < bk, and E >= 1-U
  const float E = -logf(U);
  const float key = __fdiv_rn(w, E);
  if (key > bk) {
    bk = key;
    bx = x;
  }
}

__device__ __forceinline__ void consider_given(float w, float E, int x, float &bk, int &bx, uint32_t &flags) {
  if (!(E > 0.0f)) {
    flags |= SV_DATA_BAD_EXPONENTIAL;
    return;
  }
  const float key = __fdiv_rn(w, E);
  if (key > bk) {
    bk = key;
    bx = x;
  }
}

__device__ __forceinline__ uint32_t word_of(const uint4 &w, int lane) {
  return lane == 0 ? w.x : lane == 1 ? w.y : lane == 2 ? w.z : w.w;
}

template <bool kTest, bool kResidual>
__device__ __forceinline__ void race_quad(const float4 &pv, const float4 &qv, int x, const float *Erow,
                                          const RngKey &rk, uint32_t rs, float &bk, int &bx, uint32_t &flags) {
  const float w0 = race_weight<kResidual>(pv.x, qv.x), w1 = race_weight<kResidual>(pv.y, qv.y);
  const float w2 = race_weight<kResidual>(pv.z, qv.z), w3 = race_weight<kResidual>(pv.w, qv.w);
  if (!(w0 > 0.0f || w1 > 0.0f || w2 > 0.0f || w3 > 0.0f)) return;
  if (kTest) {
    if (w0 > 0.0f) consider_given(w0, Erow[x + 0], x + 0, bk, bx, flags);
    if (w1 > 0.0f) consider_given(w1, Erow[x + 1], x + 1, bk, bx, flags);
    if (w2 > 0.0f) consider_given(w2, Erow[x + 2], x + 2, bk, bx, flags);
    if (w3 > 0.0f) consider_given(w3, Erow[x + 3], x + 3, bk, bx, flags);
  } else {
    const uint4 wd = draw_e_words(rk, rs, static_cast<uint32_t>(x) >> 2);
    if (w0 > 0.0f) consider_drawn(w0, wd.x, x + 0, bk, bx);
    if (w1 > 0.0f) consider_drawn(w1, wd.y, x + 1, bk, bx);
    if (w2 > 0.0f) consider_drawn(w2, wd.z, x + 2, bk, bx);
    if (w3 > 0.0f) consider_drawn(w3, wd.w, x + 3, bk, bx);
  }
}

template <bool kTest, bool kResidual>
__device__ __forceinline__ void race_scalar(float p, float q, int x, const float *Erow, const RngKey &rk,
                                            uint32_t rs, float &bk, int &bx, uint32_t &flags) {
  const float w = race_weight<kResidual>(p, q);
  if (!(w > 0.0f)) return;
  if (kTest) {
    consider_given(w, Erow[x], x, bk, bx, flags);
  } else {
    const uint4 wd = draw_e_words(rk, rs, static_cast<uint32_t>(x) >> 2);
    consider_drawn(w, word_of(wd, x & 3), x, bk, bx);
  }
}

// Thread-local race over this CTA's chunk [x0, x1).  Each thread visits its
// entries in increasing x, so the strict '>' keeps its lowest index on ties.
template <bool kTest, bool kResidual, bool kVec>
__device__ __forceinline__ void race_chunk(const float *prow, const float *qrow, int x0, int x1, const float *Erow,
                                           const RngKey &rk, uint32_t rs, float &bk, int &bx, uint32_t &flags) {
  const int tid = threadIdx.x;
  int xs = x0;
  if (kVec) {
    const int nq = (x1 - x0) >> 2;
    const float4 *p4 = reinterpret_cast<const float4 *>(prow + x0);
    const float4 *q4 = reinterpret_cast<const float4 *>((kResidual ? qrow : prow) + x0);
    for (int b = tid; b < nq; b += kThreads * kUnroll) {
      float4 pv[kUnroll], qv[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int k = b + u * kThreads;
        if (k < nq) {
          pv[u] = ld_stream_f4(p4 + k);
          qv[u] = kResidual ? ld_stream_f4(q4 + k) : pv[u];
        }
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int k = b + u * kThreads;
        if (k < nq) race_quad<kTest, kResidual>(pv[u], qv[u], x0 + 4 * k, Erow, rk, rs, bk, bx, flags);
      }
    }
    xs = x0 + 4 * nq;
  }
  for (int x = xs + tid; x < x1; x += kThreads) {
    const float pv = ld_stream_f1(prow + x);
    const float qv = kResidual ? ld_stream_f1(qrow + x) : pv;
    race_scalar<kTest, kResidual>(pv, qv, x, Erow, rk, rs, bk, bx, flags);
  }
}

// Thread-local argmax of a probability row chunk (greedy path).
template <bool kVec>
__device__ __forceinline__ void argmax_chunk(const float *row, int x0, int x1, unsigned long long &best,
                                             uint32_t &flags) {
  const int tid = threadIdx.x;
  int xs = x0;
  if (kVec) {
    const int nq = (x1 - x0) >> 2;
    const float4 *r4 = reinterpret_cast<const float4 *>(row + x0);
    for (int b = tid; b < nq; b += kThreads * kUnroll) {
      float4 v[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u)
        if (b + u * kThreads < nq) v[u] = ld_stream_f4(r4 + b + u * kThreads);
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int k = b + u * kThreads;
        if (k < nq) {
          const int x = x0 + 4 * k;
          const float e[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            if (isnan(e[t])) flags |= SV_DATA_BAD_VALUES;
            else best = umax64(best, pack_key(e[t], static_cast<uint32_t>(x + t)));
          }
        }
      }
    }
    xs = x0 + 4 * nq;
  }
  for (int x = xs + tid; x < x1; x += kThreads) {
    const float e = ld_stream_f1(row + x);
    if (isnan(e)) flags |= SV_DATA_BAD_VALUES;
    else best = umax64(best, pack_key(e, static_cast<uint32_t>(x)));
  }
}

template <bool kTest, bool kVec>
__global__ void __launch_bounds__(kThreads, 4) probs_kernel(const VerifyParams P) {
  pdl_enter();
  __shared__ ProbsSmem sm;
  const uint32_t ncta = cluster_nctarank(), rank = cluster_ctarank();
  const int i = static_cast<int>(blockIdx.x / ncta);
  const int tid = threadIdx.x;
  const int G = P.G, V = P.V;
  const float *p = static_cast<const float *>(P.target);
  const float *q = static_cast<const float *>(P.draft);
  const int64_t ts = P.target_stride, ds = P.draft_stride;

  // a0: ragged decode ("SpecDecodeMetadata": cu_num_draft_tokens)
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
  const int64_t tb = s + i;  // first target row of request i
  const float temp = P.temperature ? P.temperature[i] : 1.0f;
  if (valid && !temperature_ok(temp)) {
    req_bits |= SV_DATA_BAD_PARAM;
    valid = false;
  }
  int64_t stop_b = 0, stop_e = 0;
  if (valid && P.stop_cu && !list_range(P.stop_cu, P.stop_total, i, stop_b, stop_e)) {
    req_bits |= SV_DATA_BAD_LIST;
    valid = false;
  }
  const bool greedy = valid && temp == 0.0f;

  int x0, x1;
  chunk_of(V, rank, ncta, x0, x1);
  int A = 0;
  int32_t last_tok = -1;
  int step = 0;

  if (greedy) {
    for (int j = 0;; ++j) {
      unsigned long long best = 0;
      uint32_t fl = 0;
      argmax_chunk<kVec>(p + (tb + j) * ts, x0, x1, best, fl);
      const KeyFlags r = cluster_reduce(KeyFlags{best, fl}, sm.red, step++, ncta);
      if (r.flags & SV_DATA_BAD_VALUES) {
        req_bits |= SV_DATA_BAD_VALUES;
        valid = false;
        break;
      }
      const int gj = static_cast<int>(key_index(r.key));
      if (tid == 0) sm.tok[j] = gj;
      if (j == g) {  // every draft matched: the last row's argmax is the bonus
        A = g;
        break;
      }
      const int y = P.ids[s + j];
      if (y < 0 || y >= V) {
        req_bits |= SV_DATA_BAD_DRAFT_ID;
        valid = false;
        break;
      }
      if (y != gj) {  // first mismatch: the target's argmax replaces it
        A = j;
        break;
      }
    }
  } else if (valid) {
    if (g > 0 && q == nullptr) {
      req_bits |= SV_DATA_MISSING_DRAFT;
      valid = false;
    } else {
      const RngKey rk{P.seed_lo, P.seed_hi, P.off_lo, P.off_hi};
      const uint32_t rs = P.req_base + static_cast<uint32_t>(i);
      if (tid == 0) {
        sm.stop = g;
        sm.stop_bad = 0;
        sm.bad_rates = 0;
      }
      __syncthreads();
      // a2: gather-and-accept scan, all positions at once (synthetic mode:
      // the preset rate replaces the probability test and nothing is gathered)
      const float *rates = P.rates;
      float py = 0.0f, qy = 0.0f;
      bool bad = false;
      if (tid < g) {
        const int y = P.ids[s + tid];
        bad = (y < 0 || y >= V);
        bool stop = bad;
        const float u = kTest ? P.uniforms[s + tid] : draw_uniform(rk, rs, static_cast<uint32_t>(tid));
        if (rates) {
          const float rj = rates[tid];
          if (!(rj >= 0.0f && rj <= 1.0f) || (tid > 0 && rj > rates[tid - 1])) sm.bad_rates = 1;
          if (!bad) stop = !(u < rj);
        } else if (!bad) {
          py = p[(tb + tid) * ts + y];
          qy = q[(s + tid) * ds + y];
          stop = !(__fmul_rn(u, qy) < py);
        }
        if (stop) atomicMin(&sm.stop, tid);
      }
      __syncthreads();
      const int a = sm.stop;
      if (tid == a && bad) sm.stop_bad = 1;
      __syncthreads();
      if (sm.bad_rates) {
        req_bits |= SV_DATA_BAD_PARAM;
        valid = false;
      } else if (sm.stop_bad) {
        req_bits |= SV_DATA_BAD_DRAFT_ID;
        valid = false;
      } else {
        A = a;
        if (rank == 0 && tid < g && tid <= A && !rates) {
          if (P.dbg_py) P.dbg_py[s + tid] = py;
          if (P.dbg_qy) P.dbg_qy[s + tid] = qy;
        }
        // a3 / a4: one race over the row of the first rejection or the bonus row
        const float *prow = p + (tb + A) * ts;
        const float *Erow = kTest ? P.exponentials + static_cast<int64_t>(i) * P.exp_stride : nullptr;
        float bk = 0.0f;
        int bx = -1;
        uint32_t fl = 0;
        if (A < g)
          race_chunk<kTest, true, kVec>(prow, q + (s + A) * ds, x0, x1, Erow, rk, rs, bk, bx, fl);
        else
          race_chunk<kTest, false, kVec>(prow, nullptr, x0, x1, Erow, rk, rs, bk, bx, fl);
        KeyFlags r = cluster_reduce(KeyFlags{bx >= 0 ? pack_key(bk, bx) : 0ull, fl}, sm.red, step++, ncta);
        if (r.key == 0ull && A < g) {  // no positive residual key: same race over p
          bk = 0.0f;
          bx = -1;
          fl = 0;
          race_chunk<kTest, false, kVec>(prow, nullptr, x0, x1, Erow, rk, rs, bk, bx, fl);
          const KeyFlags r2 =
              cluster_reduce(KeyFlags{bx >= 0 ? pack_key(bk, bx) : 0ull, fl}, sm.red, step++, ncta);
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
      }
    }
  }
  __syncthreads();

  // a6 / a7: outputs and KV rollback, written by the cluster's first CTA
  if (rank == 0) {
    const int A0 = A;
    auto tok = [&](int k) -> int32_t { return greedy ? sm.tok[k] : (k == A0 ? last_tok : P.ids[s + k]); };
    if (valid && P.stop_cu) A = stop_commit(A0, tok, P.stop_ids, stop_b, stop_e, &sm.stop_first);
    emit_request(i, G, g, A, valid, tb, req_bits, tok, P.out, P.nacc, P.ncomp, P.slots, P.status);
  }
  cluster_sync();  // peers may still be reading this CTA's reduction slot
}

template <bool kTest, bool kVec>
cudaError_t launch_one(const VerifyParams &p, int cluster, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p.N) * static_cast<unsigned>(cluster), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  cfg.attrs = attr;
  cfg.numAttrs = launch_attrs(attr, static_cast<unsigned>(cluster), p.pdl);
  return cudaLaunchKernelEx(&cfg, probs_kernel<kTest, kVec>, p);
}

template <bool kTest, bool kVec>
cudaError_t enable_one(int max_cluster) {
  if (max_cluster > 8)
    return cudaFuncSetAttribute(probs_kernel<kTest, kVec>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  return cudaSuccess;
}

}  // namespace

cudaError_t enable_probs_kernels(int max_cluster) {
  cudaError_t e;
  if ((e = enable_one<true, true>(max_cluster)) != cudaSuccess) return e;
  if ((e = enable_one<true, false>(max_cluster)) != cudaSuccess) return e;
  if ((e = enable_one<false, true>(max_cluster)) != cudaSuccess) return e;
  return enable_one<false, false>(max_cluster);
}

cudaError_t launch_probs(const VerifyParams &p, int cluster, bool vec, cudaStream_t stream) {
  const bool test = p.exponentials != nullptr;
  if (test) return vec ? launch_one<true, true>(p, cluster, stream) : launch_one<true, false>(p, cluster, stream);
  return vec ? launch_one<false, true>(p, cluster, stream) : launch_one<false, false>(p, cluster, stream);
}

}  // namespace sv
