// sv_trunc.cuh -- top-k / top-p truncation of the target and draft rows.
//
// "Speculative Decoding: Medusa, MTP, EAGLE, DFlash, DDTree, and DSpark",
// section 1: temperature, truncation, penalties and grammar constraints must
// be incorporated consistently, so the acceptance test and the residual use
// the distributions the target and the drafter actually sample from.  Here a
// request's top_k and top_p are applied alike to its target and draft rows:
//   temperature first, p = softmax(x / T);
//   top-k (0 < K < V): keep every logit >= the K-th largest (ties kept);
//   top-p (0 < P < 1), on the top-k survivors renormalised: keep a logit while
//     the mass of the survivors with a strictly larger logit is below P;
//   the output row holds the kept logits and -inf elsewhere, so softmax of it
//   is the truncated, renormalised distribution and the verify round runs on
//   it unchanged.
// Both rules keep the logits at or above a threshold, found exactly by a radix
// descent over order-preserving keys of the logits, 8 bits a level (2 levels
// for bf16, 4 for fp32): top-k from element counts, top-p from masses
// 2^(c (x - max)) held as 2^-40 fixed-point integers.  Counts and masses are
// integer sums, so the threshold does not depend on the order of the atomics.
// Rows of greedy requests (T = 0), rows holding NaN, and rows whose top_p is
// NaN or <= 0 (which also sets SPECVERIFY_STATUS_BAD_TRUNC) are copied.
#pragma once

#include "sv_kernels.cuh"

namespace sv {

constexpr int kTruncThreads = 1024;
constexpr uint32_t kStBadTrunc = 1024u;

struct TruncParams {
  const void* target_in;
  const void* draft_in;
  void* target_out;
  void* draft_out;
  const int32_t* num_draft;
  const float* temperature;
  const int32_t* top_k;
  const float* top_p;
  int batch, total_draft, vocab;
  int32_t* status;  // nullable device word (atomicOr)
};

// Order-preserving key of a logit: larger logit, larger key (-inf lowest;
// -0 and +0 compare equal, so they share a key).  bf16 logits carry their
// information in the upper 16 bits.
template <typename E>
__device__ __forceinline__ uint32_t trunc_key(float x) {
  uint32_t u = __float_as_uint(x);
  if (u == 0x80000000u) u = 0u;
  const uint32_t k = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return E::kBytes == 2 ? (k >> 16) : k;
}

// The digit a warp-0 scan picks from 256 bins, lanes holding 8 bins each.
// mode 0 (top-k): the highest digit d with sum_{digits >= d} cnt >= need;
// mode 1 (top-p): the lowest digit d with cnt[d] > 0 and mass above d < target.
// Returns the digit and, in *above, the count or mass of the digits above it.
__device__ int pick_digit(const unsigned int* cnt, const unsigned long long* mass, int mode,
                          unsigned long long need, double target, unsigned long long* above) {
  const int lane = threadIdx.x & 31;
  unsigned long long loc[8];
  unsigned long long sum = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int d = lane * 8 + j;
    loc[j] = mode == 0 ? (unsigned long long)cnt[d] : mass[d];
    sum += loc[j];
  }
  // exclusive suffix scan over lanes: the total of the digits held by higher lanes
  unsigned long long incl = sum;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const unsigned long long o = __shfl_down_sync(0xffffffffu, incl, off);
    if (lane + off < 32) incl += o;
  }
  unsigned long long run = incl - sum;  // above this lane's digits
  int best = mode == 0 ? -1 : 256;
  unsigned long long best_above = 0;
#pragma unroll
  for (int j = 7; j >= 0; --j) {
    const int d = lane * 8 + j;
    if (mode == 0) {
      if (best < 0 && run + loc[j] >= need) {
        best = d;
        best_above = run;
      }
    } else if (cnt[d] > 0u && (double)run < target) {
      best = d;  // keeps the lowest such digit of this lane
      best_above = run;
    }
    run += loc[j];
  }
  // across lanes: the highest (mode 0) or lowest (mode 1) digit found
  int pick = best;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const int o = __shfl_xor_sync(0xffffffffu, pick, off);
    pick = mode == 0 ? max(pick, o) : min(pick, o);
  }
  const unsigned owner = __ballot_sync(0xffffffffu, best == pick);
  *above = __shfl_sync(0xffffffffu, best_above, owner ? __ffs(owner) - 1 : 0);
  return min(max(pick, 0), 255);  // always found for a consistent histogram
}

template <typename E, bool kAligned>
__global__ void __launch_bounds__(kTruncThreads) sv_truncate(TruncParams P) {
  __shared__ unsigned int s_cnt[256];
  __shared__ unsigned long long s_mass[256];
  __shared__ float s_red[kTruncThreads / 32];
  __shared__ unsigned int s_nan;
  __shared__ int s_digit;
  __shared__ unsigned long long s_above;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int kLevels = E::kBytes;  // 8-bit digits of the key
  const int V = P.vocab;
  const size_t row_bytes = (size_t)V * E::kBytes;
  const int nvec = (int)(row_bytes / 16);
  const long long n_t = (long long)P.batch + P.total_draft;
  const long long rows = n_t + (P.draft_in ? P.total_draft : 0);
  // request of the current row: a cursor over the target layout (k_r + 1 rows
  // per request), then over the draft layout (k_r rows); rows only increase
  int r_cur = -1;
  long long r_end = 0;  // rows before r_end belong to requests <= r_cur
  bool draft_phase = false;
  for (long long row = blockIdx.x; row < rows; row += gridDim.x) {
    const bool is_draft = row >= n_t;
    const long long local = is_draft ? row - n_t : row;
    if (is_draft != draft_phase) {
      draft_phase = is_draft;
      r_cur = -1;
      r_end = 0;
    }
    while (local >= r_end && r_cur < P.batch - 1) {
      ++r_cur;
      r_end += max(P.num_draft[r_cur], 0) + (is_draft ? 0 : 1);
    }
    const char* in = reinterpret_cast<const char*>(is_draft ? P.draft_in : P.target_in) +
                     (size_t)local * row_bytes;
    char* out = reinterpret_cast<char*>(is_draft ? P.draft_out : P.target_out) +
                (size_t)local * row_bytes;
    const float T = P.temperature[r_cur];
    const int K = P.top_k[r_cur];
    const float Pp = P.top_p[r_cur];
    const bool bad = !(Pp > 0.f);
    const bool use_k = K > 0 && K < V;
    const bool use_p = Pp < 1.f;
    bool copy = bad || !(T > 0.f) || (!use_k && !use_p);
    if (bad && tid == 0 && P.status) atomicOr(reinterpret_cast<unsigned int*>(P.status), kStBadTrunc);

    // visit every element of the row: f(x) (vector loads on aligned rows)
    auto each = [&](auto&& f) {
      if (kAligned) {
        const uint4* rv = reinterpret_cast<const uint4*>(in);
        for (int i = tid; i < nvec; i += kTruncThreads) {
          float x[E::kVec];
          E::unpack(ld_stream(rv + i), x);
#pragma unroll
          for (int e = 0; e < E::kVec; ++e) f(x[e]);
        }
      } else {
        for (int v = tid; v < V; v += kTruncThreads) f(E::load1(in, v));
      }
    };

    uint32_t tau = 0u;  // keep keys >= tau
    if (!copy) {
      // ---- pass 0: maximum, NaN, the first top-k level ---------------------------
      if (tid < 256) s_cnt[tid] = 0u;
      if (tid == 0) s_nan = 0u;
      __syncthreads();
      float mx = kNegInf;
      bool nan = false;
      const int shift0 = 8 * (kLevels - 1);
      each([&](float x) {
        nan |= x != x;
        mx = fmaxf(mx, x);
        if (use_k) atomicAdd(&s_cnt[trunc_key<E>(x) >> shift0], 1u);
      });
      if (__any_sync(0xffffffffu, nan) && lane == 0) s_nan = 1u;
      mx = warp_max(mx);
      if (lane == 0) s_red[warp] = mx;
      __syncthreads();
      if (warp == 0) {
        float m = lane < kTruncThreads / 32 ? s_red[lane] : kNegInf;
        m = warp_max(m);
        if (lane == 0) s_red[0] = m;
      }
      __syncthreads();
      mx = s_red[0];
      copy = s_nan != 0u;
      __syncthreads();
      if (!copy && use_k) {
        // ---- top-k: the key of the K-th largest logit, one level at a time -------
        unsigned long long need = (unsigned long long)K;
        uint32_t prefix = 0u;
        for (int L = 0; L < kLevels; ++L) {
          const int shift = 8 * (kLevels - 1 - L);
          if (L > 0) {
            if (tid < 256) s_cnt[tid] = 0u;
            __syncthreads();
            each([&](float x) {
              const uint32_t k = trunc_key<E>(x);
              if ((k >> (shift + 8)) == prefix) atomicAdd(&s_cnt[(k >> shift) & 0xffu], 1u);
            });
            __syncthreads();
          }
          if (warp == 0) {
            unsigned long long above;
            const int d = pick_digit(s_cnt, nullptr, 0, need, 0.0, &above);
            if (lane == 0) {
              s_digit = d;
              s_above = above;
            }
          }
          __syncthreads();
          prefix = (prefix << 8) | (uint32_t)s_digit;
          need -= s_above;
          __syncthreads();
        }
        tau = prefix;
      }
      if (!copy && use_p) {
        // ---- top-p on the survivors: masses 2^(c (x - mx)) in 2^-40 fixed point --
        const float c = kLog2e / T;
        const float cm = c * mx;
        double target = 0.0;
        unsigned long long above_all = 0ull;
        uint32_t prefix = 0u;
        const uint32_t tau_k = tau;
        for (int L = 0; L < kLevels; ++L) {
          const int shift = 8 * (kLevels - 1 - L);
          if (tid < 256) {
            s_cnt[tid] = 0u;
            s_mass[tid] = 0ull;
          }
          __syncthreads();
          each([&](float x) {
            const uint32_t k = trunc_key<E>(x);
            if (k >= tau_k && (L == 0 || (k >> (shift + 8)) == prefix)) {
              const float w = fast_ex2(fmaf(x, c, -cm));
              const unsigned long long q = __float2ull_rn(w * 0x1p40f);
              const int d = (k >> shift) & 0xff;
              atomicAdd(&s_cnt[d], 1u);
              if (q) atomicAdd(&s_mass[d], q);
            }
          });
          __syncthreads();
          if (warp == 0) {
            if (L == 0) {
              unsigned long long tot = 0ull;
              for (int d = lane; d < 256; d += 32) tot += s_mass[d];
#pragma unroll
              for (int off = 16; off > 0; off >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, off);
              target = (double)Pp * (double)tot;
            }
            unsigned long long above;
            const int d = pick_digit(s_cnt, s_mass, 1, 0ull, target - (double)above_all, &above);
            if (lane == 0) {
              s_digit = d;
              s_above = above;
            }
          }
          __syncthreads();
          prefix = (prefix << 8) | (uint32_t)s_digit;
          above_all += s_above;
          __syncthreads();
        }
        tau = max(tau, prefix);
      }
    }
    // ---- output: the kept logits, -inf elsewhere (or the row as it is) ----------
    if (kAligned) {
      const uint4* rv = reinterpret_cast<const uint4*>(in);
      uint4* ov = reinterpret_cast<uint4*>(out);
      for (int i = tid; i < nvec; i += kTruncThreads) {
        uint4 q = ld_stream(rv + i);
        if (!copy) {
          float x[E::kVec];
          E::unpack(q, x);
          uint32_t* w = reinterpret_cast<uint32_t*>(&q);
#pragma unroll
          for (int e = 0; e < E::kVec; ++e) {
            if (trunc_key<E>(x[e]) >= tau) continue;
            if (E::kBytes == 4) {
              w[e] = 0xff800000u;
            } else {
              const int h = e >> 1;
              w[h] = (e & 1) ? ((w[h] & 0x0000ffffu) | 0xff800000u) : ((w[h] & 0xffff0000u) | 0xff80u);
            }
          }
        }
        ov[i] = q;
      }
    } else {
      for (int v = tid; v < V; v += kTruncThreads) {
        if (E::kBytes == 4) {
          const float x = E::load1(in, v);
          reinterpret_cast<float*>(out)[v] =
              (copy || trunc_key<E>(x) >= tau) ? x : __uint_as_float(0xff800000u);
        } else {
          const unsigned short h = reinterpret_cast<const unsigned short*>(in)[v];
          const float x = __uint_as_float((uint32_t)h << 16);
          reinterpret_cast<unsigned short*>(out)[v] =
              (copy || trunc_key<E>(x) >= tau) ? h : (unsigned short)0xff80u;
        }
      }
    }
    __syncthreads();
  }
}

}  // namespace sv
