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
// Both rules keep the logits at or above a threshold on order-preserving keys
// of the logits, found exactly in one of two ways:
//   bf16 rows with 16-byte vectors first take the window histogram: a bf16
//     logit is fixed by its 16-bit key, so counts of the exact keys in the 8
//     high-byte bins at and below the maximum's give top-k from counts and
//     top-p from masses count * 2^(c (x_key - max)), summed in fp64 in a fixed
//     order; these passes work on packed words, two logits at a time;
//   other rows, and bf16 rows whose threshold lies below the window, take a
//     radix descent, 8 bits a level (2 levels for bf16, 4 for fp32): top-k from
//     element counts, top-p from masses held as 2^-40 fixed-point integers.
// Counts and fixed-point masses are integer sums and the fp64 sums run in a
// fixed order, so the threshold does not depend on the order of the atomics.
// Rows of greedy requests (T = 0), rows holding NaN, and rows whose top_p is
// NaN or <= 0 (which also sets SPECVERIFY_STATUS_BAD_TRUNC) are copied.
//
// One kernel, three uses: copy mode writes the truncated rows; threshold mode
// writes one threshold key per row instead (0 for a row kept whole); list mode
// is threshold mode over the rows of one verify wave (its row and bonus
// lists), launched before that wave of a truncated round.
#pragma once

#include "sv_kernels.cuh"

namespace sv {

constexpr int kTruncThreads = 512;  // two CTAs per SM: one's scans overlap the other's loads
constexpr int kTruncLoads = 8;  // 16-byte loads in flight per thread (packed passes)
constexpr int kPackedOutLoads = 1;  // ... and in the packed output pass
constexpr int kOutLoads = 1;    // ... and in the output pass
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
  // Threshold mode (both set, outputs unused): each row's order-key threshold
  // is written here instead of a truncated copy (0 for a row kept whole).
  uint32_t* thr_target;
  uint32_t* thr_draft;
  // List mode (threshold mode within a verify round, lists set): the rows are
  // those of one wave, its row list and its bonus list, not the whole window.
  const Entry* lists;   // the wave's row list
  const int* list_cnt;  // its length
  const Entry* blists;  // the wave's bonus list
  const int* blist_cnt;
};

// The output pass is the last touch of a row: its loads and the stores of the
// output row are marked evict-first (cache streaming), so they do not push out
// of L2 the rows other CTAs are still taking their earlier passes over.
__device__ __forceinline__ uint4 ld_last_use(const uint4* p) {
  uint4 r;
  asm volatile("ld.global.cs.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}
__device__ __forceinline__ void st_streaming(uint4* p, uint4 v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

// The digit a warp-0 scan picks from 256 bins, lanes holding 8 bins each.
// mode 0 (top-k): the highest digit d with sum_{digits >= d} cnt >= need;
// mode 1 (top-p): the lowest digit d with cnt[d] > 0 and scale * (mass above
// d) < target.  Returns the digit and, in *above, the count or mass of the
// digits above it.
__device__ int pick_digit(const unsigned int* cnt, const unsigned long long* mass, int mode,
                          unsigned long long need, double target, double scale,
                          unsigned long long* above) {
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
    } else if (cnt[d] > 0u && (double)run * scale < target) {
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

// Counts one element per lane into this warp's own histogram (lanes with
// !valid add nothing): no other warp shares the histogram, so atomics only
// meet those of the same warp.
__device__ __forceinline__ void count_add(unsigned int* whist, bool valid, int d) {
  if (valid) atomicAdd(&whist[d], 1u);
}

constexpr int kWin = 8;  // octave bins the first top-p level resolves below the maximum

// ---------------------------------------------------------------------------
// The window histogram of bf16 rows.  A bf16 logit is fixed by its 16-bit key,
// so counts of exact keys give both rules at once: top-k from counts of the
// keys at or above a key, top-p from masses count * 2^(c (x_key - max)).  The
// window is the kWinBins high-byte bins at and below the maximum's (kWinKeys
// keys); one pass counts the row's keys there (the other elements only add
// their masses to a per-thread sum), and the thresholds come from block-wide
// suffix scans over the window in a fixed order.  A row whose threshold lies
// below the window goes on to the radix descent.
// ---------------------------------------------------------------------------
constexpr int kWinBins = 8;
constexpr int kWinKeys = kWinBins * 256;
constexpr int kWinPerThread = kWinKeys / kTruncThreads;  // window keys a thread holds
static_assert(kWinPerThread * kTruncThreads == kWinKeys, "whole window keys per thread");

// The bf16 logit of a 16-bit order key (trunc_key<BF16> inverted).
__device__ __forceinline__ float key_logit(uint32_t key) {
  const uint32_t h = (key & 0x8000u) ? (key & 0x7fffu) : (~key & 0xffffu);
  return __uint_as_float(h << 16);
}

// Block-wide sum over the threads with larger index (exclusive suffix), in a
// fixed order; *total gets the sum over all threads.  All threads call it.
template <typename T>
__device__ __forceinline__ T block_suffix_excl(T v, T* s_part, T* total) {
  constexpr int kW = kTruncThreads / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  T x = v;  // inclusive suffix inside the warp
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const T o = __shfl_down_sync(0xffffffffu, x, off);
    if (lane + off < 32) x += o;
  }
  T ex = __shfl_down_sync(0xffffffffu, x, 1);
  if (lane == 31) ex = T(0);
  if (lane == 0) s_part[warp] = x;
  __syncthreads();
  if (warp == 0) {
    const T w = lane < kW ? s_part[lane] : T(0);
    T y = w;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const T o = __shfl_down_sync(0xffffffffu, y, off);
      if (lane + off < 32) y += o;
    }
    T ye = __shfl_down_sync(0xffffffffu, y, 1);
    if (lane == 31) ye = T(0);
    if (lane < kW) s_part[lane] = ye;
    if (lane == 0) s_part[kW] = y;
  }
  __syncthreads();
  const T r = ex + s_part[warp];
  *total = s_part[kW];
  __syncthreads();
  return r;
}

// Block-wide max (or min) of an int; all threads call it.
__device__ __forceinline__ int block_extreme(int v, bool is_max, int* s_part) {
  constexpr int kW = kTruncThreads / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const int o = __shfl_xor_sync(0xffffffffu, v, off);
    v = is_max ? max(v, o) : min(v, o);
  }
  if (lane == 0) s_part[warp] = v;
  __syncthreads();
  int r = s_part[0];
  for (int w = 1; w < kW; ++w) r = is_max ? max(r, s_part[w]) : min(r, s_part[w]);
  __syncthreads();
  return r;
}

// The thresholds of one bf16 row from its window histogram: *tau gets the
// 16-bit key to keep from (0 keeps everything).  Returns false, leaving *tau,
// when the row needs the radix descent: a non-finite maximum, fewer than K
// elements in the window, or a top-p boundary below the window.
//   kfloor: a key at or below the K-th largest (0 when unknown): with top-k
//   on, keys below it cannot survive and are not counted.
template <typename EachVec>
__device__ bool window_thresholds(EachVec&& each_vec, int V, float mx, float T, bool use_k, int K,
                                  bool use_p, float Pp, uint32_t kfloor, unsigned int* s_hist,
                                  double* s_dpart, unsigned int* s_upart, int* s_ipart,
                                  uint32_t* tau) {
  if (!(mx > kNegInf && mx < 3.0e38f)) return false;
  const int tid = threadIdx.x;
  const int hb_top = (int)(trunc_key<BF16>(mx) >> 8);
  const int lo = max(hb_top - (kWinBins - 1), 0);
  const float c = kLog2e / T;
  const float cm = c * mx;
#pragma unroll
  for (int j = 0; j < kWinPerThread; ++j) s_hist[kWinPerThread * tid + j] = 0u;
  __syncthreads();
  float below = 0.f;  // mass of this thread's elements below the window
  const uint32_t kb = (uint32_t)lo << 8;  // the window's lowest key
  const uint32_t kc = use_k ? max(kb, kfloor) : kb;  // the lowest key counted
  const bool tail_mass = use_p && !use_k;  // survivors below the window exist
  each_vec([&](bool ok, uint4 q) {
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t k2 = bf16x2_keys(w[j]);
#pragma unroll
      for (int h = 0; h < 2; ++h) {  // the lower-addressed logit is the low half
        const uint32_t k = h ? (k2 >> 16) : (k2 & 0xffffu);
        if (ok && k >= kc) {
          atomicAdd(&s_hist[k - kb], 1u);  // below 2048: no key exceeds the maximum's
        } else if (ok && tail_mass && k < kb) {
          const float x = __uint_as_float(h ? (w[j] & 0xffff0000u) : (w[j] << 16));
          below += fast_ex2(fmaf(x, c, -cm));
        }
      }
    }
  });
  __syncthreads();
  // -0 was keyed apart, just below +0: its count joins +0's, as equal logits
  if (tid == 0 && kb <= 0x7fffu && 0x8000u - kb < (uint32_t)kWinKeys) {
    s_hist[0x8000u - kb] += s_hist[0x7fffu - kb];
    s_hist[0x7fffu - kb] = 0u;
  }
  __syncthreads();
  // thread t holds window keys i = kWinPerThread t + j (key = (lo << 8) + i); the
  // scans run from the highest key down
  constexpr int kP = kWinPerThread;
  const int ib = kP * tid;
  unsigned int n[kP], n_own = 0u;
#pragma unroll
  for (int j = 0; j < kP; ++j) {
    n[j] = s_hist[ib + j];
    n_own += n[j];
  }
  unsigned int n_win;
  const unsigned int n_above = block_suffix_excl<unsigned int>(n_own, s_upart, &n_win);
  int first = 0;  // lowest window index a survivor of top-k may have
  if (use_k) {
    if (n_win < (unsigned int)K) return false;
    // the highest key with at least K elements at or above it
    unsigned int run = n_above;
    int cand = -1;
#pragma unroll
    for (int j = kP - 1; j >= 0; --j) {
      run += n[j];
      if (cand < 0 && run >= (unsigned int)K) cand = ib + j;
    }
    first = block_extreme(cand, true, s_ipart);
  }
  int pick = first;
  if (use_p) {
    double w[kP], w_own = 0.0;
#pragma unroll
    for (int j = 0; j < kP; ++j) {
      w[j] = (n[j] && ib + j >= first)
                 ? (double)n[j] * (double)fast_ex2(fmaf(key_logit((lo << 8) + ib + j), c, -cm))
                 : 0.0;
      w_own += w[j];
    }
    double m_win;
    const double m_above = block_suffix_excl<double>(w_own, s_dpart, &m_win);
    // survivors below the window exist only without a top-k cut inside it
    const bool tail = !use_k && n_win < (unsigned int)V;
    double m_tail = 0.0;
    if (tail) {
      const float wb = group_sum<32>(below);
      if ((tid & 31) == 0) s_dpart[tid >> 5] = (double)wb;
      __syncthreads();
      for (int wi = 0; wi < kTruncThreads / 32; ++wi) m_tail += s_dpart[wi];
      __syncthreads();
    }
    const double target = (double)Pp * (m_win + m_tail);
    if (tail && m_win < target) return false;
    // the lowest survivor key whose strictly larger survivors weigh below target
    double run = m_above;
    int lowest = kWinKeys;
#pragma unroll
    for (int j = kP - 1; j >= 0; --j) {
      if (n[j] && ib + j >= first && run < target) lowest = ib + j;
      run += w[j];
    }
    pick = block_extreme(lowest, false, s_ipart);
    pick = max(pick, first);
  }
  *tau = (uint32_t)((lo << 8) + pick);
  return true;
}

template <typename E, bool kAligned>
__global__ void __launch_bounds__(kTruncThreads, 2) sv_truncate(TruncParams P) {
  constexpr int kWarps = kTruncThreads / 32;
  __shared__ unsigned int s_whist[kWarps][256];  // per-warp counts
  __shared__ unsigned int s_cnt[256];
  __shared__ unsigned long long s_mass[256];
  __shared__ float s_wsum[kWarps][2 * kWin + 2];
  __shared__ float s_red[kWarps];
  __shared__ unsigned int s_nan;
  __shared__ int s_digit;
  __shared__ unsigned long long s_above;
  __shared__ double s_dval[2];
  // bf16 rows: exact keys of the 8 high-byte bins at and below the maximum's
  __shared__ unsigned int s_hist[kWinKeys];
  __shared__ double s_dpart[kWarps + 1];
  __shared__ unsigned int s_upart[kWarps + 1];
  __shared__ int s_ipart[kWarps];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // bf16 rows with 16-byte vectors take the window histogram first
  constexpr bool kFast = E::kBytes == 2 && kAligned;
  constexpr int kLevels = E::kBytes;  // 8-bit digits of the key
  const int V = P.vocab;
  const size_t row_bytes = (size_t)V * E::kBytes;
  const int nvec = (int)(row_bytes / 16);
  const long long n_t = (long long)P.batch + P.total_draft;
  const bool list_mode = P.lists != nullptr;
  const int n_list = list_mode ? *P.list_cnt : 0;
  const long long rows =
      list_mode ? (long long)n_list + *P.blist_cnt : n_t + (P.draft_in ? P.total_draft : 0);
  // request of the current row: a cursor over the target layout (k_r + 1 rows
  // per request), then over the draft layout (k_r rows); rows only increase
  int r_cur = -1;
  long long r_end = 0;  // rows before r_end belong to requests <= r_cur
  bool draft_phase = false;
  for (long long row = blockIdx.x; row < rows; row += gridDim.x) {
    bool is_draft;
    long long local;  // row index in the target or the draft layout
    if (list_mode) {
      // a wave entry: request r, position pos, the request's first draft row d0
      const Entry en = row < n_list ? P.lists[row] : P.blists[row - n_list];
      r_cur = en.meta & 0x1fff;
      is_draft = ((en.meta >> 13) & 1) != 0;
      const int pos = (en.meta >> 20) & 31;
      local = is_draft ? (long long)en.d0 + pos : (long long)en.d0 + r_cur + pos;
    } else {
      is_draft = row >= n_t;
      local = is_draft ? row - n_t : row;
      if (is_draft != draft_phase) {
        draft_phase = is_draft;
        r_cur = -1;
        r_end = 0;
      }
      while (local >= r_end && r_cur < P.batch - 1) {
        ++r_cur;
        r_end += max(P.num_draft[r_cur], 0) + (is_draft ? 0 : 1);
      }
    }
    const char* in = reinterpret_cast<const char*>(is_draft ? P.draft_in : P.target_in) +
                     (size_t)local * row_bytes;
    const float T = P.temperature[r_cur];
    const int K = P.top_k[r_cur];
    const float Pp = P.top_p[r_cur];
    const bool bad = !(Pp > 0.f);
    const bool use_k = K > 0 && K < V;
    const bool use_p = Pp < 1.f;
    bool copy = bad || !(T > 0.f) || (!use_k && !use_p);
    if (bad && tid == 0 && P.status) atomicOr(reinterpret_cast<unsigned int*>(P.status), kStBadTrunc);

    // visit every element of the row: f(ok, x), warp-uniform (every lane of a
    // warp runs the same iterations; ok is false past the row's end); vector
    // loads on aligned rows, nl of them issued before any is used (a thread
    // still visits its vectors i = tid + j * kTruncThreads in order of j)
    auto each_n = [&](auto nl, auto&& f) {
      constexpr int kN = decltype(nl)::value;
      if (kAligned) {
        const uint4* rv = reinterpret_cast<const uint4*>(in);
        for (int i0 = warp * 32; i0 < nvec; i0 += kN * kTruncThreads) {
          uint4 q[kN];
#pragma unroll
          for (int u = 0; u < kN; ++u) {
            const int i = i0 + u * kTruncThreads + lane;
            q[u] = i < nvec ? ld_stream(rv + i) : E::pad();
          }
#pragma unroll
          for (int u = 0; u < kN; ++u) {
            const bool ok = i0 + u * kTruncThreads + lane < nvec;
            float x[E::kVec];
            E::unpack(q[u], x);
#pragma unroll
            for (int e = 0; e < E::kVec; ++e) f(ok, x[e]);
          }
        }
      } else {
        for (int v0 = warp * 32; v0 < V; v0 += kTruncThreads) {
          const int v = v0 + lane;
          const bool ok = v < V;
          f(ok, ok ? E::load1(in, v) : kNegInf);
        }
      }
    };
    // the radix descent's passes (register-heavy) keep one load in flight; the
    // window histogram's passes, kTruncLoads
    auto each = [&](auto&& f) { each_n(std::integral_constant<int, 1>{}, f); };
    // visit every 16-byte vector of an aligned row: g(ok, q), kTruncLoads loads in
    // flight per thread (past the row's end: ok false and q the -inf padding)
    auto each_vec = [&](auto&& g) {
      const uint4* rv = reinterpret_cast<const uint4*>(in);
      for (int i0 = warp * 32; i0 < nvec; i0 += kTruncLoads * kTruncThreads) {
        uint4 q[kTruncLoads];
#pragma unroll
        for (int u = 0; u < kTruncLoads; ++u) {
          const int i = i0 + u * kTruncThreads + lane;
          q[u] = i < nvec ? ld_stream(rv + i) : E::pad();
        }
#pragma unroll
        for (int u = 0; u < kTruncLoads; ++u) g(i0 + u * kTruncThreads + lane < nvec, q[u]);
      }
    };
    auto each_deep = [&](auto&& f) {
      each_n(std::integral_constant<int, kFast ? kTruncLoads : 1>{}, f);
    };
    // the per-warp counts, zeroed before / summed into s_cnt after a pass
    auto clear_counts = [&]() {
      for (int i = lane; i < 256; i += 32) s_whist[warp][i] = 0u;
      if (tid < 256) {
        s_cnt[tid] = 0u;
        s_mass[tid] = 0ull;
      }
      __syncthreads();
    };
    auto sum_counts = [&]() {
      __syncthreads();
      if (tid < 256) {
        unsigned int c = 0u;
        for (int w = 0; w < kWarps; ++w) c += s_whist[w][tid];
        s_cnt[tid] += c;
      }
      __syncthreads();
    };

    uint32_t tau = 0u;  // keep keys >= tau
    if (!copy) {
      // ---- pass 0: maximum, NaN, the first top-k level ---------------------------
      if (tid == 0) s_nan = 0u;
      clear_counts();
      float mx = kNegInf;
      bool nan = false;
      uint32_t kx_t = 0u;  // this thread's largest key (packed bf16 pass)
      const int shift0 = 8 * (kLevels - 1);
      if constexpr (kFast) {
        // packed keys, two logits a word: their largest and smallest (the -inf
        // padding moves neither test)
        uint32_t kmax = 0u, kmin = 0xffffffffu;
        each_vec([&](bool, uint4 q) {
          const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint32_t k2 = bf16x2_keys(w[j]);
            kmax = max_u16x2(kmax, k2);
            kmin = min_u16x2(kmin, k2);
          }
        });
        const uint32_t kx = max(kmax & 0xffffu, kmax >> 16);
        const uint32_t kn = min(kmin & 0xffffu, kmin >> 16);
        nan = kx > 0xff80u || kn < 0x007fu;  // above +inf's key or below -inf's
        mx = nan ? kNegInf : key_logit(kx);
        kx_t = kx;
      } else {
        each_deep([&](bool ok, float x) {
          nan |= ok && x != x;
          mx = fmaxf(mx, x);
          if (use_k) count_add(s_whist[warp], ok, (int)(trunc_key<E>(x) >> shift0));
        });
      }
      if (__any_sync(0xffffffffu, nan) && lane == 0) s_nan = 1u;
      mx = warp_max(mx);
      if (lane == 0) s_red[warp] = mx;
      sum_counts();
      if (warp == 0) {
        float m = lane < kWarps ? s_red[lane] : kNegInf;
        m = warp_max(m);
        if (lane == 0) s_red[0] = m;
      }
      __syncthreads();
      mx = s_red[0];
      copy = s_nan != 0u;
      __syncthreads();
      bool done = false;  // the thresholds were found by the window histogram
      if constexpr (kFast) {
        // top-k floor: the threads' maxima are distinct elements, so the high
        // byte h with at least K of them in bins >= h bounds the K-th largest
        // key from below (a thread that saw only padding counts as -inf,
        // which can only lower the floor)
        uint32_t kfloor = 0u;
        if (!copy && use_k && K <= kTruncThreads) {
          atomicAdd(&s_cnt[kx_t >> 8], 1u);
          __syncthreads();
          if (warp == 0) {
            unsigned long long above;
            const int d = pick_digit(s_cnt, nullptr, 0, (unsigned long long)K, 0.0, 1.0, &above);
            if (lane == 0) s_digit = d;
          }
          __syncthreads();
          kfloor = (uint32_t)s_digit << 8;
          if (tid < 256) s_cnt[tid] = 0u;
          __syncthreads();
        }
        if (!copy) {
          done = window_thresholds(each_vec, P.vocab, mx, T, use_k, K, use_p, Pp, kfloor, s_hist,
                                   s_dpart, s_upart, s_ipart, &tau);
          if (!done && use_k) {
            // the radix descent below starts from the level-0 counts
            clear_counts();
            each([&](bool ok, float x) {
              count_add(s_whist[warp], ok, (int)(trunc_key<E>(x) >> shift0));
            });
            sum_counts();
          }
        }
      }
      if (!copy && !done && use_k) {
        // ---- top-k: the key of the K-th largest logit, one level at a time -------
        unsigned long long need = (unsigned long long)K;
        uint32_t prefix = 0u;
        for (int L = 0; L < kLevels; ++L) {
          const int shift = 8 * (kLevels - 1 - L);
          if (L > 0) {
            clear_counts();
            each([&](bool ok, float x) {
              const uint32_t k = trunc_key<E>(x);
              count_add(s_whist[warp], ok && (k >> (shift + 8)) == prefix,
                        (int)((k >> shift) & 0xffu));
            });
            sum_counts();
          }
          if (warp == 0) {
            unsigned long long above;
            const int d = pick_digit(s_cnt, nullptr, 0, need, 0.0, 1.0, &above);
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
      if (!copy && !done && use_p) {
        // ---- top-p on the survivors, masses w = 2^(c (x - mx)) ---------------------
        const float c = kLog2e / T;
        const float cm = c * mx;
        const uint32_t tau_k = tau;
        // first level: per-thread sums over kWin octave bins from the maximum's
        // digit down, and one sum below them (fixed order: deterministic); the
        // window slides down while the boundary lies below it
        const int d_top = (int)(trunc_key<E>(mx) >> shift0);
        double above_all = 0.0, target = 0.0;
        int d0 = -1;
        for (int base = d_top; base >= 0 && d0 < 0; base -= kWin) {
          float acc[kWin], below = 0.f, nbelow = 0.f, cnt[kWin];
#pragma unroll
          for (int j = 0; j < kWin; ++j) acc[j] = cnt[j] = 0.f;
          each([&](bool ok, float x) {
            const uint32_t k = trunc_key<E>(x);
            if (!(ok && k >= tau_k)) return;
            const float w = fast_ex2(fmaf(x, c, -cm));
            const int j = base - (int)(k >> shift0);
            if (j >= kWin) {
              below += w;
              nbelow += 1.f;
            }
#pragma unroll
            for (int i = 0; i < kWin; ++i)
              if (j == i) {
                acc[i] += w;
                cnt[i] += 1.f;
              }
          });
          // block sums in a fixed order
#pragma unroll
          for (int i = 0; i < kWin; ++i) {
            acc[i] = group_sum<32>(acc[i]);
            cnt[i] = group_sum<32>(cnt[i]);
          }
          below = group_sum<32>(below);
          nbelow = group_sum<32>(nbelow);
          if (lane == 0) {
#pragma unroll
            for (int i = 0; i < kWin; ++i) {
              s_wsum[warp][i] = acc[i];
              s_wsum[warp][kWin + i] = cnt[i];
            }
            s_wsum[warp][2 * kWin] = below;
            s_wsum[warp][2 * kWin + 1] = nbelow;
          }
          __syncthreads();
          if (tid == 0) {
            double a[kWin], n[kWin], bl = 0.0, bn = 0.0;
            for (int i = 0; i < kWin; ++i) a[i] = n[i] = 0.0;
            for (int w = 0; w < kWarps; ++w) {
              for (int i = 0; i < kWin; ++i) {
                a[i] += s_wsum[w][i];
                n[i] += s_wsum[w][kWin + i];
              }
              bl += s_wsum[w][2 * kWin];
              bn += s_wsum[w][2 * kWin + 1];
            }
            if (base == d_top) {
              double total = bl;
              for (int i = 0; i < kWin; ++i) total += a[i];
              target = (double)Pp * total;
            }
            // the lowest digit of the window with elements and mass above < target
            int pick = -1;
            double above = above_all, pick_above = 0.0;
            for (int i = 0; i < kWin && base - i >= 0; ++i) {
              if (n[i] > 0.0) {
                if (above < target) {
                  pick = base - i;
                  pick_above = above;
                } else {
                  break;
                }
              }
              above += a[i];
            }
            // the boundary is below the window only if the mass of the window and
            // of everything above it is still below the target and elements
            // remain below it
            const bool lower = above < target && bn > 0.0 && base - kWin >= 0;
            s_digit = lower ? -1 : pick;
            s_dval[0] = lower ? above : pick_above;
            s_dval[1] = target;
          }
          __syncthreads();
          d0 = s_digit;
          above_all = s_dval[0];
          target = s_dval[1];
          __syncthreads();
        }
        // further levels inside the chosen bin: fixed-point masses (2^-40) with
        // shared atomics, only for the elements of that bin
        uint32_t prefix = (uint32_t)max(d0, 0);
        for (int L = 1; L < kLevels; ++L) {
          const int shift = 8 * (kLevels - 1 - L);
          clear_counts();
          each([&](bool ok, float x) {
            const uint32_t k = trunc_key<E>(x);
            const bool in = ok && k >= tau_k && (k >> (shift + 8)) == prefix;
            if (in) {
              const float w = fast_ex2(fmaf(x, c, -cm));
              const int d = (int)((k >> shift) & 0xffu);
              atomicAdd(&s_mass[d], __float2ull_rn(w * 0x1p40f));
            }
            count_add(s_whist[warp], in, (int)((k >> shift) & 0xffu));
          });
          sum_counts();
          if (warp == 0) {
            unsigned long long above;
            const int d = pick_digit(s_cnt, s_mass, 1, 0ull, target - above_all, 0x1p-40, &above);
            if (lane == 0) {
              s_digit = d;
              s_above = above;
            }
          }
          __syncthreads();
          prefix = (prefix << 8) | (uint32_t)s_digit;
          above_all += (double)s_above * 0x1p-40;
          __syncthreads();
        }
        tau = max(tau, prefix);
      }
    }
    if (P.thr_target) {
      // threshold mode: the verify round masks the row as it loads it
      if (tid == 0) (is_draft ? P.thr_draft : P.thr_target)[local] = copy ? 0u : tau;
      __syncthreads();
      continue;
    }
    // ---- output: the kept logits, -inf elsewhere (or the row as it is) ----------
    char* out = reinterpret_cast<char*>(is_draft ? P.draft_out : P.target_out) +
                (size_t)local * row_bytes;
    if constexpr (kFast) {
      // packed: -0 keys just below +0 here, so a threshold at +0 moves below it
      const uint4* rv = reinterpret_cast<const uint4*>(in);
      uint4* ov = reinterpret_cast<uint4*>(out);
      const uint32_t tk = tau == 0x8000u ? 0x7fffu : tau;
      const uint32_t t2 = tk | (tk << 16);
      for (int i0 = tid; i0 < nvec; i0 += kPackedOutLoads * kTruncThreads) {
        uint4 qs[kPackedOutLoads];
#pragma unroll
        for (int u = 0; u < kPackedOutLoads; ++u) {
          const int i = i0 + u * kTruncThreads;
          if (i < nvec) qs[u] = ld_last_use(rv + i);
        }
#pragma unroll
        for (int u = 0; u < kPackedOutLoads; ++u) {
          const int i = i0 + u * kTruncThreads;
          if (i >= nvec) break;
          uint4 q = qs[u];
          if (!copy) {
            q.x = keep_bf16x2(q.x, t2);
            q.y = keep_bf16x2(q.y, t2);
            q.z = keep_bf16x2(q.z, t2);
            q.w = keep_bf16x2(q.w, t2);
          }
          st_streaming(ov + i, q);
        }
      }
    } else if (kAligned) {
      const uint4* rv = reinterpret_cast<const uint4*>(in);
      uint4* ov = reinterpret_cast<uint4*>(out);
      for (int i0 = tid; i0 < nvec; i0 += kOutLoads * kTruncThreads) {
        uint4 qs[kOutLoads];
#pragma unroll
        for (int u = 0; u < kOutLoads; ++u) {
          const int i = i0 + u * kTruncThreads;
          if (i < nvec) qs[u] = ld_last_use(rv + i);
        }
#pragma unroll
        for (int u = 0; u < kOutLoads; ++u) {
          const int i = i0 + u * kTruncThreads;
          if (i >= nvec) break;
          uint4 q = qs[u];
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
          st_streaming(ov + i, q);
        }
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
