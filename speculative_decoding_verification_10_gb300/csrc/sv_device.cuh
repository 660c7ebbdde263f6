// sv_device.cuh -- device building blocks of the verify kernels (sm_103a).
//
// Counter-based randomness, vector loads, and the per-thread accumulators of
// the three row reductions the verify step needs:
//   * online max / sum-exp of x/T (the softmax normaliser of p_i and q_i),
//   * argmax with lowest index (greedy rows),
//   * the best (score, index) of the exponential race
//     argmax_v (log2 w_v - log2 E_v)  ==  argmin_v E_v / w_v
//     (correction and bonus draws; "Speculative Decoding: Medusa, MTP, EAGLE,
//     DFlash, DDTree, and DSpark", section 1).
// Every quantity is kept in the base-2 log domain: c = log2(e)/T, so
// exp(x/T - m) = 2^(c*x - m2) and the MUFU ex2/lg2 units do the work.
#pragma once

#include <cstdint>

#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace sv {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kNegInf = -__builtin_huge_valf();

// ---------------------------------------------------------------------------
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11).  Counter
// (floor(v/4), position, request lo, stream | request hi << 8), key = seed.
// ---------------------------------------------------------------------------
struct PhiloxKey {
  uint32_t k0, k1;
};

__device__ __forceinline__ uint4 philox4x32_10(uint4 c, PhiloxKey key) {
  uint32_t k0 = key.k0, k1 = key.k1;
#pragma unroll
  for (int round = 0; round < 10; ++round) {
    const uint32_t lo0 = c.x * 0xD2511F53u;
    const uint32_t hi0 = __umulhi(c.x, 0xD2511F53u);
    const uint32_t lo1 = c.z * 0xCD9E8D57u;
    const uint32_t hi1 = __umulhi(c.z, 0xCD9E8D57u);
    c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return c;
}

__device__ __forceinline__ uint32_t word_of(uint4 r, int i) {
  return i == 0 ? r.x : (i == 1 ? r.y : (i == 2 ? r.z : r.w));
}

// Acceptance uniform of one draft position: word 0 of stream 0, as
// (w >> 8) * 2^-24 -- exactly representable in fp32.
__device__ __forceinline__ float accept_uniform(PhiloxKey key, uint32_t pos, uint32_t req_lo,
                                                uint32_t req_hi) {
  const uint4 r = philox4x32_10(make_uint4(0u, pos, req_lo, 0u | (req_hi << 8)), key);
  return (float)(r.x >> 8) * 0x1p-24f;
}

__device__ __forceinline__ float fast_ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float fast_lg2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Race exponential E = -ln(U), U = (w + 1/2) 2^-32, without branches or
// library calls.  Where d = 1 - U = (~w + 1/2) 2^-32 is below 1/8, E is the
// series d + d^2/2 + ... + d^8/8 (its remainder is below 1.2e-8 of E), from
// d formed exactly from ~w; elsewhere U itself is accurate to 2^-24 and
// |log2 U| > 0.19, so E = -ln 2 log2 U with the hardware lg2 keeps a relative
// error near 1e-6 at worst (1e-7 for U below one half).
__device__ __forceinline__ float race_exponential(uint32_t w) {
  const float d = fmaf((float)(~w), 0x1p-32f, 0x1p-33f);
  float s = 0.125f;
  s = fmaf(s, d, 0.14285715f);
  s = fmaf(s, d, 0.16666667f);
  s = fmaf(s, d, 0.2f);
  s = fmaf(s, d, 0.25f);
  s = fmaf(s, d, 0.33333334f);
  s = fmaf(s, d, 0.5f);
  s = fmaf(s, d, 1.0f);
  const float u = fmaf((float)w, 0x1p-32f, 0x1p-33f);
  return d < 0.125f ? s * d : -fast_lg2(u) * kLn2;
}

// Upper bound of -log2(E) for the race exponential of word w, from integer
// operations only, with a margin of 1e-3 over the computed -log2(E):
//   w <  2^31:  U < 1/2, so E > ln 2 and -log2 E < 0.5288;
//   w >= 2^31:  d = 1 - U = (~w + 1/2) 2^-32 > 2^-(1 + clz(~w)) and E > d,
//               so -log2 E < 1 + clz(~w)   (clz(0) = 32 covers ~w = 0).
// Because rounding is monotonic, fmaf(x, c, race_gain_bound(w)) is never
// below the computed score fmaf(x, c, -log2 E): elements whose bound cannot
// reach the best score so far can skip the exponential entirely.
//   (For w < 2^31, ~w >= 2^31 gives clz = 0 and the bound 1.001, which is
//   looser than 0.529 but still valid, so one branch-free formula serves.)
__device__ __forceinline__ float race_gain_bound(uint32_t w) {
  return (float)__clz(~w) + 1.001f;
}

// Sum over aligned groups of kLanes lanes (every lane gets its group's sum).
template <int kLanes>
__device__ __forceinline__ float group_sum(float v) {
#pragma unroll
  for (int off = kLanes / 2; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
  return v;
}

// ---------------------------------------------------------------------------
// Asynchronous global -> shared copies (cp.async, 16 bytes, L2 only).  Each
// thread waits for its own copies with cp.async.wait_group, a hardware wait.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  const uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem) : "memory");
}
// The copy only where `on` holds, as a predicated instruction (no branch).
__device__ __forceinline__ void cp_async16_if(void* smem, const void* gmem, bool on) {
  const uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %2, 0;\n\t"
      "@p cp.async.cg.shared.global [%0], [%1], 16;\n\t}" ::"r"(s),
      "l"(gmem), "r"((int)on)
      : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}

// GPU-scope release/acquire fence: a writer's fence before its counter RMW and
// the reader's fence after the RMW that completes the count order the
// writer's earlier stores before the reader's later loads (the counter's RMWs
// carry the order from every writer to the last one).  Lighter than the
// sequentially consistent fence, which these hand-offs do not need.
__device__ __forceinline__ void fence_acq_rel_gpu() {
  asm volatile("fence.acq_rel.gpu;" ::: "memory");
}

// Named CTA barriers (hardware, no polling): `arrive` counts the calling warp
// in and goes on, `sync` counts it in and waits until `n` threads have come.
// Both order the caller's earlier memory accesses before the barrier's
// completion for every participating thread.
__device__ __forceinline__ void named_bar_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
__device__ __forceinline__ void named_bar_arrive(int id, int n) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// Publishing a count in shared memory: a release store by the writer, an
// acquire load by the readers (orders only what these two accesses need, unlike
// a fence, which would also wait for the reader's copies in flight).
__device__ __forceinline__ int ld_acquire_shared(const int* p) {
  int v;
  const uint32_t a = (uint32_t)__cvta_generic_to_shared(p);
  asm volatile("ld.acquire.cta.shared::cta.b32 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_shared(int* p, int v) {
  const uint32_t a = (uint32_t)__cvta_generic_to_shared(p);
  asm volatile("st.release.cta.shared::cta.b32 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}

// ---------------------------------------------------------------------------
// Loads.  Logit rows are streamed once: 16-byte non-coherent loads that skip L1.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 r;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(p));
  return r;
}

// Element types: fp32 (4 per 16 B) and bf16 (8 per 16 B).
struct F32 {
  static constexpr int kVec = 4;
  static constexpr int kBytes = 4;
  __device__ static __forceinline__ void unpack(uint4 v, float (&x)[kVec]) {
    x[0] = __uint_as_float(v.x);
    x[1] = __uint_as_float(v.y);
    x[2] = __uint_as_float(v.z);
    x[3] = __uint_as_float(v.w);
  }
  __device__ static __forceinline__ uint4 pad() {
    const uint32_t n = 0xff800000u;  // -inf
    return make_uint4(n, n, n, n);
  }
  __device__ static __forceinline__ float load1(const void* row, int i) {
    return __ldg(reinterpret_cast<const float*>(row) + i);
  }
};

struct BF16 {
  static constexpr int kVec = 8;
  static constexpr int kBytes = 2;
  __device__ static __forceinline__ void unpack(uint4 v, float (&x)[kVec]) {
    // little-endian: the lower-addressed element is the low half
    x[0] = __uint_as_float(v.x << 16);
    x[1] = __uint_as_float(v.x & 0xffff0000u);
    x[2] = __uint_as_float(v.y << 16);
    x[3] = __uint_as_float(v.y & 0xffff0000u);
    x[4] = __uint_as_float(v.z << 16);
    x[5] = __uint_as_float(v.z & 0xffff0000u);
    x[6] = __uint_as_float(v.w << 16);
    x[7] = __uint_as_float(v.w & 0xffff0000u);
  }
  __device__ static __forceinline__ uint4 pad() {
    const uint32_t n = 0xff80ff80u;  // -inf, -inf
    return make_uint4(n, n, n, n);
  }
  __device__ static __forceinline__ float load1(const void* row, int i) {
    const unsigned short h = __ldg(reinterpret_cast<const unsigned short*>(row) + i);
    return __uint_as_float((uint32_t)h << 16);
  }
};

// Two bf16 logits packed in a 32-bit word, worked on together.  Their order
// keys: a positive logit gets its bits with the top bit set, a negative one its
// bits inverted, so keys compare as the logits do (-inf lowest; a positive NaN
// keys above +inf, a negative one below -inf).  Unlike trunc_key, -0 keeps
// its own key 0x7fff, just below +0's 0x8000.
__device__ __forceinline__ uint32_t bf16x2_keys(uint32_t w) {
  const uint32_t neg = (w >> 15) & 0x00010001u;  // sign of each half, moved to its bit 0
  return w ^ ((neg * 0x7fffu) | 0x80008000u);
}
__device__ __forceinline__ uint32_t max_u16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t min_u16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("min.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
// The word with each half whose key is below the threshold (t2: the 16-bit
// key in both halves) replaced by -inf.
__device__ __forceinline__ uint32_t keep_bf16x2(uint32_t w, uint32_t t2) {
  const uint32_t k = bf16x2_keys(w);
  const uint32_t d = max_u16x2(k, t2) ^ k;  // a half is zero where its key >= the threshold
  const uint32_t nz = (((d & 0x7fff7fffu) + 0x7fff7fffu) | d) & 0x80008000u;
  const uint32_t drop = (nz >> 15) * 0xffffu;  // 0xffff in each half to drop
  return (w & ~drop) | (0xff80ff80u & drop);
}

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

// Truncation on load: a truncated row keeps the logits whose order key is at
// or above the row's threshold key and reads -inf for the others, so every
// pass over the row sees the truncated distribution.  A threshold key of 0
// keeps the row as it is (its callers test for it, so a NaN stays visible).
// The test is the logit comparison x >= x_thr, x_thr the logit of the key: on
// the rows that get a threshold (no NaN) it keeps exactly the keys >= thr, -0
// and +0 comparing equal as they share a key.
// The threshold logit of a key, as the masks take it: bf16 in both halves of
// a word, fp32 as its bits.
template <typename E>
__device__ __forceinline__ uint32_t mask_bits(uint32_t key) {
  if (E::kBytes == 2) {
    const uint32_t h = (key & 0x8000u) ? (key & 0x7fffu) : (~key & 0xffffu);
    return h | (h << 16);
  }
  return (key & 0x80000000u) ? (key & 0x7fffffffu) : ~key;
}
template <typename E>
__device__ __forceinline__ float mask1(float x, uint32_t key) {
  if (key == 0u) return x;
  const uint32_t b = mask_bits<E>(key);
  const float t = __uint_as_float(E::kBytes == 2 ? (b << 16) : b);
  return x >= t ? x : kNegInf;
}
// A vector with `bits` = mask_bits(key) of a key that is not 0: bf16 pairs
// compared and selected two at a time (a compare mask and one bit select).
template <typename E>
__device__ __forceinline__ void mask_vec(uint4& v, uint32_t bits) {
  uint32_t* w = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    if (E::kBytes == 2) {
      const unsigned m = __hge2_mask(*reinterpret_cast<const __nv_bfloat162*>(&w[e]),
                                     *reinterpret_cast<const __nv_bfloat162*>(&bits));
      w[e] = (w[e] & m) | (0xff80ff80u & ~m);
    } else {
      w[e] = __uint_as_float(w[e]) >= __uint_as_float(bits) ? w[e] : 0xff800000u;
    }
  }
}

// ---------------------------------------------------------------------------
// Accumulators.  Each is a per-thread state with an element update and a
// commutative, associative merge; results do not depend on how a row is split.
// ---------------------------------------------------------------------------

// Online softmax normaliser in base 2: m = max_v c*x_v, s = sum_v 2^(c*x_v - m).
struct SoftmaxAcc {
  float m, s;
  __device__ __forceinline__ void init() {
    m = kNegInf;
    s = 0.f;
  }
  template <int N>
  __device__ __forceinline__ void add(const float (&x)[N], float c) {
    float mx = x[0];
#pragma unroll
    for (int e = 1; e < N; ++e) mx = fmaxf(mx, x[e]);
    const float vm = mx * c;
    if (vm > m) {
      s *= fast_ex2(m - vm);
      m = vm;
    }
    if (m != kNegInf) {
      float s0 = 0.f, s1 = 0.f;
#pragma unroll
      for (int e = 0; e < N; e += 2) {
        s0 += fast_ex2(fmaf(x[e], c, -m));
        if (e + 1 < N) s1 += fast_ex2(fmaf(x[e + 1], c, -m));
      }
      s += s0 + s1;
    }
  }
  __device__ __forceinline__ void add1(float x, float c) {
    float a[1] = {x};
    add<1>(a, c);
  }
  __device__ static __forceinline__ SoftmaxAcc merge(SoftmaxAcc a, SoftmaxAcc b) {
    SoftmaxAcc r;
    r.m = fmaxf(a.m, b.m);
    if (r.m == kNegInf) {
      r.s = a.s + b.s;  // both empty (or NaN carried)
    } else {
      r.s = a.s * fast_ex2(a.m - r.m) + b.s * fast_ex2(b.m - r.m);
    }
    return r;
  }
  __device__ __forceinline__ SoftmaxAcc shfl_xor(int lane_mask) const {
    SoftmaxAcc o;
    o.m = __shfl_xor_sync(0xffffffffu, m, lane_mask);
    o.s = __shfl_xor_sync(0xffffffffu, s, lane_mask);
    return o;
  }
};

// Softmax normaliser with a lazy reference: m is fixed from the first finite
// vector a thread sees, and only raised when a vector's terms overflow (a
// term 2^(c*x - m) above 2^100).  Terms far below m underflow to 0, which is
// harmless: the element that set m contributes 1 to s.  The sum is kept as a
// float2 and updated with packed FMA/ADD (two lanes per instruction).
struct LazySoftmax {
  float m;
  float2 s;
  __device__ __forceinline__ void init() {
    m = kNegInf;
    s = make_float2(0.f, 0.f);
  }
  template <int N>
  __device__ __forceinline__ float vmax(const float (&x)[N]) {
    float mx = x[0];
#pragma unroll
    for (int e = 1; e < N; ++e) mx = fmaxf(mx, x[e]);
    return mx;
  }
  // terms of one vector relative to the current m, summed in pairs
  template <int N>
  __device__ __forceinline__ float2 terms(const float (&x)[N], float c) const {
    const float2 cc = make_float2(c, c), nm = make_float2(-m, -m);
    float2 acc = make_float2(0.f, 0.f);
#pragma unroll
    for (int e = 0; e < N; e += 2) {
      const float2 t = __ffma2_rn(make_float2(x[e], x[e + 1]), cc, nm);
      acc = __fadd2_rn(acc, make_float2(fast_ex2(t.x), fast_ex2(t.y)));
    }
    return acc;
  }
  template <int N>
  __device__ __forceinline__ void add(const float (&x)[N], float c) {
    if (m == kNegInf) {
      const float vm = vmax(x) * c;
      if (vm == kNegInf) return;  // nothing finite yet (NaN falls through)
      m = vm;
    }
    float2 t = terms(x, c);
    if (!(t.x + t.y <= 0x1p100f)) {
      // overflow (or NaN): raise m to this vector's maximum and redo it
      const float vm = fmaxf(vmax(x) * c, m);
      const float sc = fast_ex2(m - vm);
      s = make_float2(s.x * sc, s.y * sc);
      m = vm;
      t = terms(x, c);
    }
    s = __fadd2_rn(s, t);
  }
  __device__ __forceinline__ void add1(float x, float c) {
    float a[2] = {x, kNegInf};
    add<2>(a, c);
  }
  // Two vectors with one overflow check.  A failed check (the sum left
  // (0, 2^100], including m = -inf, which makes the terms inf or NaN) raises m
  // to the running maximum and redoes both vectors; NaN logits leave s NaN.
  template <int N>
  __device__ __forceinline__ void add2(const float (&x0)[N], const float (&x1)[N], float c) {
    float2 t = __fadd2_rn(terms(x0, c), terms(x1, c));
    if (!(t.x + t.y <= 0x1p100f)) {
      const float vm = fmaxf(fmaxf(vmax(x0), vmax(x1)) * c, m);
      if (vm == kNegInf) return;  // nothing finite yet
      const float sc = fast_ex2(m - vm);
      s = make_float2(s.x * sc, s.y * sc);
      m = vm;
      t = __fadd2_rn(terms(x0, c), terms(x1, c));
    }
    s = __fadd2_rn(s, t);
  }
  __device__ __forceinline__ SoftmaxAcc result() const {
    SoftmaxAcc r;
    r.m = m;
    r.s = s.x + s.y;
    return r;
  }
};

// Best (value, index): larger value wins, lower index on ties; idx -1 = none.
struct BestAcc {
  float v;
  int idx;
  uint32_t nan;
  __device__ __forceinline__ void init() {
    v = kNegInf;
    idx = -1;
    nan = 0u;
  }
  __device__ __forceinline__ void take(float val, int i) {
    // callers feed indices in increasing order, so strict '>' keeps the lowest
    if (val > v) {
      v = val;
      idx = i;
    }
  }
  // the full order (value, then lower index): for callers without index order
  __device__ __forceinline__ void take_cmp(float val, int i) {
    if (better(val, i, v, idx)) {
      v = val;
      idx = i;
    }
  }
  __device__ static __forceinline__ bool better(float va, int ia, float vb, int ib) {
    return va > vb || (va == vb && (uint32_t)ia < (uint32_t)ib);
  }
  __device__ static __forceinline__ BestAcc merge(BestAcc a, BestAcc b) {
    BestAcc r = better(b.v, b.idx, a.v, a.idx) ? b : a;
    r.nan = a.nan | b.nan;
    return r;
  }
  __device__ __forceinline__ BestAcc shfl_xor(int lane_mask) const {
    BestAcc o;
    o.v = __shfl_xor_sync(0xffffffffu, v, lane_mask);
    o.idx = __shfl_xor_sync(0xffffffffu, idx, lane_mask);
    o.nan = __shfl_xor_sync(0xffffffffu, nan, lane_mask);
    return o;
  }
};

template <typename Acc>
__device__ __forceinline__ Acc warp_reduce(Acc a) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) a = Acc::merge(a, a.shfl_xor(off));
  return a;
}

// Block-wide reduction; the result is valid in thread 0.  `scratch` holds one
// Acc per warp.
template <typename Acc, int kThreads>
__device__ __forceinline__ Acc block_reduce(Acc a, Acc* scratch) {
  constexpr int kWarps = kThreads / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  a = warp_reduce(a);
  if (lane == 0) scratch[warp] = a;
  __syncthreads();
  if (warp == 0) {
    Acc b = scratch[lane < kWarps ? lane : 0];
    if (lane >= kWarps) b.init();
    a = warp_reduce(b);
  }
  __syncthreads();
  return a;
}

}  // namespace sv
