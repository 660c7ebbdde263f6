// sv_kernels.cuh -- the fused verify kernel: one persistent launch per round.
//
// Work items.  The logit rows of the batch are numbered request by request,
//     request r:  t_0 d_0 t_1 d_1 ... t_{k-1} d_{k-1} t_k     (2 k_r + 1 rows)
// so row n of request r is n - (r + 2 drf_off(r)); every row is split into
// `nch` vocab chunks and item = row * nch + chunk.  CTA b takes items
// b, b + grid, b + 2 grid, ...  Draft rows of greedy requests are skipped.
//
// Per item the CTA reduces its chunk to a 16-byte partial:
//   sampling target row i < k, draft row i : softmax normaliser (m, S) of c*x,
//                                            c = log2(e)/T   (p_i, q_i)
//   sampling target row k                  : bonus race argmax c*x_v - log2 E_v
//   greedy target row                      : argmax (lowest index)
// The CTA that completes a row (atomic counter) merges its partials; the CTA
// that completes a request runs the acceptance scan in one warp, writes all of
// the request's outputs and, on a rejection at position j, publishes a
// residual job: the draw from [p_j - q_j]_+ over the rows t_j, d_j, split
// into nch chunks that any CTA may claim.  Claims are checked between items, so
// the two rows are re-read while they are still in L2.
//
// Memory pipeline.  Each thread streams its 16-byte vectors of successive
// items through a private ring of shared memory with cp.async (kStages stages
// of kStageVecs vectors); it only ever reads back what it copied itself, so
// the ring needs no block barrier, and cp.async.wait_group is a hardware wait.
// Loads run kStages-1 stages ahead, across item boundaries.
//
// No CTA waits for another, except that a CTA with no items left polls the
// residual queue for at most P.spin_limit rounds before it exits; exiting is
// always safe because the CTA that publishes a residual job drains it itself.
// The last CTA to exit resets the shared counters for the next round.
#pragma once

#include "sv_device.cuh"

namespace sv {

constexpr int kThreads = 256;
constexpr int kStages = 6;
constexpr int kStageVecs = 2;
constexpr int kMaxBatch = 4096;   // requests per launch (prefix sums live in shared memory)
constexpr int kResUnroll = 4;

enum RowKind : int { kSkip = -1, kSoftmax = 0, kArgmax = 1, kRace = 2 };
enum ReqMode : int { kBadTemp = 0, kGreedy = 1, kSampling = 2 };

// Status bits (equal to the SPECVERIFY_STATUS_* values of the header).
constexpr uint32_t kStBadToken = 1u, kStBadK = 2u, kStBadTemp = 4u, kStNonfinite = 8u,
                   kStBadTotal = 16u, kStNoDraft = 64u;

struct __align__(16) Partial {
  float a;       // softmax: m  | best: value
  float b;       // softmax: S  | unused
  int idx;       // best: index | unused
  uint32_t bad;  // NaN seen
};

// Shared counters of a round (reset by the last CTA to exit).
enum Counter : int {
  kCntReserve = 0,    // residual slots reserved
  kCntPublished = 1,  // residual chunks published
  kCntClaimed = 2,    // residual chunks claimed
  kCntReqDone = 3,    // requests scanned
  kCntExit = 4,       // CTAs finished
  kCntStatus = 5,     // status bits of this round
  kCntLastStatus = 6, // status bits of the previous round
  kCntCount = 8
};

struct Params {
  const void* target;
  const void* draft;
  const int32_t* tokens;
  const int32_t* num_draft;
  const float* temperature;
  const int64_t* request_ids;
  PhiloxKey key;
  int batch, total_draft, max_k, vocab;
  int nch;      // chunks per row
  int nper;     // 16-byte vectors per thread per chunk (multiple of kStageVecs)
  int n_items;  // (batch + 2 total_draft) * nch
  int spin_limit;
  int32_t* accepted_len;
  int32_t* committed;
  uint8_t* flags;
  float* p_y;
  float* q_y;
  float* u_dbg;
  int32_t* req_status;
  Partial* part;       // [rows * nch]
  Partial* rowres;     // [rows]
  int* row_cnt;        // [rows]
  int* req_cnt;        // [batch]
  unsigned long long* res_slots;  // [batch]: r | j << 24 | chunks left << 32
  Partial* part2;      // [batch * nch]
  int* res_cnt;        // [batch]
  int* ctr;            // [kCntCount]
};

__device__ __forceinline__ Partial ld_cg(const Partial* p) {
  const int4 v = __ldcg(reinterpret_cast<const int4*>(p));
  return Partial{__int_as_float(v.x), __int_as_float(v.y), v.z, (uint32_t)v.w};
}

__device__ __forceinline__ int ld_volatile(const int* p) {
  return *reinterpret_cast<const volatile int*>(p);
}

__device__ __forceinline__ int req_mode(float t) {
  if (t == 0.f) return kGreedy;
  return (t >= 1.17549435e-38f && t <= 3.40282347e+38f) ? kSampling : kBadTemp;
}

// ---------------------------------------------------------------------------
// Work-item decoding (prefix sums of num_draft in shared memory).
// ---------------------------------------------------------------------------
struct Item {
  const char* row;  // element 0 of the logit row
  int kind;
  int r, pos, n, ch;
  float c;
};

template <typename E>
__device__ __forceinline__ Item decode_item(const Params& P, const int* s_doff, int item) {
  Item it;
  const int n = item / P.nch;
  it.n = n;
  it.ch = item - n * P.nch;
  // largest r with r + 2 drf_off(r) <= n
  int lo = 0, hi = P.batch - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (mid + 2 * s_doff[mid] <= n) lo = mid;
    else hi = mid - 1;
  }
  const int r = lo;
  const int d0 = s_doff[r];
  const int k = s_doff[r + 1] - d0;
  const int l = n - (r + 2 * d0);
  const float t = __ldg(P.temperature + r);
  const int mode = req_mode(t);
  const bool is_draft = (l < 2 * k) && (l & 1);
  const int pos = l < 2 * k ? (l >> 1) : k;
  it.r = r;
  it.pos = pos;
  it.c = mode == kSampling ? kLog2e / t : 0.f;
  const size_t row_bytes = (size_t)P.vocab * E::kBytes;
  if (is_draft) {
    it.kind = (mode == kSampling && P.draft != nullptr) ? kSoftmax : kSkip;
    it.row = reinterpret_cast<const char*>(P.draft) + (size_t)(d0 + pos) * row_bytes;
  } else {
    it.kind = mode == kSampling ? (pos < k ? kSoftmax : kRace) : kArgmax;
    it.row = reinterpret_cast<const char*>(P.target) + (size_t)(d0 + r + pos) * row_bytes;
  }
  return it;
}

// Rows a request contributes to its completion counter.
__device__ __forceinline__ int rows_of_request(const Params& P, int k, int mode) {
  return (mode == kSampling && P.draft != nullptr) ? 2 * k + 1 : k + 1;
}

// Aligned-vector geometry of a row and the vector range of chunk ch.
template <typename E>
struct Geom {
  int head, nvec, tail, vbeg, vend;
  __device__ __forceinline__ void init(const char* row, int vocab, int ch, int chv) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(row);
    int h = (int)(((16u - (uint32_t)(a & 15u)) & 15u) / E::kBytes);
    if (h > vocab) h = vocab;
    head = h;
    nvec = (vocab - h) / E::kVec;
    tail = vocab - h - nvec * E::kVec;
    vbeg = ch * chv;
    vend = min(nvec, vbeg + chv);
  }
  __device__ __forceinline__ const uint4* vecs(const char* row) const {
    return reinterpret_cast<const uint4*>(row + (size_t)head * E::kBytes);
  }
};

// ---------------------------------------------------------------------------
// The per-thread copy ring.
// ---------------------------------------------------------------------------
template <typename E>
struct LoadCursor {
  int j;             // ordinal of the current item among this CTA's items
  int st;            // stage within the item
  const uint4* base;
  int vbeg, vend;
  bool active;

  __device__ __forceinline__ void seek(const Params& P, const int* s_doff) {
    active = false;
    for (;;) {
      const int item = blockIdx.x + j * gridDim.x;
      if (item >= P.n_items) return;
      const Item it = decode_item<E>(P, s_doff, item);
      if (it.kind != kSkip) {
        Geom<E> g;
        g.init(it.row, P.vocab, it.ch, P.nper * kThreads);
        base = g.vecs(it.row);
        vbeg = g.vbeg;
        vend = g.vend;
        st = 0;
        active = true;
        return;
      }
      ++j;
    }
  }

  // copy the next stage into ring slot `slot` and commit one group
  __device__ __forceinline__ void issue(const Params& P, const int* s_doff, uint4* ring, int slot) {
    if (active) {
#pragma unroll
      for (int u = 0; u < kStageVecs; ++u) {
        const int vi = vbeg + (st * kStageVecs + u) * kThreads + (int)threadIdx.x;
        if (vi < vend) cp_async16(ring + (slot * kStageVecs + u) * kThreads + threadIdx.x, base + vi);
      }
    }
    cp_async_commit();
    if (active && ++st == P.nper / kStageVecs) {
      ++j;
      seek(P, s_doff);
    }
  }
};

// Streams the chunk's vectors out of the ring: for each stage, wait for it,
// refill the ring one stage ahead, then hand the thread's vectors to f(x, e0).
template <typename E, typename F>
__device__ __forceinline__ void consume_item(const Params& P, const int* s_doff, uint4* ring,
                                             LoadCursor<E>& lc, int& g_stage, const Geom<E>& g,
                                             F&& f) {
  const int spi = P.nper / kStageVecs;
  for (int st = 0; st < spi; ++st) {
    cp_async_wait<kStages - 2>();
    const int slot = g_stage % kStages;
    uint4 v[kStageVecs];
#pragma unroll
    for (int u = 0; u < kStageVecs; ++u) v[u] = ring[(slot * kStageVecs + u) * kThreads + threadIdx.x];
    lc.issue(P, s_doff, ring, (g_stage + kStages - 1) % kStages);
    ++g_stage;
#pragma unroll
    for (int u = 0; u < kStageVecs; ++u) {
      const int vi = g.vbeg + (st * kStageVecs + u) * kThreads + (int)threadIdx.x;
      float x[E::kVec];
      E::unpack(vi < g.vend ? v[u] : E::pad(), x);
      f(x, g.head + vi * E::kVec);
    }
  }
}

// Philox words for elements e0 .. e0+N-1 where e0 % 4 == OFF (race stream 1).
template <int N, int OFF>
struct RaceWords {
  static constexpr int kBlocks = (OFF + N + 3) / 4;
  uint4 r[kBlocks];
  __device__ __forceinline__ void make(int e0, uint32_t pos, uint32_t req_lo, uint32_t req_hi,
                                       PhiloxKey key) {
    const uint32_t b0 = (uint32_t)e0 >> 2;
#pragma unroll
    for (int b = 0; b < kBlocks; ++b)
      r[b] = philox4x32_10(make_uint4(b0 + b, pos, req_lo, 1u | (req_hi << 8)), key);
  }
  __device__ __forceinline__ uint32_t word(int e) const {
    return word_of(r[(OFF + e) >> 2], (OFF + e) & 3);
  }
};

__device__ __forceinline__ uint32_t race_word1(int e, uint32_t pos, uint32_t req_lo,
                                               uint32_t req_hi, PhiloxKey key) {
  const uint4 r = philox4x32_10(make_uint4((uint32_t)e >> 2, pos, req_lo, 1u | (req_hi << 8)), key);
  return word_of(r, e & 3);
}

// Race candidate with the integer bound; `thr` is the best exact score the
// warp has seen (an element that cannot reach it cannot win).
__device__ __forceinline__ void race_take(BestAcc& acc, float thr, float x, float c, uint32_t w,
                                          int e) {
  acc.nan |= (x != x);
  if (fmaf(x, c, race_gain_bound(w)) >= thr) {
    const float s = fmaf(x, c, -fast_lg2(race_exponential(w)));
    acc.take(s, e);
  }
}

struct RequestKey {
  uint32_t lo, hi;
};

__device__ __forceinline__ RequestKey request_key(const Params& P, int r) {
  const uint64_t id = P.request_ids ? (uint64_t)P.request_ids[r] : (uint64_t)r;
  return RequestKey{(uint32_t)id, (uint32_t)(id >> 32)};
}

// ---------------------------------------------------------------------------
// Per-kind chunk reductions (ring-fed).
// ---------------------------------------------------------------------------
template <typename E>
__device__ __forceinline__ SoftmaxAcc item_softmax(const Params& P, const int* s_doff, uint4* ring,
                                                   LoadCursor<E>& lc, int& gs, const Item& it,
                                                   const Geom<E>& g) {
  SoftmaxAcc acc;
  acc.init();
  if (it.ch == 0 && (int)threadIdx.x < g.head) acc.add1(E::load1(it.row, threadIdx.x), it.c);
  consume_item<E>(P, s_doff, ring, lc, gs, g,
                  [&](const float(&x)[E::kVec], int) { acc.add(x, it.c); });
  if (it.ch == P.nch - 1 && (int)threadIdx.x < g.tail)
    acc.add1(E::load1(it.row, g.head + g.nvec * E::kVec + threadIdx.x), it.c);
  return acc;
}

template <typename E>
__device__ __forceinline__ BestAcc item_argmax(const Params& P, const int* s_doff, uint4* ring,
                                               LoadCursor<E>& lc, int& gs, const Item& it,
                                               const Geom<E>& g) {
  BestAcc acc;
  acc.init();
  if (it.ch == 0 && (int)threadIdx.x < g.head) {
    const float x = E::load1(it.row, threadIdx.x);
    acc.nan |= (x != x);
    acc.take(x, threadIdx.x);
  }
  consume_item<E>(P, s_doff, ring, lc, gs, g, [&](const float(&x)[E::kVec], int e0) {
    float mx = x[0];
    uint32_t nan = (x[0] != x[0]);
#pragma unroll
    for (int e = 1; e < E::kVec; ++e) {
      mx = fmaxf(mx, x[e]);
      nan |= (x[e] != x[e]);
    }
    acc.nan |= nan;
    if (mx > acc.v) {
      int first = 0;
#pragma unroll
      for (int e = E::kVec - 1; e >= 0; --e)
        if (x[e] == mx) first = e;
      acc.v = mx;
      acc.idx = e0 + first;
    }
  });
  if (it.ch == P.nch - 1 && (int)threadIdx.x < g.tail) {
    const int e = g.head + g.nvec * E::kVec + threadIdx.x;
    const float x = E::load1(it.row, e);
    acc.nan |= (x != x);
    acc.take(x, e);
  }
  return acc;
}

template <typename E, int OFF>
__device__ __forceinline__ BestAcc item_race(const Params& P, const int* s_doff, uint4* ring,
                                             LoadCursor<E>& lc, int& gs, const Item& it,
                                             const Geom<E>& g, RequestKey rk) {
  BestAcc acc;
  acc.init();
  const uint32_t pos = (uint32_t)it.pos;
  float thr = kNegInf;
  if (it.ch == 0 && (int)threadIdx.x < g.head) {
    const int e = threadIdx.x;
    race_take(acc, kNegInf, E::load1(it.row, e), it.c, race_word1(e, pos, rk.lo, rk.hi, P.key), e);
  }
  consume_item<E>(P, s_doff, ring, lc, gs, g, [&](const float(&x)[E::kVec], int e0) {
    RaceWords<E::kVec, OFF> rw;
    rw.make(e0, pos, rk.lo, rk.hi, P.key);
#pragma unroll
    for (int e = 0; e < E::kVec; ++e) race_take(acc, thr, x[e], it.c, rw.word(e), e0 + e);
    thr = warp_max(acc.v);
  });
  if (it.ch == P.nch - 1 && (int)threadIdx.x < g.tail) {
    const int e = g.head + g.nvec * E::kVec + threadIdx.x;
    race_take(acc, kNegInf, E::load1(it.row, e), it.c, race_word1(e, pos, rk.lo, rk.hi, P.key), e);
  }
  return acc;
}

// ---------------------------------------------------------------------------
// Residual draw ("Speculative Decoding: Medusa, MTP, EAGLE, DFlash, DDTree,
// and DSpark", section 1: at the first rejection, sample from the normalised
// positive residual [p_j - q_j]_+).  Score log2 w_v - log2 E_v over w_v > 0.
// Bound: w_v <= p_v = 2^(c x_v - M_p) / S_p, so an element whose
// c x_v - M_p - log2 S_p + (bound on -log2 E_v) cannot reach the warp's best
// is skipped (a 1/64 margin covers the fp32 rounding of the exact path).
// ---------------------------------------------------------------------------
struct ResidualRow {
  float c, mp, inv_sp, mq, inv_sq, kbound;
};

__device__ __forceinline__ void residual_take(BestAcc& acc, float thr, float x, float z,
                                              const ResidualRow& rr, uint32_t w, int e) {
  if (fmaf(x, rr.c, race_gain_bound(w) + rr.kbound) >= thr) {
    const float p = fast_ex2(fmaf(x, rr.c, -rr.mp)) * rr.inv_sp;
    const float q = fast_ex2(fmaf(z, rr.c, -rr.mq)) * rr.inv_sq;
    const float wv = p - q;
    if (wv > 0.f) acc.take(fast_lg2(wv) - fast_lg2(race_exponential(w)), e);
  }
}

template <typename E, int OFF>
__device__ __forceinline__ BestAcc residual_chunk_vec(const Params& P, const char* trow,
                                                      const char* drow, const Geom<E>& g,
                                                      const ResidualRow& rr, uint32_t pos,
                                                      RequestKey rk) {
  BestAcc acc;
  acc.init();
  float thr = kNegInf;
  const uint4* tp = g.vecs(trow);
  const uint4* dp = g.vecs(drow);
  // uniform trip count across the block (warp_max below needs every lane)
  for (int v0 = g.vbeg; v0 < g.vend; v0 += kThreads * kResUnroll) {
    uint4 dt[kResUnroll], dd[kResUnroll];
#pragma unroll
    for (int u = 0; u < kResUnroll; ++u) {
      const int vi = v0 + u * kThreads + (int)threadIdx.x;
      dt[u] = vi < g.vend ? __ldcg(tp + vi) : E::pad();
      dd[u] = vi < g.vend ? __ldcg(dp + vi) : E::pad();
    }
#pragma unroll
    for (int u = 0; u < kResUnroll; ++u) {
      float x[E::kVec], z[E::kVec];
      E::unpack(dt[u], x);
      E::unpack(dd[u], z);
      const int e0 = g.head + (v0 + u * kThreads + (int)threadIdx.x) * E::kVec;
      RaceWords<E::kVec, OFF> rw;
      rw.make(e0, pos, rk.lo, rk.hi, P.key);
#pragma unroll
      for (int e = 0; e < E::kVec; ++e) residual_take(acc, thr, x[e], z[e], rr, rw.word(e), e0 + e);
      thr = warp_max(acc.v);
    }
  }
  return acc;
}

// One residual chunk; rows that do not share their 16-byte phase use plain
// element loads.
template <typename E>
__device__ BestAcc residual_chunk(const Params& P, int r, int j, int ch, const int* s_doff,
                                  const Partial& rt, const Partial& rd) {
  const size_t row_bytes = (size_t)P.vocab * E::kBytes;
  const int d0 = s_doff[r];
  const char* trow = reinterpret_cast<const char*>(P.target) + (size_t)(d0 + r + j) * row_bytes;
  const char* drow = reinterpret_cast<const char*>(P.draft) + (size_t)(d0 + j) * row_bytes;
  const float t = __ldg(P.temperature + r);
  ResidualRow rr;
  rr.c = kLog2e / t;
  rr.mp = rt.a;
  rr.inv_sp = 1.f / rt.b;
  rr.mq = rd.a;
  rr.inv_sq = 1.f / rd.b;
  // margin: 1/64 plus a few ulps of |M_p| (the exact path rounds at that scale)
  rr.kbound = -rt.a - fast_lg2(rt.b) + 0.015625f + fabsf(rt.a) * 0x1p-20f;
  const RequestKey rk = request_key(P, r);
  const uint32_t pos = (uint32_t)j;
  const int chv = P.nper * kThreads;
  Geom<E> gt, gd;
  gt.init(trow, P.vocab, ch, chv);
  gd.init(drow, P.vocab, ch, chv);
  BestAcc acc;
  if (gt.head == gd.head) {
    switch (gt.head & 3) {
      case 0: acc = residual_chunk_vec<E, 0>(P, trow, drow, gt, rr, pos, rk); break;
      case 1: acc = residual_chunk_vec<E, 1>(P, trow, drow, gt, rr, pos, rk); break;
      case 2: acc = residual_chunk_vec<E, 2>(P, trow, drow, gt, rr, pos, rk); break;
      default: acc = residual_chunk_vec<E, 3>(P, trow, drow, gt, rr, pos, rk); break;
    }
    if (ch == 0 && (int)threadIdx.x < gt.head) {
      const int e = threadIdx.x;
      residual_take(acc, kNegInf, E::load1(trow, e), E::load1(drow, e), rr,
                    race_word1(e, pos, rk.lo, rk.hi, P.key), e);
    }
    if (ch == P.nch - 1 && (int)threadIdx.x < gt.tail) {
      const int e = gt.head + gt.nvec * E::kVec + threadIdx.x;
      residual_take(acc, kNegInf, E::load1(trow, e), E::load1(drow, e), rr,
                    race_word1(e, pos, rk.lo, rk.hi, P.key), e);
    }
  } else {
    acc.init();
    const int e_beg = ch == 0 ? 0 : gt.head + gt.vbeg * E::kVec;
    const int e_end = ch == P.nch - 1 ? P.vocab : gt.head + gt.vend * E::kVec;
    for (int e = e_beg + threadIdx.x; e < e_end; e += kThreads)
      residual_take(acc, kNegInf, E::load1(trow, e), E::load1(drow, e), rr,
                    race_word1(e, pos, rk.lo, rk.hi, P.key), e);
  }
  return acc;
}

// Fallback when the residual has no mass (p <= q everywhere, i.e. p == q):
// draw from p_j with the same exponentials.  Whole row, one CTA; rare.
template <typename E>
__device__ BestAcc fallback_row(const Params& P, int r, int j, const int* s_doff) {
  const size_t row_bytes = (size_t)P.vocab * E::kBytes;
  const char* trow = reinterpret_cast<const char*>(P.target) +
                     (size_t)(s_doff[r] + r + j) * row_bytes;
  const float c = kLog2e / __ldg(P.temperature + r);
  const RequestKey rk = request_key(P, r);
  BestAcc acc;
  acc.init();
  for (int e = threadIdx.x; e < P.vocab; e += kThreads)
    race_take(acc, kNegInf, E::load1(trow, e), c, race_word1(e, (uint32_t)j, rk.lo, rk.hi, P.key), e);
  return acc;
}

// ---------------------------------------------------------------------------
// Outputs of one request, and the acceptance scan (one warp).
// ---------------------------------------------------------------------------
__device__ __forceinline__ void write_skipped(const Params& P, int r, int d0, int k, uint32_t rs,
                                              int lane) {
  const int width = P.max_k + 1;
  for (int i = lane; i < width; i += 32) P.committed[(size_t)r * width + i] = -1;
  const float nan = __int_as_float(0x7fc00000);
  for (int i = lane; i < k; i += 32) {
    P.flags[d0 + i] = 0;
    if (P.p_y) P.p_y[d0 + i] = nan;
    if (P.q_y) P.q_y[d0 + i] = nan;
    if (P.u_dbg) P.u_dbg[d0 + i] = nan;
  }
  if (lane == 0) {
    P.accepted_len[r] = -1;
    if (P.req_status) P.req_status[r] = (int32_t)rs;
    if (rs) atomicOr(reinterpret_cast<unsigned int*>(P.ctr + kCntStatus), rs);
  }
}

// "Speculative Decoding: Medusa, MTP, EAGLE, DFlash, DDTree, and DSpark",
// section 1: accept y_i with probability min(1, p_i(y_i)/q_i(y_i)), left to
// right, stopping at the first rejection (tested as u_i q_i(y_i) < p_i(y_i));
// greedy rounds keep y_i while it equals the target argmax.  Lane i handles
// draft position i.  Returns (via the queue) the residual job, if any.
template <typename E>
__device__ void scan_request(const Params& P, int r, const int* s_doff) {
  const int lane = threadIdx.x & 31;
  const int d0 = s_doff[r];
  const int k = s_doff[r + 1] - d0;
  const int t0 = d0 + r;                  // first target row
  const int n0 = r + 2 * d0;              // first entry of the request's rows
  const int width = P.max_k + 1;
  const float t = __ldg(P.temperature + r);
  const int mode = req_mode(t);
  const size_t row_bytes = (size_t)P.vocab * E::kBytes;

  uint32_t rs = 0u;
  if (mode == kBadTemp) rs |= kStBadTemp;
  int y = -1;
  if (lane < k) {
    y = P.tokens[d0 + lane];
    if (y < 0 || y >= P.vocab) rs |= kStBadToken;
  }
  if (!rs && mode == kSampling && k > 0 && P.draft == nullptr) rs |= kStNoDraft;
  rs = __reduce_or_sync(0xffffffffu, rs);

  bool accept = true;
  uint32_t bad = 0u;
  int tok = -1;
  float py = 0.f, qy = 0.f, u = 0.f;
  if (!rs) {
    if (mode == kGreedy) {
      if (lane <= k) {
        // target row i sits at entry 2i of the request's rows (draft entries unused)
        const Partial pr = ld_cg(P.rowres + n0 + 2 * lane);
        bad = pr.bad;
        tok = pr.idx;
        if (lane < k) accept = (y == tok);
      }
    } else {
      if (lane < k) {
        const Partial pt = ld_cg(P.rowres + n0 + 2 * lane);
        const Partial pd = ld_cg(P.rowres + n0 + 2 * lane + 1);
        bad = pt.bad | pd.bad;
        const char* trow = reinterpret_cast<const char*>(P.target) + (size_t)(t0 + lane) * row_bytes;
        const char* drow = reinterpret_cast<const char*>(P.draft) + (size_t)(d0 + lane) * row_bytes;
        const float c = kLog2e / t;
        const float tp = fmaf(E::load1(trow, y), c, -pt.a);  // log2(p(y) S_p)
        const float tq = fmaf(E::load1(drow, y), c, -pd.a);  // log2(q(y) S_q)
        const RequestKey rk = request_key(P, r);
        u = accept_uniform(P.key, (uint32_t)lane, rk.lo, rk.hi);
        // u q(y) < p(y), both sides scaled by S_p S_q 2^-max(tp, tq) > 0
        if (tp == kNegInf) {
          accept = false;
        } else if (tq == kNegInf) {
          accept = true;
        } else {
          const float mx = fmaxf(tp, tq);
          accept = u * (fast_ex2(tq - mx) * pt.b) < fast_ex2(tp - mx) * pd.b;
        }
        py = fast_ex2(tp) / pt.b;
        qy = fast_ex2(tq) / pd.b;
      } else if (lane == k) {
        const Partial pr = ld_cg(P.rowres + n0 + 2 * k);
        bad = pr.bad;
        tok = pr.idx;  // bonus race winner
      }
    }
    if (__any_sync(0xffffffffu, bad != 0u)) rs = kStNonfinite;
  }
  if (rs) {
    write_skipped(P, r, d0, k, rs, lane);
    return;
  }
  const uint32_t rej = __ballot_sync(0xffffffffu, lane < k && !accept);
  const int A = rej ? __ffs(rej) - 1 : k;
  const int tok_at_A = __shfl_sync(0xffffffffu, tok, A);
  const bool residual = (mode == kSampling) && A < k;
  if (lane < width) {  // width = max_k + 1 <= 32; lane i holds y_i
    const int v = lane < A ? y : ((lane == A && !residual) ? tok_at_A : -1);
    P.committed[(size_t)r * width + lane] = v;
  }
  const float nan = __int_as_float(0x7fc00000);
  if (lane < k) {
    P.flags[d0 + lane] = lane < A ? 1 : 0;
    if (P.p_y) P.p_y[d0 + lane] = mode == kSampling ? py : nan;
    if (P.q_y) P.q_y[d0 + lane] = mode == kSampling ? qy : nan;
    if (P.u_dbg) P.u_dbg[d0 + lane] = mode == kSampling ? u : nan;
  }
  if (lane == 0) {
    P.accepted_len[r] = A;
    if (P.req_status) P.req_status[r] = 0;
    if (residual) {
      const int slot = atomicAdd(P.ctr + kCntReserve, 1);
      const unsigned long long word = (unsigned long long)(uint32_t)r |
                                      ((unsigned long long)(uint32_t)A << 24) | (1ull << 31) |
                                      ((unsigned long long)(uint32_t)P.nch << 32);
      __threadfence();
      atomicExch(P.res_slots + slot, word);
      atomicAdd(P.ctr + kCntPublished, P.nch);
    }
  }
}

// ---------------------------------------------------------------------------
// Residual queue: claim one chunk (thread 0), returns false if none is ready.
// Slot word: r (bits 0-23) | j (24-30) | published (31) | chunks left (32-63).
// *first_live skips slots this CTA has already seen exhausted.
// ---------------------------------------------------------------------------
__device__ __forceinline__ bool claim_residual(const Params& P, int* first_live, int* slot,
                                               int* r, int* j, int* ch) {
  const int reserved = ld_volatile(P.ctr + kCntReserve);
  for (int s = *first_live; s < reserved; ++s) {
    unsigned long long w = *reinterpret_cast<volatile unsigned long long*>(P.res_slots + s);
    if ((w & (1ull << 31)) && (w >> 32) == 0ull && s == *first_live) ++*first_live;
    while ((w >> 32) != 0ull) {
      const unsigned long long old = atomicCAS(P.res_slots + s, w, w - (1ull << 32));
      if (old == w) {
        atomicAdd(P.ctr + kCntClaimed, 1);
        *slot = s;
        *r = (int)(w & 0xffffffull);
        *j = (int)((w >> 24) & 0x7full);
        *ch = (int)(w >> 32) - 1;
        return true;
      }
      w = old;
    }
  }
  return false;
}

// ---------------------------------------------------------------------------
// The kernel.
// ---------------------------------------------------------------------------
template <typename E>
__global__ void __launch_bounds__(kThreads, 3) sv_verify(Params P) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  uint4* ring = reinterpret_cast<uint4*>(smem_raw);
  int* s_doff = reinterpret_cast<int*>(smem_raw + sizeof(uint4) * kStages * kStageVecs * kThreads);
  __shared__ SoftmaxAcc s_red_sm[kThreads / 32];
  __shared__ BestAcc s_red_b[kThreads / 32];
  __shared__ int s_flag, s_claim[4];
  __shared__ uint32_t s_layout;
  const int tid = threadIdx.x;
  const int lane = tid & 31;

  // --- prefix sums of num_draft, and the layout check -----------------------
  if (tid == 0) s_layout = 0u;
  __syncthreads();
  int carry = 0;
  for (int base = 0; base < P.batch; base += kThreads) {
    const int r = base + tid;
    const int k = r < P.batch ? P.num_draft[r] : 0;
    if (k < 0 || k > P.max_k) atomicOr(&s_layout, kStBadK);
    const int kk = (k < 0 || k > P.max_k) ? 0 : k;
    // block inclusive scan
    int v = kk;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, v, off);
      if (lane >= off) v += o;
    }
    __shared__ int s_w[kThreads / 32 + 1];
    if (lane == 31) s_w[tid >> 5] = v;
    __syncthreads();
    if (tid < 32) {
      int w = tid < kThreads / 32 ? s_w[tid] : 0;
      int wi = w;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, wi, off);
        if (lane >= off) wi += o;
      }
      if (tid < kThreads / 32) s_w[tid] = wi - w;
      if (tid == kThreads / 32 - 1) s_w[kThreads / 32] = wi;
    }
    __syncthreads();
    if (r < P.batch) s_doff[r] = carry + s_w[tid >> 5] + v - kk;
    carry += s_w[kThreads / 32];
    __syncthreads();
  }
  if (tid == 0) {
    s_doff[P.batch] = carry;
    if (!s_layout && carry != P.total_draft) s_layout = kStBadTotal;
  }
  __syncthreads();
  const uint32_t layout = s_layout;

  if (layout) {
    // untrustworthy layout: nothing is verified; CTA 0 reports it
    if (blockIdx.x == 0) {
      const int width = P.max_k + 1;
      for (int i = tid; i < P.batch * width; i += kThreads) P.committed[i] = -1;
      for (int r = tid; r < P.batch; r += kThreads) {
        P.accepted_len[r] = -1;
        if (P.req_status) P.req_status[r] = (int32_t)layout;
      }
      const float nan = __int_as_float(0x7fc00000);
      for (int d = tid; d < P.total_draft; d += kThreads) {
        P.flags[d] = 0;
        if (P.p_y) P.p_y[d] = nan;
        if (P.q_y) P.q_y[d] = nan;
        if (P.u_dbg) P.u_dbg[d] = nan;
      }
      if (tid == 0) atomicOr(reinterpret_cast<unsigned int*>(P.ctr + kCntStatus), layout);
    }
  } else {
    // --- the item loop ------------------------------------------------------
    LoadCursor<E> lc;
    lc.j = 0;
    lc.seek(P, s_doff);
    for (int s = 0; s < kStages - 1; ++s) lc.issue(P, s_doff, ring, s);
    int gs = 0;
    const int chv = P.nper * kThreads;
    int first_live = 0;  // thread 0: residual slots below this are exhausted

    for (int jj = 0;; ++jj) {
      const int item = blockIdx.x + jj * gridDim.x;
      const bool have_item = item < P.n_items;

      // residual jobs first (their rows are still in L2)
      for (;;) {
        if (tid == 0) {
          const int avail = ld_volatile(P.ctr + kCntPublished) - ld_volatile(P.ctr + kCntClaimed);
          int slot = -1, r = 0, j = 0, ch = 0;
          bool got = false;
          if (avail > 0) got = claim_residual(P, &first_live, &slot, &r, &j, &ch);
          if (!got && !have_item) {
            // no items left: wait (bounded) while requests are still being scanned
            for (int spin = 0; spin < P.spin_limit && !got; ++spin) {
              if (ld_volatile(P.ctr + kCntReqDone) == P.batch &&
                  ld_volatile(P.ctr + kCntPublished) == ld_volatile(P.ctr + kCntClaimed))
                break;
              __nanosleep(256);
              if (ld_volatile(P.ctr + kCntPublished) != ld_volatile(P.ctr + kCntClaimed))
                got = claim_residual(P, &first_live, &slot, &r, &j, &ch);
            }
          }
          s_claim[0] = got ? slot : -1;
          s_claim[1] = r;
          s_claim[2] = j;
          s_claim[3] = ch;
        }
        __syncthreads();
        const int slot = s_claim[0];
        if (slot < 0) break;
        const int r = s_claim[1], j = s_claim[2], ch = s_claim[3];
        __threadfence();
        const int n0 = r + 2 * s_doff[r];
        const Partial rt = ld_cg(P.rowres + n0 + 2 * j);
        const Partial rd = ld_cg(P.rowres + n0 + 2 * j + 1);
        BestAcc a = residual_chunk<E>(P, r, j, ch, s_doff, rt, rd);
        a = block_reduce<BestAcc, kThreads>(a, s_red_b);
        if (tid == 0) {
          P.part2[(size_t)slot * P.nch + ch] = Partial{a.v, 0.f, a.idx, 0u};
          __threadfence();
          s_flag = (atomicAdd(P.res_cnt + slot, 1) == P.nch - 1) ? 1 : 0;
        }
        __syncthreads();
        if (s_flag) {
          // last chunk of this residual job: merge and commit the token
          __threadfence();
          BestAcc m;
          m.init();
          if (tid < 32) {
            for (int q = lane; q < P.nch; q += 32) {
              const Partial pq = ld_cg(P.part2 + (size_t)slot * P.nch + q);
              BestAcc b;
              b.v = pq.a;
              b.idx = pq.idx;
              b.nan = 0u;
              m = BestAcc::merge(m, b);
            }
            m = warp_reduce(m);
            if (lane == 0) s_claim[0] = m.idx;
          }
          __syncthreads();
          int token = s_claim[0];
          if (token < 0) {
            BestAcc f = fallback_row<E>(P, r, j, s_doff);
            f = block_reduce<BestAcc, kThreads>(f, s_red_b);
            if (tid == 0) s_claim[0] = f.idx;
            __syncthreads();
            token = s_claim[0];
          }
          if (tid == 0) {
            P.committed[(size_t)r * (P.max_k + 1) + j] = token;
            P.res_cnt[slot] = 0;
          }
        }
        __syncthreads();
      }
      if (!have_item) break;

      const Item it = decode_item<E>(P, s_doff, item);
      if (it.kind == kSkip) continue;
      Geom<E> g;
      g.init(it.row, P.vocab, it.ch, chv);

      Partial out;
      if (it.kind == kSoftmax) {
        SoftmaxAcc a = item_softmax<E>(P, s_doff, ring, lc, gs, it, g);
        a = block_reduce<SoftmaxAcc, kThreads>(a, s_red_sm);
        out = Partial{a.m, a.s, -1, 0u};
      } else {
        BestAcc a;
        if (it.kind == kArgmax) {
          a = item_argmax<E>(P, s_doff, ring, lc, gs, it, g);
        } else {
          const RequestKey rk = request_key(P, it.r);
          switch (g.head & 3) {
            case 0: a = item_race<E, 0>(P, s_doff, ring, lc, gs, it, g, rk); break;
            case 1: a = item_race<E, 1>(P, s_doff, ring, lc, gs, it, g, rk); break;
            case 2: a = item_race<E, 2>(P, s_doff, ring, lc, gs, it, g, rk); break;
            default: a = item_race<E, 3>(P, s_doff, ring, lc, gs, it, g, rk); break;
          }
        }
        a = block_reduce<BestAcc, kThreads>(a, s_red_b);
        out = Partial{a.v, 0.f, a.idx, a.nan};
      }

      if (tid == 0) {
        P.part[item] = out;
        __threadfence();
        s_flag = (atomicAdd(P.row_cnt + it.n, 1) == P.nch - 1) ? 1 : 0;
      }
      __syncthreads();
      if (s_flag && tid < 32) {
        // this CTA completed row n: merge its chunk partials
        __threadfence();
        Partial res;
        if (it.kind == kSoftmax) {
          SoftmaxAcc a;
          a.init();
          for (int q = lane; q < P.nch; q += 32) {
            const Partial pq = ld_cg(P.part + (size_t)it.n * P.nch + q);
            SoftmaxAcc b;
            b.m = pq.a;
            b.s = pq.b;
            a = SoftmaxAcc::merge(a, b);
          }
          a = warp_reduce(a);
          const bool bad = !(a.s > 0.f) || !(a.s < 3.0e38f) || !(a.m > kNegInf) ||
                           !(a.m < 3.0e38f);
          res = Partial{a.m, a.s, -1, bad ? 1u : 0u};
        } else {
          BestAcc a;
          a.init();
          for (int q = lane; q < P.nch; q += 32) {
            const Partial pq = ld_cg(P.part + (size_t)it.n * P.nch + q);
            BestAcc b;
            b.v = pq.a;
            b.idx = pq.idx;
            b.nan = pq.bad;
            a = BestAcc::merge(a, b);
          }
          a = warp_reduce(a);
          const bool bad = a.nan != 0u || a.idx < 0 || !(a.v < 3.0e38f);
          res = Partial{a.v, 0.f, a.idx, bad ? 1u : 0u};
        }
        int last_row = 0;
        if (lane == 0) {
          P.rowres[it.n] = res;
          P.row_cnt[it.n] = 0;
          __threadfence();
          const int d0 = s_doff[it.r];
          const int k = s_doff[it.r + 1] - d0;
          const int need = rows_of_request(P, k, req_mode(__ldg(P.temperature + it.r)));
          last_row = (atomicAdd(P.req_cnt + it.r, 1) == need - 1) ? 1 : 0;
        }
        last_row = __shfl_sync(0xffffffffu, last_row, 0);
        if (last_row) {
          __threadfence();
          scan_request<E>(P, it.r, s_doff);
          if (lane == 0) {
            P.req_cnt[it.r] = 0;
            __threadfence();
            atomicAdd(P.ctr + kCntReqDone, 1);
          }
        }
      }
      __syncthreads();
    }
    cp_async_wait_all();
  }

  // --- the last CTA out resets the round's shared state ----------------------
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    if (atomicAdd(P.ctr + kCntExit, 1) == (int)gridDim.x - 1) {
      __threadfence();
      const int reserved = ld_volatile(P.ctr + kCntReserve);
      for (int s = 0; s < reserved; ++s) P.res_slots[s] = 0ull;
      P.ctr[kCntLastStatus] = ld_volatile(P.ctr + kCntStatus);
      P.ctr[kCntStatus] = 0;
      P.ctr[kCntReserve] = 0;
      P.ctr[kCntPublished] = 0;
      P.ctr[kCntClaimed] = 0;
      P.ctr[kCntReqDone] = 0;
      __threadfence();
      P.ctr[kCntExit] = 0;
    }
  }
}

}  // namespace sv
