// sv_kernels.cuh -- the fused verify kernel: one persistent launch per round.
//
// Rows and items.  The logit rows of the batch are numbered request by request,
//     request r:  t_0 d_0 t_1 d_1 ... t_{k-1} d_{k-1} t_k     (2 k_r + 1 entries)
// so entry n of request r is n - (r + 2 drf_off(r)).  Each entry is split into
// `nch` vocab chunks: item = n * nch + chunk.  Items are claimed in increasing
// order from one global counter, so all chunks of a request are read at about
// the same time.  Draft entries of greedy requests are skipped.
//
// Per item the CTA reduces its chunk to a 16-byte partial:
//   sampling target row i < k, draft row i : softmax normaliser (m, S) of c*x,
//                                            c = log2(e)/T   (p_i, q_i)
//   sampling target row k                  : bonus race argmax c*x_v - log2 E_v
//   greedy (or bad-temperature) target row : argmax (lowest index)
// The CTA that completes an entry merges its partials; the CTA that completes
// a request runs the acceptance scan, writes all of its outputs and, on a
// rejection at position j, publishes a residual job: the draw from
// [p_j - q_j]_+ over rows t_j and d_j, in nch chunks any CTA may claim.  Jobs
// are claimed ahead of new items, while those two rows are still in L2.
//
// CTA layout: 7 compute warps and 1 control warp, one __syncthreads per work
// unit.  Compute warps stream the unit's bytes and leave one partial per warp
// in shared memory.  During the next unit the control warp combines them and
// does all latency-bound global work: partial stores, completion counters,
// merges, the acceptance scan, claiming items and residual jobs.
//
// Memory pipeline.  Each compute thread streams its 16-byte vectors of
// successive items through a private ring of shared memory with cp.async
// (kStages stages of kStageVecs vectors), kStages-1 stages ahead and across
// item boundaries; it only reads back what it copied itself, and
// cp.async.wait_group is a hardware wait.
//
// No CTA waits for another, except that the control warp of a CTA with no
// work left polls the job queue for at most P.spin_limit rounds in all;
// exiting is always safe because the CTA that publishes a job drains it
// itself.  The last CTA to exit resets the shared counters for the next round.
#pragma once

#include "sv_device.cuh"

namespace sv {

constexpr int kComputeWarps = 7;
constexpr int kThreads = kComputeWarps * 32;   // compute threads
constexpr int kBlock = kThreads + 32;          // + the control warp
constexpr int kStages = 8;
constexpr int kStageVecs = 2;
constexpr int kQueue = 16;                     // item queue entries (power of 2)
constexpr int kMaxBatch = 4096;                // requests per launch
constexpr int kResUnroll = 2;

enum RowKind : int { kSkip = -1, kSoftmax = 0, kArgmax = 1, kRace = 2 };
enum ReqMode : int { kBadTemp = 0, kGreedy = 1, kSampling = 2 };
enum UnitType : int { kUnitEnd = 0, kUnitIdle = 1, kUnitItem = 2, kUnitResidual = 3,
                      kUnitFallback = 4 };

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
  kCntItems = 0,      // items claimed
  kCntReserve = 1,    // job slots reserved
  kCntPublished = 2,  // job chunks published
  kCntClaimed = 3,    // job chunks claimed
  kCntReqDone = 4,    // requests scanned
  kCntExit = 5,       // CTAs finished
  kCntStatus = 6,     // status bits of this round
  kCntLastStatus = 7, // status bits of the previous round
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
  int fill;     // items kept claimed ahead: enough to cover kStages-1 stages, + 1
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
  unsigned long long* res_slots;  // [2 * batch] job words
  Partial* part2;      // [2 * batch * nch]
  int* res_cnt;        // [2 * batch]
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

struct RequestKey {
  uint32_t lo, hi;
};

__device__ __forceinline__ RequestKey request_key(const Params& P, int r) {
  const uint64_t id = P.request_ids ? (uint64_t)P.request_ids[r] : (uint64_t)r;
  return RequestKey{(uint32_t)id, (uint32_t)(id >> 32)};
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

// A claimed item, decoded once by the control warp.
struct __align__(16) QItem {
  const char* row;   // element 0 of the logit row
  int item, n, r, kind, ch, pos;
  float c;
  int head, nvec, tail, vbeg, vend;
  uint32_t req_lo, req_hi;
};

// A residual (or fallback) job chunk.
struct __align__(16) Job {
  const char* trow;
  const char* drow;
  int slot, r, j, ch;
  float c, mp, inv_sp, mq, inv_sq, kbound;
  uint32_t req_lo, req_hi;
};

struct __align__(16) Unit {
  int type;
  int qidx;   // kUnitItem: queue entry
  int pad[2];
  Job job;    // kUnitResidual / kUnitFallback
};

template <typename E>
__device__ __forceinline__ void decode_item(const Params& P, const int* s_doff, int item,
                                            QItem& it) {
  const int n = item / P.nch;
  it.item = item;
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
  it.head = it.nvec = it.tail = it.vbeg = it.vend = 0;
  it.req_lo = it.req_hi = 0u;
  if (it.kind != kSkip) {
    Geom<E> g;
    g.init(it.row, P.vocab, it.ch, P.nper * kThreads);
    it.head = g.head;
    it.nvec = g.nvec;
    it.tail = g.tail;
    it.vbeg = g.vbeg;
    it.vend = g.vend;
    const RequestKey rk = request_key(P, r);
    it.req_lo = rk.lo;
    it.req_hi = rk.hi;
  }
}

// Entries a request contributes to its completion counter.
__device__ __forceinline__ int rows_of_request(const Params& P, int k, int mode) {
  return (mode == kSampling && P.draft != nullptr) ? 2 * k + 1 : k + 1;
}

// ---------------------------------------------------------------------------
// The per-thread copy ring (compute threads).
// ---------------------------------------------------------------------------
template <typename E>
struct LoadCursor {
  int q;             // queue index of the item being loaded
  int st;            // stage within it
  const uint4* base;
  int vbeg, vend;
  bool active;

  // s_qend: items the control warp has queued, or -1 - n once the supply is
  // exhausted at n items.  The control warp keeps P.fill items queued beyond
  // the unit being processed, which covers the kStages-1 stages the cursor
  // runs ahead, so every entry the cursor opens is already written.
  __device__ __forceinline__ void open(const QItem* queue, const int* s_qend) {
    const int qe = *reinterpret_cast<const volatile int*>(s_qend);
    __threadfence_block();
    const int avail = qe >= 0 ? qe : -1 - qe;
    active = q < avail;
    if (active) {
      const QItem& it = queue[q & (kQueue - 1)];
      base = reinterpret_cast<const uint4*>(it.row + (size_t)it.head * E::kBytes);
      vbeg = it.vbeg;
      vend = it.vend;
      st = 0;
    }
  }

  // copy the next stage into ring slot `slot` and commit one group
  __device__ __forceinline__ void issue(const Params& P, const QItem* queue, const int* s_qend,
                                        uint4* ring, int slot) {
    if (!active) open(queue, s_qend);
    if (active) {
#pragma unroll
      for (int u = 0; u < kStageVecs; ++u) {
        const int vi = vbeg + (st * kStageVecs + u) * kThreads + (int)threadIdx.x;
        if (vi < vend) cp_async16(ring + (slot * kStageVecs + u) * kThreads + threadIdx.x, base + vi);
      }
    }
    cp_async_commit();
    if (active && ++st == P.nper / kStageVecs) {
      ++q;
      open(queue, s_qend);
    }
  }
};

// Streams the item's vectors out of the ring: for each stage, wait for it,
// refill the ring one stage ahead, then hand the thread's vectors to f(x, e0).
template <typename E, typename F>
__device__ __forceinline__ void consume_item(const Params& P, const QItem* queue,
                                             const int* s_qend, uint4* ring, LoadCursor<E>& lc,
                                             int& g_stage, const QItem& it, F&& f) {
  const int spi = P.nper / kStageVecs;
  for (int st = 0; st < spi; ++st) {
    cp_async_wait<kStages - 2>();
    const int slot = g_stage % kStages;
    uint4 v[kStageVecs];
#pragma unroll
    for (int u = 0; u < kStageVecs; ++u) v[u] = ring[(slot * kStageVecs + u) * kThreads + threadIdx.x];
    lc.issue(P, queue, s_qend, ring, (g_stage + kStages - 1) % kStages);
    ++g_stage;
#pragma unroll
    for (int u = 0; u < kStageVecs; ++u) {
      const int vi = it.vbeg + (st * kStageVecs + u) * kThreads + (int)threadIdx.x;
      float x[E::kVec];
      E::unpack(vi < it.vend ? v[u] : E::pad(), x);
      f(x, it.head + vi * E::kVec);
    }
  }
}

// Calls f(e, word) for the race words (stream 1) of elements e0 .. e0+N-1,
// where e0 % 4 == OFF; each Philox block is made just before its first use so
// that at most one block is live.
template <int N, int OFF, typename F>
__device__ __forceinline__ void for_each_race_word(int e0, uint32_t pos, uint32_t req_lo,
                                                   uint32_t req_hi, PhiloxKey key, F&& f) {
  const uint32_t b0 = (uint32_t)e0 >> 2;
  uint4 blk = philox4x32_10(make_uint4(b0, pos, req_lo, 1u | (req_hi << 8)), key);
#pragma unroll
  for (int e = 0; e < N; ++e) {
    if (e > 0 && ((OFF + e) & 3) == 0)
      blk = philox4x32_10(make_uint4(b0 + ((OFF + e) >> 2), pos, req_lo, 1u | (req_hi << 8)), key);
    f(e, word_of(blk, (OFF + e) & 3));
  }
}

__device__ __forceinline__ uint32_t race_word1(int e, uint32_t pos, uint32_t req_lo,
                                               uint32_t req_hi, PhiloxKey key) {
  const uint4 r = philox4x32_10(make_uint4((uint32_t)e >> 2, pos, req_lo, 1u | (req_hi << 8)), key);
  return word_of(r, e & 3);
}

// Bonus/fallback race candidate: the integer bound decides whether the exact
// exponential is needed; `thr` is the best exact score the warp has seen.
__device__ __forceinline__ void race_take(BestAcc& acc, float thr, float x, float c, uint32_t w,
                                          int e) {
  acc.nan |= (x != x);
  if (fmaf(x, c, race_gain_bound(w)) >= thr) {
    const float s = fmaf(x, c, -fast_lg2(race_exponential(w)));
    acc.take(s, e);
  }
}

// ---------------------------------------------------------------------------
// Per-kind item reductions (compute threads, ring-fed).
// ---------------------------------------------------------------------------
template <typename E>
__device__ __forceinline__ SoftmaxAcc item_softmax(const Params& P, const QItem* queue,
                                                   const int* s_qend, uint4* ring,
                                                   LoadCursor<E>& lc, int& gs, const QItem& it) {
  LazySoftmax acc;
  acc.init();
  if (it.ch == 0 && (int)threadIdx.x < it.head) acc.add1(E::load1(it.row, threadIdx.x), it.c);
  consume_item<E>(P, queue, s_qend, ring, lc, gs, it,
                  [&](const float(&x)[E::kVec], int) { acc.add(x, it.c); });
  if (it.ch == P.nch - 1 && (int)threadIdx.x < it.tail)
    acc.add1(E::load1(it.row, it.head + it.nvec * E::kVec + threadIdx.x), it.c);
  return acc.result();
}

template <typename E>
__device__ __forceinline__ BestAcc item_argmax(const Params& P, const QItem* queue,
                                               const int* s_qend, uint4* ring, LoadCursor<E>& lc,
                                               int& gs, const QItem& it) {
  BestAcc acc;
  acc.init();
  if (it.ch == 0 && (int)threadIdx.x < it.head) {
    const float x = E::load1(it.row, threadIdx.x);
    acc.nan |= (x != x);
    acc.take(x, threadIdx.x);
  }
  consume_item<E>(P, queue, s_qend, ring, lc, gs, it, [&](const float(&x)[E::kVec], int e0) {
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
  if (it.ch == P.nch - 1 && (int)threadIdx.x < it.tail) {
    const int e = it.head + it.nvec * E::kVec + threadIdx.x;
    const float x = E::load1(it.row, e);
    acc.nan |= (x != x);
    acc.take(x, e);
  }
  return acc;
}

template <typename E, int OFF>
__device__ __forceinline__ BestAcc item_race(const Params& P, const QItem* queue,
                                             const int* s_qend, uint4* ring, LoadCursor<E>& lc,
                                             int& gs, const QItem& it) {
  BestAcc acc;
  acc.init();
  const uint32_t pos = (uint32_t)it.pos;
  float thr = kNegInf;
  if (it.ch == 0 && (int)threadIdx.x < it.head) {
    const int e = threadIdx.x;
    race_take(acc, kNegInf, E::load1(it.row, e), it.c,
              race_word1(e, pos, it.req_lo, it.req_hi, P.key), e);
  }
  consume_item<E>(P, queue, s_qend, ring, lc, gs, it, [&](const float(&x)[E::kVec], int e0) {
    for_each_race_word<E::kVec, OFF>(e0, pos, it.req_lo, it.req_hi, P.key,
                                     [&](int e, uint32_t w) {
                                       race_take(acc, thr, x[e], it.c, w, e0 + e);
                                     });
    thr = warp_max(acc.v);
  });
  if (it.ch == P.nch - 1 && (int)threadIdx.x < it.tail) {
    const int e = it.head + it.nvec * E::kVec + threadIdx.x;
    race_take(acc, kNegInf, E::load1(it.row, e), it.c,
              race_word1(e, pos, it.req_lo, it.req_hi, P.key), e);
  }
  return acc;
}

// ---------------------------------------------------------------------------
// Residual draw ("Speculative Decoding: Medusa, MTP, EAGLE, DFlash, DDTree,
// and DSpark", section 1: at the first rejection, sample from the normalised
// positive residual [p_j - q_j]_+).  Score log2 w_v - log2 E_v over w_v > 0.
// Bound: w_v <= p_v = 2^(c x_v - M_p) / S_p, so an element whose
// c x_v + kbound + (bound on -log2 E_v) cannot reach the warp's best is
// skipped (kbound carries a margin for the fp32 rounding of the exact path).
// A fallback job (residual without mass, i.e. p == q) races on p_j instead.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void residual_take(BestAcc& acc, float thr, float x, float z,
                                              const Job& jb, uint32_t w, int e) {
  if (fmaf(x, jb.c, race_gain_bound(w) + jb.kbound) >= thr) {
    const float p = fast_ex2(fmaf(x, jb.c, -jb.mp)) * jb.inv_sp;
    const float q = fast_ex2(fmaf(z, jb.c, -jb.mq)) * jb.inv_sq;
    const float wv = p - q;
    if (wv > 0.f) acc.take(fast_lg2(wv) - fast_lg2(race_exponential(w)), e);
  }
}

template <typename E, bool kFallback, int OFF>
__device__ __forceinline__ BestAcc job_chunk_vec(const Params& P, const Job& jb, const Geom<E>& g) {
  BestAcc acc;
  acc.init();
  float thr = kNegInf;
  const uint4* tp = g.vecs(jb.trow);
  const uint4* dp = kFallback ? tp : g.vecs(jb.drow);
  const uint32_t pos = (uint32_t)jb.j;
  // uniform trip count across the compute warps (warp_max needs every lane)
  for (int v0 = g.vbeg; v0 < g.vend; v0 += kThreads * kResUnroll) {
    uint4 dt[kResUnroll], dd[kResUnroll];
#pragma unroll
    for (int u = 0; u < kResUnroll; ++u) {
      const int vi = v0 + u * kThreads + (int)threadIdx.x;
      dt[u] = vi < g.vend ? __ldcg(tp + vi) : E::pad();
      dd[u] = (!kFallback && vi < g.vend) ? __ldcg(dp + vi) : E::pad();
    }
#pragma unroll
    for (int u = 0; u < kResUnroll; ++u) {
      float x[E::kVec], z[E::kVec];
      E::unpack(dt[u], x);
      E::unpack(dd[u], z);
      const int e0 = g.head + (v0 + u * kThreads + (int)threadIdx.x) * E::kVec;
      for_each_race_word<E::kVec, OFF>(e0, pos, jb.req_lo, jb.req_hi, P.key,
                                       [&](int e, uint32_t w) {
                                         if (kFallback) race_take(acc, thr, x[e], jb.c, w, e0 + e);
                                         else residual_take(acc, thr, x[e], z[e], jb, w, e0 + e);
                                       });
      thr = warp_max(acc.v);
    }
  }
  return acc;
}

template <typename E, bool kFallback>
__device__ BestAcc job_chunk(const Params& P, const Job& jb) {
  const int chv = P.nper * kThreads;
  Geom<E> gt, gd;
  gt.init(jb.trow, P.vocab, jb.ch, chv);
  gd.init(kFallback ? jb.trow : jb.drow, P.vocab, jb.ch, chv);
  const uint32_t pos = (uint32_t)jb.j;
  auto one = [&](BestAcc& acc, int e) {
    const uint32_t w = race_word1(e, pos, jb.req_lo, jb.req_hi, P.key);
    const float x = E::load1(jb.trow, e);
    if (kFallback) race_take(acc, kNegInf, x, jb.c, w, e);
    else residual_take(acc, kNegInf, x, E::load1(jb.drow, e), jb, w, e);
  };
  BestAcc acc;
  if (gt.head == gd.head) {
    switch (gt.head & 3) {
      case 0: acc = job_chunk_vec<E, kFallback, 0>(P, jb, gt); break;
      case 1: acc = job_chunk_vec<E, kFallback, 1>(P, jb, gt); break;
      case 2: acc = job_chunk_vec<E, kFallback, 2>(P, jb, gt); break;
      default: acc = job_chunk_vec<E, kFallback, 3>(P, jb, gt); break;
    }
    if (jb.ch == 0 && (int)threadIdx.x < gt.head) one(acc, threadIdx.x);
    if (jb.ch == P.nch - 1 && (int)threadIdx.x < gt.tail)
      one(acc, gt.head + gt.nvec * E::kVec + threadIdx.x);
  } else {
    // rows with different 16-byte phases: plain element loads over the chunk
    acc.init();
    const int e_beg = jb.ch == 0 ? 0 : gt.head + gt.vbeg * E::kVec;
    const int e_end = jb.ch == P.nch - 1 ? P.vocab : gt.head + gt.vend * E::kVec;
    for (int e = e_beg + threadIdx.x; e < e_end; e += kThreads) one(acc, e);
  }
  return acc;
}

// ---------------------------------------------------------------------------
// Outputs of one request, and the acceptance scan (the control warp).
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

// Publishes a job (residual or fallback) for request r at position j.
__device__ __forceinline__ void publish_job(const Params& P, int r, int j, bool fallback) {
  const int slot = atomicAdd(P.ctr + kCntReserve, 1);
  const unsigned long long word = (unsigned long long)(uint32_t)r |
                                  ((unsigned long long)(uint32_t)j << 24) |
                                  (fallback ? (1ull << 30) : 0ull) | (1ull << 31) |
                                  ((unsigned long long)(uint32_t)P.nch << 32);
  __threadfence();
  atomicExch(P.res_slots + slot, word);
  atomicAdd(P.ctr + kCntPublished, P.nch);
}

// "Speculative Decoding: Medusa, MTP, EAGLE, DFlash, DDTree, and DSpark",
// section 1: accept y_i with probability min(1, p_i(y_i)/q_i(y_i)), left to
// right, stopping at the first rejection (tested as u_i q_i(y_i) < p_i(y_i));
// greedy rounds keep y_i while it equals the target argmax.  Lane i handles
// draft position i (k <= 31).  A rejection publishes the residual job.
template <typename E>
__device__ void scan_request(const Params& P, int r, const int* s_doff) {
  const int lane = threadIdx.x & 31;
  const int d0 = s_doff[r];
  const int k = s_doff[r + 1] - d0;
  const int t0 = d0 + r;                  // first target row
  const int n0 = r + 2 * d0;              // first entry of the request
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
        // target row i sits at entry 2i of the request (draft entries unused)
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
    if (residual) publish_job(P, r, A, false);
  }
}

// ---------------------------------------------------------------------------
// Job queue: claim one chunk (control lane 0), false if none is ready.
// Slot word: r (bits 0-23) | j (24-29) | fallback (30) | published (31) |
// chunks left (32-63).  *first_live skips slots already seen exhausted.
// ---------------------------------------------------------------------------
__device__ __forceinline__ bool claim_job(const Params& P, int* first_live, int* slot, int* r,
                                          int* j, int* ch, bool* fallback) {
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
        *j = (int)((w >> 24) & 0x3full);
        *fallback = (w >> 30) & 1ull;
        *ch = (int)(w >> 32) - 1;
        return true;
      }
      w = old;
    }
  }
  return false;
}

// ---------------------------------------------------------------------------
// Control-warp helpers.
// ---------------------------------------------------------------------------
struct Ctrl {
  int q_head;      // items queued so far
  int q_used;      // items handed out as units
  bool exhausted;  // no more items to claim
  int first_live;
  int spins;
};

// Keep P.fill items queued ahead of q_used (lane 0 claims and decodes).
template <typename E>
__device__ __forceinline__ void fill_queue(const Params& P, const int* s_doff, QItem* queue,
                                           int* s_qend, Ctrl& cs) {
  const int lane = threadIdx.x & 31;
  while (!cs.exhausted && cs.q_head < cs.q_used + P.fill) {
    const int need = cs.q_used + P.fill - cs.q_head;
    int base = 0;
    if (lane == 0) base = atomicAdd(P.ctr + kCntItems, need);
    base = __shfl_sync(0xffffffffu, base, 0);
    for (int i = 0; i < need; ++i) {
      const int item = base + i;
      if (item >= P.n_items) {
        cs.exhausted = true;
        break;
      }
      int kept = 0;
      if (lane == 0) {
        QItem it;
        decode_item<E>(P, s_doff, item, it);
        if (it.kind != kSkip) {
          queue[cs.q_head & (kQueue - 1)] = it;
          kept = 1;
        }
      }
      cs.q_head += __shfl_sync(0xffffffffu, kept, 0);
    }
  }
  __syncwarp();
  if (lane == 0) {
    __threadfence_block();  // queue entries before the count that publishes them
    *reinterpret_cast<volatile int*>(s_qend) = cs.exhausted ? -1 - cs.q_head : cs.q_head;
  }
  __syncwarp();
}

// Fill in a residual / fallback job for (slot, r, j, ch) (lane 0).
template <typename E>
__device__ __forceinline__ void make_job(const Params& P, const int* s_doff, int slot, int r,
                                         int j, int ch, bool fallback, Job& jb) {
  const size_t row_bytes = (size_t)P.vocab * E::kBytes;
  const int d0 = s_doff[r];
  const int n0 = r + 2 * d0;
  jb.trow = reinterpret_cast<const char*>(P.target) + (size_t)(d0 + r + j) * row_bytes;
  jb.drow = reinterpret_cast<const char*>(P.draft) + (size_t)(d0 + j) * row_bytes;
  jb.slot = slot;
  jb.r = r;
  jb.j = j;
  jb.ch = ch;
  jb.c = kLog2e / __ldg(P.temperature + r);
  const RequestKey rk = request_key(P, r);
  jb.req_lo = rk.lo;
  jb.req_hi = rk.hi;
  if (!fallback) {
    __threadfence();
    const Partial rt = ld_cg(P.rowres + n0 + 2 * j);
    const Partial rd = ld_cg(P.rowres + n0 + 2 * j + 1);
    jb.mp = rt.a;
    jb.inv_sp = 1.f / rt.b;
    jb.mq = rd.a;
    jb.inv_sq = 1.f / rd.b;
    // margin: 1/64 plus a few ulps of |M_p| (the exact path rounds at that scale)
    jb.kbound = -rt.a - fast_lg2(rt.b) + 0.015625f + fabsf(rt.a) * 0x1p-20f;
  } else {
    jb.mp = jb.inv_sp = jb.mq = jb.inv_sq = jb.kbound = 0.f;
  }
}

// Combine the compute warps' partials of a finished unit (control warp).
__device__ __forceinline__ Partial combine_best(const Partial* mb) {
  const int lane = threadIdx.x & 31;
  BestAcc a;
  a.init();
  if (lane < kComputeWarps) {
    const Partial p = mb[lane];
    a.v = p.a;
    a.idx = p.idx;
    a.nan = p.bad;
  }
  a = warp_reduce(a);
  return Partial{a.v, 0.f, a.idx, a.nan};
}

__device__ __forceinline__ Partial combine_softmax(const Partial* mb) {
  const int lane = threadIdx.x & 31;
  SoftmaxAcc a;
  a.init();
  if (lane < kComputeWarps) {
    a.m = mb[lane].a;
    a.s = mb[lane].b;
  }
  a = warp_reduce(a);
  return Partial{a.m, a.s, -1, 0u};
}

// Completion of an item unit: partial out, and the last arrivals merge the
// entry and scan the request.
template <typename E>
__device__ void complete_item(const Params& P, const int* s_doff, const QItem& it,
                              const Partial* mb) {
  const int lane = threadIdx.x & 31;
  const Partial p = it.kind == kSoftmax ? combine_softmax(mb) : combine_best(mb);
  int last = 0;
  if (lane == 0) {
    P.part[it.item] = p;
    __threadfence();
    last = (atomicAdd(P.row_cnt + it.n, 1) == P.nch - 1) ? 1 : 0;
  }
  last = __shfl_sync(0xffffffffu, last, 0);
  if (!last) return;
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
    const bool bad = !(a.s > 0.f) || !(a.s < 3.0e38f) || !(a.m > kNegInf) || !(a.m < 3.0e38f);
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
  if (!last_row) return;
  __threadfence();
  scan_request<E>(P, it.r, s_doff);
  if (lane == 0) {
    P.req_cnt[it.r] = 0;
    __threadfence();
    atomicAdd(P.ctr + kCntReqDone, 1);
  }
}

// Completion of a job unit: the last chunk picks the token (or hands the
// request to a fallback job when the residual had no mass).
struct JobRef {
  int slot, r, j, ch;
};
__device__ void complete_job(const Params& P, const JobRef& jb, bool fallback, const Partial* mb) {
  const int lane = threadIdx.x & 31;
  const Partial p = combine_best(mb);
  int last = 0;
  if (lane == 0) {
    P.part2[(size_t)jb.slot * P.nch + jb.ch] = p;
    __threadfence();
    last = (atomicAdd(P.res_cnt + jb.slot, 1) == P.nch - 1) ? 1 : 0;
  }
  last = __shfl_sync(0xffffffffu, last, 0);
  if (!last) return;
  __threadfence();
  BestAcc a;
  a.init();
  for (int q = lane; q < P.nch; q += 32) {
    const Partial pq = ld_cg(P.part2 + (size_t)jb.slot * P.nch + q);
    BestAcc b;
    b.v = pq.a;
    b.idx = pq.idx;
    b.nan = 0u;
    a = BestAcc::merge(a, b);
  }
  a = warp_reduce(a);
  if (lane == 0) {
    P.res_cnt[jb.slot] = 0;
    if (a.idx >= 0 || fallback) {
      P.committed[(size_t)jb.r * (P.max_k + 1) + jb.j] = a.idx;
    } else {
      publish_job(P, jb.r, jb.j, true);
    }
  }
}

// ---------------------------------------------------------------------------
// The kernel.
// ---------------------------------------------------------------------------
template <typename E>
__global__ void __maxnreg__(128) sv_verify(Params P) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  uint4* ring = reinterpret_cast<uint4*>(smem_raw);
  int* s_doff = reinterpret_cast<int*>(smem_raw + sizeof(uint4) * kStages * kStageVecs * kThreads);
  __shared__ QItem queue[kQueue];
  __shared__ Unit s_unit[2];
  __shared__ Partial mailbox[2][kComputeWarps];
  __shared__ int s_w[kBlock / 32 + 1];
  __shared__ int s_qend;
  __shared__ uint32_t s_layout;
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const bool control = warp == kComputeWarps;

  // --- prefix sums of num_draft, and the layout check (all threads) -----------
  if (tid == 0) s_layout = 0u;
  __syncthreads();
  int carry = 0;
  for (int base = 0; base < P.batch; base += kBlock) {
    const int r = base + tid;
    const int k = r < P.batch ? P.num_draft[r] : 0;
    const bool badk = k < 0 || k > P.max_k;
    if (badk) atomicOr(&s_layout, kStBadK);
    const int kk = badk ? 0 : k;
    int v = kk;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, v, off);
      if (lane >= off) v += o;
    }
    if (lane == 31) s_w[warp] = v;
    __syncthreads();
    if (tid < 32) {
      const int w = tid < kBlock / 32 ? s_w[tid] : 0;
      int wi = w;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, wi, off);
        if (lane >= off) wi += o;
      }
      if (tid < kBlock / 32) s_w[tid] = wi - w;
      if (tid == kBlock / 32 - 1) s_w[kBlock / 32] = wi;
    }
    __syncthreads();
    if (r < P.batch) s_doff[r] = carry + s_w[warp] + v - kk;
    carry += s_w[kBlock / 32];
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
      for (int i = tid; i < P.batch * width; i += kBlock) P.committed[i] = -1;
      for (int r = tid; r < P.batch; r += kBlock) {
        P.accepted_len[r] = -1;
        if (P.req_status) P.req_status[r] = (int32_t)layout;
      }
      const float nan = __int_as_float(0x7fc00000);
      for (int d = tid; d < P.total_draft; d += kBlock) {
        P.flags[d] = 0;
        if (P.p_y) P.p_y[d] = nan;
        if (P.q_y) P.q_y[d] = nan;
        if (P.u_dbg) P.u_dbg[d] = nan;
      }
      if (tid == 0) atomicOr(reinterpret_cast<unsigned int*>(P.ctr + kCntStatus), layout);
    }
  } else {
    Ctrl cs;
    cs.q_head = cs.q_used = 0;
    cs.exhausted = false;
    cs.first_live = 0;
    cs.spins = 0;
    // control: the unit the compute warps are processing
    int cur_type = kUnitIdle, cur_qidx = 0;
    JobRef cur_job{0, 0, 0, 0};
    if (control) {
      fill_queue<E>(P, s_doff, queue, &s_qend, cs);
      if (lane == 0) s_unit[0].type = kUnitIdle;
    }
    __syncthreads();

    LoadCursor<E> lc;
    int gs = 0;
    if (!control) {
      lc.q = 0;
      lc.active = false;
      lc.open(queue, &s_qend);
      for (int s = 0; s < kStages - 1; ++s) lc.issue(P, queue, &s_qend, ring, s);
    }

    for (int u = 0;; ++u) {
      if (!control) {
        // ---- compute warps: process unit u ---------------------------------
        const int type = s_unit[u & 1].type;
        if (type == kUnitItem) {
          const QItem it = queue[s_unit[u & 1].qidx & (kQueue - 1)];
          Partial out;
          if (it.kind == kSoftmax) {
            SoftmaxAcc a = item_softmax<E>(P, queue, &s_qend, ring, lc, gs, it);
            a = warp_reduce(a);
            out = Partial{a.m, a.s, -1, 0u};
          } else {
            BestAcc a;
            if (it.kind == kArgmax) {
              a = item_argmax<E>(P, queue, &s_qend, ring, lc, gs, it);
            } else {
              switch (it.head & 3) {
                case 0: a = item_race<E, 0>(P, queue, &s_qend, ring, lc, gs, it); break;
                case 1: a = item_race<E, 1>(P, queue, &s_qend, ring, lc, gs, it); break;
                case 2: a = item_race<E, 2>(P, queue, &s_qend, ring, lc, gs, it); break;
                default: a = item_race<E, 3>(P, queue, &s_qend, ring, lc, gs, it); break;
              }
            }
            a = warp_reduce(a);
            out = Partial{a.v, 0.f, a.idx, a.nan};
          }
          if (lane == 0) mailbox[u & 1][warp] = out;
        } else if (type == kUnitResidual || type == kUnitFallback) {
          const Job jb = s_unit[u & 1].job;
          BestAcc a = type == kUnitResidual ? job_chunk<E, false>(P, jb)
                                            : job_chunk<E, true>(P, jb);
          a = warp_reduce(a);
          if (lane == 0) mailbox[u & 1][warp] = Partial{a.v, 0.f, a.idx, a.nan};
        }
      } else {
        // ---- control warp: finish unit u-1, schedule unit u+1 ----------------
        const int prev_type = cur_type, prev_qidx = cur_qidx;
        const JobRef prev_job = cur_job;
        cur_type = s_unit[u & 1].type;
        cur_qidx = s_unit[u & 1].qidx;
        cur_job = JobRef{s_unit[u & 1].job.slot, s_unit[u & 1].job.r, s_unit[u & 1].job.j,
                         s_unit[u & 1].job.ch};
        if (prev_type == kUnitItem) {
          complete_item<E>(P, s_doff, queue[prev_qidx & (kQueue - 1)], mailbox[(u - 1) & 1]);
        } else if (prev_type == kUnitResidual || prev_type == kUnitFallback) {
          complete_job(P, prev_job, prev_type == kUnitFallback, mailbox[(u - 1) & 1]);
        }
        // keep the items the compute warps may stream during unit u+1 queued
        fill_queue<E>(P, s_doff, queue, &s_qend, cs);
        // next unit: a claimable job first, then the next queued item
        int next_type = kUnitIdle;
        if (lane == 0) {
          Unit nx;
          nx.type = kUnitIdle;
          int slot, r, j, ch;
          bool fb;
          bool got = false;
          if (ld_volatile(P.ctr + kCntPublished) != ld_volatile(P.ctr + kCntClaimed))
            got = claim_job(P, &cs.first_live, &slot, &r, &j, &ch, &fb);
          if (got) {
            nx.type = fb ? kUnitFallback : kUnitResidual;
            make_job<E>(P, s_doff, slot, r, j, ch, fb, nx.job);
          } else if (cs.q_used < cs.q_head) {
            nx.type = kUnitItem;
            nx.qidx = cs.q_used;
          } else if (cur_type == kUnitIdle) {
            // nothing in flight here: finished once every request is scanned
            // and every job claimed; otherwise wait a little for new jobs
            const bool done = ld_volatile(P.ctr + kCntReqDone) == P.batch &&
                              ld_volatile(P.ctr + kCntPublished) == ld_volatile(P.ctr + kCntClaimed);
            if (done || cs.spins >= P.spin_limit) {
              nx.type = kUnitEnd;
            } else {
              ++cs.spins;
              __nanosleep(500);
            }
          }
          s_unit[(u + 1) & 1] = nx;
          next_type = nx.type;
        }
        next_type = __shfl_sync(0xffffffffu, next_type, 0);
        cs.spins = __shfl_sync(0xffffffffu, cs.spins, 0);
        cs.first_live = __shfl_sync(0xffffffffu, cs.first_live, 0);
        if (next_type == kUnitItem) ++cs.q_used;
        __syncwarp();
      }
      __syncthreads();
      if (s_unit[(u + 1) & 1].type == kUnitEnd) break;
    }
    if (!control) cp_async_wait_all();
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
      P.ctr[kCntItems] = 0;
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
