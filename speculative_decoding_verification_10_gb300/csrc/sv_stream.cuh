// sv_stream.cuh -- the verify round as one persistent launch after the plan:
// the decisions feed a queue of rows, and all CTAs consume it in bands.
//
// Positions are decided left to right and nothing after the first rejection
// is read ("Speculative Decoding: Medusa, MTP, EAGLE, DFlash, DDTree, and
// DSpark", section 1), so the rows a round needs are only known as it goes.
// Here they are kept in two append-only queues:
//   * the row queue: the plan puts position 0 of every request there; a
//     decision that accepts position i appends the rows of position i+1
//     (t_{i+1} and d_{i+1} when sampling, the bonus row t_k at i+1 = k, the
//     target row when greedy);
//   * the urgent queue: a rejection at position j appends the correction draw
//     over [p_j - q_j]_+, which streams t_j and d_j again.
// The queues are consumed in bands.  Band b is formed once, by the first CTA
// that needs it: all urgent entries queued so far, then row entries up to
// about 64 KB per CTA, cut only between positions.  Every CTA then takes the
// same flat share of the band as the wave kernel does of a wave (contiguous
// race blocks, CTA c takes [c T / G, (c + 1) T / G)), so all CTAs sweep the
// queue front to back together.  A rejected row pair comes back through the
// urgent queue two or three bands (tens of MB) after it was read, so the
// correction pass is served from L2, and there is no launch, fill or drain
// between positions.
//
// Waits.  A CTA waits only where another CTA's progress is required: for a
// band that nobody can form yet (its rows depend on decisions still in
// flight), for a band another CTA is forming, and for the ready tag of a queue
// entry that has been reserved but not yet written.  Every such wait is a
// bounded poll; when one runs out the CTA sets SPECVERIFY_STATUS_TIMEOUT and
// returns, and the others run out in turn.  A CTA never waits while it holds a
// finished segment it has not counted: the control warp counts it first and
// hands the compute warps an idle unit meanwhile.
#pragma once

#include "sv_kernels.cuh"

namespace sv {

constexpr int kBandSpanBytes = 131072; // a CTA's share of a full band
constexpr int kBandMaxRows = 1024;     // entries of a full band, at most
constexpr int kSpinLimit = 1 << 20;    // polls of one bounded wait
constexpr int kIdleLimit = 1 << 21;    // consecutive idle units before giving up

enum StreamUnit : int { kSIdle = -1, kSEnd = -2 };

// ---- global-memory ordering ----------------------------------------------------
__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ int ld_acquire_s32(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_u32(uint32_t* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void st_release_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ int ld_relaxed_s32(const int* p) {
  int v;
  asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ uint32_t ld_relaxed_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
// Counting with release: the partial stored before it is visible to whoever
// completes the count (who then fences before reading the partials).  Later
// accesses of the counting thread need not wait for it.
__device__ __forceinline__ unsigned long long atom_add_release(unsigned long long* p,
                                                                unsigned long long v) {
  unsigned long long old;
  asm volatile("atom.release.gpu.global.add.u64 %0, [%1], %2;"
               : "=l"(old)
               : "l"(p), "l"(v)
               : "memory");
  return old;
}
__device__ __forceinline__ void red_release_add(int* p, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Bounded wait (warp-collective) until every entry of [a, b) of a queue shows
// this round's ready tag; the fence after the polls orders this warp's later
// accesses after the writers'.
__device__ bool wait_ready_range(const uint32_t* tags, int a, int b, uint32_t epoch) {
  const int lane = threadIdx.x & 31;
  for (int spin = 0; spin < kSpinLimit; ++spin) {
    bool ok = true;
    for (int e = a + lane; e < b; e += 32) ok &= ld_relaxed_u32(tags + e) == epoch;
    if (__all_sync(0xffffffffu, ok)) {
      __threadfence();
      return true;
    }
    __nanosleep(64);
  }
  return false;
}

__device__ __forceinline__ void cp_async_wait_dyn(int n) {
  switch (n) {
    case 0: cp_async_wait<0>(); break;
    case 1: cp_async_wait<1>(); break;
    case 2: cp_async_wait<2>(); break;
    case 3: cp_async_wait<3>(); break;
    case 4: cp_async_wait<4>(); break;
    case 5: cp_async_wait<5>(); break;
    default: cp_async_wait<6>(); break;
  }
}

// ---------------------------------------------------------------------------
// Bands.
// ---------------------------------------------------------------------------
enum BandLook : int { kLookFormed = 0, kLookEnd = 1, kLookOpen = 2, kLookBusy = 3, kLookFailed = 4 };

// The split of a band over its CTAs, in units of one row's race block: an
// urgent entry streams two rows and counts 2 nb units, a row entry nb; the
// urgent entries come first.  CTA v takes units [v U / G, (v + 1) U / G), so
// every CTA streams the same bytes.  Block k of an urgent entry belongs to the
// CTA that holds the entry's unit 2k (shares are at least two units long, so
// the CTAs holding blocks of one entry are consecutive and each holds one).
struct BandSplit {
  unsigned long long U, UU;  // all units, urgent units
  int G, nb;
  __device__ __forceinline__ void init(int nu, int nn, int nb_, int min_span, int grid) {
    nb = nb_;
    UU = 2ull * (unsigned long long)nb * (unsigned long long)nu;
    U = UU + (unsigned long long)nb * (unsigned long long)nn;
    const unsigned long long g = U / (unsigned long long)min_span;
    G = (int)(g < 1ull ? 1ull : (g > (unsigned long long)grid ? (unsigned long long)grid : g));
    if (U == 0ull) G = 0;
  }
  __device__ __forceinline__ void from_item(const QItem& it, int nb_) {
    nb = nb_;
    U = it.sT;
    G = it.sG;
    UU = 2ull * (unsigned long long)nb * (unsigned long long)it.snu;
  }
  __device__ __forceinline__ unsigned long long begin(int v) const {
    return (unsigned long long)v * U / (unsigned long long)G;
  }
  __device__ __forceinline__ int cta_of(unsigned long long x) const {
    return (int)(((x + 1ull) * (unsigned long long)G - 1ull) / U);
  }
  // the first unit of block k of entry e
  __device__ __forceinline__ unsigned long long unit(bool urgent, int e, int k) const {
    return urgent ? 2ull * (unsigned long long)nb * (unsigned long long)e + 2ull * (unsigned long long)k
                  : UU + (unsigned long long)nb * (unsigned long long)e + (unsigned long long)k;
  }
  __device__ __forceinline__ int first_cta(bool urgent, int e) const {
    return cta_of(unit(urgent, e, 0));
  }
  __device__ __forceinline__ int segments(bool urgent, int e) const {
    return cta_of(unit(urgent, e, nb - 1)) - first_cta(urgent, e) + 1;
  }
};

// Band b as this warp may use it (warp-collective).  (u0, n0) is where band
// b-1 ended and `word` band b's word as last read.  An open band is formed
// here when a full band's worth of rows is queued, when half of one is and
// the caller has nothing left queued (`hungry`), or when anything is and the
// caller has nothing to do (`idle`); it becomes the end band once every
// request is finished.  Returns kLookFormed / kLookEnd with *u1, *n1 set;
// kLookOpen when the band cannot be formed now; kLookBusy when its word
// changed under us or another CTA is forming it (read it again); kLookFailed
// when a wait ran out.
__device__ int look_band(const Params& P, int b, int u0, int n0, unsigned long long word,
                         bool hungry, bool idle, int* u1, int* n1) {
  const int lane = threadIdx.x & 31;
  const uint32_t epoch = P.epoch;
  if ((uint32_t)(word >> 32) == epoch) {
    const uint32_t pl = (uint32_t)word;
    if (pl == kBandFormingMark) return kLookBusy;
    if (pl == kBandEndMark) {
      *u1 = u0;
      *n1 = n0;
      return kLookEnd;
    }
    *u1 = band_u1(pl);
    *n1 = band_n1(pl);
    return kLookFormed;
  }
  // open: lane 0 decides and takes it; the queue counts are read before the
  // finished count (a request is finished only after its last rows were
  // banded, so "nothing queued and every request finished" is final)
  unsigned long long* w = &P.bands[b].word;
  int act = 0, ur = 0, nr = 0;  // 0 leave open, 1 form, 2 end, 3 changed
  if (lane == 0) {
    // the three counts in one round trip; the fence makes the reads acquire
    ur = ld_relaxed_s32(P.ctr + kCntURes);
    nr = ld_relaxed_s32(P.ctr + kCntNRes);
    const int done = ld_relaxed_s32(P.ctr + kCntDone);
    __threadfence();
    const int avail = 2 * (ur - u0) + (nr - n0);
    if (avail > 0) {
      act = (avail >= P.band_rows || (hungry && 2 * avail >= P.band_rows) || idle) ? 1 : 0;
    } else {
      // re-read in order: nothing queued, then every request finished
      act = ld_acquire_s32(P.ctr + kCntDone) >= __ldcg(P.ctr + kCntLive) ? 2 : 0;
      (void)done;
    }
    if (act != 0 &&
        atomicCAS(w, word, ((unsigned long long)epoch << 32) | kBandFormingMark) != word)
      act = 3;
  }
  act = __shfl_sync(0xffffffffu, act, 0);
  if (act == 0) return kLookOpen;
  if (act == 3) return kLookBusy;
  const unsigned long long tag = (unsigned long long)epoch << 32;
  if (act == 2) {
    if (lane == 0) st_release_u64(w, tag | kBandEndMark);
    *u1 = u0;
    *n1 = n0;
    return kLookEnd;
  }
  ur = __shfl_sync(0xffffffffu, ur, 0);
  nr = __shfl_sync(0xffffffffu, nr, 0);
  int n_end = nr;
  const int want = max(0, P.band_rows - 2 * (ur - u0));
  if (n_end - n0 > want) {
    n_end = n0 + want;
    if (n_end > n0) {
      // a position's target and draft rows were reserved together: never cut
      // between them
      if (!wait_ready_range(P.ready_n, n_end - 1, n_end, epoch)) return kLookFailed;
      const int meta = __ldcg(&P.lists[n_end - 1].meta);
      if (((meta >> 14) & 1) && !((meta >> 13) & 1)) ++n_end;
    }
  }
  // every entry of the band is written before the band is published, so the
  // CTAs that cut it read the entries without waiting
  if (!wait_ready_range(P.ready_u, u0, ur, epoch) || !wait_ready_range(P.ready_n, n0, n_end, epoch))
    return kLookFailed;
  __syncwarp();
  if (lane == 0) st_release_u64(w, tag | band_payload(ur, n_end));
  *u1 = ur;
  *n1 = n_end;
  return kLookFormed;
}

// ---------------------------------------------------------------------------
// The copy ring of the compute threads: as the wave kernel's, but a stage is
// only counted once it is issued, so the ring may run dry while the queue
// waits for a band and fill up again when it comes.
// ---------------------------------------------------------------------------
struct StreamRing {
  int issued, consumed;  // stages
  int q;                 // queue index of the item being loaded
  int seen;              // queued items known to this thread
  int left;              // its stages still to copy
  const uint4* b0;
  const uint4* b1;
  int i0, i1, step, vend;
  bool active;

  __device__ __forceinline__ void init() {
    issued = consumed = 0;
    q = 0;
    seen = 0;
    active = false;
  }
  // Polls the queue count with a plain load and takes the acquire (which
  // orders the reads of the new entries) only when it has grown.
  __device__ __forceinline__ bool open(const QItem* queue, const int* s_qend) {
    if (q >= seen) {
      if (*reinterpret_cast<const volatile int*>(s_qend) <= q) return active = false;
      seen = ld_acquire_shared(s_qend);
    }
    active = true;
    {
      const QItem& it = queue[q & (kQueue - 1)];
      const bool pair = it.kind == kResidual;
      b0 = reinterpret_cast<const uint4*>(it.row);
      b1 = reinterpret_cast<const uint4*>(pair ? it.row2 : it.row);
      i0 = it.vbeg + (int)threadIdx.x;
      i1 = pair ? i0 : i0 + kThreads;
      step = pair ? kThreads : kStageVecs * kThreads;
      vend = it.vend;
      left = it.nst;
    }
    return active;
  }
  __device__ __forceinline__ bool issue(const QItem* queue, const int* s_qend, uint4* ring) {
    if (!active && !open(queue, s_qend)) return false;
    uint4* dst = ring + (issued & (kStages - 1)) * kStageVecs * kThreads + threadIdx.x;
    if (i0 < vend) cp_async16(dst, b0 + i0);
    if (i1 < vend) cp_async16(dst + kThreads, b1 + i1);
    cp_async_commit();
    ++issued;
    i0 += step;
    i1 += step;
    if (--left == 0) {
      ++q;
      active = false;
    }
    return true;
  }
  __device__ __forceinline__ void top_up(const QItem* queue, const int* s_qend, uint4* ring) {
    while (issued - consumed < kStages - 1 && issue(queue, s_qend, ring)) {
    }
  }
  // the next stage of the item being reduced (its item is always queued)
  __device__ __forceinline__ void take(const QItem* queue, const int* s_qend, uint4* ring,
                                       uint4& v0, uint4& v1) {
    if (issued == consumed) issue(queue, s_qend, ring);
    cp_async_wait_dyn(issued - consumed - 1);
    const uint4* src = ring + (consumed & (kStages - 1)) * kStageVecs * kThreads + threadIdx.x;
    v0 = src[0];
    v1 = src[kThreads];
    ++consumed;
    top_up(queue, s_qend, ring);
  }
};

// ---------------------------------------------------------------------------
// Queue appends and the end of a request (control warp).
// ---------------------------------------------------------------------------
__device__ __forceinline__ void request_done(const Params& P) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) red_release_add(P.ctr + kCntDone, 1);
}

// The rows of position `next` of an accepted request, appended to the row
// queue as one reservation.
__device__ void publish_rows(const Params& P, const ReqInfo& q, int next) {
  const int lane = threadIdx.x & 31;
  const bool sampling = q.c > 0.f;
  const int n = wave_rows(P, sampling, q.k, next);  // depth 1: one or two rows
  int at = 0;
  if (lane == 0) at = atomicAdd(P.ctr + kCntNRes, n);
  at = __shfl_sync(0xffffffffu, at, 0);
  if (lane < n) {
    P.lists[at + lane] = wave_entry(P, sampling, q.r, q.d0, q.k, q.c, q.rk, next, lane, at, P.tokens);
    st_release_u32(P.ready_n + at + lane, P.epoch);
  }
}

// ---------------------------------------------------------------------------
// Decisions ("Speculative Decoding: Medusa, MTP, EAGLE, DFlash, DDTree, and
// DSpark", section 1): accept y_i with probability min(1, p_i(y_i)/q_i(y_i)),
// tested as u_i q_i(y_i) < p_i(y_i); at the first rejection draw from
// [p_i - q_i]_+ (queued as urgent); after k acceptances draw the bonus from
// p_k; greedy rounds keep y_i while it equals the target argmax.
// ---------------------------------------------------------------------------
template <typename E>
__device__ void decide_stream(const Params& P, const ReqInfo& q, int i, const RowRes& t,
                              const RowRes& d, int y) {
  const int lane = threadIdx.x & 31;
  const size_t row_bytes = (size_t)P.vocab * E::kBytes;
  const bool sampling = q.c > 0.f;
  if (!sampling) {
    if (t.bad) {
      skip_request_warp(P, q.r, q.d0, q.k, kStNonfinite);
      request_done(P);
      return;
    }
    if (!(i < q.k && y == t.idx)) {
      finish_request(P, q.r, q.d0, q.k, i, t.idx, true);
      request_done(P);
      return;
    }
  } else if (i == q.k) {
    if (t.bad || t.idx < 0) {
      skip_request_warp(P, q.r, q.d0, q.k, kStNonfinite);
      request_done(P);
      return;
    }
    const char* trow =
        reinterpret_cast<const char*>(P.target) + (size_t)(q.d0 + q.r + i) * row_bytes;
    const ResidualRow rr{q.c, 0.f, 0.f, 0.f, 0.f};
    const int token = inner_race<E, false>(P, trow, nullptr, t.idx, rr, (uint32_t)i, q.rk);
    finish_request(P, q.r, q.d0, q.k, i, token, false);
    request_done(P);
    return;
  } else {
    if (t.bad || d.bad) {
      skip_request_warp(P, q.r, q.d0, q.k, kStNonfinite);
      request_done(P);
      return;
    }
    const float tp = fmaf(t.xy, q.c, -t.a);  // log2(p(y) S_p)
    const float tq = fmaf(d.xy, q.c, -d.a);  // log2(q(y) S_q)
    const float u = accept_uniform(P.key, (uint32_t)i, q.rk.lo, q.rk.hi);
    // u q(y) < p(y), both sides scaled by S_p S_q 2^-max(tp, tq) > 0
    bool accept;
    if (tp == kNegInf) {
      accept = false;
    } else if (tq == kNegInf) {
      accept = true;
    } else {
      const float mx = fmaxf(tp, tq);
      accept = u * (fast_ex2(tq - mx) * t.b) < fast_ex2(tp - mx) * d.b;
    }
    if (lane == 0) {
      if (P.p_y) P.p_y[q.d0 + i] = fast_ex2(tp) / t.b;
      if (P.q_y) P.q_y[q.d0 + i] = fast_ex2(tq) / d.b;
      if (P.u_dbg) P.u_dbg[q.d0 + i] = u;
    }
    if (!accept) {
      // first rejection at i: the correction draw goes to the urgent queue
      finish_request(P, q.r, q.d0, q.k, i, -1, false);
      if (lane == 0) {
        const int at = atomicAdd(P.ctr + kCntURes, 1);
        ResEntry re;
        re.r = q.r;
        re.j = i;
        re.d0 = q.d0;
        re.pad = 0;
        re.c = q.c;
        re.mp = t.a;
        re.inv_sp = 1.f / t.b;
        re.mq = d.a;
        re.inv_sq = 1.f / d.b;
        re.req_lo = q.rk.lo;
        re.req_hi = q.rk.hi;
        re.pad2 = 0u;
        P.res[at] = re;
        st_release_u32(P.ready_u + at, P.epoch);
      }
      return;
    }
  }
  publish_rows(P, q, i + 1);
}

// Counting a finished segment, in two stages so that the control warp can
// look for more work while the count is in flight: stage 1 combines the
// warps' partials, stores the segment's partial and issues the count; stage 2
// learns whether this segment completed its position (or residual draw) and,
// if so, merges the partials and decides.
struct Pending {
  int mode;     // 0 nothing, 1 a position or draw of one segment, 2 counted
  Partial p;    // the segment's combined partial
  unsigned long long old;  // lane 0: the count before this segment
  int target;   // segments to count
};

template <typename E>
__device__ void complete_begin(const Params& P, const QItem& it, const Partial* mb, float xy,
                               Pending& pd) {
  const int lane = threadIdx.x & 31;
  BandSplit bs;
  bs.from_item(it, P.nb);
  if (it.kind == kResidual) {
    pd.p = combine_best(mb);
    pd.target = bs.segments(true, it.e);
  } else {
    if (it.kind == kSoftmax) {
      pd.p = combine_softmax(mb);
      pd.p.idx = __float_as_int(xy);
      pd.p.bad = it.yv >= 0 ? 1u : 0u;
    } else {
      pd.p = combine_best(mb);
    }
    const int et = (it.paired && it.is_draft) ? it.e - 1 : it.e;
    pd.target = bs.segments(false, et) + (it.paired ? bs.segments(false, et + 1) : 0);
  }
  pd.mode = pd.target == 1 ? 1 : 2;
  if (pd.mode == 2 && lane == 0) {
    unsigned long long* cnt;
    if (it.kind == kResidual) {
      P.srpart[it.g] = pd.p;
      cnt = P.rcnt + it.r;
    } else {
      P.spart[it.g] = pd.p;
      cnt = P.pos_cnt + (size_t)it.pos * P.stride + it.r;
    }
    pd.old = atom_add_release(cnt, 1ull);
  }
}

template <typename E>
__device__ void complete_end(const Params& P, const QItem& it, const Pending& pd) {
  const int lane = threadIdx.x & 31;
  if (pd.mode == 2) {
    int last = 0;
    if (lane == 0) last = pd.old + 1ull == (unsigned long long)pd.target;
    if (!__shfl_sync(0xffffffffu, last, 0)) return;
    __threadfence();  // the acquire side of the count: every partial is visible
  }
  BandSplit bs;
  bs.from_item(it, P.nb);
  if (it.kind == kResidual) {
    // the correction draw: block race merged, element race in the winning
    // block (a residual without mass in fp32, i.e. p == q, draws from p_j)
    RowRes best, unused;
    if (pd.mode == 1) {
      best = single_res(pd.p, kResidual);
    } else {
      merge_rows(P.srpart + (size_t)(it.e0 + it.e) * P.seg_max_res, pd.target, nullptr, 0, false,
                 kResidual, best, unused);
    }
    const int j = it.pos;
    const RequestKey rk{it.req_lo, it.req_hi};
    int token;
    if (best.idx >= 0) {
      const ResidualRow rr{it.c, it.mp, it.inv_sp, it.mq, it.inv_sq};
      token = inner_race<E, true>(P, it.row, it.row2, best.idx, rr, (uint32_t)j, rk);
    } else {
      const ResidualRow rr{it.c, 0.f, 0.f, 0.f, 0.f};
      const BestAcc br = warp_block_race<E>(P, it.row, it.c, (uint32_t)j, rk);
      token = inner_race<E, false>(P, it.row, nullptr, br.idx, rr, (uint32_t)j, rk);
    }
    if (lane == 0) P.committed[(size_t)it.r * (P.max_k + 1) + j] = token;
    request_done(P);
    return;
  }
  const int et = (it.paired && it.is_draft) ? it.e - 1 : it.e;
  const int tkind = it.paired ? kSoftmax : it.kind;
  RowRes t, d{0.f, 0.f, 0.f, -1, false};
  if (pd.mode == 1) {
    t = single_res(pd.p, tkind);
  } else {
    const Partial* pt = P.spart + (size_t)(it.e0 + et) * P.seg_max;
    const int nt = bs.segments(false, et);
    merge_rows(pt, nt, pt + P.seg_max, it.paired ? pd.target - nt : 0, it.paired != 0, tkind,
               t, d);
  }
  const ReqInfo q{it.r, it.d0, it.k, 0, it.c, RequestKey{it.req_lo, it.req_hi}};
  decide_stream<E>(P, q, it.pos, t, d, it.y);
}

// ---------------------------------------------------------------------------
// Segment generation (control warp): walks the bands in order, skipping those
// that give this CTA no share, and cuts its shares (urgent entries first) at
// row boundaries.  Band b numbers the CTAs from a rotation rot_b (CTA c is
// (c - rot_b) mod grid in it; rot_{b+1} = rot_b + the CTAs band b uses), so a
// run of small bands is spread over the whole grid instead of the first CTAs.
// ---------------------------------------------------------------------------
struct StreamGen {
  int b;          // next band to look at
  int b_ok;       // a band with a share for this CTA may be cut up to here
  int u0, n0;     // where band b - 1 ended
  int rot;        // rotation of band b
  int win_base;   // bands [win_base, win_base + 32) have their words in `win`
  unsigned long long win;  // lane i: word of band win_base + i as read
  bool ended, failed;
  bool have;      // a band is being cut
  int hb, hu0, hn0, v;     // its index, start, and this CTA's number in it
  int hnu;        // its urgent entries
  BandSplit bs;   // its split
  unsigned long long x, x1;  // the part of this CTA's share still to cut
  int q_head, q_used, q_next;
  int idle;
};

__device__ __forceinline__ void gen_init(StreamGen& g) {
  g.b = g.b_ok = 0;
  g.u0 = g.n0 = 0;
  g.rot = 0;
  g.win_base = -64;
  g.win = 0ull;
  g.ended = g.failed = g.have = false;
  g.q_head = g.q_used = g.q_next = 0;
  g.idle = 0;
}

// Keeps the queue filled (up to kQueue - 2 segments ahead of the oldest one
// not yet counted); returns without waiting when the next band cannot be used
// yet.  `in_flight` is the number of queued segments the compute warps have
// not all finished, `b_cur` the band of the oldest of them.  A new band is
// looked for only when at most one segment is in flight, a band is cut only
// if it is at most one band past b_cur, and a band with fewer rows than half
// a full one is formed only by a CTA with nothing in flight.
template <typename E>
__device__ void fill_stream(const Params& P, QItem* queue, int* s_qend, StreamGen& g,
                            int in_flight, int b_cur) {
  const int lane = threadIdx.x & 31;
  const int grid = (int)gridDim.x;
  const bool idle = in_flight == 0;
  while (!g.ended && !g.failed && g.q_head < g.q_used + kQueue - 2) {
    if (!g.have) {
      if (in_flight > 1) break;  // enough queued for now
      if (g.b >= P.band_cap) {
        g.failed = true;
        break;
      }
      if (g.b < g.win_base || g.b >= g.win_base + 32) {
        // the words of the next 32 bands in one round trip
        g.win_base = g.b;
        const int bi = g.b + lane;
        g.win = bi < P.band_cap ? ld_acquire_u64(&P.bands[bi].word) : 0ull;
      }
      const unsigned long long word = __shfl_sync(0xffffffffu, g.win, g.b - g.win_base);
      int u1 = 0, n1 = 0;
      int look = look_band(P, g.b, g.u0, g.n0, word, true, idle, &u1, &n1);
      // a band another CTA is forming is ready within microseconds: wait for
      // it (bounded) rather than start the next item without prefetch
      for (int w = 0; look == kLookBusy && w < 64; ++w) {
        __nanosleep(128);
        const unsigned long long wd =
            __shfl_sync(0xffffffffu, lane == 0 ? ld_acquire_u64(&P.bands[g.b].word) : 0ull, 0);
        look = look_band(P, g.b, g.u0, g.n0, wd, true, idle, &u1, &n1);
      }
      if (look == kLookOpen || look == kLookBusy) {
        g.win_base = -64;  // read it again next time
        break;
      }
      if (look == kLookFailed) {
        g.failed = true;
        break;
      }
      if (look == kLookEnd) {
        g.ended = true;
        break;
      }
      BandSplit bs;
      bs.init(u1 - g.u0, n1 - g.n0, P.nb, P.min_span, grid);
      const int used = bs.G;
      const int v = ((int)blockIdx.x - g.rot + grid) % grid;
      if (v >= used) {
        // no share here: on to the next band
        g.b_ok = max(g.b_ok, g.b + 1);
        g.u0 = u1;
        g.n0 = n1;
        g.rot = (g.rot + used) % grid;
        ++g.b;
        continue;
      }
      if (in_flight > 0 && g.b > b_cur + 1) break;  // at most one band ahead
      g.have = true;
      g.hb = g.b;
      g.hu0 = g.u0;
      g.hn0 = g.n0;
      g.hnu = u1 - g.u0;
      g.v = v;
      g.bs = bs;
      g.x = bs.begin(v);
      g.x1 = bs.begin(v + 1);
      g.u0 = u1;
      g.n0 = n1;
      g.rot = (g.rot + used) % grid;
      ++g.b;
    }
    // cut the next segments of this CTA's share (all lanes alike): whole
    // urgent entries' blocks held by this CTA, then row blocks
    const int room = min(8, kQueue - 2 - (g.q_head - g.q_used));
    const BandSplit& bs = g.bs;
    const unsigned long long ub = 2ull * (unsigned long long)P.nb;
    int n = 0, my_urgent = 0, my_e = 0, my_b0 = 0, my_b1 = 0;
    while (n < room && g.x < g.x1) {
      int urgent, e, k0, k1;
      unsigned long long next;
      if (g.x < bs.UU) {
        urgent = 1;
        e = (int)(g.x / ub);
        const unsigned long long s0 = (unsigned long long)e * ub;
        next = g.x1 < s0 + ub ? g.x1 : s0 + ub;
        k0 = (int)((g.x - s0 + 1ull) / 2ull);  // blocks whose first unit is in the share
        k1 = (int)((next - s0 + 1ull) / 2ull);
      } else {
        urgent = 0;
        e = (int)((g.x - bs.UU) / (unsigned long long)P.nb);
        const unsigned long long s0 = bs.UU + (unsigned long long)e * P.nb;
        next = g.x1 < s0 + P.nb ? g.x1 : s0 + P.nb;
        k0 = (int)(g.x - s0);
        k1 = (int)(next - s0);
      }
      g.x = next;
      if (k0 >= k1) continue;  // only the last unit of an urgent entry
      if (lane == n) {
        my_urgent = urgent;
        my_e = e;
        my_b0 = k0;
        my_b1 = k1;
      }
      ++n;
    }
    if (lane < n) {
      const int base = my_urgent ? g.hu0 : g.hn0;
      QItem it;
      decode_segment<E, true>(P, my_urgent ? 0 : 1, my_e, my_b0, my_b1, it, P.res + g.hu0,
                              P.lists + g.hn0, base);
      // partial slot: the entry's own block, indexed by the segment's place
      // among the entry's segments
      const int smax = my_urgent ? P.seg_max_res : P.seg_max;
      it.g = (base + my_e) * smax + (g.v - bs.first_cta(my_urgent != 0, my_e));
      it.sT = bs.U;
      it.sG = bs.G;
      it.snu = g.hnu;
      it.band = g.hb;
      queue[(g.q_head + lane) & (kQueue - 1)] = it;
    }
    g.q_head += n;
    in_flight += n;
    if (g.x >= g.x1) g.have = false;
  }
  __syncwarp();
  if (lane == 0) st_release_shared(s_qend, g.q_head);
  __syncwarp();
}

// ---------------------------------------------------------------------------
// The stream launch (16-byte aligned rows): every CTA resident at once, one
// launch per round after the plan.  Inside a CTA the compute warps and the
// control warp are decoupled: the control warp publishes segments in the
// shared queue (s_qend), each compute warp streams them in order and
// publishes its progress (s_wdone[warp]), and the control warp counts a
// segment once every compute warp is past it.  No CTA-wide barrier is taken
// per segment, so control latency only matters when the queue runs dry.
// ---------------------------------------------------------------------------
template <typename E>
__global__ void __maxnreg__(128) sv_stream(Params P) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  uint4* ring = reinterpret_cast<uint4*>(smem_raw);
  __shared__ QItem queue[kQueue];
  __shared__ Partial mailbox[kQueue][kComputeWarps];
  __shared__ float s_xy[kQueue];
  __shared__ int s_qend;
  __shared__ int s_wdone[kComputeWarps];
  __shared__ int s_end;
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;

  pdl_launch_dependents();
  pdl_wait();  // the plan's queue and counters are complete
  if (tid == 0) {
    s_qend = 0;
    s_end = 0;
  }
  if (tid < kComputeWarps) s_wdone[tid] = 0;
  __syncthreads();

  if (warp < kComputeWarps) {
    // ---- compute warps: stream the queued segments in order --------------------
    StreamRing sr;
    sr.init();
    const volatile int* vq = &s_qend;
    for (int q = 0;;) {
      if (*vq <= q) {
        if (ld_acquire_shared(&s_end)) break;
        sr.top_up(queue, &s_qend, ring);  // prefetch whatever was queued meanwhile
        __nanosleep(64);
        continue;
      }
      (void)ld_acquire_shared(&s_qend);  // orders the reads of item q
      const QItem& it = queue[q & (kQueue - 1)];
      auto take = [&](uint4& a, uint4& b) { sr.take(queue, &s_qend, ring, a, b); };
      const Partial out = seg_reduce<E>(P, it, &s_xy[q & (kQueue - 1)], take);
      if (lane == 0) mailbox[q & (kQueue - 1)][warp] = out;
      ++q;
      __syncwarp();
      if (lane == 0) st_release_shared(&s_wdone[warp], q);
    }
    cp_async_wait_all();
    return;
  }

  // ---- control warp ------------------------------------------------------------
  StreamGen g;
  gen_init(g);
  for (;;) {
    // the compute warps' progress: segments [0, wmin) are finished by all
    int wmin = lane < kComputeWarps ? ld_acquire_shared(&s_wdone[lane]) : 0x7fffffff;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) wmin = min(wmin, __shfl_xor_sync(0xffffffffu, wmin, off));
    bool progress = false;
    // count the oldest finished segment (stage 1), queue ahead while its count
    // is in flight, then finish counting it (stage 2)
    Pending pd;
    pd.mode = 0;
    const int done_item = g.q_used < wmin ? g.q_used : -1;
    if (done_item >= 0)
      complete_begin<E>(P, queue[done_item & (kQueue - 1)], mailbox[done_item & (kQueue - 1)],
                        s_xy[done_item & (kQueue - 1)], pd);
    const int in_flight = g.q_head - wmin;
    const int b_cur = in_flight > 0 ? queue[wmin & (kQueue - 1)].band : 0;
    const int head0 = g.q_head;
    fill_stream<E>(P, queue, &s_qend, g, in_flight, b_cur);
    if (done_item >= 0) {
      complete_end<E>(P, queue[done_item & (kQueue - 1)], pd);
      g.q_used = done_item + 1;
      progress = true;
    }
    if (g.q_head != head0) progress = true;
    if ((g.ended || g.failed) && g.q_used == g.q_head) break;
    if (progress) {
      g.idle = 0;
    } else {
      if (++g.idle > kIdleLimit && !g.failed) g.failed = true;
      __nanosleep(g.idle < 16 ? 32 * g.idle : 512);
    }
  }
  if (g.failed && lane == 0)
    atomicOr(reinterpret_cast<unsigned int*>(P.ctr + kCntStatus), kStTimeout);
  __syncwarp();
  if (lane == 0) st_release_shared(&s_end, 1);
}

}  // namespace sv
