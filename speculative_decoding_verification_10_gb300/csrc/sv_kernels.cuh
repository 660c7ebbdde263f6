// sv_kernels.cuh -- the fused verify kernel: one persistent launch per round.
//
// Left to right, and no further than needed.  A round verifies the positions
// of each request left to right and discards everything after the first
// rejection ("Speculative Decoding: Medusa, MTP, EAGLE, DFlash, DDTree, and
// DSpark", section 1), so it only needs the rows of positions 0..A (and the
// bonus row when all k are accepted).  Work is therefore ordered by position:
// wave i holds, for every request, target row t_i and draft row d_i (slot
// n = i * 2B + 2r + is_draft), each split into `nch` vocab chunks (item =
// n * nch + chunk), claimed in increasing order from one global counter.  A
// request that is already decided has its later items skipped at claim time.
//
// Per item the CTA reduces its chunk to a 16-byte partial:
//   sampling target row i < k, draft row i : softmax normaliser (m, S) of c*x,
//                                            c = log2(e)/T   (p_i, q_i)
//   sampling target row k                  : block race of the bonus draw
//   greedy (or bad-temperature) target row : argmax (lowest index)
// The CTA that completes a slot merges its partials and counts the slot
// towards its position; position i of a request is decided by whichever CTA
// brings that count to (rows of position i) + (1 if i > 0, the "position i-1
// accepted" signal), so each position is decided exactly once, in order, as
// soon as both its rows and its predecessor are done.  A rejection at j
// publishes a residual job over rows t_j and d_j (still in L2), in nch chunks
// any CTA may claim; jobs are claimed ahead of new items.  Completion
// counters carry the round's epoch in their high word, so counters left
// partial by skipped work need no reset.
//
// CTA layout: 7 compute warps and 1 control warp, one __syncthreads per work
// unit.  Compute warps stream the unit's bytes and leave one partial per warp
// in shared memory.  During the next unit the control warp combines them and
// does all latency-bound global work: partial stores, completion counters,
// merges, decisions, claiming items and residual jobs.
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
constexpr int kResUnroll = 4;

enum RowKind : int { kSkip = -1, kSoftmax = 0, kArgmax = 1, kRace = 2 };
enum ReqMode : int { kBadTemp = 0, kGreedy = 1, kSampling = 2 };
enum UnitType : int { kUnitEnd = 0, kUnitIdle = 1, kUnitItem = 2, kUnitResidual = 3 };

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
  kCntReqDone = 4,    // requests decided
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
  int nch;      // chunks per row (items)
  int nper;     // 16-byte vectors per thread per chunk (multiple of kStageVecs)
  int jnch;     // chunks per row of a residual job
  int jnper;    // 16-byte vectors per thread per job chunk
  int fill;     // items kept claimed ahead: enough to cover kStages-1 stages, + 1
  int spin_limit;
  uint32_t epoch;  // this round's tag for completion counters and `done`
  int32_t* accepted_len;
  int32_t* committed;
  uint8_t* flags;
  float* p_y;
  float* q_y;
  float* u_dbg;
  int32_t* req_status;
  Partial* part;       // [slots * nch], slots = (max_k + 1) * 2 * batch
  Partial* rowres;     // [slots]
  unsigned long long* row_cnt;  // [slots] epoch | chunks merged
  unsigned long long* pos_cnt;  // [batch * (max_k + 1)] epoch | rows merged (+1 signal)
  uint32_t* done;      // [batch] epoch of the round that decided the request
  unsigned long long* res_slots;  // [batch] job words
  Partial* part2;      // [batch * jnch]
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

// Adds one to an epoch-tagged counter and returns the count of this epoch: a
// counter last touched in an earlier round is first raised to (epoch, 0).  The
// two atomics of one thread on one address are performed in program order.
__device__ __forceinline__ uint32_t epoch_add(unsigned long long* c, uint32_t epoch) {
  atomicMax(c, (unsigned long long)epoch << 32);
  return (uint32_t)atomicAdd(c, 1ull) + 1u;
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
  float c, mp, inv_sp, mq, inv_sq;
  uint32_t req_lo, req_hi;
};

struct __align__(16) Unit {
  int type;
  int qidx;   // kUnitItem: queue entry
  int pad[2];
  Job job;    // kUnitResidual
};

// slot n = i * 2B + 2r + is_draft
__device__ __forceinline__ int slot_of(const Params& P, int i, int r, int is_draft) {
  return i * 2 * P.batch + 2 * r + is_draft;
}

template <typename E>
__device__ __forceinline__ void decode_item(const Params& P, const int* s_doff, int item,
                                            QItem& it) {
  const int n = item / P.nch;
  it.item = item;
  it.n = n;
  it.ch = item - n * P.nch;
  const int i = n / (2 * P.batch);
  const int rem = n - i * 2 * P.batch;
  const int r = rem >> 1;
  const bool is_draft = rem & 1;
  const int d0 = s_doff[r];
  const int k = s_doff[r + 1] - d0;
  const float t = __ldg(P.temperature + r);
  const int mode = req_mode(t);
  it.r = r;
  it.pos = i;
  it.c = mode == kSampling ? kLog2e / t : 0.f;
  const size_t row_bytes = (size_t)P.vocab * E::kBytes;
  if (i > k) {
    it.kind = kSkip;
    it.row = nullptr;
  } else if (is_draft) {
    it.kind = (mode == kSampling && i < k && P.draft != nullptr) ? kSoftmax : kSkip;
    it.row = reinterpret_cast<const char*>(P.draft) + (size_t)(d0 + i) * row_bytes;
  } else {
    it.kind = mode == kSampling ? (i < k ? kSoftmax : kRace) : kArgmax;
    it.row = reinterpret_cast<const char*>(P.target) + (size_t)(d0 + r + i) * row_bytes;
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

// The count that decides position i of a request: its rows, plus the signal
// that position i-1 was accepted (i > 0).
__device__ __forceinline__ uint32_t position_target(const Params& P, int i, int k, int mode) {
  const uint32_t rows = (mode == kSampling && i < k && P.draft != nullptr) ? 2u : 1u;
  return rows + (i > 0 ? 1u : 0u);
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

// ---------------------------------------------------------------------------
// Two-level exponential race: blocks of kRaceBlock vocab ids.  The block race
// picks argmax_b log2 W_b - log2 E2_b over blocks with mass W_b > 0 (Philox
// stream 2, indexed by block); the element race inside the winning block picks
// argmax_v log2 w_v - log2 E1_v (stream 1, indexed by vocab id).  Lowest index
// on ties at both levels.
// ---------------------------------------------------------------------------
constexpr int kRaceBlock = 128;

__device__ __forceinline__ uint32_t race_word(uint32_t stream, int idx, uint32_t pos,
                                              RequestKey rk, PhiloxKey key) {
  const uint4 r = philox4x32_10(make_uint4((uint32_t)idx >> 2, pos, rk.lo, stream | (rk.hi << 8)), key);
  return word_of(r, idx & 3);
}

// -log2 E for a race word (the additive "gain" of an element or block).
__device__ __forceinline__ float race_gain(uint32_t w) { return -fast_lg2(race_exponential(w)); }

template <int kLanes>
__device__ __forceinline__ float group_max(float v) {
#pragma unroll
  for (int off = kLanes / 2; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
  return v;
}
template <int kLanes>
__device__ __forceinline__ float group_sum(float v) {
#pragma unroll
  for (int off = kLanes / 2; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

// Block gains of a warp's vector groups, made 32 groups at a time: lane L
// holds the gains of the kBlocksPerGroup blocks of group g0 + L.  A vector
// group is the warp's 32 consecutive vectors (32 * kVec ids, block aligned).
template <typename E>
struct GroupGains {
  static constexpr int kBlocksPerGroup = 32 * E::kVec / kRaceBlock;   // 2 (bf16) or 1 (fp32)
  static constexpr int kLanesPerBlock = kRaceBlock / E::kVec;          // 16 or 32
  float lo, hi;
  // first element of group g of warp w, for a chunk starting at vector vbeg
  __device__ static __forceinline__ int group_elem(int vbeg, int g, int w) {
    return (vbeg + g * kThreads + w * 32) * E::kVec;
  }
  __device__ __forceinline__ void make(int vbeg, int g0, int w, uint32_t pos, RequestKey rk,
                                       PhiloxKey key) {
    const int lane = threadIdx.x & 31;
    const int b = group_elem(vbeg, g0 + lane, w) / kRaceBlock;
    const uint4 r = philox4x32_10(make_uint4((uint32_t)b >> 2, pos, rk.lo, 2u | (rk.hi << 8)), key);
    lo = race_gain(word_of(r, b & 3));
    hi = kBlocksPerGroup > 1 ? race_gain(word_of(r, (b & 3) + 1)) : lo;  // b is even here
  }
  // the gain of this lane's block in group g (all lanes call it)
  __device__ __forceinline__ float get(int g) const {
    const int src = g & 31;
    const float a = __shfl_sync(0xffffffffu, lo, src);
    const float c = __shfl_sync(0xffffffffu, hi, src);
    return ((threadIdx.x & 31) / kLanesPerBlock) ? c : a;
  }
};

// Bonus race over one vector group: block weight W_b = sum 2^(c x_v) (kept as
// log2: block max + log2 of the rescaled sum), score log2 W_b + gain.
template <typename E>
__device__ __forceinline__ void group_bonus(BestAcc& acc, const float (&x)[E::kVec], int e_lane,
                                            float c, float gain) {
  constexpr int kL = GroupGains<E>::kLanesPerBlock;
  float mx = x[0];
#pragma unroll
  for (int e = 1; e < E::kVec; ++e) mx = fmaxf(mx, x[e]);
  const float m = group_max<kL>(mx) * c;
  float s = 0.f;
  if (m > kNegInf) {
    const float2 cc = make_float2(c, c), nm = make_float2(-m, -m);
    float2 a2 = make_float2(0.f, 0.f);
#pragma unroll
    for (int e = 0; e < E::kVec; e += 2) {
      const float2 t = __ffma2_rn(make_float2(x[e], x[e + 1]), cc, nm);
      a2 = __fadd2_rn(a2, make_float2(fast_ex2(t.x), fast_ex2(t.y)));
    }
    s = a2.x + a2.y;
  } else if (m != m) {
    s = m;  // a block of NaNs
  }
  s = group_sum<kL>(s);
  acc.nan |= (s != s);
  if (s > 0.f) acc.take_cmp(m + fast_lg2(s) + gain, e_lane / kRaceBlock);
}

// Residual race over one vector group: W_b = sum max(p_v - q_v, 0).
struct ResidualRow {
  float c, mp, inv_sp, mq, inv_sq;
};

template <typename E>
__device__ __forceinline__ void group_residual(BestAcc& acc, const float (&x)[E::kVec],
                                               const float (&z)[E::kVec], int e_lane,
                                               const ResidualRow& rr, float gain) {
  constexpr int kL = GroupGains<E>::kLanesPerBlock;
  const float2 cc = make_float2(rr.c, rr.c), nm = make_float2(-rr.mp, -rr.mq);
  const float2 inv = make_float2(rr.inv_sp, rr.inv_sq);
  float s = 0.f;
#pragma unroll
  for (int e = 0; e < E::kVec; ++e) {
    const float2 t = __ffma2_rn(make_float2(x[e], z[e]), cc, nm);
    const float2 pq = __fmul2_rn(make_float2(fast_ex2(t.x), fast_ex2(t.y)), inv);
    s += fmaxf(pq.x - pq.y, 0.f);
  }
  s = group_sum<kL>(s);
  if (s > 0.f) acc.take_cmp(fast_lg2(s) + gain, e_lane / kRaceBlock);
}

// Element race inside block b (one warp, lane l takes ids 128 b + 4 l .. +3):
// bonus/fallback weights 2^(c x_v) (kResid false) or residual [p - q]_+.
template <typename E, bool kResid>
__device__ __forceinline__ int inner_race(const Params& P, const char* trow, const char* drow,
                                          int b, const ResidualRow& rr, uint32_t pos,
                                          RequestKey rk) {
  const int lane = threadIdx.x & 31;
  const int v0 = b * kRaceBlock + 4 * lane;
  const uint4 r = philox4x32_10(make_uint4((uint32_t)v0 >> 2, pos, rk.lo, 1u | (rk.hi << 8)), P.key);
  BestAcc acc;
  acc.init();
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int v = v0 + i;
    if (v < P.vocab) {
      const float x = E::load1(trow, v);
      const float g = race_gain(word_of(r, i));
      if (kResid) {
        const float p = fast_ex2(fmaf(x, rr.c, -rr.mp)) * rr.inv_sp;
        const float q = fast_ex2(fmaf(E::load1(drow, v), rr.c, -rr.mq)) * rr.inv_sq;
        const float w = p - q;
        if (w > 0.f) acc.take(fast_lg2(w) + g, v);
      } else {
        acc.take(fmaf(x, rr.c, g), v);
      }
    }
  }
  acc = warp_reduce(acc);
  return acc.idx;
}

// The whole two-level race over one row by one warp, with plain loads (rows
// that are not 16-byte aligned, and the rare fallback).  Weights as in
// inner_race.  Reports NaN / +inf in the row through acc.nan.
template <typename E, bool kResid>
__device__ BestAcc slow_block_race(const Params& P, const char* trow, const char* drow,
                                   const ResidualRow& rr, uint32_t pos, RequestKey rk) {
  const int lane = threadIdx.x & 31;
  const int nblocks = (P.vocab + kRaceBlock - 1) / kRaceBlock;
  BestAcc acc;
  acc.init();
  for (int b = lane; b < nblocks; b += 32) {
    const int v_end = min(P.vocab, (b + 1) * kRaceBlock);
    float s = 0.f, m = kNegInf;
    if (kResid) {
      for (int v = b * kRaceBlock; v < v_end; ++v) {
        const float p = fast_ex2(fmaf(E::load1(trow, v), rr.c, -rr.mp)) * rr.inv_sp;
        const float q = fast_ex2(fmaf(E::load1(drow, v), rr.c, -rr.mq)) * rr.inv_sq;
        s += fmaxf(p - q, 0.f);
      }
      m = 0.f;
    } else {
      for (int v = b * kRaceBlock; v < v_end; ++v) {
        const float x = E::load1(trow, v);
        acc.nan |= (x != x) || (x == -kNegInf);
        m = fmaxf(m, x);
      }
      m *= rr.c;
      if (m > kNegInf)
        for (int v = b * kRaceBlock; v < v_end; ++v) s += fast_ex2(fmaf(E::load1(trow, v), rr.c, -m));
    }
    if (s > 0.f) acc.take(m + fast_lg2(s) + race_gain(race_word(2u, b, pos, rk, P.key)), b);
  }
  acc = warp_reduce(acc);
  return acc;
}

// Rows whose vector groups line up with the race blocks.
template <typename E>
__device__ __forceinline__ bool row_fast(const char* row, int vocab) {
  return ((reinterpret_cast<uintptr_t>(row) & 15u) == 0u) && (vocab % E::kVec == 0);
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

// Bonus race item: block race over the chunk's vector groups.  Rows that are
// not block aligned stream through the ring without work and are raced later
// by the slow path (partial index -2).
template <typename E>
__device__ __forceinline__ BestAcc item_race(const Params& P, const QItem* queue,
                                             const int* s_qend, uint4* ring, LoadCursor<E>& lc,
                                             int& gs, const QItem& it) {
  BestAcc acc;
  acc.init();
  if (!(it.head == 0 && it.tail == 0)) {
    consume_item<E>(P, queue, s_qend, ring, lc, gs, it, [&](const float(&)[E::kVec], int) {});
    acc.idx = -2;
    return acc;
  }
  const int w = threadIdx.x >> 5;
  const RequestKey rk{it.req_lo, it.req_hi};
  GroupGains<E> gg;
  int g = 0;
  consume_item<E>(P, queue, s_qend, ring, lc, gs, it, [&](const float(&x)[E::kVec], int e0) {
    if ((g & 31) == 0) gg.make(it.vbeg, g, w, (uint32_t)it.pos, rk, P.key);
    group_bonus<E>(acc, x, e0, it.c, gg.get(g));
    ++g;
  });
  return acc;
}

// ---------------------------------------------------------------------------
// Residual job chunk ("Speculative Decoding: Medusa, MTP, EAGLE, DFlash,
// DDTree, and DSpark", section 1: at the first rejection, sample from the
// normalised positive residual [p_j - q_j]_+): the block race over the chunk,
// rows t_j and d_j read through L2 (both are block aligned: jobs are only
// published for such rows).
// ---------------------------------------------------------------------------
template <typename E>
__device__ BestAcc job_chunk(const Params& P, const Job& jb) {
  const int chv = P.jnper * kThreads;
  Geom<E> g;
  g.init(jb.trow, P.vocab, jb.ch, chv);
  const uint4* tp = g.vecs(jb.trow);
  const uint4* dp = g.vecs(jb.drow);
  const ResidualRow rr{jb.c, jb.mp, jb.inv_sp, jb.mq, jb.inv_sq};
  const RequestKey rk{jb.req_lo, jb.req_hi};
  const int w = threadIdx.x >> 5;
  BestAcc acc;
  acc.init();
  GroupGains<E> gg;
  int gi = 0;
  // uniform trip count across the compute warps (the shuffles need every lane)
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
      if ((gi & 31) == 0) gg.make(g.vbeg, gi, w, (uint32_t)jb.j, rk, P.key);
      const int e0 = (v0 + u * kThreads + (int)threadIdx.x) * E::kVec;
      group_residual<E>(acc, x, z, e0, rr, gg.get(gi));
      ++gi;
    }
  }
  return acc;
}

// ---------------------------------------------------------------------------
// Outputs of one request, and the acceptance scan (the control warp).
// ---------------------------------------------------------------------------
// Publishes the residual job of request r at position j.
__device__ __forceinline__ void publish_job(const Params& P, int r, int j) {
  const int slot = atomicAdd(P.ctr + kCntReserve, 1);
  const unsigned long long word = (unsigned long long)(uint32_t)r |
                                  ((unsigned long long)(uint32_t)j << 24) | (1ull << 31) |
                                  ((unsigned long long)(uint32_t)P.jnch << 32);
  __threadfence();
  atomicExch(P.res_slots + slot, word);
  atomicAdd(P.ctr + kCntPublished, P.jnch);
}

// Outputs of a decided request (the control warp): accepted prefix, the extra
// token (-1 while a residual job still has to draw it), flags, NaN debug values
// after position A; then the request is marked done.
__device__ void finish_request(const Params& P, int r, int d0, int k, int A, int token,
                               bool pending) {
  const int lane = threadIdx.x & 31;
  const int width = P.max_k + 1;
  if (lane < width) {  // width <= 32
    const int v = lane < A ? P.tokens[d0 + lane] : (lane == A && !pending ? token : -1);
    P.committed[(size_t)r * width + lane] = v;
  }
  const float nan = __int_as_float(0x7fc00000);
  if (lane < k) {
    P.flags[d0 + lane] = lane < A ? 1 : 0;
    if (lane > A) {
      if (P.p_y) P.p_y[d0 + lane] = nan;
      if (P.q_y) P.q_y[d0 + lane] = nan;
      if (P.u_dbg) P.u_dbg[d0 + lane] = nan;
    }
  }
  if (lane == 0) {
    P.accepted_len[r] = A;
    if (P.req_status) P.req_status[r] = 0;
    if (pending) publish_job(P, r, A);
    __threadfence();
    *reinterpret_cast<volatile uint32_t*>(P.done + r) = P.epoch;
    atomicAdd(P.ctr + kCntReqDone, 1);
  }
}

// A request that cannot be verified: -1 outputs, flags 0, NaN debug values.
__device__ void skip_request(const Params& P, int r, int d0, int k, uint32_t rs) {
  const int lane = threadIdx.x & 31;
  const int width = P.max_k + 1;
  if (lane < width) P.committed[(size_t)r * width + lane] = -1;
  const float nan = __int_as_float(0x7fc00000);
  if (lane < k) {
    P.flags[d0 + lane] = 0;
    if (P.p_y) P.p_y[d0 + lane] = nan;
    if (P.q_y) P.q_y[d0 + lane] = nan;
    if (P.u_dbg) P.u_dbg[d0 + lane] = nan;
  }
  if (lane == 0) {
    P.accepted_len[r] = -1;
    if (P.req_status) P.req_status[r] = (int32_t)rs;
    atomicOr(reinterpret_cast<unsigned int*>(P.ctr + kCntStatus), rs);
    __threadfence();
    *reinterpret_cast<volatile uint32_t*>(P.done + r) = P.epoch;
    atomicAdd(P.ctr + kCntReqDone, 1);
  }
}

// Decides position i of request r (the control warp; its rows are merged and
// positions 0..i-1 were accepted).  "Speculative Decoding: Medusa, MTP, EAGLE,
// DFlash, DDTree, and DSpark", section 1: accept y_i with probability
// min(1, p_i(y_i)/q_i(y_i)), tested as u_i q_i(y_i) < p_i(y_i); at the first
// rejection draw from [p_i - q_i]_+, after k acceptances draw the bonus from
// p_k; greedy rounds keep y_i while it equals the target argmax.  Returns true
// when position i was accepted and position i+1 comes next.
template <typename E>
__device__ bool decide_position(const Params& P, int r, int i, const int* s_doff) {
  const int lane = threadIdx.x & 31;
  const int d0 = s_doff[r];
  const int k = s_doff[r + 1] - d0;
  const float t = __ldg(P.temperature + r);
  const int mode = req_mode(t);
  const size_t row_bytes = (size_t)P.vocab * E::kBytes;

  if (i == 0) {
    // inputs are checked once, before the first decision
    uint32_t rs = 0u;
    if (mode == kBadTemp) rs |= kStBadTemp;
    if (lane < k) {
      const int y = P.tokens[d0 + lane];
      if (y < 0 || y >= P.vocab) rs |= kStBadToken;
    }
    if (!rs && mode == kSampling && k > 0 && P.draft == nullptr) rs |= kStNoDraft;
    rs = __reduce_or_sync(0xffffffffu, rs);
    if (rs) {
      skip_request(P, r, d0, k, rs);
      return false;
    }
  }
  const Partial pt = ld_cg(P.rowres + slot_of(P, i, r, 0));
  if (mode == kGreedy) {
    if (pt.bad) {
      skip_request(P, r, d0, k, kStNonfinite);
      return false;
    }
    if (i < k && P.tokens[d0 + i] == pt.idx) return true;
    finish_request(P, r, d0, k, i, pt.idx, false);
    return false;
  }
  const RequestKey rk = request_key(P, r);
  const float c = kLog2e / t;
  const char* trow = reinterpret_cast<const char*>(P.target) + (size_t)(d0 + r + i) * row_bytes;
  ResidualRow rr{c, 0.f, 0.f, 0.f, 0.f};
  if (i == k) {
    // every draft accepted: the bonus draw (block race done in the row pass,
    // index -2 when the row is left to the slow path)
    int token = -1;
    if (pt.bad || pt.idx == -1) {
      skip_request(P, r, d0, k, kStNonfinite);
      return false;
    }
    if (pt.idx >= 0) {
      token = inner_race<E, false>(P, trow, nullptr, pt.idx, rr, (uint32_t)k, rk);
    } else {
      const BestAcc br = slow_block_race<E, false>(P, trow, nullptr, rr, (uint32_t)k, rk);
      if (br.nan || br.idx < 0) {
        skip_request(P, r, d0, k, kStNonfinite);
        return false;
      }
      token = inner_race<E, false>(P, trow, nullptr, br.idx, rr, (uint32_t)k, rk);
    }
    finish_request(P, r, d0, k, k, token, false);
    return false;
  }
  const Partial pd = ld_cg(P.rowres + slot_of(P, i, r, 1));
  if (pt.bad || pd.bad) {
    skip_request(P, r, d0, k, kStNonfinite);
    return false;
  }
  const char* drow = reinterpret_cast<const char*>(P.draft) + (size_t)(d0 + i) * row_bytes;
  const int y = P.tokens[d0 + i];
  const float tp = fmaf(E::load1(trow, y), c, -pt.a);  // log2(p(y) S_p)
  const float tq = fmaf(E::load1(drow, y), c, -pd.a);  // log2(q(y) S_q)
  const float u = accept_uniform(P.key, (uint32_t)i, rk.lo, rk.hi);
  // u q(y) < p(y), both sides scaled by S_p S_q 2^-max(tp, tq) > 0
  bool accept;
  if (tp == kNegInf) {
    accept = false;
  } else if (tq == kNegInf) {
    accept = true;
  } else {
    const float mx = fmaxf(tp, tq);
    accept = u * (fast_ex2(tq - mx) * pt.b) < fast_ex2(tp - mx) * pd.b;
  }
  if (lane == 0) {
    if (P.p_y) P.p_y[d0 + i] = fast_ex2(tp) / pt.b;
    if (P.q_y) P.q_y[d0 + i] = fast_ex2(tq) / pd.b;
    if (P.u_dbg) P.u_dbg[d0 + i] = u;
  }
  if (accept) return true;
  // first rejection at i: the residual draw
  if (row_fast<E>(trow, P.vocab) && row_fast<E>(drow, P.vocab)) {
    finish_request(P, r, d0, k, i, -1, true);  // a residual job draws the token
    return false;
  }
  rr = ResidualRow{c, pt.a, 1.f / pt.b, pd.a, 1.f / pd.b};
  BestAcc br = slow_block_race<E, true>(P, trow, drow, rr, (uint32_t)i, rk);
  int token;
  if (br.idx >= 0) {
    token = inner_race<E, true>(P, trow, drow, br.idx, rr, (uint32_t)i, rk);
  } else {
    // the residual has no mass (p == q): draw from p_i instead
    rr = ResidualRow{c, 0.f, 0.f, 0.f, 0.f};
    br = slow_block_race<E, false>(P, trow, nullptr, rr, (uint32_t)i, rk);
    token = inner_race<E, false>(P, trow, nullptr, br.idx, rr, (uint32_t)i, rk);
  }
  finish_request(P, r, d0, k, i, token, false);
  return false;
}

// Counts one merged row (or the accept signal) towards position i of request
// r; whoever completes the count decides, and an acceptance signals the next
// position, which may already have all its rows.
template <typename E>
__device__ void count_position(const Params& P, int r, int i, const int* s_doff) {
  const int lane = threadIdx.x & 31;
  const int d0 = s_doff[r];
  const int k = s_doff[r + 1] - d0;
  const int mode = req_mode(__ldg(P.temperature + r));
  const int width = P.max_k + 1;
  for (;;) {
    uint32_t cnt = 0;
    if (lane == 0) cnt = epoch_add(P.pos_cnt + (size_t)r * width + i, P.epoch);
    cnt = __shfl_sync(0xffffffffu, cnt, 0);
    if (cnt != position_target(P, i, k, mode)) return;
    __threadfence();
    if (!decide_position<E>(P, r, i, s_doff)) return;
    ++i;  // accepted: signal position i + 1
  }
}

// ---------------------------------------------------------------------------
// Job queue: claim one chunk (control lane 0), false if none is ready.
// Slot word: r (bits 0-23) | j (24-29) | published (31) | chunks left (32-63).
// *first_live skips slots already seen exhausted.
// ---------------------------------------------------------------------------
__device__ __forceinline__ bool claim_job(const Params& P, int* first_live, int* slot, int* r,
                                          int* j, int* ch) {
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

// Keep P.fill items queued ahead of q_used.  Items are claimed up to 8 at a
// time and decoded by separate lanes; items of decided requests are dropped.
template <typename E>
__device__ __forceinline__ void fill_queue(const Params& P, const int* s_doff, QItem* queue,
                                           int* s_qend, Ctrl& cs, int n_items) {
  const int lane = threadIdx.x & 31;
  while (!cs.exhausted && cs.q_head < cs.q_used + P.fill) {
    const int room = kQueue - 1 - (cs.q_head - cs.q_used);
    const int grab = min(8, room);
    int base = 0;
    if (lane == 0) base = atomicAdd(P.ctr + kCntItems, grab);
    base = __shfl_sync(0xffffffffu, base, 0);
    const int item = base + lane;
    bool keep = false;
    QItem it;
    if (lane < grab && item < n_items) {
      decode_item<E>(P, s_doff, item, it);
      keep = it.kind != kSkip &&
             *reinterpret_cast<const volatile uint32_t*>(P.done + it.r) != P.epoch;
    }
    const uint32_t mask = __ballot_sync(0xffffffffu, keep);
    if (keep) queue[(cs.q_head + __popc(mask & ((1u << lane) - 1u))) & (kQueue - 1)] = it;
    cs.q_head += __popc(mask);
    if (base + grab >= n_items) cs.exhausted = true;
  }
  __syncwarp();
  if (lane == 0) {
    __threadfence_block();  // queue entries before the count that publishes them
    *reinterpret_cast<volatile int*>(s_qend) = cs.exhausted ? -1 - cs.q_head : cs.q_head;
  }
  __syncwarp();
}

// Fill in the residual job chunk (slot, r, j, ch) (lane 0).
template <typename E>
__device__ __forceinline__ void make_job(const Params& P, const int* s_doff, int slot, int r,
                                         int j, int ch, Job& jb) {
  const size_t row_bytes = (size_t)P.vocab * E::kBytes;
  const int d0 = s_doff[r];
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
  __threadfence();
  const Partial rt = ld_cg(P.rowres + slot_of(P, j, r, 0));
  const Partial rd = ld_cg(P.rowres + slot_of(P, j, r, 1));
  jb.mp = rt.a;
  jb.inv_sp = 1.f / rt.b;
  jb.mq = rd.a;
  jb.inv_sq = 1.f / rd.b;
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
  // a whole-row item is its own row result; chunks are merged by the last one
  int last = 1;
  if (P.nch > 1) {
    if (lane == 0) {
      P.part[it.item] = p;
      __threadfence();
      last = (epoch_add(P.row_cnt + it.n, P.epoch) == (uint32_t)P.nch) ? 1 : 0;
    }
    last = __shfl_sync(0xffffffffu, last, 0);
    if (!last) return;
    __threadfence();
  }
  Partial res;
  if (it.kind == kSoftmax) {
    SoftmaxAcc a;
    a.init();
    if (P.nch == 1 && lane == 0) {
      a.m = p.a;
      a.s = p.b;
    }
    for (int q = lane; P.nch > 1 && q < P.nch; q += 32) {
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
    if (P.nch == 1 && lane == 0) {
      a.v = p.a;
      a.idx = p.idx;
      a.nan = p.bad;
    }
    for (int q = lane; P.nch > 1 && q < P.nch; q += 32) {
      const Partial pq = ld_cg(P.part + (size_t)it.n * P.nch + q);
      BestAcc b;
      b.v = pq.a;
      b.idx = pq.idx;
      b.nan = pq.bad;
      a = BestAcc::merge(a, b);
    }
    a = warp_reduce(a);
    // argmax rows need a finite maximum; race rows carry a block index (-1: no
    // block with mass, -2: left to the slow path), judged by the scan
    const bool bad = it.kind == kRace ? a.nan != 0u
                                      : (a.nan != 0u || a.idx < 0 || !(a.v < 3.0e38f));
    res = Partial{a.v, 0.f, a.idx, bad ? 1u : 0u};
  }
  if (lane == 0) {
    P.rowres[it.n] = res;
    __threadfence();
  }
  __syncwarp();
  count_position<E>(P, it.r, it.pos, s_doff);
}

// Completion of a job unit: the last chunk merges the block race, runs the
// element race in the winning block and commits the token (a residual without
// mass, i.e. p == q, draws from p_j instead, by the slow path).
struct JobRef {
  int slot, r, j, ch;
};
template <typename E>
__device__ void complete_job(const Params& P, const int* s_doff, const JobRef& jb,
                             const Partial* mb) {
  const int lane = threadIdx.x & 31;
  const Partial p = combine_best(mb);
  int last = 0;
  if (lane == 0) {
    P.part2[(size_t)jb.slot * P.jnch + jb.ch] = p;
    __threadfence();
    last = (atomicAdd(P.res_cnt + jb.slot, 1) == P.jnch - 1) ? 1 : 0;
  }
  last = __shfl_sync(0xffffffffu, last, 0);
  if (!last) return;
  __threadfence();
  BestAcc a;
  a.init();
  for (int q = lane; q < P.jnch; q += 32) {
    const Partial pq = ld_cg(P.part2 + (size_t)jb.slot * P.jnch + q);
    BestAcc b;
    b.v = pq.a;
    b.idx = pq.idx;
    b.nan = 0u;
    a = BestAcc::merge(a, b);
  }
  a = warp_reduce(a);
  const size_t row_bytes = (size_t)P.vocab * E::kBytes;
  const int d0 = s_doff[jb.r];
  const char* trow = reinterpret_cast<const char*>(P.target) + (size_t)(d0 + jb.r + jb.j) * row_bytes;
  const char* drow = reinterpret_cast<const char*>(P.draft) + (size_t)(d0 + jb.j) * row_bytes;
  const float c = kLog2e / __ldg(P.temperature + jb.r);
  const RequestKey rk = request_key(P, jb.r);
  int token;
  if (a.idx >= 0) {
    const Partial pt = ld_cg(P.rowres + slot_of(P, jb.j, jb.r, 0));
    const Partial pd = ld_cg(P.rowres + slot_of(P, jb.j, jb.r, 1));
    const ResidualRow rr{c, pt.a, 1.f / pt.b, pd.a, 1.f / pd.b};
    token = inner_race<E, true>(P, trow, drow, a.idx, rr, (uint32_t)jb.j, rk);
  } else {
    const ResidualRow rr{c, 0.f, 0.f, 0.f, 0.f};
    const BestAcc br = slow_block_race<E, false>(P, trow, nullptr, rr, (uint32_t)jb.j, rk);
    token = inner_race<E, false>(P, trow, nullptr, br.idx, rr, (uint32_t)jb.j, rk);
  }
  if (lane == 0) {
    P.res_cnt[jb.slot] = 0;
    P.committed[(size_t)jb.r * (P.max_k + 1) + jb.j] = token;
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
  __shared__ int s_kmax;
  __shared__ uint32_t s_layout;
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const bool control = warp == kComputeWarps;

  // --- prefix sums of num_draft, and the layout check (all threads) -----------
  if (tid == 0) {
    s_layout = 0u;
    s_kmax = 0;
  }
  __syncthreads();
  int carry = 0;
  for (int base = 0; base < P.batch; base += kBlock) {
    const int r = base + tid;
    const int k = r < P.batch ? P.num_draft[r] : 0;
    const bool badk = k < 0 || k > P.max_k;
    if (badk) atomicOr(&s_layout, kStBadK);
    const int kk = badk ? 0 : k;
    if (kk > 0) atomicMax(&s_kmax, kk);
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
  // waves 0..max_k of this batch, two slots per request each
  const int n_items = (s_kmax + 1) * 2 * P.batch * P.nch;

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
      fill_queue<E>(P, s_doff, queue, &s_qend, cs, n_items);
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
              a = item_race<E>(P, queue, &s_qend, ring, lc, gs, it);
            }
            a = warp_reduce(a);
            out = Partial{a.v, 0.f, a.idx, a.nan};
          }
          if (lane == 0) mailbox[u & 1][warp] = out;
        } else if (type == kUnitResidual) {
          const Job jb = s_unit[u & 1].job;
          BestAcc a = job_chunk<E>(P, jb);
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
        } else if (prev_type == kUnitResidual) {
          complete_job<E>(P, s_doff, prev_job, mailbox[(u - 1) & 1]);
        }
        // keep the items the compute warps may stream during unit u+1 queued
        fill_queue<E>(P, s_doff, queue, &s_qend, cs, n_items);
        // next unit: a claimable job first, then the next queued item
        int next_type = kUnitIdle;
        if (lane == 0) {
          Unit nx;
          nx.type = kUnitIdle;
          int slot, r, j, ch;
          bool got = false;
          if (ld_volatile(P.ctr + kCntPublished) != ld_volatile(P.ctr + kCntClaimed))
            got = claim_job(P, &cs.first_live, &slot, &r, &j, &ch);
          if (got) {
            nx.type = kUnitResidual;
            make_job<E>(P, s_doff, slot, r, j, ch, nx.job);
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
