// sv_kernels.cuh -- the verify round as a plan launch and a short sequence of
// wave launches.
//
// Left to right, and no further than needed.  A round tests the draft
// positions of each request left to right and discards everything after the
// first rejection ("Speculative Decoding: Medusa, MTP, EAGLE, DFlash, DDTree,
// and DSpark", section 1), so only the rows of positions 0..A are needed, plus
// the bonus row when all k drafts are accepted.  The round is therefore run as
// waves of D positions: wave w streams, for every request still alive at
// position w*D, its rows of positions w*D .. w*D+D-1 -- target row t_i and
// draft row d_i (sampling, i < k), the bonus row t_k (sampling, i = k) or
// target row t_i (greedy) -- and decides them in order.  A request that
// survives the wave is appended to the list of wave w+1; a rejected one to the
// residual list, whose rows t_j and d_j the next wave reads again (first,
// while they may still sit in L2) to draw the correction token.  D = 1 reads
// exactly the needed rows; a larger D trades rows read past a rejection for
// fewer launches, which pays for small batches.
//
// Inside a wave the work is split flat: the wave's rows form one sequence of
// vocab blocks (128 vocab ids), and CTA c takes the contiguous range
// [c*T/G, (c+1)*T/G) of it, so every CTA streams the same number of bytes
// whatever the row lengths.  A CTA's range cuts into a few row segments; each
// segment reduces to one 16-byte partial.  A position is decided by the CTA
// that brings its count to the total: the segments of its rows, plus one for
// "the previous position of this wave was accepted".  No CTA ever waits for
// another, there is no work claiming, and the segment count of any row follows
// from the split arithmetic alone.
//
// CTA layout: 7 compute warps and 1 control warp, one __syncthreads per
// segment.  Compute warps stream the segment and leave one partial per warp in
// shared memory; during the next segment the control warp combines them and
// does every latency-bound step: partial stores, the completion counts, the
// merges, the decisions, the list appends and the outputs.  Consecutive waves
// overlap their launch with programmatic dependent launch.
//
// Memory pipeline (16-byte aligned rows): each compute thread streams its
// vectors of successive segments through a private shared-memory ring with
// cp.async, kStages-1 stages ahead and across segment boundaries, and only
// reads back what it copied itself.  Rows that are not 16-byte aligned take a
// scalar path with the same structure.
#pragma once

#include <cstddef>

#include "sv_device.cuh"

namespace sv {

constexpr int kComputeWarps = 7;
constexpr int kThreads = kComputeWarps * 32;   // compute threads
constexpr int kBlock = kThreads + 32;          // + the control warp
constexpr int kStages = 8;
constexpr int kStageVecs = 2;
constexpr int kQueue = 16;                     // segment queue entries (power of 2)
constexpr int kMaxBatch = 4096;                // requests per round
constexpr int kMaxK = 31;                      // draft positions per request
constexpr int kPlanThreads = 1024;
constexpr int kPlanTokens = 4096;              // draft tokens the plan stages in shared memory
constexpr int kVocabBlock = 128;               // vocab ids per block of the flat split
constexpr int kMinSpanBytes = 16384;           // smallest share of a wave per CTA

enum RowKind : int { kSoftmax = 0, kArgmax = 1, kRace = 2, kResidual = 3 };
enum ReqMode : int { kBadTemp = 0, kGreedy = 1, kSampling = 2 };
// Mailbox slots between the compute warps and the control warp, and the named
// barriers that hand them over (0 is __syncthreads).
constexpr int kMailSlots = 4;
constexpr int kBarReady = 1;          // kBarReady + slot: partials of the slot are in
constexpr int kBarFree = 1 + kMailSlots;  // kBarFree + slot: the slot may be refilled
constexpr int kCtaThreads = kThreads + 32;

// Status bits (equal to the SPECVERIFY_STATUS_* values of the header).
constexpr uint32_t kStBadToken = 1u, kStBadK = 2u, kStBadTemp = 4u, kStNonfinite = 8u,
                   kStBadTotal = 16u, kStNoDraft = 64u,
                   kStBadConf = 512u;

// Number of waves of a round with positions 0..max_k taken D at a time: one
// per group of D positions, plus one for the residual draws of the last group
// when it can reject (D > 1).
__host__ __device__ constexpr int wave_count(int max_k, int depth) {
  return (max_k + depth) / depth + (depth > 1 ? 1 : 0);
}

// One row of a wave's list, written by the plan launch or by the CTA that
// accepted the request's last position of the previous wave.
struct __align__(16) Entry {
  int meta;         // r | is_draft << 13 | paired << 14 | k << 15 | pos << 20
  int d0;           // the request's first draft row
  float c;          // log2(e) / T; 0 for greedy requests
  int y;            // the draft token at pos; -1 at pos = k
  uint32_t req_lo;  // Philox request word
  uint32_t req_hi;
  int base;         // list index of the request's first row in this wave
  int pad;
};

__host__ __device__ __forceinline__ int entry_meta(int r, int is_draft, int paired, int k, int pos) {
  return r | (is_draft << 13) | (paired << 14) | (k << 15) | (pos << 20);
}

struct __align__(16) Partial {
  float a;       // softmax: m     | best: value
  float b;       // softmax: S     | unused
  int idx;       // softmax: x[y]  | best: index
  uint32_t bad;  // softmax: 1 when the segment holds y | best: NaN seen
};

// The merged rows of one position (a wave of several positions per request):
// target row (a = m or best value, b = S, xy = x[y], idx = best index) and
// draft row, with their NaN / non-finite flags (bit 0 target, bit 1 draft).
struct __align__(16) PosRec {
  float ta, tb, txy;
  int tidx;
  float da, db, dxy;
  uint32_t bad;
};

// A rejected request waiting for its correction draw (written by the deciding
// CTA of wave w, read by wave w+1).
struct __align__(16) ResEntry {
  int r, j, d0, pad;
  float c, mp, inv_sp, mq;
  float inv_sq;
  uint32_t req_lo, req_hi, pad2;
};

// Global counters.
enum Counter : int {
  kCntStatus = 0,
  kCntLive = 1,   // requests the plan left to verify
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
  int depth;         // D, positions per wave
  int wave;          // this launch: wave w, positions [pos0, pos1)
  int pos0, pos1;
  int n_waves;
  uint32_t epoch;    // this round's tag of the completion counters
  int nb;            // vocab blocks per row
  int nvec;          // 16-byte vectors per row (aligned rows)
  int min_span;      // fewest vocab blocks per CTA share of the row phase
  int min_span_res;  // ... and of the residual phase
  int stride;        // capacity of a request-indexed array (max_batch)
  int list_cap;      // entries per wave list: 2 * D * stride
  // Device copies of the window, same layout as target / draft, or NULL.  When
  // set (waves, 16-byte rows, logits read from host memory), every sampled
  // row a wave streams is also written here, and the correction draws of the
  // next wave read these copies instead of the host rows.
  char* tee_target;
  char* tee_draft;
  int trimmed;              // num_draft is the window layout; verify trimmed windows
  const float* confidence;  // trimmed runs: c_i per draft position of the window layout
  const float* cost;        // trimmed runs: cost of one verified position, per request
  int32_t* verified_k;      // trimmed runs: the window verified per request (out)
  int32_t* accepted_len;
  int32_t* committed;
  uint8_t* flags;
  float* p_y;
  float* q_y;
  float* u_dbg;
  int32_t* req_status;
  // Truncated rounds: the order-key threshold of every target / draft row of
  // the window (the logits below it read as -inf), or NULL.
  const uint32_t* thr_t;
  const uint32_t* thr_d;
  Entry* lists;                 // [n_waves * list_cap] rows of each wave (bonus rows apart)
  int* list_cnt;                // [n_waves]
  Entry* blists;                // [n_waves * stride] bonus rows of each wave
  int* blist_cnt;               // [n_waves]
  ResEntry* res;                // [n_waves * stride] rejections of each wave
  int* res_cnt;                 // [n_waves]
  unsigned long long* pos_cnt;  // [(max_k + 1) * stride] epoch | count of a position
  unsigned long long* rcnt;     // [stride] epoch | residual segments merged
  Partial* part;                // [grid + list_cap] row segment partials
  Partial* bpart;               // [grid + stride] bonus-row segment partials
  Partial* rpart;               // [grid + stride] residual segment partials
  int* ctr;                     // [kCntCount]
  PosRec* recs;                 // [(max_k + 1) * stride] merged rows of multi-position waves
  unsigned long long* rdy;      // [n_waves * stride] epoch | positions of a request merged
};

__device__ __forceinline__ Partial ld_cg(const Partial* p) {
  const int4 v = __ldcg(reinterpret_cast<const int4*>(p));
  return Partial{__int_as_float(v.x), __int_as_float(v.y), v.z, (uint32_t)v.w};
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

// ---------------------------------------------------------------------------
// The flat split of one phase of a wave: n rows of nb vocab blocks, T = n * nb
// blocks over G CTAs; CTA c takes blocks [c*T/G, (c+1)*T/G).
// ---------------------------------------------------------------------------
struct Split {
  unsigned long long T;
  int G;
  __device__ __forceinline__ void init(int n, int nb, int min_span, int grid) {
    T = (unsigned long long)n * (unsigned long long)nb;
    const unsigned long long g = T / (unsigned long long)min_span;
    G = (int)(g < 1ull ? 1ull : (g > (unsigned long long)grid ? (unsigned long long)grid : g));
    if (n == 0) G = 0;
  }
  __device__ __forceinline__ unsigned long long begin(int c) const {
    return (unsigned long long)c * T / (unsigned long long)G;
  }
  // the CTA whose share holds block x
  __device__ __forceinline__ int cta_of(unsigned long long x) const {
    return (int)(((x + 1ull) * (unsigned long long)G - 1ull) / T);
  }
  __device__ __forceinline__ int first_cta(int e, int nb) const {
    return cta_of((unsigned long long)e * nb);
  }
  __device__ __forceinline__ int last_cta(int e, int nb) const {
    return cta_of((unsigned long long)(e + 1) * nb - 1ull);
  }
  __device__ __forceinline__ int segments(int e, int nb) const {
    return last_cta(e, nb) - first_cta(e, nb) + 1;
  }
};

// A segment of the CTA's share, decoded once by the control warp.
struct __align__(16) QItem {
  const char* row;   // the row (target row of a residual segment)
  const char* row2;  // draft row of a residual segment
  int kind;          // RowKind of this segment
  int e;             // list (or residual list) entry
  int r, d0, k, y;   // request, its first draft row, k, the draft token at pos (or -1)
  int pos;           // the position the row belongs to (Philox position)
  int base;          // list index of the request's first row in this wave
  int paired, is_draft;
  int vbeg, vend;    // vectors (aligned rows) or vocab blocks (scalar path)
  int nst;           // ring stages (aligned rows)
  int g;             // partial index: CTA + entry
  int yv;            // vector (aligned) or vocab block (scalar) holding y, -1 if none
  float c;           // log2(e) / T
  float mp, inv_sp, mq, inv_sq;  // residual segments: normalisers of p_j and q_j
  uint32_t req_lo, req_hi;
  int e0;    // entry e of the phase is partial slot CTA + e0 + e
  int phase;  // 0 correction draws, 1 rows, 2 bonus rows
  uint32_t thr, thr2;  // truncation thresholds of row and row2 (0: none)
  char* tee;  // where a softmax segment's row is copied (Params::tee_*), or NULL
};


// ---------------------------------------------------------------------------
// Exponential race over vocab ids.  A categorical draw from weights w_v >= 0
// is argmin_{v: w_v > 0} E_v / w_v, E_v the race exponential of the Philox
// stream-1 word of vocab id v at the draw's (request, position), lowest index
// on ties; in the base-2 log domain it is the argmax of the score
//   s_v = log2 w_v + gain_v,   gain_v = -log2 E_v.
// E_v / w_v is exponential with rate w_v, so the winner is an exact sample of
// w / sum w, and the order in which ids are visited does not change it.
//
// Every id needs its word (one Philox call gives the words of four
// consecutive ids), but not its exponential: race_gain_bound(word) bounds the
// gain from integer operations, so an id whose bounded score cannot beat the
// thread's best so far is passed over without a logarithm, and a group of
// four whose largest logit plus the largest possible gain (kMaxGain) cannot
// beat it is passed over without the Philox call.  Both skips are exact: a
// skipped id's computed score is never above the best it is compared with.
// ---------------------------------------------------------------------------
constexpr float kMaxGain = 33.001f;   // >= race_gain_bound(w) for every word w
constexpr float kBoundSlack = 1e-3f;  // margin of the fast log2 p_v bound below

// Words of ids 4 g .. 4 g + 3 (stream 1).
__device__ __forceinline__ uint4 race_words(uint32_t g, uint32_t pos, RequestKey rk,
                                            PhiloxKey key) {
  return philox4x32_10(make_uint4(g, pos, rk.lo, 1u | (rk.hi << 8)), key);
}

// -log2 E for a race word.
__device__ __forceinline__ float race_gain(uint32_t w) { return -fast_lg2(race_exponential(w)); }

// IEEE max that propagates NaN (a NaN logit is then seen by the group test).
__device__ __forceinline__ float fmax_nan(float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}

template <typename E>
__device__ __forceinline__ void group_max(const float (&x)[E::kVec], int h, float& mx) {
  mx = fmax_nan(fmax_nan(x[h], x[h + 1]), fmax_nan(x[h + 2], x[h + 3]));
}

// Bonus race (weights 2^(c x_v), unnormalised) over one vector of kVec
// consecutive ids starting at id e0 (a multiple of 4); ids must come in
// increasing order per thread.  A NaN or +inf logit marks the row bad.
template <typename E>
__device__ __forceinline__ void race_vec(BestAcc& acc, const float (&x)[E::kVec], int e0, float c,
                                         uint32_t pos, RequestKey rk, PhiloxKey key) {
#pragma unroll
  for (int h = 0; h < E::kVec; h += 4) {
    float mx;
    group_max<E>(x, h, mx);
    acc.nan |= !(mx < -kNegInf);
    if (fmaf(mx, c, kMaxGain) > acc.v) {
      const uint4 r = race_words((uint32_t)(e0 + h) >> 2, pos, rk, key);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t w = word_of(r, i);
        if (fmaf(x[h + i], c, race_gain_bound(w)) > acc.v)
          acc.take(fmaf(x[h + i], c, race_gain(w)), e0 + h + i);
      }
    }
  }
}

// Residual race over [p - q]_+ (the normalisers of p_j and q_j known) for one
// vector of each row.  log2 p_v + kBoundSlack = fmaf(x, c, rr.lp) bounds
// log2 (p_v - q_v) from above.
struct ResidualRow {
  float c, mp, inv_sp, mq, inv_sq;
  float lp;  // -mp + log2(inv_sp) + kBoundSlack
};

template <typename E>
__device__ __forceinline__ void residual_vec(BestAcc& acc, const float (&x)[E::kVec],
                                             const float (&z)[E::kVec], int e0,
                                             const ResidualRow& rr, uint32_t pos, RequestKey rk,
                                             PhiloxKey key) {
#pragma unroll
  for (int h = 0; h < E::kVec; h += 4) {
    const float mx = fmaxf(fmaxf(x[h], x[h + 1]), fmaxf(x[h + 2], x[h + 3]));
    if (fmaf(mx, rr.c, rr.lp) + kMaxGain > acc.v) {
      const uint4 r = race_words((uint32_t)(e0 + h) >> 2, pos, rk, key);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t w = word_of(r, i);
        if (fmaf(x[h + i], rr.c, rr.lp) + race_gain_bound(w) > acc.v) {
          const float p = fast_ex2(fmaf(x[h + i], rr.c, -rr.mp)) * rr.inv_sp;
          const float q = fast_ex2(fmaf(z[h + i], rr.c, -rr.mq)) * rr.inv_sq;
          const float d = p - q;
          if (d > 0.f) acc.take(fast_lg2(d) + race_gain(w), e0 + h + i);
        }
      }
    }
  }
}

__device__ __forceinline__ ResidualRow residual_row(float c, float mp, float inv_sp, float mq,
                                                    float inv_sq) {
  return ResidualRow{c, mp, inv_sp, mq, inv_sq, -mp + fast_lg2(inv_sp) + kBoundSlack};
}

// N Philox blocks of stream 1 (ids 4 g[i] .. 4 g[i] + 3) with their rounds
// interleaved: independent dependency chains the scheduler overlaps.
template <int N>
__device__ __forceinline__ void race_words_n(uint4 (&r)[N], const uint32_t (&g)[N], uint32_t pos,
                                             RequestKey rk, PhiloxKey key) {
#pragma unroll
  for (int i = 0; i < N; ++i) r[i] = make_uint4(g[i], pos, rk.lo, 1u | (rk.hi << 8));
  uint32_t k0 = key.k0, k1 = key.k1;
#pragma unroll
  for (int round = 0; round < 10; ++round) {
#pragma unroll
    for (int i = 0; i < N; ++i) {
      const uint4 c = r[i];
      const uint64_t p0 = (uint64_t)c.x * 0xD2511F53u;
      const uint64_t p1 = (uint64_t)c.z * 0xCD9E8D57u;
      r[i] = make_uint4((uint32_t)(p1 >> 32) ^ c.y ^ k0, (uint32_t)p1,
                        (uint32_t)(p0 >> 32) ^ c.w ^ k1, (uint32_t)p0);
    }
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
}

// Largest of the 4 N words of N Philox blocks.
template <int N>
__device__ __forceinline__ uint32_t max_word(const uint4 (&r)[N]) {
  uint32_t m = max(max(r[0].x, r[0].y), max(r[0].z, r[0].w));
#pragma unroll
  for (int i = 1; i < N; ++i) m = max(m, max(max(r[i].x, r[i].y), max(r[i].z, r[i].w)));
  return m;
}

// The race's best score so far, shared by the warps that reduce one segment
// (a shared-memory word per mailbox slot, raised with atomicMax): every warp
// then prunes with the best any of them has found.  Floats map to unsigned
// words in the same order.
__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t b = __float_as_uint(f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float from_order_key(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}
constexpr uint32_t kOrderKeyNegInf = 0x007fffffu;  // order_key(-inf)

// kOn = false (the build for logits read from host memory, whose streaming
// measured slower with the shared word in the kernel) keeps each warp's best
// to itself.
template <bool kOn>
struct SharedBest {
  uint32_t* word;  // the segment's mailbox-slot word
  __device__ __forceinline__ float load() const {
    return kOn ? from_order_key(*reinterpret_cast<volatile uint32_t*>(word)) : kNegInf;
  }
  __device__ __forceinline__ void raise(float v) const {
    if (kOn && (threadIdx.x & 31) == 0) atomicMax(word, order_key(v));
  }
};

// Smallest gain any word can have: E < 22.9, so -log2 E > -4.52.
constexpr float kMinGain = -4.52f;

// A race score enters the best only when finite: an id of zero weight (a
// logit of -inf, or a residual that underflows) never wins, even against an
// empty best of -inf.
__device__ __forceinline__ void take_finite(BestAcc& acc, float score, int i) {
  if (score > kNegInf) acc.take_cmp(score, i);
}

// Bonus race over one stage of the copy ring: vectors x0 (ids e0 ..) and x1
// (ids e1 ..), kVec ids each.  `wbest` is the best score of the warp so far
// (warp-uniform, raised after a stage where some lane took an element): an id
// whose bounded score is below it cannot be the row's winner, so every lane
// tests against the warp's best, not only its own.  The test keeps ties
// (>=), which take_cmp then orders by index.  Call with the whole warp.
// kSkipEmpty (truncated rounds): a stage of -inf logits has no id to race.
template <typename E, bool kShare, bool kSkipEmpty>
__device__ __forceinline__ void race_stage(BestAcc& acc, float& wbest, const SharedBest<kShare>& sb,
                                           const float (&x0)[E::kVec],
                                           const float (&x1)[E::kVec], int e0, int e1, float c,
                                           uint32_t pos, RequestKey rk, PhiloxKey key) {
  constexpr int G = E::kVec / 4;  // Philox blocks per vector
  float mx = x0[0];
#pragma unroll
  for (int i = 1; i < E::kVec; ++i) mx = fmax_nan(mx, x0[i]);
#pragma unroll
  for (int i = 0; i < E::kVec; ++i) mx = fmax_nan(mx, x1[i]);
  acc.nan |= !(mx < -kNegInf);  // NaN or +inf
  wbest = fmaxf(wbest, sb.load());
  if (wbest == kNegInf) {
    // first stage: the largest logit seen, with the smallest gain any word can
    // have, is a score some id reaches, so the winner's score is at least that
    const float lo = warp_max(mx < -kNegInf ? mx : kNegInf) * c + kMinGain;
    if (lo > kNegInf) wbest = lo - kBoundSlack;
  }
  if (!__any_sync(0xffffffffu, (!kSkipEmpty || mx > kNegInf) && fmaf(mx, c, kMaxGain) >= wbest))
    return;
  uint32_t g[2 * G];
#pragma unroll
  for (int j = 0; j < G; ++j) {
    g[j] = (uint32_t)(e0 >> 2) + j;
    g[G + j] = (uint32_t)(e1 >> 2) + j;
  }
  uint4 r[2 * G];
  race_words_n<2 * G>(r, g, pos, rk, key);
  // the stage's largest logit with its largest word bounds every id's score
  // from above (both terms are monotone), so one test stands for all of them
  const bool pass = fmaf(mx, c, race_gain_bound(max_word<2 * G>(r))) >= wbest;
  if (pass) {
#pragma unroll
    for (int i = 0; i < E::kVec; ++i) {
      const uint32_t w = word_of(r[i >> 2], i & 3);
      if (fmaf(x0[i], c, race_gain_bound(w)) >= wbest)
        take_finite(acc, fmaf(x0[i], c, race_gain(w)), e0 + i);
    }
#pragma unroll
    for (int i = 0; i < E::kVec; ++i) {
      const uint32_t w = word_of(r[G + (i >> 2)], i & 3);
      if (fmaf(x1[i], c, race_gain_bound(w)) >= wbest)
        take_finite(acc, fmaf(x1[i], c, race_gain(w)), e1 + i);
    }
  }
  if (__any_sync(0xffffffffu, pass)) {
    wbest = fmaxf(wbest, warp_max(acc.v));
    sb.raise(wbest);
  }
}

// Residual race over one stage: vector x of t_j and z of d_j, the same kVec
// ids from e0.  fmaf(x, c, rr.lp) bounds log2 (p_v - q_v) from above, so the
// two exponentials are only taken for ids that pass.  Call with the whole warp.
template <typename E, bool kShare, bool kSkipEmpty>
__device__ __forceinline__ void residual_stage(BestAcc& acc, float& wbest,
                                               const SharedBest<kShare>& sb,
                                               const float (&x)[E::kVec],
                                               const float (&z)[E::kVec], int e0,
                                               const ResidualRow& rr, uint32_t pos,
                                               RequestKey rk, PhiloxKey key) {
  constexpr int G = E::kVec / 4;
  float mx = x[0];
#pragma unroll
  for (int i = 1; i < E::kVec; ++i) mx = fmaxf(mx, x[i]);
  wbest = fmaxf(wbest, sb.load());
  if (!__any_sync(0xffffffffu,
                  (!kSkipEmpty || mx > kNegInf) && fmaf(mx, rr.c, rr.lp) + kMaxGain >= wbest))
    return;
  uint32_t g[G];
#pragma unroll
  for (int j = 0; j < G; ++j) g[j] = (uint32_t)(e0 >> 2) + j;
  uint4 r[G];
  race_words_n<G>(r, g, pos, rk, key);
  // one bound for the whole vector: its largest logit with its largest word
  const bool pass = fmaf(mx, rr.c, rr.lp) + race_gain_bound(max_word<G>(r)) >= wbest;
  if (pass) {
#pragma unroll
    for (int i = 0; i < E::kVec; ++i) {
      const uint32_t w = word_of(r[i >> 2], i & 3);
      if (fmaf(x[i], rr.c, rr.lp) + race_gain_bound(w) >= wbest) {
        const float p = fast_ex2(fmaf(x[i], rr.c, -rr.mp)) * rr.inv_sp;
        const float q = fast_ex2(fmaf(z[i], rr.c, -rr.mq)) * rr.inv_sq;
        const float d = p - q;
        if (d > 0.f) take_finite(acc, fast_lg2(d) + race_gain(w), e0 + i);
      }
    }
  }
  if (__any_sync(0xffffffffu, pass)) {
    wbest = fmaxf(wbest, warp_max(acc.v));
    sb.raise(wbest);
  }
}

// The race over a whole row by one warp with plain loads (lane l takes ids
// 128 b + 4 l .. + 3): the draw from p_j when a residual turns out to have no
// mass in fp32 (p <= q everywhere), an edge case.
template <typename E>
__device__ int warp_row_race(const Params& P, const char* trow, float c, uint32_t pos,
                             RequestKey rk, uint32_t thr) {
  const int lane = threadIdx.x & 31;
  BestAcc acc;
  acc.init();
  for (int v0 = 4 * lane; v0 < P.vocab; v0 += 128) {
    float x[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      x[i] = v0 + i < P.vocab ? mask1<E>(E::load1(trow, v0 + i), thr) : kNegInf;
    // a group that cannot beat this lane's best (all -inf, in a truncated
    // row) needs no Philox call
    const float mx = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
    if (!(mx > kNegInf && fmaf(mx, c, kMaxGain) >= acc.v)) continue;
    const uint4 r = race_words((uint32_t)v0 >> 2, pos, rk, P.key);
#pragma unroll
    for (int i = 0; i < 4; ++i) acc.take(fmaf(x[i], c, race_gain(word_of(r, i))), v0 + i);
  }
  return warp_reduce(acc).idx;
}

// ---------------------------------------------------------------------------
// The per-thread copy ring (compute threads, aligned rows).  Stage s of a
// segment holds two vectors per thread: vectors vbeg + 2 s kThreads + tid and
// + kThreads of a single row, or vector vbeg + s kThreads + tid of t_j and of
// d_j for a residual segment.
// ---------------------------------------------------------------------------
struct LoadCursor {
  int q;      // queue index of the segment being loaded
  int left;   // its stages still to copy
  const uint4* b0;
  const uint4* b1;
  int i0, i1, step, vend;
  bool active;

  // s_qend: segments the control warp has queued, or -1 - n once all n are.
  __device__ __forceinline__ void open(const QItem* queue, const int* s_qend) {
    const int qe = ld_acquire_shared(s_qend);
    const int avail = qe >= 0 ? qe : -1 - qe;
    active = q < avail;
    if (active) {
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
  }

  // copy the next stage into ring slot `slot` and commit one group
  __device__ __forceinline__ void issue(const QItem* queue, const int* s_qend, uint4* ring,
                                        int slot) {
    if (!active) open(queue, s_qend);
    if (active) {
      uint4* dst = ring + slot * kStageVecs * kThreads + threadIdx.x;
      cp_async16_if(dst, b0 + i0, i0 < vend);
      cp_async16_if(dst + kThreads, b1 + i1, i1 < vend);
      i0 += step;
      i1 += step;
      if (--left == 0) {
        ++q;
        open(queue, s_qend);
      }
    }
    cp_async_commit();
  }
};

// Reads one stage of the ring (after its copies landed) and refills the ring
// one stage ahead.
__device__ __forceinline__ void ring_take(const QItem* queue, const int* s_qend, uint4* ring,
                                          LoadCursor& lc, int& g_stage, uint4& v0, uint4& v1) {
  cp_async_wait<kStages - 2>();
  const int slot = g_stage & (kStages - 1);
  const uint4* src = ring + slot * kStageVecs * kThreads + threadIdx.x;
  v0 = src[0];
  v1 = src[kThreads];
  lc.issue(queue, s_qend, ring, (g_stage + kStages - 1) & (kStages - 1));
  ++g_stage;
}

// ---------------------------------------------------------------------------
// Segment reductions (compute threads).  Each returns this warp's partial; a
// softmax segment that holds the draft token y also leaves x[y] in *s_xy.
// ---------------------------------------------------------------------------
// `take(v0, v1)` hands over the next stage of the segment from the copy ring.
// kTrunc: the build for truncated rounds, which masks the rows on load.
template <typename E, bool kShare, bool kTrunc, typename Take>
__device__ __forceinline__ Partial seg_reduce(const Params& P, const QItem& itm, float* s_xy,
                                              uint32_t* s_best, Take& take) {
  const int tid = threadIdx.x;
  // the segment's fields in registers (the queue is shared memory, which the
  // copy ring's memory clobbers would otherwise make the loop reload)
  const int kind = itm.kind, vbeg = itm.vbeg, vend = itm.vend, nst = itm.nst, pos = itm.pos;
  const float c = itm.c;
  const uint32_t thr = itm.thr, thr2 = itm.thr2;  // truncation (0: none)
  const uint32_t tb = mask_bits<E>(thr), tb2 = mask_bits<E>(thr2);
  const RequestKey rk{itm.req_lo, itm.req_hi};
  const int per = kind == kResidual ? kThreads : kStageVecs * kThreads;
  const int nfull = (vend - vbeg) / per;
  if (kind == kSoftmax) {
    LazySoftmax acc;
    acc.init();
    // x[y] comes from the thread whose vectors hold it, loaded before the
    // stages so that its latency hides under them (no test inside the loop)
    const int yv = itm.yv;
    const bool own_y = yv >= vbeg && yv < vend && (yv - vbeg) % kThreads == tid;
    float xy = 0.f;
    if (own_y) xy = kTrunc ? mask1<E>(E::load1(itm.row, itm.y), thr) : E::load1(itm.row, itm.y);
    // the stages: plain, with the copy to the device staging, or truncated
    // (a loop of its own for each, so the common one carries no test)
    auto stages = [&](auto mode) {
      constexpr int kMode = decltype(mode)::value;
      uint4* tee = reinterpret_cast<uint4*>(itm.tee);
      for (int st = 0; st < nst; ++st) {
        uint4 v0, v1;
        take(v0, v1);
        const int vi = vbeg + st * kStageVecs * kThreads + tid;
        if (kMode == 1) {
          if (vi < vend) tee[vi] = v0;
          if (vi + kThreads < vend) tee[vi + kThreads] = v1;
        }
        if (kMode == 2) {
          mask_vec<E>(v0, tb);
          mask_vec<E>(v1, tb);
        }
        if (st >= nfull) {
          if (vi >= vend) v0 = E::pad();
          if (vi + kThreads >= vend) v1 = E::pad();
        }
        float x0[E::kVec], x1[E::kVec];
        E::unpack(v0, x0);
        E::unpack(v1, x1);
        acc.add2(x0, x1, c);
      }
    };
    if constexpr (kTrunc) {
      if (thr)
        stages(std::integral_constant<int, 2>{});
      else
        stages(std::integral_constant<int, 0>{});
    } else {
      if (itm.tee)
        stages(std::integral_constant<int, 1>{});
      else
        stages(std::integral_constant<int, 0>{});
    }
    if (own_y) *s_xy = xy;
    SoftmaxAcc a = warp_reduce(acc.result());
    return Partial{a.m, a.s, -1, 0u};
  }
  BestAcc acc;
  acc.init();
  if (kind == kArgmax) {
    auto vec = [&](const float(&x)[E::kVec], int e0) {
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
    };
    for (int st = 0; st < nst; ++st) {
      uint4 v[kStageVecs];
      take(v[0], v[1]);
      const int vi = vbeg + st * kStageVecs * kThreads + tid;
      if (kTrunc && thr) {
        mask_vec<E>(v[0], tb);
        mask_vec<E>(v[1], tb);
      }
      if (st >= nfull) {
        if (vi >= vend) v[0] = E::pad();
        if (vi + kThreads >= vend) v[1] = E::pad();
      }
      float x[E::kVec];
      E::unpack(v[0], x);
      vec(x, vi * E::kVec);
      E::unpack(v[1], x);
      vec(x, (vi + kThreads) * E::kVec);
    }
  } else if (kind == kRace) {
    float wbest = kNegInf;
    for (int st = 0; st < nst; ++st) {
      uint4 v[kStageVecs];
      take(v[0], v[1]);
      const int vi = vbeg + st * kStageVecs * kThreads + tid;
      if (kTrunc && thr) {
        mask_vec<E>(v[0], tb);
        mask_vec<E>(v[1], tb);
      }
      if (st >= nfull) {
        if (vi >= vend) v[0] = E::pad();
        if (vi + kThreads >= vend) v[1] = E::pad();
      }
      float x0[E::kVec], x1[E::kVec];
      E::unpack(v[0], x0);
      E::unpack(v[1], x1);
      race_stage<E, kShare, kTrunc>(acc, wbest, SharedBest<kShare>{s_best}, x0, x1, vi * E::kVec,
                                    (vi + kThreads) * E::kVec, c, (uint32_t)pos, rk, P.key);
    }
  } else {
    const ResidualRow rr = residual_row(c, itm.mp, itm.inv_sp, itm.mq, itm.inv_sq);
    float wbest = kNegInf;
    for (int st = 0; st < nst; ++st) {
      uint4 v[kStageVecs];
      take(v[0], v[1]);
      const int vi = vbeg + st * kThreads + tid;
      if (kTrunc) {
        if (thr) mask_vec<E>(v[0], tb);
        if (thr2) mask_vec<E>(v[1], tb2);
      }
      if (st >= nfull && vi >= vend) {
        v[0] = E::pad();
        v[1] = E::pad();
      }
      float x[E::kVec], z[E::kVec];
      E::unpack(v[0], x);
      E::unpack(v[1], z);
      residual_stage<E, kShare, kTrunc>(acc, wbest, SharedBest<kShare>{s_best}, x, z,
                                        vi * E::kVec, rr, (uint32_t)pos, rk, P.key);
    }
  }
  acc = warp_reduce(acc);
  return Partial{acc.v, 0.f, acc.idx, acc.nan};
}

// Scalar path (rows not 16-byte aligned): warp w takes vocab blocks
// vbeg + w, vbeg + w + 7, ...; lane l the ids 128 b + l + 32 j.
template <typename E, bool kTrunc>
__device__ __forceinline__ Partial seg_scalar(const Params& P, const QItem& it, float* s_xy) {
  // one logit, masked in truncated rounds
  auto ld = [&](const char* row, int v, uint32_t thr) {
    const float x = E::load1(row, v);
    return kTrunc ? mask1<E>(x, thr) : x;
  };
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const RequestKey rk{it.req_lo, it.req_hi};
  if (it.kind == kSoftmax) {
    LazySoftmax acc;
    acc.init();
    for (int b = it.vbeg + w; b < it.vend; b += kComputeWarps)
      for (int j = 0; j < 4; ++j) {
        const int v = b * kVocabBlock + lane + 32 * j;
        if (v < P.vocab) {
          const float x = ld(it.row, v, it.thr);
          if (v == it.y) *s_xy = x;
          acc.add1(x, it.c);
        }
      }
    SoftmaxAcc a = warp_reduce(acc.result());
    return Partial{a.m, a.s, -1, 0u};
  }
  BestAcc acc;
  acc.init();
  const uint32_t pos = (uint32_t)it.pos;
  for (int b = it.vbeg + w; b < it.vend; b += kComputeWarps) {
    if (it.kind == kArgmax) {
      for (int j = 0; j < 4; ++j) {
        const int v = b * kVocabBlock + lane + 32 * j;
        if (v < P.vocab) {
          const float x = ld(it.row, v, it.thr);
          acc.nan |= (x != x);
          acc.take(x, v);
        }
      }
      continue;
    }
    // race rows: lane l takes ids 128 b + 4 l .. + 3 (one Philox call)
    const int v0 = b * kVocabBlock + 4 * lane;
    float x[4], z[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      x[i] = v0 + i < P.vocab ? ld(it.row, v0 + i, it.thr) : kNegInf;
      z[i] = (it.kind == kResidual && v0 + i < P.vocab) ? ld(it.row2, v0 + i, it.thr2) : kNegInf;
    }
    if (it.kind == kRace) {
      race_vec<F32>(acc, x, v0, it.c, pos, rk, P.key);
    } else {
      const ResidualRow rr = residual_row(it.c, it.mp, it.inv_sp, it.mq, it.inv_sq);
      residual_vec<F32>(acc, x, z, v0, rr, pos, rk, P.key);
    }
  }
  acc = warp_reduce(acc);
  return Partial{acc.v, 0.f, acc.idx, acc.nan};
}

// ---------------------------------------------------------------------------
// Wave lists.
// ---------------------------------------------------------------------------
// Rows a request alive at position s has in the wave that starts there:
// positions s .. min(s + D - 1, k), two rows each below k when sampling, one
// (the bonus or greedy row) otherwise.
__device__ __forceinline__ int wave_rows(const Params& P, bool sampling, int k, int s) {
  const int last = min(s + P.depth - 1, k);
  if (!sampling) return last - s + 1;
  return 2 * (min(s + P.depth, k) - s) + (last == k ? 1 : 0);
}
// Whether the last of those rows is a bonus row (sampling, position k in the
// wave); bonus rows go to the wave's bonus list, the others to its row list.
__device__ __forceinline__ bool wave_has_bonus(const Params& P, bool sampling, int k, int s) {
  return sampling && min(s + P.depth - 1, k) == k;
}

// The j-th of those rows, as a list entry.
__device__ __forceinline__ Entry wave_entry(const Params& P, bool sampling, int r, int d0, int k,
                                            float c, RequestKey rk, int s, int j, int base,
                                            const int32_t* tokens) {
  int pos, is_draft = 0, paired = 0;
  if (!sampling) {
    pos = s + j;
  } else if (j < 2 * (min(s + P.depth, k) - s)) {
    pos = s + j / 2;
    is_draft = j & 1;
    paired = 1;
  } else {
    pos = k;
  }
  Entry en;
  en.meta = entry_meta(r, is_draft, paired, k, pos);
  en.d0 = d0;
  en.c = c;
  en.y = pos < k ? tokens[d0 + pos] : -1;
  en.req_lo = rk.lo;
  en.req_hi = rk.hi;
  en.base = base;
  en.pad = 0;
  return en;
}

// The request a decision is about.
struct ReqInfo {
  int r, d0, k, base;
  float c;
  RequestKey rk;
};

// A request accepted through the last position of this wave: its rows of the
// next wave (control warp).
__device__ void append_next_wave(const Params& P, const ReqInfo& q, int next) {
  const int lane = threadIdx.x & 31;
  const bool sampling = q.c > 0.f;
  const int n = wave_rows(P, sampling, q.k, next);
  const bool bonus = wave_has_bonus(P, sampling, q.k, next);
  const int nm = n - (bonus ? 1 : 0);
  const int w1 = P.wave + 1;
  int at = 0, bat = 0;
  if (lane == 0 && nm > 0) at = atomicAdd(P.list_cnt + w1, nm);
  if (lane == 0 && bonus) bat = atomicAdd(P.blist_cnt + w1, 1);
  at = __shfl_sync(0xffffffffu, at, 0);
  bat = __shfl_sync(0xffffffffu, bat, 0);
  Entry* list = P.lists + (size_t)w1 * P.list_cap;
  for (int j = lane; j < nm; j += 32)
    list[at + j] = wave_entry(P, sampling, q.r, q.d0, q.k, q.c, q.rk, next, j, at, P.tokens);
  if (lane == 0 && bonus)
    P.blists[(size_t)w1 * P.stride + bat] =
        wave_entry(P, sampling, q.r, q.d0, q.k, q.c, q.rk, next, nm, bat, P.tokens);
}

// ---------------------------------------------------------------------------
// Outputs of one request (the control warp).
// ---------------------------------------------------------------------------
// Accepted prefix, the extra token (-1 while the next wave still has to draw
// it), flags, and NaN debug values where no acceptance test was made: after
// position A, and everywhere for greedy requests.
__device__ void finish_request(const Params& P, int r, int d0, int k, int A, int token,
                               bool greedy) {
  const int lane = threadIdx.x & 31;
  const int width = P.max_k + 1;
  if (lane < width) {  // width <= 32
    const int v = lane < A ? P.tokens[d0 + lane] : (lane == A ? token : -1);
    P.committed[(size_t)r * width + lane] = v;
  }
  const float nan = __int_as_float(0x7fc00000);
  if (lane < k) {
    P.flags[d0 + lane] = lane < A ? 1 : 0;
    if (lane > A || greedy) {
      if (P.p_y) P.p_y[d0 + lane] = nan;
      if (P.q_y) P.q_y[d0 + lane] = nan;
      if (P.u_dbg) P.u_dbg[d0 + lane] = nan;
    }
  }
  if (lane == 0) {
    P.accepted_len[r] = A;
    if (P.req_status) P.req_status[r] = 0;
  }
}

// A request that cannot be verified (one thread): -1 outputs, flags 0, NaN
// debug values, its status bits.
__device__ void skip_request_thread(const Params& P, int r, int d0, int k, uint32_t rs) {
  const int width = P.max_k + 1;
  for (int i = 0; i < width; ++i) P.committed[(size_t)r * width + i] = -1;
  const float nan = __int_as_float(0x7fc00000);
  for (int i = 0; i < k; ++i) {
    P.flags[d0 + i] = 0;
    if (P.p_y) P.p_y[d0 + i] = nan;
    if (P.q_y) P.q_y[d0 + i] = nan;
    if (P.u_dbg) P.u_dbg[d0 + i] = nan;
  }
  P.accepted_len[r] = -1;
  if (P.req_status) P.req_status[r] = (int32_t)rs;
  atomicOr(reinterpret_cast<unsigned int*>(P.ctr + kCntStatus), rs);
}

// The same from the control warp (a row read in this wave held NaN/+inf).
__device__ void skip_request_warp(const Params& P, int r, int d0, int k, uint32_t rs) {
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
  }
}

// ---------------------------------------------------------------------------
// Merging (control warp).
// ---------------------------------------------------------------------------
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

// A whole row: softmax (a = m, b = S, xy = x[y]) or best (a = value, idx).
struct RowRes {
  float a, b, xy;
  int idx;
  bool bad;
};

__device__ __forceinline__ RowRes softmax_res(SoftmaxAcc a, float xy) {
  const bool bad = !(a.s > 0.f) || !(a.s < 3.0e38f) || !(a.m > kNegInf) || !(a.m < 3.0e38f);
  return RowRes{a.m, a.s, xy, -1, bad};
}

// argmax rows need a finite maximum; race rows carry a block index (-1: no
// block with mass), judged by the decision
__device__ __forceinline__ RowRes best_res(BestAcc a, int kind) {
  const bool bad = kind == kArgmax ? (a.nan != 0u || a.idx < 0 || !(a.v < 3.0e38f))
                                   : a.nan != 0u;
  return RowRes{a.v, 0.f, 0.f, a.idx, bad};
}

__device__ __forceinline__ RowRes single_res(const Partial& p, int kind) {
  if (kind == kSoftmax) {
    SoftmaxAcc a;
    a.m = p.a;
    a.s = p.b;
    return softmax_res(a, __int_as_float(p.idx));
  }
  BestAcc a;
  a.v = p.a;
  a.idx = p.idx;
  a.nan = p.bad;
  return best_res(a, kind);
}

// The rows of one position from their segments' partials: the target row at
// list entry et (kind tkind) and, when paired, the draft row at et + 1 -- all
// partials loaded lane-parallel in one pass.
// The nt partials of the target row are pt[0..nt), the nd of the draft row
// pd[0..nd).
__device__ void merge_rows(const Partial* pt, int nt, const Partial* pd, int nd, bool paired,
                           int tkind, RowRes& t, RowRes& d) {
  const int lane = threadIdx.x & 31;
  SoftmaxAcc st, sd;
  st.init();
  sd.init();
  BestAcc bt;
  bt.init();
  float xyt = 0.f, xyd = 0.f;
  bool ht = false, hd = false;
  for (int q = lane; q < nt + nd; q += 32) {
    const bool is_t = q < nt;
    const Partial pp = ld_cg(is_t ? pt + q : pd + (q - nt));
    if (is_t && tkind != kSoftmax) {
      BestAcc x;
      x.v = pp.a;
      x.idx = pp.idx;
      x.nan = pp.bad;
      bt = BestAcc::merge(bt, x);
    } else {
      SoftmaxAcc x;
      x.m = pp.a;
      x.s = pp.b;
      if (is_t) {
        st = SoftmaxAcc::merge(st, x);
        if (pp.bad) {
          ht = true;
          xyt = __int_as_float(pp.idx);
        }
      } else {
        sd = SoftmaxAcc::merge(sd, x);
        if (pp.bad) {
          hd = true;
          xyd = __int_as_float(pp.idx);
        }
      }
    }
  }
  const float nan = __int_as_float(0x7fc00000);
  if (tkind == kSoftmax) {
    st = warp_reduce(st);
    const unsigned hm = __ballot_sync(0xffffffffu, ht);
    const float xy = __shfl_sync(0xffffffffu, xyt, hm ? __ffs(hm) - 1 : 0);
    t = softmax_res(st, hm ? xy : nan);
  } else {
    t = best_res(warp_reduce(bt), tkind);
  }
  if (paired) {
    sd = warp_reduce(sd);
    const unsigned hm = __ballot_sync(0xffffffffu, hd);
    const float xy = __shfl_sync(0xffffffffu, xyd, hm ? __ffs(hm) - 1 : 0);
    d = softmax_res(sd, hm ? xy : nan);
  }
}

// The same for the segments of a wave's flat split: segment s of entry e
// (s counted from the entry's first CTA c) left its partial at parts[c + s + e].
__device__ void merge_position(const Params& P, const Partial* parts, const Split& sp, int et,
                               bool paired, int tkind, RowRes& t, RowRes& d) {
  const int nt = sp.segments(et, P.nb);
  const int nd = paired ? sp.segments(et + 1, P.nb) : 0;
  const int ct = sp.first_cta(et, P.nb);
  const int cd = paired ? sp.first_cta(et + 1, P.nb) : 0;
  merge_rows(parts + ct + et, nt, parts + cd + et + 1, nd, paired, tkind, t, d);
}

// ---------------------------------------------------------------------------
// Decisions (control warp).  "Speculative Decoding: Medusa, MTP, EAGLE,
// DFlash, DDTree, and DSpark", section 1: accept y_i with probability
// min(1, p_i(y_i)/q_i(y_i)), tested as u_i q_i(y_i) < p_i(y_i); at the first
// rejection draw from [p_i - q_i]_+ (queued for the next wave), after k
// acceptances draw the bonus from p_k; greedy rounds keep y_i while it equals
// the target argmax.
//
// Decides position i of request q from its merged rows and, while positions
// are accepted, hands on to the next one: inside the wave by counting the
// "accepted" signal towards that position (whoever completes its count
// decides it), past the wave by appending the request to the next wave.
// ---------------------------------------------------------------------------
// The records of a request's positions in this wave, lane j holding position
// pos0 + j (one round trip for the whole chain), and the draft token there.
struct WaveRecs {
  int4 a, b;
  int y;
};
__device__ __forceinline__ WaveRecs load_wave_recs(const Params& P, const ReqInfo& q) {
  const int lane = threadIdx.x & 31;
  const int i = P.pos0 + lane;
  WaveRecs w;
  w.a = w.b = make_int4(0, 0, 0, 0);
  w.y = -1;
  if (i < P.pos1 && i <= q.k) {
    const int4* src = reinterpret_cast<const int4*>(P.recs + (size_t)i * P.stride + q.r);
    w.a = __ldcg(src);
    w.b = __ldcg(src + 1);
    if (i < q.k) w.y = P.tokens[q.d0 + i];
  }
  return w;
}
// position pos0 + j of the loaded records (all lanes call it)
__device__ __forceinline__ void rec_of(const WaveRecs& w, int j, RowRes& t, RowRes& d, int& y) {
  int4 a, b;
  a.x = __shfl_sync(0xffffffffu, w.a.x, j);
  a.y = __shfl_sync(0xffffffffu, w.a.y, j);
  a.z = __shfl_sync(0xffffffffu, w.a.z, j);
  a.w = __shfl_sync(0xffffffffu, w.a.w, j);
  b.x = __shfl_sync(0xffffffffu, w.b.x, j);
  b.y = __shfl_sync(0xffffffffu, w.b.y, j);
  b.z = __shfl_sync(0xffffffffu, w.b.z, j);
  b.w = __shfl_sync(0xffffffffu, w.b.w, j);
  y = __shfl_sync(0xffffffffu, w.y, j);
  t = RowRes{__int_as_float(a.x), __int_as_float(a.y), __int_as_float(a.z), a.w, (b.w & 1) != 0};
  d = RowRes{__int_as_float(b.x), __int_as_float(b.y), __int_as_float(b.z), -1, (b.w & 2) != 0};
}

// Decides position i of request q from its merged rows and, while positions
// are accepted inside the wave, the ones after it from their records (every
// position of the request in this wave has been merged when this runs).
template <typename E>
__device__ void decide_chain(const Params& P, const Split& sp, const ReqInfo& q, int i, RowRes t,
                             RowRes d, int y, const WaveRecs* recs = nullptr) {
  (void)sp;
  const int lane = threadIdx.x & 31;
  const bool sampling = q.c > 0.f;
  for (;;) {
    if (!sampling) {
      if (t.bad) {
        skip_request_warp(P, q.r, q.d0, q.k, kStNonfinite);
        return;
      }
      if (!(i < q.k && y == t.idx)) {
        finish_request(P, q.r, q.d0, q.k, i, t.idx, true);
        return;
      }
    } else if (i == q.k) {
      // every draft accepted: the bonus race's winner over the whole row
      if (t.bad || t.idx < 0) {
        skip_request_warp(P, q.r, q.d0, q.k, kStNonfinite);
        return;
      }
      finish_request(P, q.r, q.d0, q.k, i, t.idx, false);
      return;
    } else {
      if (t.bad || d.bad) {
        skip_request_warp(P, q.r, q.d0, q.k, kStNonfinite);
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
        // first rejection at i: the next wave draws the correction
        finish_request(P, q.r, q.d0, q.k, i, -1, false);
        if (lane == 0) {
          const int at = atomicAdd(P.res_cnt + P.wave, 1);
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
          P.res[(size_t)P.wave * P.stride + at] = re;
        }
        return;
      }
    }
    // position i accepted (i < k)
    const int next = i + 1;
    if (next >= P.pos1) {
      append_next_wave(P, q, next);
      return;
    }
    rec_of(*recs, next - P.pos0, t, d, y);  // several positions: all merged and loaded
    if (sampling) y = -1;
    i = next;
  }
}

// Completion of a row segment: partial out; the CTA that completes the count
// of the segment's position merges the position's rows and decides it.
template <typename E>
__device__ void complete_row(const Params& P, const Split& sp, Partial* parts, const QItem& it,
                             const Partial* mb, float xy) {
  const int lane = threadIdx.x & 31;
  Partial p;
  if (it.kind == kSoftmax) {
    p = combine_softmax(mb);
    p.idx = __float_as_int(xy);
    p.bad = it.yv >= 0 ? 1u : 0u;
  } else {
    p = combine_best(mb);
  }
  const int i = it.pos;
  const int et = (it.paired && it.is_draft) ? it.e - 1 : it.e;
  const int tkind = it.paired ? kSoftmax : it.kind;
  const int target = sp.segments(et, P.nb) + (it.paired ? sp.segments(et + 1, P.nb) : 0);
  RowRes t, d{0.f, 0.f, 0.f, -1, false};
  if (target == 1) {
    t = single_res(p, tkind);
  } else {
    int last = 0;
    if (lane == 0) {
      parts[it.g] = p;
      fence_acq_rel_gpu();
      last = epoch_add(P.pos_cnt + (size_t)i * P.stride + it.r, P.epoch) == (uint32_t)target;
      if (last) fence_acq_rel_gpu();  // acquire: every writer's data is visible here
    }
    last = __shfl_sync(0xffffffffu, last, 0);
    if (!last) return;
    __syncwarp();  // ... and, past the warp barrier, to every lane
    merge_position(P, parts, sp, et, it.paired != 0, tkind, t, d);
  }
  const ReqInfo q{it.r, it.d0, it.k, it.base, it.c, RequestKey{it.req_lo, it.req_hi}};
  // positions of this request in this wave: each is merged where its last
  // segment lands, in parallel; the last one merged decides them left to right
  const int n_pos = min(P.pos1, it.k + 1) - P.pos0;
  if (n_pos <= 1) {
    decide_chain<E>(P, sp, q, i, t, d, it.y);
    return;
  }
  int last = 0;
  if (lane == 0) {
    const int4 a = make_int4(__float_as_int(t.a), __float_as_int(t.b), __float_as_int(t.xy), t.idx);
    const int4 b = make_int4(__float_as_int(d.a), __float_as_int(d.b), __float_as_int(d.xy),
                             (t.bad ? 1 : 0) | (d.bad ? 2 : 0));
    int4* dst = reinterpret_cast<int4*>(P.recs + (size_t)i * P.stride + it.r);
    dst[0] = a;
    dst[1] = b;
    fence_acq_rel_gpu();
    last = epoch_add(P.rdy + (size_t)P.wave * P.stride + it.r, P.epoch) == (uint32_t)n_pos;
    if (last) fence_acq_rel_gpu();  // acquire: every position's record is visible here
  }
  last = __shfl_sync(0xffffffffu, last, 0);
  if (!last) return;
  __syncwarp();  // ... and, past the warp barrier, to every lane
  const WaveRecs recs = load_wave_recs(P, q);
  RowRes t0, d0;
  int y0;
  rec_of(recs, 0, t0, d0, y0);
  if (it.c != 0.f) y0 = -1;
  decide_chain<E>(P, sp, q, P.pos0, t0, d0, y0, &recs);
}

// Completion of a residual segment: the CTA completing the count merges the
// race over the row's segments and commits the correction token (a residual
// without mass in fp32, i.e. p <= q everywhere, draws from p_j instead).
template <typename E>
__device__ void complete_residual(const Params& P, const Split& sp, const QItem& it,
                                  const Partial* mb) {
  const int lane = threadIdx.x & 31;
  const Partial p = combine_best(mb);
  const int n = sp.segments(it.e, P.nb);
  RowRes best;
  if (n == 1) {
    best = single_res(p, kResidual);
  } else {
    int last = 0;
    if (lane == 0) {
      P.rpart[it.g] = p;
      fence_acq_rel_gpu();
      last = epoch_add(P.rcnt + it.r, P.epoch) == (uint32_t)n;
      if (last) fence_acq_rel_gpu();  // acquire: every writer's data is visible here
    }
    last = __shfl_sync(0xffffffffu, last, 0);
    if (!last) return;
    __syncwarp();  // ... and, past the warp barrier, to every lane
    RowRes unused;
    merge_position(P, P.rpart, sp, it.e, false, kResidual, best, unused);
  }
  const int j = it.pos;
  int token = best.idx;
  if (token < 0)
    token = warp_row_race<E>(P, it.row, it.c, (uint32_t)j, RequestKey{it.req_lo, it.req_hi},
                             it.thr);
  if (lane == 0) P.committed[(size_t)it.r * (P.max_k + 1) + j] = token;
}

// ---------------------------------------------------------------------------
// Segment generation (control warp): the CTA's share of the residual phase,
// then of the row phase, cut at row boundaries and decoded lane-parallel.
// ---------------------------------------------------------------------------
// A CTA takes its share of three phases, each split flat over the grid on its
// own so that every CTA gets the same part of each kind of work: the
// correction draws (ALU-bound), the bonus rows (ALU-bound races) and the
// other rows (bound by memory).
constexpr int kPhases = 3;
struct SegGen {
  int step;                   // 0, 1, 2: phases 0, 2, 1 in turn; kPhases once done
  unsigned long long x, x1;   // next block, end of the share
  int q_head, q_used;
  __device__ __forceinline__ int phase() const { return step == 0 ? 0 : (step == 1 ? 2 : 1); }
  // the CTA's share of its current phase (empty when it has none)
  __device__ __forceinline__ void open(const Split* sp) {
    const int ph = step < kPhases ? phase() : 0;
    if (step < kPhases && (int)blockIdx.x < sp[ph].G) {
      x = sp[ph].begin(blockIdx.x);
      x1 = sp[ph].begin(blockIdx.x + 1);
    } else {
      x = x1 = 0ull;
    }
  }
};

// Queue entries are read from L2 (another CTA may have written them during
// this launch).
__device__ __forceinline__ Entry ldcg_entry(const Entry* p) {
  const int4 a = __ldcg(reinterpret_cast<const int4*>(p));
  const int4 b = __ldcg(reinterpret_cast<const int4*>(p) + 1);
  Entry e;
  e.meta = a.x;
  e.d0 = a.y;
  e.c = __int_as_float(a.z);
  e.y = a.w;
  e.req_lo = (uint32_t)b.x;
  e.req_hi = (uint32_t)b.y;
  e.base = b.z;
  e.pad = b.w;
  return e;
}
__device__ __forceinline__ ResEntry ldcg_res(const ResEntry* p) {
  const int4 a = __ldcg(reinterpret_cast<const int4*>(p));
  const int4 b = __ldcg(reinterpret_cast<const int4*>(p) + 1);
  const int4 c = __ldcg(reinterpret_cast<const int4*>(p) + 2);
  ResEntry r;
  r.r = a.x;
  r.j = a.y;
  r.d0 = a.z;
  r.pad = a.w;
  r.c = __int_as_float(b.x);
  r.mp = __int_as_float(b.y);
  r.inv_sp = __int_as_float(b.z);
  r.mq = __int_as_float(b.w);
  r.inv_sq = __int_as_float(c.x);
  r.req_lo = (uint32_t)c.y;
  r.req_hi = (uint32_t)c.z;
  r.pad2 = (uint32_t)c.w;
  return r;
}

// Entry e of a phase is res[e] (phase 0) or list[e] (phase 1: the row list,
// phase 2: the bonus list); its segment partials go to slot CTA + e0 + e.
template <typename E, bool kAligned>
__device__ void decode_segment(const Params& P, int phase, int e, int b0, int b1, QItem& it,
                               const ResEntry* res, const Entry* list, int e0) {
  const size_t row_bytes = (size_t)P.vocab * E::kBytes;
  it.e = e;
  it.g = (int)blockIdx.x + e0 + e;
  it.e0 = e0;
  it.phase = phase;
  it.mp = it.inv_sp = it.mq = it.inv_sq = 0.f;
  it.row2 = nullptr;
  it.tee = nullptr;
  it.thr = it.thr2 = 0u;
  if (phase == 0) {
    const ResEntry re = ldcg_res(res + e);
    it.r = re.r;
    it.kind = kResidual;
    it.d0 = re.d0;
    it.k = 0;
    it.y = -1;
    it.pos = re.j;
    it.base = 0;
    it.paired = 0;
    it.is_draft = 0;
    it.c = re.c;
    it.mp = re.mp;
    it.inv_sp = re.inv_sp;
    it.mq = re.mq;
    it.inv_sq = re.inv_sq;
    it.req_lo = re.req_lo;
    it.req_hi = re.req_hi;
    // the rows were streamed (and, with a tee, copied) in an earlier wave
    const char* tb = kAligned && P.tee_target ? P.tee_target : reinterpret_cast<const char*>(P.target);
    const char* db = kAligned && P.tee_target ? P.tee_draft : reinterpret_cast<const char*>(P.draft);
    it.row = tb + (size_t)(re.d0 + re.r + re.j) * row_bytes;
    it.row2 = db + (size_t)(re.d0 + re.j) * row_bytes;
    if (P.thr_t) {
      it.thr = __ldcg(P.thr_t + re.d0 + re.r + re.j);
      it.thr2 = __ldcg(P.thr_d + re.d0 + re.j);
    }
  } else {
    const Entry en = ldcg_entry(list + e);
    const int r = en.meta & 0x1fff;
    it.r = r;
    it.is_draft = (en.meta >> 13) & 1;
    it.paired = (en.meta >> 14) & 1;
    it.k = (en.meta >> 15) & 31;
    it.pos = (en.meta >> 20) & 31;
    it.d0 = en.d0;
    it.c = en.c;
    it.y = en.y;
    it.base = en.base;
    it.req_lo = en.req_lo;
    it.req_hi = en.req_hi;
    it.kind = en.c == 0.f ? kArgmax : (it.is_draft || it.pos < it.k ? kSoftmax : kRace);
    const size_t off = it.is_draft ? (size_t)(en.d0 + it.pos) * row_bytes
                                   : (size_t)(en.d0 + r + it.pos) * row_bytes;
    it.row = (it.is_draft ? reinterpret_cast<const char*>(P.draft)
                          : reinterpret_cast<const char*>(P.target)) + off;
    if (P.thr_t)
      it.thr = __ldcg(it.is_draft ? P.thr_d + en.d0 + it.pos : P.thr_t + en.d0 + r + it.pos);
    if (kAligned && P.tee_target && it.kind == kSoftmax)
      it.tee = (it.is_draft ? P.tee_draft : P.tee_target) + off;
  }
  if (kAligned) {
    constexpr int kVPB = kVocabBlock / E::kVec;
    it.vbeg = b0 * kVPB;
    it.vend = min(b1 * kVPB, P.nvec);
    const int per = it.kind == kResidual ? kThreads : kThreads * kStageVecs;
    it.nst = (it.vend - it.vbeg + per - 1) / per;
    const int vy = it.y >= 0 ? it.y / E::kVec : -1;
    it.yv = (it.kind == kSoftmax && vy >= it.vbeg && vy < it.vend) ? vy : -1;
  } else {
    it.vbeg = b0;
    it.vend = b1;
    it.nst = 0;
    const int by = it.y >= 0 ? it.y / kVocabBlock : -1;
    it.yv = (it.kind == kSoftmax && by >= b0 && by < b1) ? by : -1;
  }
}

// Keeps the queue filled: once fewer than kRefillAt segments are queued past
// the completed ones it refills up to kQueue - 2, decoding up to 8 segments at
// a time, one per lane (one round trip for the list entries of several
// completions).  kRefillAt covers what the compute warps may touch before the
// next refill: they stream at most kMailSlots - 1 segments past the completed
// ones, and their copy cursor reaches at most kStages - 1 segments (each is at
// least one stage) past the one they stream.
constexpr int kRefillAt = kMailSlots + kStages - 1;
static_assert(kRefillAt <= kQueue - 2, "the refill level fits the queue");

template <typename E, bool kAligned>
__device__ void fill_queue(const Params& P, const Split* sp, QItem* queue, int* s_qend,
                           SegGen& sg) {
  const int lane = threadIdx.x & 31;
  if (sg.step < kPhases && sg.q_head >= sg.q_used + kRefillAt) return;
  while (sg.step < kPhases && sg.q_head < sg.q_used + kQueue - 2) {
    const int room = min(8, kQueue - 2 - (sg.q_head - sg.q_used));
    // cut the next `room` segments (all lanes alike); lane j keeps the j-th
    int n = 0, my_phase = 0, my_e = 0, my_b0 = 0, my_b1 = 0;
    while (n < room && sg.step < kPhases) {
      if (sg.x >= sg.x1) {
        // next phase: the share of this CTA in it
        ++sg.step;
        sg.open(sp);
        continue;
      }
      const int e = (int)(sg.x / (unsigned long long)P.nb);
      const unsigned long long row0 = (unsigned long long)e * P.nb;
      const int b0 = (int)(sg.x - row0);
      const unsigned long long end = sg.x1 < row0 + P.nb ? sg.x1 : row0 + P.nb;
      const int b1 = (int)(end - row0);
      if (lane == n) {
        my_phase = sg.phase();
        my_e = e;
        my_b0 = b0;
        my_b1 = b1;
      }
      sg.x = end;
      ++n;
    }
    QItem it;
    if (lane < n)
      decode_segment<E, kAligned>(P, my_phase, my_e, my_b0, my_b1, it,
                                  P.res + (P.wave > 0 ? (size_t)(P.wave - 1) * P.stride : 0),
                                  my_phase == 2 ? P.blists + (size_t)P.wave * P.stride
                                                : P.lists + (size_t)P.wave * P.list_cap,
                                  0);
    if (lane < n) queue[(sg.q_head + lane) & (kQueue - 1)] = it;
    sg.q_head += n;
  }
  __syncwarp();
  if (lane == 0) {
    // queue entries before the count that publishes them
    st_release_shared(s_qend, sg.step >= kPhases ? -1 - sg.q_head : sg.q_head);
  }
  __syncwarp();
}

__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ---------------------------------------------------------------------------
// Confidence-based window trimming ("Speculative Decoding: Medusa, MTP,
// EAGLE, DFlash, DDTree, and DSpark", section 5, DSpark): with conditional
// confidences c_i the estimated probability of accepting through position j
// is s_j = prod_{i<=j} c_i and verifying a prefix of length k has estimated
// progress 1 + sum_{j<=k} s_j.  The window kept is the k in [0, K] that
// maximises 1 + sum_{j<=k} s_j - cost * k, the shortest on ties, evaluated in
// fp64 without contraction.  -1 when a confidence is NaN or outside [0, 1],
// or the cost is NaN.
// ---------------------------------------------------------------------------
__device__ int trim_window(const Params& P, int r, int d0, int K) {
  const double lam = (double)P.cost[r];
  bool bad = lam != lam;
  for (int i = 0; i < K; ++i) {
    const double c = (double)P.confidence[d0 + i];
    if (!(c >= 0.0 && c <= 1.0)) bad = true;
  }
  if (bad) return -1;
  double best = 1.0, s = 1.0, value = 1.0;
  int best_k = 0;
  for (int j = 1; j <= K; ++j) {
    s = __dmul_rn(s, (double)P.confidence[d0 + j - 1]);
    value = __dadd_rn(value, __dsub_rn(s, lam));
    if (value > best) {
      best = value;
      best_k = j;
    }
  }
  return best_k;
}

// ---------------------------------------------------------------------------
// The plan launch (one CTA): draft offsets, the layout and input checks, the
// outputs of requests that cannot be verified, and the rows of wave 0.  In a
// trimmed run num_draft is the window layout K_r and each request verifies
// its trimmed window k_r <= K_r in place (rows past k_r are never read).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kPlanThreads) sv_plan(Params P) {
  __shared__ int s_w[kPlanThreads / 32 + 1];
  __shared__ uint32_t s_layout;
  __shared__ int s_doff[kMaxBatch + 1];
  __shared__ int32_t s_tok[kPlanTokens];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int kW = kPlanThreads / 32;
  constexpr int kPer = kMaxBatch / kPlanThreads;  // requests a thread takes

  pdl_launch_dependents();  // wave 0 may be scheduled; it waits for this grid
  // The small inputs in one round trip: every thread's num_draft and
  // temperature, and the draft tokens (total_draft of them, valid memory
  // whatever num_draft holds) into shared memory when they fit; the checks
  // and the list entries then read them there.
  const bool tok_shared = P.total_draft <= kPlanTokens;
  for (int i = tid; tok_shared && i < P.total_draft; i += kPlanThreads) s_tok[i] = P.tokens[i];
  const int32_t* tokens = tok_shared ? s_tok : P.tokens;
  int k_in[kPer];
  float t_in[kPer];
#pragma unroll
  for (int b = 0; b < kPer; ++b) {
    const int r = b * kPlanThreads + tid;
    k_in[b] = r < P.batch ? P.num_draft[r] : 0;
    t_in[b] = r < P.batch ? P.temperature[r] : 0.f;
  }
  if (tid == 0) {
    s_layout = 0u;
    P.ctr[kCntStatus] = 0;
    P.ctr[kCntLive] = 0;
  }
  for (int i = tid; i < P.n_waves; i += kPlanThreads) {
    P.list_cnt[i] = 0;
    P.blist_cnt[i] = 0;
    P.res_cnt[i] = 0;
  }
  __syncthreads();

  // block-wide exclusive scan of v (all threads call it); *total gets the sum
  auto scan = [&](int v, int* total) {
    int incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += o;
    }
    if (lane == 31) s_w[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      const int w = s_w[lane];
      int wi = w;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, wi, off);
        if (lane >= off) wi += o;
      }
      s_w[lane] = wi - w;
      if (lane == 31) s_w[kW] = wi;
    }
    __syncthreads();
    const int excl = s_w[warp] + incl - v;
    *total = s_w[kW];
    __syncthreads();
    return excl;
  };

  // draft-row offsets, and the checks that make the layout trustworthy
  int carry = 0;
#pragma unroll
  for (int b = 0; b < kPer; ++b) {
    const int base = b * kPlanThreads;
    if (base >= P.batch) break;
    const int r = base + tid;
    const int k = k_in[b];
    const bool badk = k < 0 || k > P.max_k;
    if (badk) atomicOr(&s_layout, kStBadK);
    const int kk = badk ? 0 : k;
    int tot;
    const int ex = scan(kk, &tot);
    if (r < P.batch) s_doff[r] = carry + ex;
    carry += tot;
  }
  if (tid == 0) {
    s_doff[P.batch] = carry;
    if (!s_layout && carry != P.total_draft) s_layout = kStBadTotal;
  }
  __syncthreads();
  const uint32_t layout = s_layout;
  if (layout) {
    // nothing is verified
    const int width = P.max_k + 1;
    for (int i = tid; i < P.batch * width; i += kPlanThreads) P.committed[i] = -1;
    for (int r = tid; r < P.batch; r += kPlanThreads) {
      P.accepted_len[r] = -1;
      if (P.req_status) P.req_status[r] = (int32_t)layout;
    }
    const float nan = __int_as_float(0x7fc00000);
    for (int d = tid; d < P.total_draft; d += kPlanThreads) {
      P.flags[d] = 0;
      if (P.p_y) P.p_y[d] = nan;
      if (P.q_y) P.q_y[d] = nan;
      if (P.u_dbg) P.u_dbg[d] = nan;
    }
    if (tid == 0) P.ctr[kCntStatus] = (int)layout;
    return;
  }

  // per request: the input checks, then its rows of wave 0 (the bonus row, if
  // the wave reaches position k, in the bonus list)
  int written = 0, bwritten = 0, live = 0;
#pragma unroll
  for (int b = 0; b < kPer; ++b) {
    const int base = b * kPlanThreads;
    if (base >= P.batch) break;
    const int r = base + tid;
    int n = 0, d0 = 0, k = 0;
    float c = 0.f;
    bool sampling = false, bonus = false;
    if (r < P.batch) {
      d0 = s_doff[r];
      const int K = s_doff[r + 1] - d0;  // the window's layout
      k = K;
      uint32_t rs = 0u;
      if (P.trimmed) {
        k = trim_window(P, r, d0, K);
        if (P.verified_k) P.verified_k[r] = k;
        if (k < 0) {
          rs = kStBadConf;
        } else {
          // positions past the trimmed window: never verified
          const float nan = __int_as_float(0x7fc00000);
          for (int i = k; i < K; ++i) {
            P.flags[d0 + i] = 0;
            if (P.p_y) P.p_y[d0 + i] = nan;
            if (P.q_y) P.q_y[d0 + i] = nan;
            if (P.u_dbg) P.u_dbg[d0 + i] = nan;
          }
        }
      }
      const float t = t_in[b];
      const int mode = req_mode(t);
      if (!rs) {
        if (mode == kBadTemp) rs |= kStBadTemp;
        for (int i = 0; i < k; ++i) {
          const int y = tokens[d0 + i];
          if (y < 0 || y >= P.vocab) rs |= kStBadToken;
        }
        if (!rs && mode == kSampling && k > 0 && P.draft == nullptr) rs |= kStNoDraft;
      }
      if (rs) {
        skip_request_thread(P, r, d0, K, rs);
      } else {
        sampling = mode == kSampling;
        c = sampling ? kLog2e / t : 0.f;
        n = wave_rows(P, sampling, k, 0);
        bonus = wave_has_bonus(P, sampling, k, 0);
      }
    }
    const int nm = n - (bonus ? 1 : 0);
    int tot, btot;
    const int at = written + scan(nm, &tot);
    const int bat = bwritten + scan(bonus ? 1 : 0, &btot);
    if (n > 0) {
      const RequestKey rk = request_key(P, r);
      for (int j = 0; j < nm; ++j)
        P.lists[at + j] = wave_entry(P, sampling, r, d0, k, c, rk, 0, j, at, tokens);
      if (bonus) P.blists[bat] = wave_entry(P, sampling, r, d0, k, c, rk, 0, nm, bat, tokens);
    }
    written += tot;
    bwritten += btot;
    live += __syncthreads_count(n > 0);
  }
  if (tid == 0) {
    P.list_cnt[0] = written;
    P.blist_cnt[0] = bwritten;
    P.ctr[kCntLive] = live;
  }
}

// ---------------------------------------------------------------------------
// The wave launch: positions [pos0, pos1) of every request alive at pos0, and
// the correction draws of the requests the previous wave rejected.
// ---------------------------------------------------------------------------
// kMinBlocks CTAs per SM bound the registers: 2 (up to 128 a thread) for
// windows that stream long shares, 3 (up to 80) for small, latency-bound ones.
// kShare: the race's best shared by the warps of a segment (see SharedBest).
// kTrunc: the build for truncated rounds (Params::thr_t set), which masks
// every row it loads with the row's threshold.
template <typename E, bool kAligned, int kMinBlocks, bool kShare = true, bool kTrunc = false>
__global__ void __launch_bounds__(kBlock, kMinBlocks) sv_wave(Params P) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  uint4* ring = reinterpret_cast<uint4*>(smem_raw);
  __shared__ QItem queue[kQueue];
  __shared__ Partial mailbox[kMailSlots][kComputeWarps];
  __shared__ float s_xy[kMailSlots];
  __shared__ uint32_t s_best[kMailSlots];  // race best of the slot's segment (order key)
  __shared__ int s_qend;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const bool control = warp == kComputeWarps;

  pdl_launch_dependents();  // the next wave may be scheduled as CTAs of this one exit
  pdl_wait();               // the previous launch's lists are complete

  const int n_rows = P.list_cnt[P.wave];
  const int n_bonus = P.blist_cnt[P.wave];
  const int n_res = P.wave > 0 ? P.res_cnt[P.wave - 1] : 0;
  Split sp[kPhases];
  sp[0].init(n_res, P.nb, P.min_span_res, gridDim.x);
  sp[1].init(n_rows, P.nb, P.min_span, gridDim.x);
  // a race costs about four times a softmax per byte: shares of a quarter
  sp[2].init(n_bonus, P.nb, max(1, P.min_span / 4), gridDim.x);
  const int c = blockIdx.x;
  if (c >= sp[0].G && c >= sp[1].G && c >= sp[2].G) return;  // no share in this wave

  SegGen sg;
  sg.step = 0;
  sg.q_head = sg.q_used = 0;
  sg.open(sp);
  if (control) fill_queue<E, kAligned>(P, sp, queue, &s_qend, sg);
  if (tid < kMailSlots) s_best[tid] = kOrderKeyNegInf;
  __syncthreads();

  // Segment u travels through mailbox slot u % kMailSlots.  The compute warps
  // arrive on kBarReady + slot when its partials are in; the control warp
  // syncs there, completes the segment, refills the queue and then arrives on
  // kBarFree + slot.  A compute warp syncs on kBarFree + (u % kMailSlots)
  // before every index u >= kMailSlots, including the index equal to the
  // final count, where it then stops; so the control warp arrives after
  // completing u exactly when u + kMailSlots <= the count.  It knows: its
  // refill leaves the queue either final or at least kRefillAt > kMailSlots
  // entries past u.  For the same reason a compute warp past that barrier
  // (or, below kMailSlots, past the initial fill) reads a published count
  // that is final or larger than its index.  The compute warps thus run up to
  // kMailSlots segments ahead of the control warp's completions (merges,
  // decisions) and do not wait for them while those are shorter than the
  // streaming.
  if (!control) {
    // ---- compute warps: stream segment after segment ---------------------------
    auto segments = [&](auto&& seg) {
      for (int u = 0;; ++u) {
        const int slot = u % kMailSlots;
        if (u >= kMailSlots) named_bar_sync(kBarFree + slot, kCtaThreads);
        const int qe = ld_acquire_shared(&s_qend);
        if (u >= (qe >= 0 ? qe : -1 - qe)) break;  // only once the count is final
        const QItem& it = queue[u & (kQueue - 1)];
        const Partial out = seg(it, slot);
        if ((tid & 31) == 0) mailbox[slot][warp] = out;
        named_bar_arrive(kBarReady + slot, kCtaThreads);
      }
    };
    if (!kAligned) {
      segments(
          [&](const QItem& it, int slot) { return seg_scalar<E, kTrunc>(P, it, &s_xy[slot]); });
    } else {
      int gs = 0;
      LoadCursor lc;
      lc.q = 0;
      lc.active = false;
      lc.open(queue, &s_qend);
      for (int s = 0; s < kStages - 1; ++s) lc.issue(queue, &s_qend, ring, s);
      auto take = [&](uint4& v0, uint4& v1) { ring_take(queue, &s_qend, ring, lc, gs, v0, v1); };
      segments([&](const QItem& it, int slot) {
        return seg_reduce<E, kShare, kTrunc>(P, it, &s_xy[slot], &s_best[slot], take);
      });
      cp_async_wait_all();
    }
  } else {
    // ---- control warp: complete segment after segment, keep the queue full ----
    for (int u = 0; u < sg.q_head; ++u) {
      const int slot = u % kMailSlots;
      named_bar_sync(kBarReady + slot, kCtaThreads);
      const QItem& pv = queue[u & (kQueue - 1)];
      if (pv.phase == 0) {
        complete_residual<E>(P, sp[0], pv, mailbox[slot]);
      } else {
        complete_row<E>(P, sp[pv.phase], pv.phase == 2 ? P.bpart : P.part, pv, mailbox[slot],
                        s_xy[slot]);
      }
      sg.q_used = u + 1;  // its queue entry may now be reused
      fill_queue<E, kAligned>(P, sp, queue, &s_qend, sg);
      if ((tid & 31) == 0) s_best[slot] = kOrderKeyNegInf;  // for segment u + kMailSlots
      if (u + kMailSlots <= sg.q_head) named_bar_arrive(kBarFree + slot, kCtaThreads);
    }
  }
}

}  // namespace sv
