// sv_kernels.cuh -- the three kernels of one verify round.
//
//   sv_plan     (1 CTA)  prefix sums of num_draft -> per-request offsets and the
//                        list of logit rows the round must read; validation;
//                        outputs pre-filled as "skipped".
//   sv_rowpass  (persistent, one CTA per (row, vocab chunk) item at a time)
//                        streams every needed logit row once.  Sampling target
//                        rows i<k and draft rows: softmax normaliser (m, S).
//                        Greedy target rows: argmax.  The last target row of a
//                        sampling request: the bonus race.  The CTA finishing a
//                        row merges its chunk partials; the CTA finishing a
//                        request runs the left-to-right acceptance scan, writes
//                        the outputs and, on a rejection, queues the residual.
//   sv_residual (persistent) the correction draw from [p_j - q_j]_+ for each
//                        queued request, split over vocab chunks; the CTA
//                        finishing a request writes its committed token.
//
// No CTA ever waits for another: hand-offs use "last arriver" atomic counters.
#pragma once

#include "sv_device.cuh"

namespace sv {

constexpr int kThreads = 256;   // row-pass / residual CTA size
constexpr int kUnroll = 4;      // 16-byte loads in flight per thread
constexpr int kPlanThreads = 1024;

enum RowKind : int { kSoftmax = 0, kArgmax = 1, kRace = 2 };
enum ReqMode : int { kSkipped = 0, kGreedy = 1, kSampling = 2 };

// Status bits (kept equal to the SPECVERIFY_STATUS_* values of the header).
constexpr uint32_t kStBadToken = 1u, kStBadK = 2u, kStBadTemp = 4u, kStNonfinite = 8u,
                   kStBadTotal = 16u, kStNoDraft = 64u;

struct __align__(16) ReqInfo {
  int tgt_off;     // first target row
  int drf_off;     // first draft row / token
  int k;           // draft positions
  int row0;        // first entry in the row list
  int nrows;       // entries in the row list (2k+1 sampling, k+1 greedy, 0 skipped)
  int mode;        // ReqMode
  float c;         // log2(e) / T (sampling only)
  uint32_t req_lo, req_hi;  // Philox request word
  int pad[3];
};

struct __align__(16) RowInfo {
  int req;        // request index in the batch
  int logit_row;  // row of target_logits (or draft_logits when is_draft)
  int pos;        // draft position i
  int kind_draft; // kind | (is_draft << 8)
};

struct __align__(16) Partial {  // per (row, chunk), and merged per row
  float a;      // softmax: m   | best: value
  float b;      // softmax: S   | unused
  int idx;      // best: index  | unused
  uint32_t bad; // NaN seen (best rows)
};

struct __align__(16) Partial2 {  // residual race and its fallback
  float va;
  int ia;
  float vb;
  int ib;
};

enum Counter : int { kCntRows = 0, kCntResid = 1, kCntStatus = 2, kCntCount = 4 };

// L2-coherent loads of records other CTAs of this grid wrote (bypass L1).
__device__ __forceinline__ Partial ld_cg(const Partial* p) {
  const int4 v = __ldcg(reinterpret_cast<const int4*>(p));
  return Partial{__int_as_float(v.x), __int_as_float(v.y), v.z, (uint32_t)v.w};
}
__device__ __forceinline__ Partial2 ld_cg(const Partial2* p) {
  const int4 v = __ldcg(reinterpret_cast<const int4*>(p));
  return Partial2{__int_as_float(v.x), v.y, __int_as_float(v.z), v.w};
}
__device__ __forceinline__ int2 ld_cg(const int2* p) { return __ldcg(p); }

struct Params {
  // inputs
  const void* target;
  const void* draft;
  const int32_t* tokens;
  const int32_t* num_draft;
  const float* temperature;
  const int64_t* request_ids;
  PhiloxKey key;
  int batch, total_draft, max_k, vocab, nch;
  // outputs
  int32_t* accepted_len;
  int32_t* committed;
  uint8_t* flags;
  float* p_y;
  float* q_y;
  float* u_dbg;
  int32_t* req_status;
  // scratch
  ReqInfo* req;
  RowInfo* rows;
  Partial* part;
  Partial* rowres;
  int* row_cnt;
  int* req_cnt;
  int2* res_list;
  Partial2* part2;
  int* res_cnt;
  int* counters;
};

// ---------------------------------------------------------------------------
// Block-wide exclusive scan of one int per thread (kPlanThreads threads).
// ---------------------------------------------------------------------------
__device__ __forceinline__ int plan_exclusive_scan(int v, int* smem, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += o;
  }
  if (lane == 31) smem[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = smem[lane];
    int wi = w;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, wi, off);
      if (lane >= off) wi += o;
    }
    smem[lane] = wi - w;   // exclusive prefix of warp totals
    if (lane == 31) smem[32] = wi;
  }
  __syncthreads();
  const int res = smem[warp] + incl - v;
  *total = smem[32];
  __syncthreads();
  return res;
}

__device__ __forceinline__ bool temperature_ok(float t) {
  // 0 (greedy) or a normal, finite positive value
  return t == 0.f || (t >= 1.17549435e-38f && t <= 3.40282347e+38f);
}

__device__ __forceinline__ void prefill_request(const Params& P, int r, int d_off, int k,
                                                uint32_t rs) {
  const int width = P.max_k + 1;
  for (int i = 0; i < width; ++i) P.committed[(size_t)r * width + i] = -1;
  P.accepted_len[r] = -1;
  for (int i = 0; i < k; ++i) {
    P.flags[d_off + i] = 0;
    const float nan = __int_as_float(0x7fc00000);
    if (P.p_y) P.p_y[d_off + i] = nan;
    if (P.q_y) P.q_y[d_off + i] = nan;
    if (P.u_dbg) P.u_dbg[d_off + i] = nan;
  }
  if (P.req_status) P.req_status[r] = (int32_t)rs;
}

// ---------------------------------------------------------------------------
// K0: plan.  One CTA of kPlanThreads threads.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kPlanThreads) sv_plan(Params P) {
  __shared__ int smem[40];
  __shared__ uint32_t s_status;
  __shared__ long long s_sum;
  __shared__ int s_badk;
  const int tid = threadIdx.x;
  if (tid == 0) {
    s_status = 0u;
    s_sum = 0;
    s_badk = 0;
  }
  __syncthreads();

  // Pass 1: is the layout trustworthy?  Every k_r in range and sum == total_draft.
  long long sum = 0;
  int badk = 0;
  for (int r = tid; r < P.batch; r += kPlanThreads) {
    const int k = P.num_draft[r];
    if (k < 0 || k > P.max_k) badk = 1;
    sum += k;
  }
  if (badk) atomicOr(&s_badk, 1);
  atomicAdd(reinterpret_cast<unsigned long long*>(&s_sum), (unsigned long long)sum);
  __syncthreads();
  uint32_t gstatus = 0u;
  if (s_badk) gstatus = kStBadK;
  else if (s_sum != (long long)P.total_draft) gstatus = kStBadTotal;
  if (gstatus) {
    const int width = P.max_k + 1;
    for (int r = tid; r < P.batch; r += kPlanThreads) {
      for (int i = 0; i < width; ++i) P.committed[(size_t)r * width + i] = -1;
      P.accepted_len[r] = -1;
      if (P.req_status) P.req_status[r] = (int32_t)gstatus;
    }
    const float nan = __int_as_float(0x7fc00000);
    for (int d = tid; d < P.total_draft; d += kPlanThreads) {
      P.flags[d] = 0;
      if (P.p_y) P.p_y[d] = nan;
      if (P.q_y) P.q_y[d] = nan;
      if (P.u_dbg) P.u_dbg[d] = nan;
    }
    if (tid == 0) {
      P.counters[kCntRows] = 0;
      P.counters[kCntResid] = 0;
      P.counters[kCntStatus] = (int)gstatus;
    }
    return;
  }

  // Pass 2: offsets, modes and the row list, one tile of requests at a time.
  int carry_t = 0, carry_d = 0, carry_rows = 0;
  uint32_t status = 0u;
  for (int base = 0; base < P.batch; base += kPlanThreads) {
    const int r = base + tid;
    const bool active = r < P.batch;
    const int k = active ? P.num_draft[r] : 0;
    int tot;
    const int t_off = carry_t + plan_exclusive_scan(active ? k + 1 : 0, smem, &tot);
    carry_t += tot;
    const int d_off = carry_d + plan_exclusive_scan(k, smem, &tot);
    carry_d += tot;

    uint32_t rs = 0u;
    int mode = kSkipped;
    float c = 0.f;
    if (active) {
      const float t = P.temperature[r];
      if (!temperature_ok(t)) rs |= kStBadTemp;
      for (int i = 0; i < k; ++i) {
        const int y = P.tokens[d_off + i];
        if (y < 0 || y >= P.vocab) rs |= kStBadToken;
      }
      if (!rs && t > 0.f && k > 0 && P.draft == nullptr) rs |= kStNoDraft;
      if (!rs) {
        mode = (t == 0.f) ? kGreedy : kSampling;
        c = (t == 0.f) ? 0.f : kLog2e / t;
      }
    }
    const int nrows = mode == kSampling ? 2 * k + 1 : (mode == kGreedy ? k + 1 : 0);
    const int row0 = carry_rows + plan_exclusive_scan(nrows, smem, &tot);
    carry_rows += tot;

    if (active) {
      status |= rs;
      const uint64_t rid = P.request_ids ? (uint64_t)P.request_ids[r] : (uint64_t)r;
      ReqInfo q;
      q.tgt_off = t_off;
      q.drf_off = d_off;
      q.k = k;
      q.row0 = row0;
      q.nrows = nrows;
      q.mode = mode;
      q.c = c;
      q.req_lo = (uint32_t)rid;
      q.req_hi = (uint32_t)(rid >> 32);
      q.pad[0] = q.pad[1] = q.pad[2] = 0;
      P.req[r] = q;
      if (mode == kSampling) {
        // interleaved t_0 d_0 t_1 d_1 ... t_k: the residual pair (t_j, d_j) is
        // read close together in time
        for (int i = 0; i < k; ++i) {
          P.rows[row0 + 2 * i] = RowInfo{r, t_off + i, i, kSoftmax};
          P.rows[row0 + 2 * i + 1] = RowInfo{r, d_off + i, i, kSoftmax | (1 << 8)};
        }
        P.rows[row0 + 2 * k] = RowInfo{r, t_off + k, k, kRace};
      } else if (mode == kGreedy) {
        for (int i = 0; i <= k; ++i) P.rows[row0 + i] = RowInfo{r, t_off + i, i, kArgmax};
      }
      prefill_request(P, r, d_off, k, rs);
      P.req_cnt[r] = 0;
      P.res_cnt[r] = 0;
    }
  }
  if (status) atomicOr(&s_status, status);
  __syncthreads();
  for (int n = tid; n < carry_rows; n += kPlanThreads) P.row_cnt[n] = 0;
  if (tid == 0) {
    P.counters[kCntRows] = carry_rows;
    P.counters[kCntResid] = 0;
    P.counters[kCntStatus] = (int)s_status;
  }
}

// ---------------------------------------------------------------------------
// Chunk geometry of a row: `head` scalar elements up to the first 16-byte
// boundary, `nvec` aligned vectors, `tail` scalar elements.  Chunk ch owns
// vectors [vbeg, vend); chunk 0 also owns the head, the last chunk the tail.
// ---------------------------------------------------------------------------
template <typename E>
struct ChunkGeom {
  int head, nvec, tail, vbeg, vend;
  __device__ __forceinline__ void init(const void* row, int vocab, int ch, int nch) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(row);
    int h = (int)(((16u - (uint32_t)(a & 15u)) & 15u) / E::kBytes);
    if (h > vocab) h = vocab;
    head = h;
    nvec = (vocab - h) / E::kVec;
    tail = vocab - h - nvec * E::kVec;
    vbeg = (int)(((long long)ch * nvec) / nch);
    vend = (int)(((long long)(ch + 1) * nvec) / nch);
  }
};

// Streams the vectors of one chunk through `f(x[kVec], first_element_index)`,
// kUnroll 16-byte loads in flight per thread, indices increasing per thread.
template <typename E, typename F>
__device__ __forceinline__ void stream_chunk(const void* row, const ChunkGeom<E>& g, F&& f) {
  const uint4* vp = reinterpret_cast<const uint4*>(reinterpret_cast<const char*>(row) +
                                                   (size_t)g.head * E::kBytes);
  for (int v0 = g.vbeg + threadIdx.x; v0 < g.vend; v0 += kThreads * kUnroll) {
    uint4 d[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int vi = v0 + u * kThreads;
      d[u] = vi < g.vend ? ld_stream(vp + vi) : E::pad();
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      float x[E::kVec];
      E::unpack(d[u], x);
      f(x, g.head + (v0 + u * kThreads) * E::kVec);
    }
  }
}

// Philox words for elements e0 .. e0+N-1 where e0 % 4 == OFF.
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

// --- per-kind chunk reductions ----------------------------------------------

template <typename E>
__device__ __forceinline__ SoftmaxAcc chunk_softmax(const void* row, const ChunkGeom<E>& g,
                                                    int ch, int nch, float c) {
  SoftmaxAcc acc;
  acc.init();
  if (ch == 0 && (int)threadIdx.x < g.head) acc.add1(E::load1(row, threadIdx.x), c);
  stream_chunk<E>(row, g, [&](const float(&x)[E::kVec], int) { acc.add(x, c); });
  if (ch == nch - 1 && (int)threadIdx.x < g.tail)
    acc.add1(E::load1(row, g.head + g.nvec * E::kVec + threadIdx.x), c);
  return acc;
}

template <typename E>
__device__ __forceinline__ BestAcc chunk_argmax(const void* row, const ChunkGeom<E>& g, int ch,
                                                int nch) {
  BestAcc acc;
  acc.init();
  auto one = [&](float x, int e) {
    acc.nan |= (x != x);
    acc.take(x, e);
  };
  if (ch == 0 && (int)threadIdx.x < g.head) one(E::load1(row, threadIdx.x), threadIdx.x);
  stream_chunk<E>(row, g, [&](const float(&x)[E::kVec], int e0) {
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
  if (ch == nch - 1 && (int)threadIdx.x < g.tail) {
    const int e = g.head + g.nvec * E::kVec + threadIdx.x;
    one(E::load1(row, e), e);
  }
  return acc;
}

// Bonus race: argmax_v c*x_v - log2(E_v)  (== argmin_v E_v / p_v).
template <typename E, int OFF>
__device__ __forceinline__ BestAcc chunk_race(const void* row, const ChunkGeom<E>& g, int ch,
                                              int nch, float c, uint32_t pos, uint32_t req_lo,
                                              uint32_t req_hi, PhiloxKey key) {
  BestAcc acc;
  acc.init();
  auto one = [&](float x, int e, uint32_t w) {
    const float s = fmaf(x, c, -fast_lg2(race_exponential(w)));
    acc.nan |= (s != s);
    acc.take(s, e);
  };
  if (ch == 0 && (int)threadIdx.x < g.head) {
    const int e = threadIdx.x;
    one(E::load1(row, e), e, race_word1(e, pos, req_lo, req_hi, key));
  }
  stream_chunk<E>(row, g, [&](const float(&x)[E::kVec], int e0) {
    RaceWords<E::kVec, OFF> rw;
    rw.make(e0, pos, req_lo, req_hi, key);
#pragma unroll
    for (int e = 0; e < E::kVec; ++e) one(x[e], e0 + e, rw.word(e));
  });
  if (ch == nch - 1 && (int)threadIdx.x < g.tail) {
    const int e = g.head + g.nvec * E::kVec + threadIdx.x;
    one(E::load1(row, e), e, race_word1(e, pos, req_lo, req_hi, key));
  }
  return acc;
}

// ---------------------------------------------------------------------------
// The acceptance scan of one request, run by one warp once all its rows are
// merged ("Speculative Decoding: Medusa, MTP, EAGLE, DFlash, DDTree, and
// DSpark", section 1: accept y_i with probability min(1, p_i(y_i)/q_i(y_i)),
// left to right, stop at the first rejection).  Lane i handles position i.
// ---------------------------------------------------------------------------
template <typename E>
__device__ void scan_request(const Params& P, int r) {
  const int lane = threadIdx.x & 31;
  const ReqInfo q = P.req[r];
  const int k = q.k;
  const int width = P.max_k + 1;
  uint32_t bad = 0u;
  bool accept = true;
  int y = -1, tok = -1;

  if (q.mode == kGreedy) {
    if (lane <= k) {
      const Partial rr = ld_cg(P.rowres + q.row0 + lane);
      bad = rr.bad;
      tok = rr.idx;  // argmax of target row `lane`
      if (lane < k) {
        y = P.tokens[q.drf_off + lane];
        accept = (y == tok);
      }
    }
  } else {
    if (lane < k) {
      const Partial rt = ld_cg(P.rowres + q.row0 + 2 * lane);
      const Partial rd = ld_cg(P.rowres + q.row0 + 2 * lane + 1);
      bad = rt.bad | rd.bad;
      y = P.tokens[q.drf_off + lane];
      const void* trow = reinterpret_cast<const char*>(P.target) +
                         (size_t)(q.tgt_off + lane) * P.vocab * E::kBytes;
      const void* drow = reinterpret_cast<const char*>(P.draft) +
                         (size_t)(q.drf_off + lane) * P.vocab * E::kBytes;
      const float tp = fmaf(E::load1(trow, y), q.c, -rt.a);   // log2 of p(y) * S_p
      const float tq = fmaf(E::load1(drow, y), q.c, -rd.a);   // log2 of q(y) * S_q
      const float u = accept_uniform(P.key, (uint32_t)lane, q.req_lo, q.req_hi);
      // u * q(y) < p(y), scaled by S_p * S_q * 2^-max(tp, tq) > 0
      if (tp == kNegInf) {
        accept = false;
      } else if (tq == kNegInf) {
        accept = true;
      } else {
        const float mx = fmaxf(tp, tq);
        accept = u * (fast_ex2(tq - mx) * rt.b) < fast_ex2(tp - mx) * rd.b;
      }
      if (P.p_y) P.p_y[q.drf_off + lane] = fast_ex2(tp) / rt.b;
      if (P.q_y) P.q_y[q.drf_off + lane] = fast_ex2(tq) / rd.b;
      if (P.u_dbg) P.u_dbg[q.drf_off + lane] = u;
    } else if (lane == k) {
      const Partial rr = ld_cg(P.rowres + q.row0 + 2 * k);
      bad = rr.bad;
      tok = rr.idx;  // bonus race winner
    }
  }
  if (__any_sync(0xffffffffu, bad != 0u)) {
    if (lane == 0) {
      atomicOr(reinterpret_cast<unsigned int*>(P.counters + kCntStatus), kStNonfinite);
      if (P.req_status) P.req_status[r] = (int32_t)kStNonfinite;
    }
    return;
  }
  const uint32_t rej = __ballot_sync(0xffffffffu, lane < k && !accept);
  const int A = rej ? __ffs(rej) - 1 : k;
  if (lane < A) {
    P.committed[(size_t)r * width + lane] = y;
    P.flags[q.drf_off + lane] = 1;
  }
  const int tok_at_A = __shfl_sync(0xffffffffu, tok, A);
  if (lane == 0) {
    P.accepted_len[r] = A;
    if (q.mode == kGreedy || A == k) {
      P.committed[(size_t)r * width + A] = tok_at_A;
    } else {
      const int slot = atomicAdd(P.counters + kCntResid, 1);
      P.res_list[slot] = make_int2(r, A);
    }
  }
}

// ---------------------------------------------------------------------------
// K1: persistent row pass.
// ---------------------------------------------------------------------------
template <typename E>
__global__ void __launch_bounds__(kThreads) sv_rowpass(Params P) {
  __shared__ SoftmaxAcc s_red_sm[kThreads / 32];
  __shared__ BestAcc s_red_b[kThreads / 32];
  __shared__ int s_flag;
  const int n_items = P.counters[kCntRows] * P.nch;

  for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
    const int n = item / P.nch;
    const int ch = item - n * P.nch;
    const RowInfo ri = P.rows[n];
    const ReqInfo q = P.req[ri.req];
    const int kind = ri.kind_draft & 0xff;
    const void* base = (ri.kind_draft >> 8) ? P.draft : P.target;
    const void* row = reinterpret_cast<const char*>(base) +
                      (size_t)ri.logit_row * P.vocab * E::kBytes;
    ChunkGeom<E> g;
    g.init(row, P.vocab, ch, P.nch);

    Partial out;
    if (kind == kSoftmax) {
      SoftmaxAcc a = chunk_softmax<E>(row, g, ch, P.nch, q.c);
      a = block_reduce<SoftmaxAcc, kThreads>(a, s_red_sm);
      out = Partial{a.m, a.s, -1, 0u};
    } else {
      BestAcc a;
      if (kind == kArgmax) {
        a = chunk_argmax<E>(row, g, ch, P.nch);
      } else {
        const uint32_t pos = (uint32_t)ri.pos;
        switch (g.head & 3) {
          case 0: a = chunk_race<E, 0>(row, g, ch, P.nch, q.c, pos, q.req_lo, q.req_hi, P.key); break;
          case 1: a = chunk_race<E, 1>(row, g, ch, P.nch, q.c, pos, q.req_lo, q.req_hi, P.key); break;
          case 2: a = chunk_race<E, 2>(row, g, ch, P.nch, q.c, pos, q.req_lo, q.req_hi, P.key); break;
          default: a = chunk_race<E, 3>(row, g, ch, P.nch, q.c, pos, q.req_lo, q.req_hi, P.key); break;
        }
      }
      a = block_reduce<BestAcc, kThreads>(a, s_red_b);
      out = Partial{a.v, 0.f, a.idx, a.nan};
    }

    if (threadIdx.x == 0) {
      P.part[item] = out;
      __threadfence();
      s_flag = (atomicAdd(P.row_cnt + n, 1) == P.nch - 1) ? 1 : 0;
    }
    __syncthreads();
    if (s_flag) {
      // this CTA finished row n: merge its chunk partials
      if (threadIdx.x < 32) {
        __threadfence();
        const int lane = threadIdx.x;
        Partial res;
        if (kind == kSoftmax) {
          SoftmaxAcc a;
          a.init();
          for (int j = lane; j < P.nch; j += 32) {
            const Partial pj = ld_cg(P.part + (size_t)n * P.nch + j);
            SoftmaxAcc b;
            b.m = pj.a;
            b.s = pj.b;
            a = SoftmaxAcc::merge(a, b);
          }
          a = warp_reduce(a);
          const bool bad = !(a.s > 0.f) || !(a.s < 3.0e38f) || a.m == kNegInf ||
                           !(a.m < 3.0e38f) || (a.m != a.m) || (a.s != a.s);
          res = Partial{a.m, a.s, -1, bad ? 1u : 0u};
        } else {
          BestAcc a;
          a.init();
          for (int j = lane; j < P.nch; j += 32) {
            const Partial pj = ld_cg(P.part + (size_t)n * P.nch + j);
            BestAcc b;
            b.v = pj.a;
            b.idx = pj.idx;
            b.nan = pj.bad;
            a = BestAcc::merge(a, b);
          }
          a = warp_reduce(a);
          const bool bad = a.nan != 0u || a.idx < 0 || !(a.v < 3.0e38f);
          res = Partial{a.v, 0.f, a.idx, bad ? 1u : 0u};
        }
        if (lane == 0) {
          P.rowres[n] = res;
          __threadfence();
          s_flag = (atomicAdd(P.req_cnt + ri.req, 1) == q.nrows - 1) ? 2 : 0;
        }
        __syncwarp();
        if (s_flag == 2) {
          __threadfence();
          scan_request<E>(P, ri.req);
        }
      }
    }
    __syncthreads();
  }
}

// ---------------------------------------------------------------------------
// K2: the correction draw for requests rejected at position j.  Weights
// w_v = [p_j(v) - q_j(v)]_+ ("Speculative Decoding: Medusa, MTP, EAGLE,
// DFlash, DDTree, and DSpark", section 1: sample from the normalised positive
// residual); race score log2(w_v) - log2(E_v).  The fallback race on p_j (used
// when the residual has no mass) shares the exponentials.
// ---------------------------------------------------------------------------
template <typename E, int OFF>
__device__ __forceinline__ Best2Acc chunk_residual_vec(const void* trow, const void* drow,
                                                       const ChunkGeom<E>& g, float c, float mp,
                                                       float inv_sp, float mq, float inv_sq,
                                                       uint32_t pos, uint32_t req_lo,
                                                       uint32_t req_hi, PhiloxKey key) {
  Best2Acc acc;
  acc.init();
  const uint4* tp = reinterpret_cast<const uint4*>(reinterpret_cast<const char*>(trow) +
                                                   (size_t)g.head * E::kBytes);
  const uint4* dp = reinterpret_cast<const uint4*>(reinterpret_cast<const char*>(drow) +
                                                   (size_t)g.head * E::kBytes);
  for (int v0 = g.vbeg + threadIdx.x; v0 < g.vend; v0 += kThreads * kUnroll) {
    uint4 dt[kUnroll], dd[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int vi = v0 + u * kThreads;
      dt[u] = vi < g.vend ? ld_stream(tp + vi) : E::pad();
      dd[u] = vi < g.vend ? ld_stream(dp + vi) : E::pad();
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      float x[E::kVec], z[E::kVec];
      E::unpack(dt[u], x);
      E::unpack(dd[u], z);
      const int e0 = g.head + (v0 + u * kThreads) * E::kVec;
      RaceWords<E::kVec, OFF> rw;
      rw.make(e0, pos, req_lo, req_hi, key);
#pragma unroll
      for (int e = 0; e < E::kVec; ++e) {
        const float lE = fast_lg2(race_exponential(rw.word(e)));
        const float p = fast_ex2(fmaf(x[e], c, -mp)) * inv_sp;
        const float qv = fast_ex2(fmaf(z[e], c, -mq)) * inv_sq;
        const float w = p - qv;
        if (w > 0.f) acc.a.take(fast_lg2(w) - lE, e0 + e);
        acc.b.take(fmaf(x[e], c, -lE), e0 + e);
      }
    }
  }
  return acc;
}

template <typename E>
__device__ __forceinline__ void residual_one(Best2Acc& acc, float x, float z, int e, float c,
                                             float mp, float inv_sp, float mq, float inv_sq,
                                             uint32_t pos, uint32_t req_lo, uint32_t req_hi,
                                             PhiloxKey key) {
  const float lE = fast_lg2(race_exponential(race_word1(e, pos, req_lo, req_hi, key)));
  const float p = fast_ex2(fmaf(x, c, -mp)) * inv_sp;
  const float qv = fast_ex2(fmaf(z, c, -mq)) * inv_sq;
  const float w = p - qv;
  if (w > 0.f) acc.a.take(fast_lg2(w) - lE, e);
  acc.b.take(fmaf(x, c, -lE), e);
}

template <typename E>
__global__ void __launch_bounds__(kThreads) sv_residual(Params P) {
  __shared__ Best2Acc s_red[kThreads / 32];
  __shared__ int s_flag;
  const int n_items = P.counters[kCntResid] * P.nch;
  for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
    const int slot = item / P.nch;
    const int ch = item - slot * P.nch;
    const int2 rj = ld_cg(P.res_list + slot);
    const int r = rj.x, j = rj.y;
    const ReqInfo q = P.req[r];
    const Partial rt = ld_cg(P.rowres + q.row0 + 2 * j);
    const Partial rd = ld_cg(P.rowres + q.row0 + 2 * j + 1);
    const void* trow = reinterpret_cast<const char*>(P.target) +
                       (size_t)(q.tgt_off + j) * P.vocab * E::kBytes;
    const void* drow = reinterpret_cast<const char*>(P.draft) +
                       (size_t)(q.drf_off + j) * P.vocab * E::kBytes;
    const float inv_sp = 1.f / rt.b, inv_sq = 1.f / rd.b;
    const uint32_t pos = (uint32_t)j;
    ChunkGeom<E> gt, gd;
    gt.init(trow, P.vocab, ch, P.nch);
    gd.init(drow, P.vocab, ch, P.nch);

    Best2Acc acc;
    acc.init();
    if (gt.head == gd.head) {
      // both rows share their 16-byte phase: vector path plus scalar head/tail
      switch (gt.head & 3) {
        case 0: acc = chunk_residual_vec<E, 0>(trow, drow, gt, q.c, rt.a, inv_sp, rd.a, inv_sq, pos, q.req_lo, q.req_hi, P.key); break;
        case 1: acc = chunk_residual_vec<E, 1>(trow, drow, gt, q.c, rt.a, inv_sp, rd.a, inv_sq, pos, q.req_lo, q.req_hi, P.key); break;
        case 2: acc = chunk_residual_vec<E, 2>(trow, drow, gt, q.c, rt.a, inv_sp, rd.a, inv_sq, pos, q.req_lo, q.req_hi, P.key); break;
        default: acc = chunk_residual_vec<E, 3>(trow, drow, gt, q.c, rt.a, inv_sp, rd.a, inv_sq, pos, q.req_lo, q.req_hi, P.key); break;
      }
      if (ch == 0 && (int)threadIdx.x < gt.head) {
        const int e = threadIdx.x;
        residual_one<E>(acc, E::load1(trow, e), E::load1(drow, e), e, q.c, rt.a, inv_sp, rd.a,
                        inv_sq, pos, q.req_lo, q.req_hi, P.key);
      }
      if (ch == P.nch - 1 && (int)threadIdx.x < gt.tail) {
        const int e = gt.head + gt.nvec * E::kVec + threadIdx.x;
        residual_one<E>(acc, E::load1(trow, e), E::load1(drow, e), e, q.c, rt.a, inv_sp, rd.a,
                        inv_sq, pos, q.req_lo, q.req_hi, P.key);
      }
    } else {
      // rows with different 16-byte phases: plain element loads over the chunk
      const int e_beg = ch == 0 ? 0 : gt.head + gt.vbeg * E::kVec;
      const int e_end = ch == P.nch - 1 ? P.vocab : gt.head + gt.vend * E::kVec;
      for (int e = e_beg + threadIdx.x; e < e_end; e += kThreads)
        residual_one<E>(acc, E::load1(trow, e), E::load1(drow, e), e, q.c, rt.a, inv_sp, rd.a,
                        inv_sq, pos, q.req_lo, q.req_hi, P.key);
    }
    acc = block_reduce<Best2Acc, kThreads>(acc, s_red);

    if (threadIdx.x == 0) {
      P.part2[item] = Partial2{acc.a.v, acc.a.idx, acc.b.v, acc.b.idx};
      __threadfence();
      s_flag = (atomicAdd(P.res_cnt + slot, 1) == P.nch - 1) ? 1 : 0;
    }
    __syncthreads();
    if (s_flag && threadIdx.x < 32) {
      __threadfence();
      const int lane = threadIdx.x;
      Best2Acc a;
      a.init();
      for (int jj = lane; jj < P.nch; jj += 32) {
        const Partial2 pj = ld_cg(P.part2 + (size_t)slot * P.nch + jj);
        Best2Acc b;
        b.a.v = pj.va;
        b.a.idx = pj.ia;
        b.a.nan = 0u;
        b.b.v = pj.vb;
        b.b.idx = pj.ib;
        b.b.nan = 0u;
        a = Best2Acc::merge(a, b);
      }
      a = warp_reduce(a);
      if (lane == 0) {
        const int token = a.a.idx >= 0 ? a.a.idx : a.b.idx;
        P.committed[(size_t)r * (P.max_k + 1) + j] = token;
      }
    }
    __syncthreads();
  }
}

}  // namespace sv
