// sv_cluster.cuh -- the verify round on thread-block clusters: one launch
// after the plan, every request's positions decided as soon as its rows are
// read, and the correction draw made while those rows are still in L2.
//
// A cluster of N CTAs works through requests one position at a time: each CTA
// streams its 1/N slice (whole race blocks) of the position's rows, the CTAs
// swap their 16-byte partials through distributed shared memory at a cluster
// barrier, and every CTA then makes the same decision from the same merged
// values ("Speculative Decoding: Medusa, MTP, EAGLE, DFlash, DDTree, and
// DSpark", section 1: accept y_i with probability min(1, p_i(y_i)/q_i(y_i)),
// stop at the first rejection, draw the correction from [p_j - q_j]_+ or the
// bonus from p_k).  A rejection is followed at once by the correction pass over
// the same slices -- a few microseconds after they were read, so it is served
// from L2 -- and only the rows of positions 0..A are ever read from HBM.
//
// Two requests are in flight per cluster (slots), their items interleaved, so
// the exchange and decision of one item overlap the streaming of the next.
// Requests are claimed from the plan's list by the cluster's rank-0 CTA one
// claim ahead (the "spare"), published through its shared memory.  All CTAs of
// a cluster run the identical item sequence: every branch that decides the
// sequence depends only on merged values all of them hold.
//
// Cluster barriers (hardware, split into arrive and wait) are the only waits:
// one phase per item, entered by every thread of every CTA in the same order,
// plus one at the start and one at the end.
#pragma once

#include "sv_kernels.cuh"

namespace sv {

constexpr int kSlots = 3;

enum CKind : int { kCPair = 0, kCArg = 1, kCRace = 2, kCResid = 3 };
enum CUnit : int { kCUEnd = 0, kCUIdle = 1, kCUItem = 2 };
// A slot is idle, starting (request taken, its list entry and tokens being
// loaded), pending (its next item known), or streaming (item in flight).
enum SlotSt : int { kSlotIdle = 0, kSlotStarting = 1, kSlotPending = 2, kSlotStreaming = 3 };

// ---- cluster primitives -------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_size() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release;" ::: "memory");
}
// arrival of a thread that publishes nothing (no ordering of its own accesses)
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire;" ::: "memory");
}
// address of `p` (this CTA's shared memory) in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t cluster_addr(const void* p, uint32_t rank) {
  const uint32_t a = (uint32_t)__cvta_generic_to_shared(p);
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
  return r;
}
__device__ __forceinline__ int4 ld_cluster_v4(uint32_t addr) {
  int4 v;
  asm volatile("ld.shared::cluster.v4.s32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}
__device__ __forceinline__ int ld_cluster_s32(uint32_t addr) {
  int v;
  asm volatile("ld.shared::cluster.s32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ Partial as_partial(int4 v) {
  return Partial{__int_as_float(v.x), __int_as_float(v.y), v.z, (uint32_t)v.w};
}

// ---- one item of the cluster kernel (queue entry) ------------------------------
// PAIR: two streams (the CTA's slice of t_i, then of d_i); ARG / RACE: one
// stream of t_i; RESID: one stream holding t_j and d_j side by side.
struct __align__(16) CItem {
  const char* row0;
  const char* row1;
  int kind;
  int slot;
  int vbeg, vend;  // this CTA's slice, in 16-byte vectors
  int nst0, nst1;  // ring stages of stream 0 and stream 1
  int yv, ye;      // vector of the slice holding y (-1: none) and its element
  int pos;         // Philox position
  float c;
  float mp, inv_sp, mq, inv_sq;
  uint32_t req_lo, req_hi;
};

// A request slot (control warp state, identical in every CTA of the cluster).
struct SlotState {
  int st;      // SlotSt
  int ent;     // request list entry
  int r, d0, k;
  float c;
  uint32_t req_lo, req_hi;
  int kind, pos;                 // the slot's next (or current) item
  float mp, inv_sp, mq, inv_sq;  // normalisers for a RESID item
};

// ---- the copy ring with catch-up ----------------------------------------------
// Stages are numbered globally; stage s lives in ring slot s % kStages.  A
// stage is issued only once its item is queued; consuming stage C first issues
// whatever is still missing up to C (the item being consumed is always
// queued), waits for C, then refills up to C + kStages - 1.
struct ClusterRing {
  int issued;  // stages issued so far
  int q;       // queue index of the item being issued
  int stream;  // its stream (0 or 1)
  int left;    // stages of that stream still to issue
  const uint4* b0;
  const uint4* b1;
  int i0, i1, step, vend;
  bool active;

  __device__ __forceinline__ bool open_stream(const CItem* queue, int qavail) {
    while (q < qavail) {
      const CItem& it = queue[q & (kQueue - 1)];
      const int nst = stream == 0 ? it.nst0 : it.nst1;
      if (nst > 0) {
        const bool side = it.kind == kCResid;
        const char* row = stream == 0 ? it.row0 : it.row1;
        b0 = reinterpret_cast<const uint4*>(row);
        b1 = reinterpret_cast<const uint4*>(side ? it.row1 : row);
        i0 = it.vbeg + (int)threadIdx.x;
        i1 = side ? i0 : i0 + kThreads;
        step = side ? kThreads : kStageVecs * kThreads;
        vend = it.vend;
        left = nst;
        return true;
      }
      if (stream == 0 && it.nst1 > 0) {
        stream = 1;
      } else {
        stream = 0;
        ++q;
      }
    }
    return false;
  }

  __device__ __forceinline__ void pump(const CItem* queue, const int* s_qend, uint4* ring,
                                       int limit) {
    // the common case: one more stage of the stream being copied
    if (issued + 1 == limit && active && left > 1) {
      uint4* dst = ring + (issued & (kStages - 1)) * kStageVecs * kThreads + threadIdx.x;
      if (i0 < vend) cp_async16(dst, b0 + i0);
      if (i1 < vend) cp_async16(dst + kThreads, b1 + i1);
      cp_async_commit();
      ++issued;
      i0 += step;
      i1 += step;
      --left;
      return;
    }
    while (issued < limit) {
      if (!active) {
        // only opening a stream looks at the queue (published items only)
        active = open_stream(queue, ld_acquire_shared(s_qend));
        if (!active) return;
      }
      uint4* dst = ring + (issued & (kStages - 1)) * kStageVecs * kThreads + threadIdx.x;
      if (i0 < vend) cp_async16(dst, b0 + i0);
      if (i1 < vend) cp_async16(dst + kThreads, b1 + i1);
      cp_async_commit();
      ++issued;
      i0 += step;
      i1 += step;
      if (--left == 0) {
        active = false;
        const CItem& it = queue[q & (kQueue - 1)];
        if (stream == 0 && it.nst1 > 0) {
          stream = 1;
        } else {
          stream = 0;
          ++q;
        }
      }
    }
  }
};

__device__ __forceinline__ void wait_pending(int n) {
  switch (n) {
    case 0: cp_async_wait<0>(); break;
    case 1: cp_async_wait<1>(); break;
    case 2: cp_async_wait<2>(); break;
    case 3: cp_async_wait<3>(); break;
    case 4: cp_async_wait<4>(); break;
    case 5: cp_async_wait<5>(); break;
    case 6: cp_async_wait<6>(); break;
    default: cp_async_wait<kStages - 1>(); break;
  }
}

// Consumes stage `cs` (the next one) into v0, v1.
__device__ __forceinline__ void cring_take(const CItem* queue, const int* s_qend, uint4* ring,
                                           ClusterRing& cr, int& cs, uint4& v0, uint4& v1) {
  if (cr.issued <= cs) cr.pump(queue, s_qend, ring, cs + 1);
  const int ahead = cr.issued - cs - 1;
  if (ahead == kStages - 2) {
    cp_async_wait<kStages - 2>();
  } else {
    wait_pending(ahead);
  }
  const uint4* src = ring + (cs & (kStages - 1)) * kStageVecs * kThreads + threadIdx.x;
  v0 = src[0];
  v1 = src[kThreads];
  ++cs;
  cr.pump(queue, s_qend, ring, cs + kStages - 1);
}

// The CTA's reduction of one item: out[0] (and out[1] for PAIR) per warp.
// The item's fields are copied to registers first: the queue lives in shared
// memory, which every copy-ring instruction's memory clobber would reload.
template <typename E>
__device__ __forceinline__ void citem_reduce(const Params& P, const CItem* queue,
                                             const int* s_qend, uint4* ring, ClusterRing& cr,
                                             int& cs, const CItem& itm, float* s_xy,
                                             Partial (&out)[2]) {
  const int w = threadIdx.x >> 5;
  const int tid = threadIdx.x;
  const int kind = itm.kind, vbeg = itm.vbeg, vend = itm.vend, nst0 = itm.nst0,
            nst1 = itm.nst1, yv = itm.yv, ye = itm.ye, pos = itm.pos;
  const float c = itm.c;
  const RequestKey rk{itm.req_lo, itm.req_hi};
  if (kind == kCPair) {
    const int nfull = (vend - vbeg) / (kStageVecs * kThreads);
#pragma unroll
    for (int s = 0; s < 2; ++s) {
      LazySoftmax acc;
      acc.init();
      const int nst = s == 0 ? nst0 : nst1;
      for (int st = 0; st < nst; ++st) {
        uint4 v0, v1;
        cring_take(queue, s_qend, ring, cr, cs, v0, v1);
        const int vi = vbeg + st * kStageVecs * kThreads + tid;
        if (st >= nfull) {
          if (vi >= vend) v0 = E::pad();
          if (vi + kThreads >= vend) v1 = E::pad();
        }
        float x0[E::kVec], x1[E::kVec];
        E::unpack(v0, x0);
        E::unpack(v1, x1);
        if (vi == yv) s_xy[s] = pick(x0, ye);
        if (vi + kThreads == yv) s_xy[s] = pick(x1, ye);
        acc.add2(x0, x1, c);
      }
      const SoftmaxAcc a = warp_reduce(acc.result());
      out[s] = Partial{a.m, a.s, -1, 0u};
    }
    return;
  }
  BestAcc acc;
  acc.init();
  if (kind == kCArg) {
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
    const int nfull = (vend - vbeg) / (kStageVecs * kThreads);
    for (int st = 0; st < nst0; ++st) {
      uint4 v0, v1;
      cring_take(queue, s_qend, ring, cr, cs, v0, v1);
      const int vi = vbeg + st * kStageVecs * kThreads + tid;
      if (st >= nfull) {
        if (vi >= vend) v0 = E::pad();
        if (vi + kThreads >= vend) v1 = E::pad();
      }
      float x[E::kVec];
      E::unpack(v0, x);
      vec(x, vi * E::kVec);
      E::unpack(v1, x);
      vec(x, (vi + kThreads) * E::kVec);
    }
  } else if (kind == kCRace) {
    GroupGains<E> gg;
    const int nfull = (vend - vbeg) / (kStageVecs * kThreads);
    for (int st = 0; st < nst0; ++st) {
      uint4 v0, v1;
      cring_take(queue, s_qend, ring, cr, cs, v0, v1);
      const int vi = vbeg + st * kStageVecs * kThreads + tid;
      if (st >= nfull) {
        if (vi >= vend) v0 = E::pad();
        if (vi + kThreads >= vend) v1 = E::pad();
      }
      const int g = st * kStageVecs;
      if ((g & 31) == 0) gg.make(vbeg, g, w, (uint32_t)pos, rk, P.key);
      float x[E::kVec];
      E::unpack(v0, x);
      group_bonus<E>(acc, x, vi * E::kVec, c, gg.get(g));
      E::unpack(v1, x);
      group_bonus<E>(acc, x, (vi + kThreads) * E::kVec, c, gg.get(g + 1));
    }
  } else {
    const ResidualRow rr{c, itm.mp, itm.inv_sp, itm.mq, itm.inv_sq};
    GroupGains<E> gg;
    const int nfull = (vend - vbeg) / kThreads;
    for (int st = 0; st < nst0; ++st) {
      uint4 v0, v1;
      cring_take(queue, s_qend, ring, cr, cs, v0, v1);
      const int vi = vbeg + st * kThreads + tid;
      if (st >= nfull && vi >= vend) {
        v0 = E::pad();
        v1 = E::pad();
      }
      if ((st & 31) == 0) gg.make(vbeg, st, w, (uint32_t)pos, rk, P.key);
      float x[E::kVec], z[E::kVec];
      E::unpack(v0, x);
      E::unpack(v1, z);
      group_residual<E>(acc, x, z, vi * E::kVec, rr, gg.get(st));
    }
  }
  acc = warp_reduce(acc);
  out[0] = Partial{acc.v, 0.f, acc.idx, acc.nan};
  out[1] = Partial{0.f, 0.f, -1, 0u};
}

// ---- control-warp side ----------------------------------------------------------
// The queue entry of a slot's next item, for CTA `rank` of `n`.
template <typename E>
__device__ __forceinline__ void make_citem(const Params& P, const SlotState& sl, const int* tok,
                                           int s, int vb, int ve, CItem& it) {
  const size_t row_bytes = (size_t)P.vocab * E::kBytes;
  const char* trow =
      reinterpret_cast<const char*>(P.target) + (size_t)(sl.d0 + sl.r + sl.pos) * row_bytes;
  const char* drow = P.draft == nullptr
                         ? nullptr
                         : reinterpret_cast<const char*>(P.draft) + (size_t)(sl.d0 + sl.pos) * row_bytes;
  const int y = (sl.kind == kCPair) ? tok[sl.pos] : -1;
  it.row0 = trow;
  it.row1 = (sl.kind == kCPair || sl.kind == kCResid) ? drow : nullptr;
  it.kind = sl.kind;
  it.slot = s;
  it.vbeg = vb;
  it.vend = ve;
  const int len = ve - vb;
  const int per = sl.kind == kCResid ? kThreads : kStageVecs * kThreads;
  it.nst0 = len > 0 ? (len + per - 1) / per : 0;
  it.nst1 = sl.kind == kCPair ? it.nst0 : 0;
  const int vy = y >= 0 ? y / E::kVec : -1;
  it.yv = (vy >= it.vbeg && vy < it.vend) ? vy : -1;
  it.ye = y >= 0 ? (y & (E::kVec - 1)) : 0;
  it.pos = sl.pos;
  it.c = sl.c;
  it.mp = sl.mp;
  it.inv_sp = sl.inv_sp;
  it.mq = sl.mq;
  it.inv_sq = sl.inv_sq;
  it.req_lo = sl.req_lo;
  it.req_hi = sl.req_hi;
}

// Loads a starting slot's list entry and draft tokens (all lanes) and gives it
// its first item.
__device__ void load_request(const Params& P, SlotState& sl, int* tok) {
  const int lane = threadIdx.x & 31;
  const Entry en = P.lists[sl.ent];
  sl.r = en.meta & 0x1fff;
  sl.k = (en.meta >> 15) & 31;
  sl.d0 = en.d0;
  sl.c = en.c;
  sl.req_lo = en.req_lo;
  sl.req_hi = en.req_hi;
  sl.pos = 0;
  sl.kind = sl.c == 0.f ? kCArg : (sl.k > 0 ? kCPair : kCRace);
  if (lane < sl.k) tok[lane] = P.tokens[sl.d0 + lane];
  sl.st = kSlotPending;
}

// The item just exchanged, merged over the cluster: every CTA gets the same.
struct CMerged {
  RowRes a, b;
};

__device__ CMerged merge_cluster(const Partial* s_part_buf, int kind, uint32_t n) {
  const int lane = threadIdx.x & 31;
  SoftmaxAcc sa, sb;
  sa.init();
  sb.init();
  BestAcc ba;
  ba.init();
  float xa = 0.f, xb = 0.f;
  bool ha = false, hb = false;
  if (lane < (int)n) {
    const Partial pa = as_partial(ld_cluster_v4(cluster_addr(s_part_buf, lane)));
    const Partial pb = as_partial(ld_cluster_v4(cluster_addr(s_part_buf + 1, lane)));
    if (kind == kCPair) {
      sa.m = pa.a;
      sa.s = pa.b;
      sb.m = pb.a;
      sb.s = pb.b;
      if (pa.bad) {
        ha = true;
        xa = __int_as_float(pa.idx);
      }
      if (pb.bad) {
        hb = true;
        xb = __int_as_float(pb.idx);
      }
    } else {
      ba.v = pa.a;
      ba.idx = pa.idx;
      ba.nan = pa.bad;
    }
  }
  CMerged m;
  const float nan = __int_as_float(0x7fc00000);
  if (kind == kCPair) {
    sa = warp_reduce(sa);
    sb = warp_reduce(sb);
    const unsigned hma = __ballot_sync(0xffffffffu, ha), hmb = __ballot_sync(0xffffffffu, hb);
    const float ya = __shfl_sync(0xffffffffu, xa, hma ? __ffs(hma) - 1 : 0);
    const float yb = __shfl_sync(0xffffffffu, xb, hmb ? __ffs(hmb) - 1 : 0);
    m.a = softmax_res(sa, hma ? ya : nan);
    m.b = softmax_res(sb, hmb ? yb : nan);
  } else {
    m.a = best_res(warp_reduce(ba), kind == kCArg ? kArgmax : kRace);
    m.b = RowRes{0.f, 0.f, 0.f, -1, false};
  }
  return m;
}

// What a decision leaves for the owning CTA to write after the next item is
// published.
enum Action : int {
  kActNone = 0,      // accepted, nothing to write yet
  kActSkip = 1,      // a read row held NaN/+inf: the request is skipped
  kActGreedy = 2,    // greedy: accepted prefix A and the target argmax
  kActBonus = 3,     // every draft accepted: element race in block `idx` of t_k
  kActReject = 4,    // first rejection at A: prefix written, correction pending
  kActResidual = 5,  // the correction: element race in block `idx` of [p_j - q_j]_+
};

struct Outcome {
  int action;
  int r, d0, k, A, idx;
  float c, mp, inv_sp, mq, inv_sq;
  uint32_t req_lo, req_hi;
  bool debug;       // an acceptance test was made at position A (or A - 1)
  int dpos;         // its position
  float p, q, u;    // p(y), q(y), u there
};

// Decides the item of slot sl (all lanes alike) and updates the slot: pending
// with its next item, or idle.  No global memory is read.
__device__ Outcome cdecide(const Params& P, SlotState& sl, const int* tok, int kind,
                           const CMerged& m) {
  Outcome o;
  o.action = kActNone;
  o.r = sl.r;
  o.d0 = sl.d0;
  o.k = sl.k;
  o.A = sl.pos;
  o.idx = -1;
  o.c = sl.c;
  o.mp = sl.mp;
  o.inv_sp = sl.inv_sp;
  o.mq = sl.mq;
  o.inv_sq = sl.inv_sq;
  o.req_lo = sl.req_lo;
  o.req_hi = sl.req_hi;
  o.debug = false;
  o.dpos = sl.pos;
  o.p = o.q = o.u = 0.f;
  const int i = sl.pos;
  if (kind == kCArg) {
    if (m.a.bad) {
      o.action = kActSkip;
      sl.st = kSlotIdle;
    } else if (i < sl.k && tok[i] == m.a.idx) {
      sl.pos = i + 1;
      sl.st = kSlotPending;
    } else {
      o.action = kActGreedy;
      o.idx = m.a.idx;
      sl.st = kSlotIdle;
    }
    return o;
  }
  if (kind == kCRace) {
    o.action = (m.a.bad || m.a.idx < 0) ? kActSkip : kActBonus;
    o.idx = m.a.idx;
    sl.st = kSlotIdle;
    return o;
  }
  if (kind == kCResid) {
    o.action = kActResidual;
    o.idx = m.a.idx;
    sl.st = kSlotIdle;
    return o;
  }
  // PAIR: the acceptance test
  const RowRes& t = m.a;
  const RowRes& d = m.b;
  if (t.bad || d.bad) {
    o.action = kActSkip;
    sl.st = kSlotIdle;
    return o;
  }
  const float tp = fmaf(t.xy, sl.c, -t.a);  // log2(p(y) S_p)
  const float tq = fmaf(d.xy, sl.c, -d.a);  // log2(q(y) S_q)
  const float u = accept_uniform(P.key, (uint32_t)i, sl.req_lo, sl.req_hi);
  bool accept;
  if (tp == kNegInf) {
    accept = false;
  } else if (tq == kNegInf) {
    accept = true;
  } else {
    const float mx = fmaxf(tp, tq);
    accept = u * (fast_ex2(tq - mx) * t.b) < fast_ex2(tp - mx) * d.b;
  }
  o.debug = true;
  o.p = fast_ex2(tp) / t.b;
  o.q = fast_ex2(tq) / d.b;
  o.u = u;
  if (accept) {
    sl.pos = i + 1;
    sl.kind = sl.pos < sl.k ? kCPair : kCRace;
    sl.st = kSlotPending;
    return o;
  }
  // first rejection at i: the correction pass over the same slices follows
  o.action = kActReject;
  sl.kind = kCResid;
  sl.mp = t.a;
  sl.inv_sp = 1.f / t.b;
  sl.mq = d.a;
  sl.inv_sq = 1.f / d.b;
  sl.st = kSlotPending;
  return o;
}

// Accepted prefix, the extra token (-1 while the correction is pending),
// flags and NaN debug values after A (or everywhere, greedy), from the slot's
// copy of the draft tokens (control warp of the owning CTA).
__device__ void cfinish(const Params& P, const Outcome& o, const int* tok, int token,
                        bool greedy) {
  const int lane = threadIdx.x & 31;
  const int width = P.max_k + 1;
  if (lane < width) {
    const int v = lane < o.A ? tok[lane] : (lane == o.A ? token : -1);
    P.committed[(size_t)o.r * width + lane] = v;
  }
  const float nan = __int_as_float(0x7fc00000);
  if (lane < o.k) {
    P.flags[o.d0 + lane] = lane < o.A ? 1 : 0;
    if (lane > o.A || greedy) {
      if (P.p_y) P.p_y[o.d0 + lane] = nan;
      if (P.q_y) P.q_y[o.d0 + lane] = nan;
      if (P.u_dbg) P.u_dbg[o.d0 + lane] = nan;
    }
  }
  if (lane == 0) {
    P.accepted_len[o.r] = o.A;
    if (P.req_status) P.req_status[o.r] = 0;
  }
}

// The owning CTA's writes for a decision (control warp).
template <typename E>
__device__ void cwrite(const Params& P, const Outcome& o, const int* tok) {
  const int lane = threadIdx.x & 31;
  if (o.debug && lane == 0) {
    if (P.p_y) P.p_y[o.d0 + o.dpos] = o.p;
    if (P.q_y) P.q_y[o.d0 + o.dpos] = o.q;
    if (P.u_dbg) P.u_dbg[o.d0 + o.dpos] = o.u;
  }
  if (o.action == kActNone) return;
  if (o.action == kActSkip) {
    skip_request_warp(P, o.r, o.d0, o.k, kStNonfinite);
    return;
  }
  if (o.action == kActGreedy) {
    cfinish(P, o, tok, o.idx, true);
    return;
  }
  if (o.action == kActReject) {
    cfinish(P, o, tok, -1, false);
    return;
  }
  const size_t row_bytes = (size_t)P.vocab * E::kBytes;
  const RequestKey rk{o.req_lo, o.req_hi};
  const char* trow =
      reinterpret_cast<const char*>(P.target) + (size_t)(o.d0 + o.r + o.A) * row_bytes;
  if (o.action == kActBonus) {
    const ResidualRow rr{o.c, 0.f, 0.f, 0.f, 0.f};
    const int token = inner_race<E, false>(P, trow, nullptr, o.idx, rr, (uint32_t)o.A, rk);
    cfinish(P, o, tok, token, false);
    return;
  }
  // kActResidual
  const char* drow = reinterpret_cast<const char*>(P.draft) + (size_t)(o.d0 + o.A) * row_bytes;
  int token;
  if (o.idx >= 0) {
    const ResidualRow rr{o.c, o.mp, o.inv_sp, o.mq, o.inv_sq};
    token = inner_race<E, true>(P, trow, drow, o.idx, rr, (uint32_t)o.A, rk);
  } else {
    const ResidualRow rr{o.c, 0.f, 0.f, 0.f, 0.f};
    const BestAcc br = warp_block_race<E>(P, trow, o.c, (uint32_t)o.A, rk);
    token = inner_race<E, false>(P, trow, nullptr, br.idx, rr, (uint32_t)o.A, rk);
  }
  if (lane == 0) P.committed[(size_t)o.r * (P.max_k + 1) + o.A] = token;
}

// Queues the next item of every pending slot, round robin (control warp).  A
// slot has at most one item queued or streaming at a time.
template <typename E>
__device__ __forceinline__ void publish_items(const Params& P, SlotState* s_slot,
                                              int (*s_tok)[32], CItem* queue, int& q_head,
                                              int& next_slot, int vb, int ve) {
  const int lane = threadIdx.x & 31;
  for (int j = 0; j < kSlots; ++j) {
    const int s = (next_slot + j) % kSlots;
    if (s_slot[s].st != kSlotPending) continue;
    CItem it;
    make_citem<E>(P, s_slot[s], s_tok[s], s, vb, ve, it);
    __syncwarp();
    if (lane == 0) {
      queue[q_head & (kQueue - 1)] = it;
      s_slot[s].st = kSlotStreaming;
    }
    __syncwarp();
    ++q_head;
  }
  next_slot = (next_slot + 1) % kSlots;
}

// The next unit: an item if one is queued and not yet started, else idle
// while a slot is busy, else the end.
__device__ __forceinline__ int next_unit(const SlotState* s_slot, int q_head, int& n_started) {
  if (q_head > n_started) {
    ++n_started;
    return kCUItem;
  }
  for (int s = 0; s < kSlots; ++s)
    if (s_slot[s].st == kSlotStreaming || s_slot[s].st == kSlotStarting) return kCUIdle;
  return kCUEnd;
}

// ---------------------------------------------------------------------------
// The cluster launch.
// ---------------------------------------------------------------------------
template <typename E>
__global__ void __maxnreg__(128) sv_cluster(Params P) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  uint4* ring = reinterpret_cast<uint4*>(smem_raw);
  __shared__ CItem queue[kQueue];
  __shared__ Partial mailbox[2][kComputeWarps][2];
  __shared__ __align__(16) Partial s_part[2][2];  // this CTA's item partials, by exchange parity
  __shared__ int s_spare[2];                      // rank 0: the claimed spare, by exchange parity
  __shared__ int s_init[kSlots];                  // rank 0: the first claims
  __shared__ int s_unit[2];                       // CUnit | slot << 8
  __shared__ float s_xy[2][2];
  __shared__ int s_qend;
  __shared__ SlotState s_slot[kSlots];
  __shared__ int s_tok[kSlots][32];
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const bool control = warp == kComputeWarps;
  const uint32_t rank = cluster_rank(), n = cluster_size();
  // this CTA's slice of every row: race blocks [rank nb / n, (rank + 1) nb / n)
  constexpr int kVPB = kRaceBlock / E::kVec;
  const int slice_vb = (int)((long long)rank * P.nb / n) * kVPB;
  const int slice_ve = min((int)((long long)(rank + 1) * P.nb / n) * kVPB, P.nvec);

  pdl_launch_dependents();
  pdl_wait();  // the plan's request list is complete

  // every CTA of the cluster is running before any distributed access
  cluster_arrive();
  cluster_wait();
  if (control && rank == 0 && lane == 0) {
    for (int s = 0; s < kSlots; ++s) {
      const int e = atomicAdd(P.ctr + kCntClaim, 1);
      s_init[s] = e < P.list_cnt[0] ? e : -1;
    }
    const int e = atomicAdd(P.ctr + kCntClaim, 1);
    s_spare[1] = e < P.list_cnt[0] ? e : -1;
  }
  cluster_arrive();
  cluster_wait();

  int n_dec = 0;      // exchanges so far (identical in all CTAs)
  int q_head = 0;     // items queued
  int n_started = 0;  // items handed to the compute warps
  int next_slot = 0;
  if (control) {
    const uint32_t leader_init = cluster_addr(s_init, 0);
    for (int s = 0; s < kSlots; ++s) {
      const int e = ld_cluster_s32(leader_init + 4u * s);
      SlotState sl;
      sl.st = kSlotIdle;
      sl.ent = e;
      if (e >= 0) load_request(P, sl, s_tok[s]);
      __syncwarp();
      if (lane == 0) s_slot[s] = sl;
      __syncwarp();
    }
    publish_items<E>(P, s_slot, s_tok, queue, q_head, next_slot, slice_vb, slice_ve);
    const int unit = next_unit(s_slot, q_head, n_started);
    if (lane == 0) {
      s_unit[0] = unit;
      st_release_shared(&s_qend, q_head);
    }
    __syncwarp();
  }
  __syncthreads();

  ClusterRing cr;
  int cs = 0;
  if (!control) {
    cr.issued = 0;
    cr.q = 0;
    cr.stream = 0;
    cr.active = false;
    cr.pump(queue, &s_qend, ring, kStages - 1);
  }

  int prev = kCUIdle;  // the unit of the previous iteration
  int q_cur = 0;       // queue index of the current unit's item (compute warps)
  for (int u = 0;; ++u) {
    // a round needs at most two units per item and k + 2 items per request;
    // every CTA of the cluster reaches the same u, between exchanges
    if (u >= P.unit_cap) {
      if (tid == 0 && rank == 0)
        atomicOr(reinterpret_cast<unsigned int*>(P.ctr + kCntStatus), kStOverrun);
      break;
    }
    const int cur = s_unit[u & 1];
    const bool prev_item = (prev & 0xff) == kCUItem;
    const bool cur_item = (cur & 0xff) == kCUItem;
    if (!control) {
      if (prev_item) cluster_arrive_relaxed();
      if (cur_item) {
        Partial out[2];
        citem_reduce<E>(P, queue, &s_qend, ring, cr, cs, queue[q_cur & (kQueue - 1)],
                        s_xy[u & 1], out);
        if (lane == 0) {
          mailbox[u & 1][warp][0] = out[0];
          mailbox[u & 1][warp][1] = out[1];
        }
        ++q_cur;
      }
      if (prev_item) cluster_wait();
    } else {
      Outcome o;
      o.action = kActNone;
      o.debug = false;
      int ps = -1;
      bool owner = false;
      if (prev_item) {
        // ---- exchange and decide the previous item -----------------------------
        const CItem& pit = queue[n_dec & (kQueue - 1)];  // items are decided in queue order
        ps = pit.slot;
        const int kind = pit.kind;
        const int par = n_dec & 1;
        {
          const Partial* mb = &mailbox[(u - 1) & 1][0][0];
          Partial p0, p1;
          if (kind == kCPair) {
            SoftmaxAcc a, b;
            a.init();
            b.init();
            if (lane < kComputeWarps) {
              a.m = mb[2 * lane].a;
              a.s = mb[2 * lane].b;
              b.m = mb[2 * lane + 1].a;
              b.s = mb[2 * lane + 1].b;
            }
            a = warp_reduce(a);
            b = warp_reduce(b);
            p0 = Partial{a.m, a.s, __float_as_int(s_xy[(u - 1) & 1][0]), pit.yv >= 0 ? 1u : 0u};
            p1 = Partial{b.m, b.s, __float_as_int(s_xy[(u - 1) & 1][1]), pit.yv >= 0 ? 1u : 0u};
          } else {
            BestAcc a;
            a.init();
            if (lane < kComputeWarps) {
              a.v = mb[2 * lane].a;
              a.idx = mb[2 * lane].idx;
              a.nan = mb[2 * lane].bad;
            }
            a = warp_reduce(a);
            p0 = Partial{a.v, 0.f, a.idx, a.nan};
            p1 = Partial{0.f, 0.f, -1, 0u};
          }
          if (lane == 0) {
            s_part[par][0] = p0;
            s_part[par][1] = p1;
          }
          __syncwarp();
        }
        cluster_arrive();
        cluster_wait();
        const CMerged m = merge_cluster(s_part[par], kind, n);
        const int spare = ld_cluster_s32(cluster_addr(&s_spare[par ^ 1], 0));
        SlotState sl = s_slot[ps];
        owner = (uint32_t)(sl.r % (int)n) == rank;
        o = cdecide(P, sl, s_tok[ps], kind, m);
        bool took = false;
        if (sl.st == kSlotIdle && spare >= 0) {
          sl.st = kSlotStarting;  // loaded after the next item is published
          sl.ent = spare;
          took = true;
        }
        if (rank == 0 && lane == 0) {
          int ns = spare;
          if (took) {
            const int e = atomicAdd(P.ctr + kCntClaim, 1);
            ns = e < P.list_cnt[0] ? e : -1;
          }
          s_spare[par] = ns;
        }
        __syncwarp();
        if (lane == 0) s_slot[ps] = sl;
        __syncwarp();
        ++n_dec;
      }
      // ---- publish first, then the writes and loads nobody waits for -----------
      publish_items<E>(P, s_slot, s_tok, queue, q_head, next_slot, slice_vb, slice_ve);
      const int pub = next_unit(s_slot, q_head, n_started);
      if (lane == 0) {
        s_unit[(u + 1) & 1] = pub;
        st_release_shared(&s_qend, q_head);
      }
      __syncwarp();
      if (ps >= 0 && owner) cwrite<E>(P, o, s_tok[ps]);
      __syncwarp();
      if (ps >= 0 && s_slot[ps].st == kSlotStarting) {
        SlotState sl = s_slot[ps];
        load_request(P, sl, s_tok[ps]);
        __syncwarp();
        if (lane == 0) s_slot[ps] = sl;
      }
      __syncwarp();
    }
    __syncthreads();
    prev = cur;
    if ((cur & 0xff) == kCUEnd) break;
  }
  if (!control) cp_async_wait_all();
  // no CTA leaves while another may still read its shared memory
  cluster_arrive();
  cluster_wait();
}

}  // namespace sv
