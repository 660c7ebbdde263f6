// sv_tree.cuh -- greedy verification of a drafted token tree.
//
// "Speculative Decoding: Medusa, MTP, EAGLE, DFlash, DDTree, and DSpark",
// section 5 (DDTree): the drafted tree uses depth-based positions and
// ancestor-only attention; verification walks the target's selected tokens,
// and when no child matches, that target token becomes the next bonus token;
// only the accepted path survives.  Section 1 gives no sampling rule for
// trees, so the selection here is greedy: the target argmax, lowest index on
// ties.
//
// Layout: request r has n_r nodes; node i has a token and a parent in
// [-1, i) (-1: child of the root, the last committed token).  Its n_r + 1
// target rows are consecutive: row 0 is the target's output at the root, row
// 1 + i its output after node i.
//
// A round is three launches:
//   sv_tree_plan   one CTA: prefix offsets of rows and nodes, the layout checks;
//   sv_tree_rows   the HBM pass: every target row is cut into chunks of
//                  kTreeChunkVecs 16-byte vectors and each chunk reduced to its
//                  first maximum (value, index, NaN seen) by one CTA;
//   sv_tree_walk   one warp per request: validates its nodes, then from the
//                  root merges the chunk partials of the current row, takes
//                  its argmax tau and moves to the lowest-index child carrying
//                  tau, until no child does (tau is then the bonus token).
// Every row is read once, also rows off the accepted path: the walk needs the
// argmax of whichever row it reaches, and reading all rows in one pass keeps
// HBM streaming instead of one dependent launch per depth.
#pragma once

#include "sv_kernels.cuh"

namespace sv {

constexpr int kTreeThreads = 256;
constexpr int kTreeVecsPerThread = 8;                                  // loads in flight
constexpr int kTreeChunkVecs = kTreeThreads * kTreeVecsPerThread * 2;  // 64 KB chunks
constexpr int kTreeWalkWarps = 8;
constexpr int kTreeRegNodes = 4;  // nodes per lane the walk keeps in registers (128 per tree)
constexpr int kTreeMaxNodes = 1024;
constexpr uint32_t kStBadParent = 32u;

struct TreeParams {
  const void* target;
  const int32_t* num_nodes;
  const int32_t* parent;
  const int32_t* tokens;
  int batch, total_nodes, max_nodes, vocab;
  int nvec;     // 16-byte vectors per row (aligned rows)
  int nchunk;   // chunks per row
  int chunk;    // elements per chunk
  int rows;     // batch + total_nodes
  int32_t* accepted_len;
  int32_t* path;       // [batch, max_nodes]
  int32_t* committed;  // [batch, max_nodes + 1]
  int32_t* req_status;
  Partial* part;       // [rows * nchunk]
  int* t_off;          // [batch + 1]
  int* n_off;          // [batch + 1]
  int* ctr;            // [0] status, [1] layout bits
};

// ---------------------------------------------------------------------------
// Plan: offsets and layout checks (one CTA of kPlanThreads).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kPlanThreads) sv_tree_plan(TreeParams P) {
  __shared__ int s_w[kPlanThreads / 32 + 1];
  __shared__ uint32_t s_layout;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int kW = kPlanThreads / 32;
  if (tid == 0) s_layout = 0u;
  __syncthreads();
  int carry = 0;
  for (int base = 0; base < P.batch; base += kPlanThreads) {
    const int r = base + tid;
    const int n = r < P.batch ? P.num_nodes[r] : 0;
    const bool bad = n < 0 || n > P.max_nodes;
    if (bad) atomicOr(&s_layout, kStBadK);
    const int v = bad ? 0 : n;
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
    const int ex = carry + s_w[warp] + incl - v;
    if (r < P.batch) {
      P.n_off[r] = ex;
      P.t_off[r] = ex + r;
    }
    carry += s_w[kW];
    __syncthreads();
  }
  if (tid == 0) {
    P.n_off[P.batch] = carry;
    P.t_off[P.batch] = carry + P.batch;
    uint32_t layout = s_layout;
    if (!layout && carry != P.total_nodes) layout = kStBadTotal;
    P.ctr[0] = (int)layout;
    P.ctr[1] = (int)layout;
  }
}

// ---------------------------------------------------------------------------
// The row pass: first maximum of every chunk of every target row.
// ---------------------------------------------------------------------------
template <typename E, bool kAligned>
__global__ void __launch_bounds__(kTreeThreads, 4) sv_tree_rows(TreeParams P) {
  __shared__ BestAcc s_red[kTreeThreads / 32];
  const int tid = threadIdx.x;
  const size_t row_bytes = (size_t)P.vocab * E::kBytes;
  const long long items = (long long)P.rows * P.nchunk;
  for (long long item = blockIdx.x; item < items; item += gridDim.x) {
    const int row = (int)(item / P.nchunk), ch = (int)(item % P.nchunk);
    const char* rp = reinterpret_cast<const char*>(P.target) + (size_t)row * row_bytes;
    BestAcc acc;
    acc.init();
    if (kAligned) {
      const uint4* rv = reinterpret_cast<const uint4*>(rp);
      const int v0 = ch * kTreeChunkVecs, v1 = min(v0 + kTreeChunkVecs, P.nvec);
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint4 buf[kTreeVecsPerThread];
#pragma unroll
        for (int j = 0; j < kTreeVecsPerThread; ++j) {
          const int vi = v0 + (half * kTreeVecsPerThread + j) * kTreeThreads + tid;
          buf[j] = vi < v1 ? ld_stream(rv + vi) : E::pad();
        }
#pragma unroll
        for (int j = 0; j < kTreeVecsPerThread; ++j) {
          const int vi = v0 + (half * kTreeVecsPerThread + j) * kTreeThreads + tid;
          float x[E::kVec];
          E::unpack(buf[j], x);
#pragma unroll
          for (int e = 0; e < E::kVec; ++e) {
            acc.nan |= (x[e] != x[e]);
            acc.take(x[e], vi * E::kVec + e);  // increasing index: strict > keeps the first
          }
        }
      }
    } else {
      const int e0 = ch * P.chunk, e1 = min(e0 + P.chunk, P.vocab);
      for (int v = e0 + tid; v < e1; v += kTreeThreads) {
        const float x = E::load1(rp, v);
        acc.nan |= (x != x);
        acc.take(x, v);
      }
    }
    acc = warp_reduce(acc);
    if ((tid & 31) == 0) s_red[tid >> 5] = acc;
    __syncthreads();
    if (tid < 32) {
      BestAcc b;
      b.init();
      if (tid < kTreeThreads / 32) b = s_red[tid];
      b = warp_reduce(b);
      if (tid == 0) P.part[item] = Partial{b.v, 0.f, b.idx, b.nan};
    }
    __syncthreads();
  }
}

// ---------------------------------------------------------------------------
// The walk: one warp per request.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kTreeWalkWarps * 32) sv_tree_walk(TreeParams P) {
  const int lane = threadIdx.x & 31;
  const int r = blockIdx.x * kTreeWalkWarps + (threadIdx.x >> 5);
  if (r >= P.batch) return;
  const int pw = P.max_nodes, cw = P.max_nodes + 1;
  int32_t* pth = P.path + (size_t)r * pw;
  int32_t* com = P.committed + (size_t)r * cw;
  const uint32_t layout = (uint32_t)P.ctr[1];
  uint32_t rs = layout;
  int a = 0;
  if (!layout) {
    const int n = P.num_nodes[r];
    const int n0 = P.n_off[r], t0 = P.t_off[r];
    const int32_t* par = P.parent + n0;
    const int32_t* tok = P.tokens + n0;
    // the first 32 * kTreeRegNodes nodes stay in registers for the whole walk
    int rp[kTreeRegNodes], rt[kTreeRegNodes];
#pragma unroll
    for (int j = 0; j < kTreeRegNodes; ++j) {
      const int i = j * 32 + lane;
      rp[j] = i < n ? par[i] : -2;
      rt[j] = i < n ? tok[i] : -1;
    }
    for (int i = lane; i < n; i += 32) {
      const int pi = i < 32 * kTreeRegNodes ? rp[i / 32] : par[i];
      const int ti = i < 32 * kTreeRegNodes ? rt[i / 32] : tok[i];
      if (pi < -1 || pi >= i) rs |= kStBadParent;
      if (ti < 0 || ti >= P.vocab) rs |= kStBadToken;
    }
    rs = __reduce_or_sync(0xffffffffu, rs);
    int cur = -1;
    while (!rs) {
      // the argmax of the current node's row, from its chunk partials
      const Partial* pp = P.part + (size_t)(t0 + cur + 1) * P.nchunk;
      BestAcc best;
      best.init();
      for (int c = lane; c < P.nchunk; c += 32) {
        const Partial q = pp[c];
        BestAcc x;
        x.v = q.a;
        x.idx = q.idx;
        x.nan = q.bad;
        best = BestAcc::merge(best, x);
      }
      best = warp_reduce(best);
      if (best.nan != 0u || best.idx < 0 || !(best.v < 3.0e38f)) {
        rs = kStNonfinite;
        break;
      }
      const int tau = best.idx;
      if (lane == 0) com[a] = tau;
      // the lowest-index child of `cur` whose token is tau
      int child = -1;
#pragma unroll
      for (int j = 0; j < kTreeRegNodes; ++j) {
        const unsigned m = __ballot_sync(0xffffffffu, rp[j] == cur && rt[j] == tau);
        if (child < 0 && m) child = j * 32 + __ffs(m) - 1;
      }
      for (int i0 = 32 * kTreeRegNodes; i0 < n && child < 0; i0 += 32) {
        const int i = i0 + lane;
        const unsigned m = __ballot_sync(0xffffffffu, i < n && par[i] == cur && tok[i] == tau);
        if (m) child = i0 + __ffs(m) - 1;
      }
      if (child < 0) break;
      if (lane == 0) pth[a] = child;
      ++a;
      cur = child;
    }
  }
  if (rs) {
    for (int d = lane; d < cw; d += 32) com[d] = -1;
    for (int d = lane; d < pw; d += 32) pth[d] = -1;
    if (lane == 0) {
      P.accepted_len[r] = -1;
      atomicOr(reinterpret_cast<unsigned int*>(P.ctr), rs);
    }
  } else {
    for (int d = a + 1 + lane; d < cw; d += 32) com[d] = -1;
    for (int d = a + lane; d < pw; d += 32) pth[d] = -1;
    if (lane == 0) P.accepted_len[r] = a;
  }
  if (P.req_status && lane == 0) P.req_status[r] = (int32_t)rs;
}

}  // namespace sv
