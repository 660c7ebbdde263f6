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
// A round is two launches:
//   sv_tree_plan   one CTA: prefix offsets of rows and nodes, the layout checks;
//   sv_tree_path   one thread-block cluster per tree: validates the tree's nodes,
//                  then from the root reads the row of the node it stands on
//                  (each CTA a slice of it), takes its argmax tau (first
//                  maximum) and moves to the lowest-index child carrying tau,
//                  until no child does (tau is then the bonus token).
// Only the rows of the accepted path are read: A + 1 rows of a tree whose
// walk accepts A nodes, one after another, each by the CS CTAs of its
// cluster (64 KB of loads in flight per CTA) while other clusters walk
// other trees.
#pragma once

#include <cooperative_groups.h>

#include "sv_kernels.cuh"

namespace sv {

constexpr int kTreeMaxNodes = 1024;
constexpr uint32_t kStBadParent = 32u;

struct TreeParams {
  const void* target;
  const int32_t* num_nodes;
  const int32_t* parent;
  const int32_t* tokens;
  int batch, total_nodes, max_nodes, vocab;
  int nvec;     // 16-byte vectors per row (aligned rows)
  int rows;     // batch + total_nodes
  int32_t* accepted_len;
  int32_t* path;       // [batch, max_nodes]
  int32_t* committed;  // [batch, max_nodes + 1]
  int32_t* req_status;
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
// The walk: one thread-block cluster of CS CTAs per tree (trees cluster c,
// c + clusters, ...).  CTA q of the cluster reduces its slice q/CS of the
// current row to a first maximum; the slices' maxima are exchanged through
// distributed shared memory, so every CTA of the cluster takes the same tau,
// the same child and the same number of steps (cluster barriers are always
// matched).  CTA 0 writes the outputs.
// ---------------------------------------------------------------------------
constexpr int kPathThreads = 512;
constexpr int kPathVecs = 8;       // 16-byte loads in flight per thread
constexpr int kPathMaxCluster = 8; // portable cluster size

// The first maximum of elements [e0, e1) of one row (all threads call it; the
// result is valid in every thread).
template <typename E, bool kAligned>
__device__ BestAcc path_slice_argmax(const TreeParams& P, const char* rp, int v0, int v1,
                                     BestAcc* s_red) {
  const int tid = threadIdx.x;
  BestAcc acc;
  acc.init();
  if (kAligned) {
    const uint4* rv = reinterpret_cast<const uint4*>(rp);
    for (int b = v0; b < v1; b += kPathVecs * kPathThreads) {
      uint4 buf[kPathVecs];
#pragma unroll
      for (int j = 0; j < kPathVecs; ++j) {
        const int vi = b + j * kPathThreads + tid;
        buf[j] = vi < v1 ? ld_stream(rv + vi) : E::pad();
      }
#pragma unroll
      for (int j = 0; j < kPathVecs; ++j) {
        const int vi = b + j * kPathThreads + tid;
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
    for (int v = v0 + tid; v < v1; v += kPathThreads) {
      const float x = E::load1(rp, v);
      acc.nan |= (x != x);
      acc.take(x, v);
    }
  }
  acc = warp_reduce(acc);
  if ((tid & 31) == 0) s_red[tid >> 5] = acc;
  __syncthreads();
  BestAcc b;
  b.init();
  if ((tid & 31) < kPathThreads / 32) b = s_red[tid & 31];
  b = warp_reduce(b);  // every warp reduces the partials alike
  __syncthreads();     // s_red is reused by the next row
  return b;
}

template <typename E, bool kAligned>
__global__ void __launch_bounds__(kPathThreads, 2) sv_tree_path(TreeParams P) {
  namespace cg = cooperative_groups;
  cg::cluster_group cl = cg::this_cluster();
  const int cs = (int)cl.num_blocks(), crank = (int)cl.block_rank();
  const int cluster = (int)blockIdx.x / cs, clusters = (int)gridDim.x / cs;
  __shared__ BestAcc s_red[kPathThreads / 32];
  __shared__ BestAcc s_slice[2];  // this CTA's slice maximum, double-buffered by step
  __shared__ int s_par[kTreeMaxNodes];
  __shared__ int s_tok[kTreeMaxNodes];
  __shared__ int s_flag[kPathThreads / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const size_t row_bytes = (size_t)P.vocab * E::kBytes;
  const int units = kAligned ? P.nvec : P.vocab;  // vectors or elements of a row
  const int u0 = (int)((long long)units * crank / cs), u1 = (int)((long long)units * (crank + 1) / cs);
  const uint32_t layout = (uint32_t)P.ctr[1];
  const int pw = P.max_nodes, cw = P.max_nodes + 1;
  int step = 0;
  for (int r = cluster; r < P.batch; r += clusters) {
    int32_t* pth = P.path + (size_t)r * pw;
    int32_t* com = P.committed + (size_t)r * cw;
    uint32_t rs = layout;
    int a = 0;
    if (!layout) {
      const int n = P.num_nodes[r];
      const int n0 = P.n_off[r], t0 = P.t_off[r];
      uint32_t bad = 0u;
      for (int i = tid; i < n; i += kPathThreads) {
        const int pi = P.parent[n0 + i], ti = P.tokens[n0 + i];
        s_par[i] = pi;
        s_tok[i] = ti;
        if (pi < -1 || pi >= i) bad |= kStBadParent;
        if (ti < 0 || ti >= P.vocab) bad |= kStBadToken;
      }
      bad = __reduce_or_sync(0xffffffffu, bad);
      if (lane == 0) s_flag[warp] = (int)bad;
      __syncthreads();
      rs = 0u;
#pragma unroll 1
      for (int w = 0; w < kPathThreads / 32; ++w) rs |= (uint32_t)s_flag[w];
      __syncthreads();
      int cur = -1;
      while (!rs) {
        const char* rp =
            reinterpret_cast<const char*>(P.target) + (size_t)(t0 + cur + 1) * row_bytes;
        const BestAcc mine = path_slice_argmax<E, kAligned>(P, rp, u0, u1, s_red);
        const int buf = step & 1;
        if (tid == 0) s_slice[buf] = mine;
        cl.sync();  // every slice maximum of this step is in place
        BestAcc best;
        best.init();
#pragma unroll 1
        for (int q = 0; q < cs; ++q) best = BestAcc::merge(best, *cl.map_shared_rank(&s_slice[buf], q));
        ++step;
        if (best.nan != 0u || best.idx < 0 || !(best.v < 3.0e38f)) {
          rs = kStNonfinite;
          break;
        }
        const int tau = best.idx;
        if (crank == 0 && tid == 0) com[a] = tau;
        // the lowest-index child of `cur` whose token is tau
        int child = -1;
        for (int i0 = 0; i0 < n && child < 0; i0 += kPathThreads) {
          const int i = i0 + tid;
          const bool match = i < n && s_par[i] == cur && s_tok[i] == tau;
          const unsigned m = __ballot_sync(0xffffffffu, match);
          if (lane == 0) s_flag[warp] = m ? i0 + warp * 32 + __ffs(m) - 1 : -1;
          __syncthreads();
#pragma unroll 1
          for (int w = 0; w < kPathThreads / 32 && child < 0; ++w) child = s_flag[w];
          __syncthreads();
        }
        if (child < 0) break;
        if (crank == 0 && tid == 0) pth[a] = child;
        ++a;
        cur = child;
      }
    }
    if (crank == 0) {
      if (rs) {
        for (int d = tid; d < cw; d += kPathThreads) com[d] = -1;
        for (int d = tid; d < pw; d += kPathThreads) pth[d] = -1;
        if (tid == 0) {
          P.accepted_len[r] = -1;
          atomicOr(reinterpret_cast<unsigned int*>(P.ctr), rs);
        }
      } else {
        for (int d = a + 1 + tid; d < cw; d += kPathThreads) com[d] = -1;
        for (int d = a + tid; d < pw; d += kPathThreads) pth[d] = -1;
        if (tid == 0) P.accepted_len[r] = a;
      }
      if (P.req_status && tid == 0) P.req_status[r] = (int32_t)rs;
    }
    __syncthreads();  // s_par / s_tok are reused by the next tree
  }
  cl.sync();  // no CTA leaves while another may still read its slice maximum
}

}  // namespace sv
