// specverify.cu -- host side of the C ABI declared in include/specverify.h.
//
// Argument checking, scratch ownership and the launches of a verify round
// (a plan launch and a few wave launches).  All device work lives in
// sv_kernels.cuh.  Two owners of scratch memory share one launch path: a
// handle (cudaMalloc at create) and a fixed-size static device arena
// (specverify_run_static, no allocation at all).
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>

#include "specverify.h"
#include "sv_kernels.cuh"
#include "sv_metrics.cuh"
#include "sv_tree.cuh"
#include "sv_trunc.cuh"

namespace {

constexpr uint32_t kLiveMagic = 0x53564c56u;  // "SVLV"
constexpr uint32_t kDeadMagic = 0x53564444u;  // "SVDD"

constexpr size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct DeviceGuard {
  int prev = -1;
  bool switched = false;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) == cudaSuccess && prev != dev) {
      switched = cudaSetDevice(dev) == cudaSuccess;
    }
  }
  ~DeviceGuard() {
    if (switched) cudaSetDevice(prev);
  }
};

// ---------------------------------------------------------------------------
// Scratch: byte offsets of every piece, sized for `mb` requests, positions
// 0..max_k, every wave depth 1..max_k+1 and a grid of at most `grid` CTAs.
// ---------------------------------------------------------------------------
// The epoch-tagged completion counters come first, so that one memset of
// `tagged` bytes clears them all.
struct ScratchLayout {
  size_t lists, lcnt, blists, blcnt, res, rcnt, pos, rescnt, part, bpart, rpart, ctr, recs, rdy;
  size_t thr_t, thr_d;
  size_t list_entries, tagged, bytes;
};

// Fewest vocab blocks in one CTA's share of a wave: rows and residual
// row pairs (each CTA streams at least 16 KB of a split).
int min_span_blocks(int elem_bytes) {
  return std::max(1, sv::kMinSpanBytes / (sv::kVocabBlock * elem_bytes));
}
int min_span_res_blocks(int elem_bytes) {
  return std::max(1, sv::kMinSpanBytes / (2 * sv::kVocabBlock * elem_bytes));
}

constexpr ScratchLayout scratch_layout(size_t mb, int max_k, size_t grid) {
  size_t list_entries = 0, max_waves = 0, max_cap = 0;
  for (int d = 1; d <= max_k + 1; ++d) {
    const size_t w = (size_t)sv::wave_count(max_k, d), cap = 2 * (size_t)d * mb;
    list_entries = std::max(list_entries, w * cap);
    max_waves = std::max(max_waves, w);
    max_cap = std::max(max_cap, cap);
  }
  ScratchLayout L{};
  size_t off = 0;
  L.pos = off;
  off = align_up(off + sizeof(unsigned long long) * ((size_t)max_k + 1) * mb, 256);
  L.rescnt = off;
  off = align_up(off + sizeof(unsigned long long) * mb, 256);
  L.rdy = off;
  off = align_up(off + sizeof(unsigned long long) * max_waves * mb, 256);
  L.tagged = off;
  L.lists = off;
  off = align_up(off + sizeof(sv::Entry) * list_entries, 256);
  L.lcnt = off;
  off = align_up(off + sizeof(int) * max_waves, 256);
  L.blists = off;
  off = align_up(off + sizeof(sv::Entry) * max_waves * mb, 256);
  L.blcnt = off;
  off = align_up(off + sizeof(int) * max_waves, 256);
  L.res = off;
  off = align_up(off + sizeof(sv::ResEntry) * max_waves * mb, 256);
  L.rcnt = off;
  off = align_up(off + sizeof(int) * max_waves, 256);
  L.part = off;
  off = align_up(off + sizeof(sv::Partial) * (grid + max_cap), 256);
  L.bpart = off;
  off = align_up(off + sizeof(sv::Partial) * (grid + mb), 256);
  L.rpart = off;
  off = align_up(off + sizeof(sv::Partial) * (grid + mb), 256);
  L.ctr = off;
  off = align_up(off + sizeof(int) * sv::kCntCount, 256);
  L.recs = off;
  off = align_up(off + sizeof(sv::PosRec) * ((size_t)max_k + 1) * mb, 256);
  L.thr_t = off;
  off = align_up(off + sizeof(uint32_t) * ((size_t)max_k + 1) * mb, 256);
  L.thr_d = off;
  off = align_up(off + sizeof(uint32_t) * (size_t)max_k * mb, 256);
  L.list_entries = list_entries;
  L.bytes = off;
  return L;
}

struct Scratch {
  sv::Entry* lists;
  int* list_cnt;
  sv::Entry* blists;
  int* blist_cnt;
  sv::Partial* bpart;
  sv::ResEntry* res;
  int* res_cnt;
  unsigned long long* pos_cnt;  // epoch-tagged: must start at zero
  unsigned long long* rcnt;     // epoch-tagged: must start at zero
  sv::Partial* part;
  sv::Partial* rpart;
  int* ctr;
  sv::PosRec* recs;
  unsigned long long* rdy;  // epoch-tagged: must start at zero
  uint32_t* thr_t;          // truncated rounds: per-row thresholds of the window
  uint32_t* thr_d;
  char* tagged;             // the epoch-tagged counters above, one block
  size_t tagged_bytes;
};

Scratch scratch_at(char* b, const ScratchLayout& L) {
  Scratch s;
  s.lists = reinterpret_cast<sv::Entry*>(b + L.lists);
  s.list_cnt = reinterpret_cast<int*>(b + L.lcnt);
  s.blists = reinterpret_cast<sv::Entry*>(b + L.blists);
  s.blist_cnt = reinterpret_cast<int*>(b + L.blcnt);
  s.bpart = reinterpret_cast<sv::Partial*>(b + L.bpart);
  s.res = reinterpret_cast<sv::ResEntry*>(b + L.res);
  s.res_cnt = reinterpret_cast<int*>(b + L.rcnt);
  s.pos_cnt = reinterpret_cast<unsigned long long*>(b + L.pos);
  s.rcnt = reinterpret_cast<unsigned long long*>(b + L.rescnt);
  s.part = reinterpret_cast<sv::Partial*>(b + L.part);
  s.rpart = reinterpret_cast<sv::Partial*>(b + L.rpart);
  s.ctr = reinterpret_cast<int*>(b + L.ctr);
  s.recs = reinterpret_cast<sv::PosRec*>(b + L.recs);
  s.rdy = reinterpret_cast<unsigned long long*>(b + L.rdy);
  s.thr_t = reinterpret_cast<uint32_t*>(b + L.thr_t);
  s.thr_d = reinterpret_cast<uint32_t*>(b + L.thr_d);
  s.tagged = b;
  s.tagged_bytes = L.tagged;
  return s;
}

size_t ring_bytes() { return sizeof(uint4) * sv::kStages * sv::kStageVecs * sv::kThreads; }

template <typename E>
const void* wave_kernel(bool aligned, bool three) {
  if (three)
    return aligned ? reinterpret_cast<const void*>(sv::sv_wave<E, true, 3>)
                   : reinterpret_cast<const void*>(sv::sv_wave<E, false, 3>);
  return aligned ? reinterpret_cast<const void*>(sv::sv_wave<E, true, 2>)
                 : reinterpret_cast<const void*>(sv::sv_wave<E, false, 2>);
}

// Grids on the current device, every CTA resident at once: the wave kernels
// (aligned and scalar rows).
struct KernelShape {
  int grid_aligned, grid_scalar;    // the wave kernel built for two CTAs per SM
  int grid3_aligned, grid3_scalar;  // ... and for three
  int sms;
};

bool kernel_shape(int device, int dtype, KernelShape* out) {
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess)
    return false;
  int occ[4] = {0, 0, 0, 0};  // [three][aligned]
  for (int v = 0; v < 4; ++v) {
    const bool aligned = (v & 1) != 0, three = (v & 2) != 0;
    const void* fn = dtype == SPECVERIFY_BF16 ? wave_kernel<sv::BF16>(aligned, three)
                                              : wave_kernel<sv::F32>(aligned, three);
    const size_t sm = aligned ? ring_bytes() : 0;
    if (cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared) != cudaSuccess ||
        cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm) !=
            cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ[v], fn, sv::kBlock, sm) !=
            cudaSuccess || occ[v] < 1)
      return false;
  }
  // the builds for logits in host memory (aligned rows only): the same shared
  // memory, launched on the same grids
  const void* host_fn[2] = {
      dtype == SPECVERIFY_BF16 ? reinterpret_cast<const void*>(sv::sv_wave<sv::BF16, true, 2, false>)
                               : reinterpret_cast<const void*>(sv::sv_wave<sv::F32, true, 2, false>),
      dtype == SPECVERIFY_BF16 ? reinterpret_cast<const void*>(sv::sv_wave<sv::BF16, true, 3, false>)
                               : reinterpret_cast<const void*>(sv::sv_wave<sv::F32, true, 3, false>)};
  for (const void* fn : host_fn)
    if (cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared) != cudaSuccess ||
        cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)ring_bytes()) != cudaSuccess)
      return false;
  // the builds for truncated rounds (two CTAs per SM, the same grids)
  const void* trunc_fn = dtype == SPECVERIFY_BF16
                             ? reinterpret_cast<const void*>(sv::sv_wave<sv::BF16, true, 2, true, true>)
                             : reinterpret_cast<const void*>(sv::sv_wave<sv::F32, true, 2, true, true>);
  if (cudaFuncSetAttribute(trunc_fn, cudaFuncAttributePreferredSharedMemoryCarveout,
                           cudaSharedmemCarveoutMaxShared) != cudaSuccess ||
      cudaFuncSetAttribute(trunc_fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)ring_bytes()) != cudaSuccess)
    return false;
  out->grid_scalar = occ[0] * sms;
  out->grid_aligned = occ[1] * sms;
  out->grid3_scalar = occ[2] * sms;
  out->grid3_aligned = occ[3] * sms;
  out->sms = sms;
  return true;
}

// What a round needs besides its arguments.
struct RunConfig {
  int device, max_batch, max_k, vocab, dtype, elem_bytes;
  int depth_setting;  // 0: chosen per run from the batch size
  KernelShape shape;
  Scratch sc;
};

// Batches whose whole verify window (every row of every position) is at most
// kShallowBytes are verified in one wave of all positions: reading rows past a
// rejection costs less than a launch per position there.  Up to kPairBytes,
// two positions per wave; above, one (measured on GB300: a 613 MB window
// verifies fastest at depth 2, a 2.4 GB one at depth 1).
constexpr double kShallowBytes = 192.0 * (1 << 20);
constexpr double kPairBytes = 1024.0 * (1 << 20);

// Positions per wave for a run of `batch` requests.
int run_depth(const RunConfig& c, int batch) {
  if (c.depth_setting > 0) return c.depth_setting;
  const double window = (double)batch * (2.0 * c.max_k + 1.0) * c.vocab * c.elem_bytes;
  if (window <= kShallowBytes) return c.max_k + 1;
  return window <= kPairBytes ? std::min(2, c.max_k + 1) : 1;
}

// The wave kernel built for three CTAs per SM (up to 80 registers a thread)
// or for two (up to 128).  Measured on GB300: windows up to kShallowBytes are
// bound by latency (a few segments per CTA, decisions at the end) and run
// fastest on the most CTAs; larger windows stream best on two per SM with the
// larger register budget.
bool wave_three(const RunConfig& c, int batch) {
  const double window = (double)batch * (2.0 * c.max_k + 1.0) * c.vocab * c.elem_bytes;
  return window <= kShallowBytes;
}

bool rows_aligned(const RunConfig& c, const void* target, const void* draft) {
  return ((size_t)c.vocab * c.elem_bytes) % 16 == 0 && ((uintptr_t)target & 15u) == 0 &&
         ((uintptr_t)draft & 15u) == 0;
}

// A wave launch that may begin while the previous launch of the stream is
// finishing (programmatic dependent launch; the kernel waits for it first).
template <typename K>
cudaError_t launch_wave(K kernel, int grid, size_t smem, cudaStream_t s, const sv::Params& P) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(sv::kBlock);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, P);
}

// One round: the plan launch, then the waves (a wave with nothing to do
// returns at once), optionally bracketed by two events.
template <typename E>
int launch_round(const RunConfig& c, sv::Params P, bool aligned, cudaStream_t s,
                 cudaEvent_t ev_start, cudaEvent_t ev_stop, const sv::TruncParams* tp) {
  if (ev_start && cudaEventRecord(ev_start, s) != cudaSuccess) return SPECVERIFY_ERR_CUDA;
  sv::sv_plan<<<1, sv::kPlanThreads, 0, s>>>(P);
  const size_t smem = aligned ? ring_bytes() : 0;
  const bool trunc = P.thr_t != nullptr;  // truncated rounds: the masking build, two CTAs per SM
  const bool three = !trunc && wave_three(c, P.batch);
  const int grid = three ? (aligned ? c.shape.grid3_aligned : c.shape.grid3_scalar)
                         : (aligned ? c.shape.grid_aligned : c.shape.grid_scalar);
  for (int w = 0; w < P.n_waves; ++w) {
    P.wave = w;
    P.pos0 = std::min(w * P.depth, c.max_k + 1);
    P.pos1 = std::min((w + 1) * P.depth, c.max_k + 1);
    // logits read in place from host memory stream faster in the build
    // without the shared race best (measured on GB300: 8.3 against 14.5 ms
    // per w4 round end to end)
    const bool host = P.tee_target != nullptr;
    if (trunc) {
      // truncated round: before each wave, the thresholds of the rows that wave
      // streams (its row and bonus lists; a correction draw re-reads rows whose
      // thresholds an earlier wave's pass wrote).  A plain launch: it waits for
      // the previous wave (or the plan, which also resets the status word its
      // bad top_p values are OR-ed into), and the wave's dependent launch waits
      // for it.
      sv::TruncParams lt = *tp;
      lt.lists = P.lists + (size_t)w * P.list_cap;
      lt.list_cnt = P.list_cnt + w;
      lt.blists = P.blists + (size_t)w * P.stride;
      lt.blist_cnt = P.blist_cnt + w;
      const int tgrid = 2 * c.shape.sms;
      if (aligned)
        sv::sv_truncate<E, true><<<tgrid, sv::kTruncThreads, 0, s>>>(lt);
      else
        sv::sv_truncate<E, false><<<tgrid, sv::kTruncThreads, 0, s>>>(lt);
    }
    cudaError_t e;
    if (trunc)
      e = aligned ? launch_wave(sv::sv_wave<E, true, 2, true, true>, grid, smem, s, P)
                  : launch_wave(sv::sv_wave<E, false, 2, true, true>, grid, smem, s, P);
    else if (three)
      e = aligned ? (host ? launch_wave(sv::sv_wave<E, true, 3, false>, grid, smem, s, P)
                          : launch_wave(sv::sv_wave<E, true, 3>, grid, smem, s, P))
                  : launch_wave(sv::sv_wave<E, false, 3>, grid, smem, s, P);
    else
      e = aligned ? (host ? launch_wave(sv::sv_wave<E, true, 2, false>, grid, smem, s, P)
                          : launch_wave(sv::sv_wave<E, true, 2>, grid, smem, s, P))
                  : launch_wave(sv::sv_wave<E, false, 2>, grid, smem, s, P);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return SPECVERIFY_ERR_CUDA;
    }
  }
  if (ev_stop && cudaEventRecord(ev_stop, s) != cudaSuccess) return SPECVERIFY_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? SPECVERIFY_OK : SPECVERIFY_ERR_CUDA;
}

struct RunArgs {
  const void* target_logits;
  const void* draft_logits;
  const int32_t* draft_tokens;
  const int32_t* num_draft;
  const float* temperature;
  uint64_t seed;
  int batch, total_draft;
  int32_t* accepted_len;
  int32_t* committed_tokens;
  uint8_t* accept_flags;
  const int64_t* request_ids;
  float* p_y;
  float* q_y;
  float* u;
  int32_t* req_status;
  const float* confidence;  // trimmed runs only (NULL when total_draft == 0)
  const float* cost;
  int32_t* verified_k;
  bool trimmed = false;
  // device copies for the rows a wave streams when the logits lie in host
  // memory (specverify_run_host reading in place), or NULL
  void* tee_target = nullptr;
  void* tee_draft = nullptr;
  // truncated rounds (specverify_run_truncated): per-request top-k / top-p
  const int32_t* top_k = nullptr;
  const float* top_p = nullptr;
};

// Checks that need no device (the batch must already be in range).
int check_args(const RunConfig& c, const RunArgs& a) {
  if (a.total_draft < 0 || (long long)a.total_draft > (long long)a.batch * c.max_k)
    return SPECVERIFY_ERR_INVALID_ARG;
  if (a.batch == 0) return SPECVERIFY_OK;
  if (!a.target_logits || !a.num_draft || !a.temperature || !a.accepted_len ||
      !a.committed_tokens)
    return SPECVERIFY_ERR_INVALID_ARG;
  if (a.total_draft > 0 && (!a.draft_tokens || !a.accept_flags)) return SPECVERIFY_ERR_INVALID_ARG;
  const uintptr_t ea = (uintptr_t)(c.elem_bytes - 1);
  if (((uintptr_t)a.target_logits & ea) || ((uintptr_t)a.draft_logits & ea))
    return SPECVERIFY_ERR_INVALID_ARG;
  return SPECVERIFY_OK;
}

// The tag of the next round.  Tags run 1, 2, ..., 2^32 - 1; a counter last
// raised in an earlier round holds a smaller tag, which the next round's
// atomicMax replaces.  Before the tag would wrap to 0, every tagged counter is
// cleared on the round's stream (ordered after the rounds before it) and the
// tags restart at 1, so no stale count can outlive the wrap.
int next_epoch(uint32_t* epoch, const Scratch& sc, cudaStream_t s) {
  if (*epoch == 0xffffffffu) {
    if (cudaMemsetAsync(sc.tagged, 0, sc.tagged_bytes, s) != cudaSuccess) {
      cudaGetLastError();
      return SPECVERIFY_ERR_CUDA;
    }
    *epoch = 0u;
  }
  ++*epoch;
  return SPECVERIFY_OK;
}

// Enqueues one round (a.batch > 0, arguments checked) on the current device.
int enqueue_round(const RunConfig& c, const RunArgs& a, uint32_t epoch, cudaStream_t s,
                  cudaEvent_t ev_start, cudaEvent_t ev_stop) {
  sv::Params P;
  std::memset(&P, 0, sizeof P);
  P.target = a.target_logits;
  P.draft = a.total_draft > 0 ? a.draft_logits : nullptr;
  P.tokens = a.draft_tokens;
  P.num_draft = a.num_draft;
  P.temperature = a.temperature;
  P.request_ids = a.request_ids;
  P.key = sv::PhiloxKey{(uint32_t)(a.seed & 0xffffffffu), (uint32_t)(a.seed >> 32)};
  P.batch = a.batch;
  P.total_draft = a.total_draft;
  P.max_k = c.max_k;
  P.vocab = c.vocab;
  P.epoch = epoch;
  P.depth = run_depth(c, a.batch);
  P.n_waves = sv::wave_count(c.max_k, P.depth);
  P.list_cap = 2 * P.depth * c.max_batch;
  P.nb = (c.vocab + sv::kVocabBlock - 1) / sv::kVocabBlock;
  P.nvec = (int)((size_t)c.vocab * c.elem_bytes / 16);
  const int block_bytes = sv::kVocabBlock * c.elem_bytes;
  (void)block_bytes;
  P.min_span = min_span_blocks(c.elem_bytes);
  P.min_span_res = min_span_res_blocks(c.elem_bytes);
  P.stride = c.max_batch;
  P.accepted_len = a.accepted_len;
  P.committed = a.committed_tokens;
  P.flags = a.accept_flags;
  P.p_y = a.p_y;
  P.q_y = a.q_y;
  P.u_dbg = a.u;
  P.req_status = a.req_status;
  P.trimmed = a.trimmed ? 1 : 0;
  P.confidence = a.confidence;
  P.cost = a.cost;
  P.verified_k = a.verified_k;
  P.lists = c.sc.lists;
  P.list_cnt = c.sc.list_cnt;
  P.blists = c.sc.blists;
  P.blist_cnt = c.sc.blist_cnt;
  P.bpart = c.sc.bpart;
  P.res = c.sc.res;
  P.res_cnt = c.sc.res_cnt;
  P.pos_cnt = c.sc.pos_cnt;
  P.rcnt = c.sc.rcnt;
  P.part = c.sc.part;
  P.rpart = c.sc.rpart;
  P.ctr = c.sc.ctr;
  P.recs = c.sc.recs;
  P.rdy = c.sc.rdy;
  // the vector path needs every row on a 16-byte boundary
  const bool aligned = rows_aligned(c, a.target_logits, P.draft);
  if (aligned && a.tee_target != nullptr) {
    // waves over host-resident logits: sampled rows are copied to the device
    // as they stream, and the correction draws read those copies
    P.tee_target = static_cast<char*>(a.tee_target);
    P.tee_draft = static_cast<char*>(a.tee_draft);
  }
  sv::TruncParams tp;
  std::memset(&tp, 0, sizeof tp);
  if (a.top_k != nullptr) {
    P.thr_t = c.sc.thr_t;
    P.thr_d = c.sc.thr_d;
    tp.target_in = a.target_logits;
    tp.draft_in = P.draft;
    tp.num_draft = a.num_draft;
    tp.temperature = a.temperature;
    tp.top_k = a.top_k;
    tp.top_p = a.top_p;
    tp.batch = a.batch;
    tp.total_draft = a.total_draft;
    tp.vocab = c.vocab;
    tp.status = c.sc.ctr + sv::kCntStatus;
    tp.thr_target = c.sc.thr_t;
    tp.thr_draft = c.sc.thr_d;
  }
  const sv::TruncParams* tpp = a.top_k != nullptr ? &tp : nullptr;
  return c.dtype == SPECVERIFY_BF16
             ? launch_round<sv::BF16>(c, P, aligned, s, ev_start, ev_stop, tpp)
             : launch_round<sv::F32>(c, P, aligned, s, ev_start, ev_stop, tpp);
}

// ---------------------------------------------------------------------------
// The static arena of specverify_run_static: a fixed-size device array, set up
// on the first call on each device (its address, the kernel grids, zeroed
// counters).  It serves callers that may not allocate device memory, such as a
// server that has reserved the GPU's memory for its own pool; every GPU that
// loads the library holds it until the process exits, and every call shares it
// (calls that overlap in time race on it).
// ---------------------------------------------------------------------------
constexpr int kStaticMaxDevices = 64;
constexpr size_t kStaticGrid = 1024;  // CTAs a wave of the static path may use
constexpr ScratchLayout kStaticLayout =
    scratch_layout(SPECVERIFY_STATIC_MAX_BATCH, SPECVERIFY_STATIC_MAX_K, kStaticGrid);

struct StaticDevice {
  bool ready;
  char* base;
  KernelShape shape[2];  // per dtype
  uint32_t epoch;
};

StaticDevice g_static_dev[kStaticMaxDevices];
std::mutex g_static_mu;

}  // namespace

// The arena (file scope, static storage on the device).
static __device__ __align__(256) unsigned char g_static_scratch[kStaticLayout.bytes];

struct specverify_ctx {
  uint32_t magic;
  RunConfig cfg;
  void* scratch;
  uint32_t epoch;
  // staging for specverify_run_host
  int host_reads;       // SPECVERIFY_HOST_READS_*
  int last_host_place;  // the last specverify_run_host: 1 read in place, 0 staged, -1 none
  void* stage;
  char* st_target;
  char* st_draft;
  int32_t* st_tokens;
  int32_t* st_num_draft;
  float* st_temperature;
  int32_t* st_accepted;
  int32_t* st_committed;
  uint8_t* st_flags;
  cudaStream_t last_stream;
  bool last_run_empty;
  // optional timing events around a round's launches
  int n_events;
  unsigned long long run_counter;
  cudaEvent_t ev_start[64];
  cudaEvent_t ev_stop[64];
};

// A greedy tree verifier: scratch for the prefix offsets and the status words.
struct specverify_tree_ctx {
  uint32_t magic;
  int device, max_batch, max_nodes, vocab, dtype, elem_bytes;
  int sms;  // one walking CTA per SM at most
  void* scratch;
  int* t_off;
  int* n_off;
  int* ctr;
  cudaStream_t last_stream;
  bool last_run_empty;
};

static int check_tree(specverify_tree_t h) {
  if (h == nullptr) return SPECVERIFY_ERR_INVALID_ARG;
  if (h->magic == kDeadMagic) return SPECVERIFY_ERR_DESTROYED;
  if (h->magic != kLiveMagic) return SPECVERIFY_ERR_INVALID_ARG;
  return SPECVERIFY_OK;
}

static int check_handle(specverify_t h) {
  if (h == nullptr) return SPECVERIFY_ERR_INVALID_ARG;
  if (h->magic == kDeadMagic) return SPECVERIFY_ERR_DESTROYED;
  if (h->magic != kLiveMagic) return SPECVERIFY_ERR_INVALID_ARG;
  return SPECVERIFY_OK;
}

static int run_impl(specverify_t h, const RunArgs& a, void* stream) {
  int rc = check_handle(h);
  if (rc != SPECVERIFY_OK) return rc;
  if (a.batch < 0 || a.batch > h->cfg.max_batch) return SPECVERIFY_ERR_INVALID_ARG;
  rc = check_args(h->cfg, a);
  if (rc != SPECVERIFY_OK) return rc;
  if (a.batch == 0) {
    h->last_run_empty = true;
    return SPECVERIFY_OK;
  }
  DeviceGuard guard(h->cfg.device);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int slot = h->n_events > 0 ? (int)(h->run_counter % (unsigned long long)h->n_events) : -1;
  h->run_counter++;
  rc = next_epoch(&h->epoch, h->cfg.sc, s);
  if (rc != SPECVERIFY_OK) return rc;
  rc = enqueue_round(h->cfg, a, h->epoch, s, slot >= 0 ? h->ev_start[slot] : nullptr,
                     slot >= 0 ? h->ev_stop[slot] : nullptr);
  h->last_stream = s;
  h->last_run_empty = false;
  return rc;
}

extern "C" {

int specverify_create_ex(specverify_t* out, int device, int max_batch, int max_k, int vocab,
                         int dtype, unsigned flags) {
  if (out == nullptr) return SPECVERIFY_ERR_INVALID_ARG;
  *out = nullptr;
  if (dtype != SPECVERIFY_F32 && dtype != SPECVERIFY_BF16) return SPECVERIFY_ERR_DTYPE;
  if (max_batch < 1 || max_batch > sv::kMaxBatch || max_k < 0 || max_k > sv::kMaxK ||
      vocab < 1 || vocab > (1 << 30))
    return SPECVERIFY_ERR_INVALID_ARG;
  if ((flags & ~(unsigned)SPECVERIFY_CREATE_HOST_STAGING) != 0u) return SPECVERIFY_ERR_INVALID_ARG;

  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess || device < 0 || device >= ndev) {
    cudaGetLastError();
    return SPECVERIFY_ERR_CUDA;
  }
  DeviceGuard guard(device);

  specverify_ctx* h = new (std::nothrow) specverify_ctx();
  if (!h) return SPECVERIFY_ERR_CUDA;
  RunConfig& c = h->cfg;
  c.device = device;
  c.max_batch = max_batch;
  c.max_k = max_k;
  c.vocab = vocab;
  c.dtype = dtype;
  c.elem_bytes = dtype == SPECVERIFY_BF16 ? 2 : 4;
  c.depth_setting = 0;
  h->last_stream = nullptr;
  h->last_run_empty = true;
  h->n_events = 0;
  h->host_reads = SPECVERIFY_HOST_READS_AUTO;
  h->last_host_place = -1;
  h->run_counter = 0;
  h->epoch = 0u;
  h->stage = nullptr;
  if (!kernel_shape(device, dtype, &c.shape)) {
    cudaGetLastError();
    delete h;
    return SPECVERIFY_ERR_CUDA;
  }
  const size_t grid_all = (size_t)std::max({c.shape.grid_aligned, c.shape.grid_scalar,
                                             c.shape.grid3_aligned, c.shape.grid3_scalar});
  const ScratchLayout L = scratch_layout((size_t)max_batch, max_k, grid_all);
  if (cudaMalloc(&h->scratch, L.bytes) != cudaSuccess) {
    cudaGetLastError();
    delete h;
    return SPECVERIFY_ERR_CUDA;
  }
  if (cudaMemset(h->scratch, 0, L.bytes) != cudaSuccess) {
    cudaGetLastError();
    cudaFree(h->scratch);
    delete h;
    return SPECVERIFY_ERR_CUDA;
  }
  c.sc = scratch_at(static_cast<char*>(h->scratch), L);

  if (flags & SPECVERIFY_CREATE_HOST_STAGING) {
    size_t so = 0;
    auto scarve = [&](size_t bytes) {
      const size_t o = so;
      so = align_up(so + bytes, 256);
      return o;
    };
    const size_t row_bytes = (size_t)vocab * c.elem_bytes;
    const size_t rows_t = (size_t)max_batch * (max_k + 1), rows_d = (size_t)max_batch * max_k;
    const size_t s_t = scarve(rows_t * row_bytes);
    const size_t s_d = scarve(rows_d * row_bytes);
    const size_t s_tok = scarve(sizeof(int32_t) * rows_d);
    const size_t s_nd = scarve(sizeof(int32_t) * max_batch);
    const size_t s_tmp = scarve(sizeof(float) * max_batch);
    const size_t s_acc = scarve(sizeof(int32_t) * max_batch);
    const size_t s_com = scarve(sizeof(int32_t) * rows_t);
    const size_t s_flg = scarve(rows_d + 1);
    if (cudaMalloc(&h->stage, so) != cudaSuccess) {
      cudaGetLastError();
      cudaFree(h->scratch);
      delete h;
      return SPECVERIFY_ERR_CUDA;
    }
    char* sb = static_cast<char*>(h->stage);
    h->st_target = sb + s_t;
    h->st_draft = sb + s_d;
    h->st_tokens = reinterpret_cast<int32_t*>(sb + s_tok);
    h->st_num_draft = reinterpret_cast<int32_t*>(sb + s_nd);
    h->st_temperature = reinterpret_cast<float*>(sb + s_tmp);
    h->st_accepted = reinterpret_cast<int32_t*>(sb + s_acc);
    h->st_committed = reinterpret_cast<int32_t*>(sb + s_com);
    h->st_flags = reinterpret_cast<uint8_t*>(sb + s_flg);
  }
  h->magic = kLiveMagic;
  *out = h;
  return SPECVERIFY_OK;
}

int specverify_create(specverify_t* out, int device, int max_batch, int max_k, int vocab,
                      int dtype) {
  return specverify_create_ex(out, device, max_batch, max_k, vocab, dtype, 0u);
}

int specverify_run(specverify_t h, const void* target_logits, const void* draft_logits,
                   const int32_t* draft_tokens, const int32_t* num_draft,
                   const float* temperature, uint64_t seed, int batch, int total_draft,
                   int32_t* accepted_len, int32_t* committed_tokens, uint8_t* accept_flags,
                   void* stream) {
  const RunArgs a{target_logits, draft_logits, draft_tokens, num_draft, temperature, seed,
                  batch, total_draft, accepted_len, committed_tokens, accept_flags,
                  nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr};
  return run_impl(h, a, stream);
}

int specverify_run_ex(specverify_t h, const void* target_logits, const void* draft_logits,
                      const int32_t* draft_tokens, const int32_t* num_draft,
                      const float* temperature, uint64_t seed, int batch, int total_draft,
                      int32_t* accepted_len, int32_t* committed_tokens, uint8_t* accept_flags,
                      const int64_t* request_ids, float* p_y, float* q_y, float* u,
                      int32_t* req_status, void* stream) {
  const RunArgs a{target_logits, draft_logits, draft_tokens, num_draft, temperature, seed,
                  batch, total_draft, accepted_len, committed_tokens, accept_flags,
                  request_ids, p_y, q_y, u, req_status, nullptr, nullptr, nullptr};
  return run_impl(h, a, stream);
}

int specverify_run_truncated(specverify_t h, const void* target_logits,
                             const void* draft_logits, const int32_t* draft_tokens,
                             const int32_t* num_draft, const float* temperature,
                             const int32_t* top_k, const float* top_p, uint64_t seed, int batch,
                             int total_draft, int32_t* accepted_len, int32_t* committed_tokens,
                             uint8_t* accept_flags, void* stream) {
  if (batch > 0 && (top_k == nullptr || top_p == nullptr)) return SPECVERIFY_ERR_INVALID_ARG;
  RunArgs a{target_logits, draft_logits, draft_tokens, num_draft, temperature, seed,
            batch, total_draft, accepted_len, committed_tokens, accept_flags,
            nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr};
  a.top_k = top_k;
  a.top_p = top_p;
  return run_impl(h, a, stream);
}

int specverify_run_trimmed(specverify_t h, const void* target_logits, const void* draft_logits,
                           const int32_t* draft_tokens, const int32_t* window,
                           const float* confidence, const float* cost, const float* temperature,
                           uint64_t seed, int batch, int total_draft, int32_t* verified_k,
                           int32_t* accepted_len, int32_t* committed_tokens,
                           uint8_t* accept_flags, float* p_y, float* q_y, float* u,
                           int32_t* req_status, void* stream) {
  if (batch > 0 && (cost == nullptr || verified_k == nullptr ||
                    (total_draft > 0 && confidence == nullptr)))
    return SPECVERIFY_ERR_INVALID_ARG;
  RunArgs a{target_logits, draft_logits, draft_tokens, window, temperature, seed,
            batch, total_draft, accepted_len, committed_tokens, accept_flags,
            nullptr, p_y, q_y, u, req_status, confidence, cost, verified_k};
  a.trimmed = true;
  return run_impl(h, a, stream);
}

// The device address of host memory that is pinned and mapped into the
// device's address space (cudaHostAlloc, or cudaHostRegister with mapping),
// if `p` lies in such memory.
static bool mapped_host(const void* p, const void** dev) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  if (at.type != cudaMemoryTypeHost || at.devicePointer == nullptr) return false;
  *dev = at.devicePointer;
  return true;
}

int specverify_run_host(specverify_t h, const void* target_logits, const void* draft_logits,
                        const int32_t* draft_tokens, const int32_t* num_draft,
                        const float* temperature, uint64_t seed, int batch, int total_draft,
                        int32_t* accepted_len, int32_t* committed_tokens,
                        uint8_t* accept_flags, void* stream) {
  int rc = check_handle(h);
  if (rc != SPECVERIFY_OK) return rc;
  if (h->stage == nullptr) return SPECVERIFY_ERR_NO_STAGING;
  const RunConfig& c = h->cfg;
  if (batch < 0 || batch > c.max_batch) return SPECVERIFY_ERR_INVALID_ARG;
  if (total_draft < 0 || (long long)total_draft > (long long)batch * c.max_k)
    return SPECVERIFY_ERR_INVALID_ARG;
  if (batch == 0) return SPECVERIFY_OK;
  if (!target_logits || !num_draft || !temperature || !accepted_len || !committed_tokens)
    return SPECVERIFY_ERR_INVALID_ARG;
  if (total_draft > 0 && (!draft_tokens || !accept_flags)) return SPECVERIFY_ERR_INVALID_ARG;

  DeviceGuard guard(c.device);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const size_t row_bytes = (size_t)c.vocab * c.elem_bytes;
  bool ok = true;
  auto h2d = [&](void* dst, const void* src, size_t n) {
    if (n && ok) ok = cudaMemcpyAsync(dst, src, n, cudaMemcpyHostToDevice, s) == cudaSuccess;
  };
  auto d2h = [&](void* dst, const void* src, size_t n) {
    if (n && ok) ok = cudaMemcpyAsync(dst, src, n, cudaMemcpyDeviceToHost, s) == cudaSuccess;
  };
  const bool has_draft = draft_logits != nullptr && total_draft > 0;
  // Logits in pinned host memory that the device maps are read where they lie
  // (over NVLink-C2C on Grace-Blackwell): only the rows the round needs cross
  // to the GPU.  Anything else is copied into the staging buffers first.
  const void* dev_target = nullptr;
  const void* dev_draft = nullptr;
  const bool in_place = h->host_reads == SPECVERIFY_HOST_READS_AUTO &&
                        mapped_host(target_logits, &dev_target) &&
                        (!has_draft || mapped_host(draft_logits, &dev_draft));
  h->last_host_place = in_place ? 1 : 0;
  if (!in_place) {
    h2d(h->st_target, target_logits, (size_t)(batch + total_draft) * row_bytes);
    if (has_draft) h2d(h->st_draft, draft_logits, (size_t)total_draft * row_bytes);
    dev_target = h->st_target;
    dev_draft = h->st_draft;
  }
  h2d(h->st_tokens, draft_tokens, sizeof(int32_t) * (size_t)total_draft);
  h2d(h->st_num_draft, num_draft, sizeof(int32_t) * (size_t)batch);
  h2d(h->st_temperature, temperature, sizeof(float) * (size_t)batch);
  if (!ok) {
    cudaGetLastError();
    return SPECVERIFY_ERR_CUDA;
  }
  RunArgs a{dev_target, has_draft ? dev_draft : nullptr, h->st_tokens,
            h->st_num_draft, h->st_temperature, seed, batch, total_draft,
            h->st_accepted, h->st_committed, h->st_flags,
            nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr};
  if (in_place && has_draft) {
    a.tee_target = h->st_target;
    a.tee_draft = h->st_draft;
  }
  rc = run_impl(h, a, stream);
  if (rc != SPECVERIFY_OK) return rc;
  d2h(accepted_len, h->st_accepted, sizeof(int32_t) * (size_t)batch);
  d2h(committed_tokens, h->st_committed, sizeof(int32_t) * (size_t)batch * (c.max_k + 1));
  d2h(accept_flags, h->st_flags, (size_t)total_draft);
  if (ok) ok = cudaStreamSynchronize(s) == cudaSuccess;
  if (!ok) {
    cudaGetLastError();
    return SPECVERIFY_ERR_CUDA;
  }
  return SPECVERIFY_OK;
}

int specverify_run_static(int device, int max_k, int vocab, int dtype,
                          const void* target_logits, const void* draft_logits,
                          const int32_t* draft_tokens, const int32_t* num_draft,
                          const float* temperature, uint64_t seed, int batch, int total_draft,
                          int32_t* accepted_len, int32_t* committed_tokens,
                          uint8_t* accept_flags, void* stream) {
  if (dtype != SPECVERIFY_F32 && dtype != SPECVERIFY_BF16) return SPECVERIFY_ERR_DTYPE;
  if (device < 0 || device >= kStaticMaxDevices || vocab < 1 || vocab > (1 << 30) || batch < 0 ||
      max_k < 0)
    return SPECVERIFY_ERR_INVALID_ARG;
  if (batch > SPECVERIFY_STATIC_MAX_BATCH || max_k > SPECVERIFY_STATIC_MAX_K)
    return SPECVERIFY_ERR_TOO_LARGE;
  RunConfig c;
  c.device = device;
  c.max_batch = SPECVERIFY_STATIC_MAX_BATCH;
  c.max_k = max_k;
  c.vocab = vocab;
  c.dtype = dtype;
  c.elem_bytes = dtype == SPECVERIFY_BF16 ? 2 : 4;
  c.depth_setting = 0;
  const RunArgs a{target_logits, draft_logits, draft_tokens, num_draft, temperature, seed,
                  batch, total_draft, accepted_len, committed_tokens, accept_flags,
                  nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr};
  int rc = check_args(c, a);
  if (rc != SPECVERIFY_OK || batch == 0) return rc;

  std::lock_guard<std::mutex> lock(g_static_mu);
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess || device >= ndev) {
    cudaGetLastError();
    return SPECVERIFY_ERR_CUDA;
  }
  DeviceGuard guard(device);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  StaticDevice& sd = g_static_dev[device];
  if (!sd.ready) {
    // set-up, once per device: the arena's address, the kernel grids, and
    // zero counters (every epoch-tagged counter must start at zero)
    void* base = nullptr;
    if (cudaGetSymbolAddress(&base, g_static_scratch) != cudaSuccess || base == nullptr ||
        !kernel_shape(device, SPECVERIFY_F32, &sd.shape[SPECVERIFY_F32]) ||
        !kernel_shape(device, SPECVERIFY_BF16, &sd.shape[SPECVERIFY_BF16]) ||
        cudaMemsetAsync(base, 0, kStaticLayout.bytes, s) != cudaSuccess) {
      cudaGetLastError();
      return SPECVERIFY_ERR_CUDA;
    }
    for (int t = 0; t < 2; ++t) {
      sd.shape[t].grid_aligned = std::min<int>(sd.shape[t].grid_aligned, (int)kStaticGrid);
      sd.shape[t].grid_scalar = std::min<int>(sd.shape[t].grid_scalar, (int)kStaticGrid);
      sd.shape[t].grid3_aligned = std::min<int>(sd.shape[t].grid3_aligned, (int)kStaticGrid);
      sd.shape[t].grid3_scalar = std::min<int>(sd.shape[t].grid3_scalar, (int)kStaticGrid);
    }
    sd.base = static_cast<char*>(base);
    sd.epoch = 0u;
    sd.ready = true;
  }
  c.shape = sd.shape[dtype];
  c.sc = scratch_at(sd.base, kStaticLayout);
  rc = next_epoch(&sd.epoch, c.sc, s);
  if (rc != SPECVERIFY_OK) return rc;
  return enqueue_round(c, a, sd.epoch, s, nullptr, nullptr);
}

int specverify_debug_set_epoch(specverify_t h, uint32_t epoch) {
  int rc = check_handle(h);
  if (rc != SPECVERIFY_OK) return rc;
  DeviceGuard guard(h->cfg.device);
  if (cudaDeviceSynchronize() != cudaSuccess ||
      cudaMemset(h->cfg.sc.tagged, 0, h->cfg.sc.tagged_bytes) != cudaSuccess ||
      cudaDeviceSynchronize() != cudaSuccess) {
    cudaGetLastError();
    return SPECVERIFY_ERR_CUDA;
  }
  h->epoch = epoch;
  return SPECVERIFY_OK;
}

int specverify_static_debug_set_epoch(int device, uint32_t epoch) {
  if (device < 0 || device >= kStaticMaxDevices) return SPECVERIFY_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_static_mu);
  StaticDevice& sd = g_static_dev[device];
  if (!sd.ready) return SPECVERIFY_ERR_INVALID_ARG;
  DeviceGuard guard(device);
  const Scratch sc = scratch_at(sd.base, kStaticLayout);
  if (cudaDeviceSynchronize() != cudaSuccess ||
      cudaMemset(sc.tagged, 0, sc.tagged_bytes) != cudaSuccess ||
      cudaDeviceSynchronize() != cudaSuccess) {
    cudaGetLastError();
    return SPECVERIFY_ERR_CUDA;
  }
  sd.epoch = epoch;
  return SPECVERIFY_OK;
}

int specverify_status(specverify_t h, int32_t* status_out) {
  int rc = check_handle(h);
  if (rc != SPECVERIFY_OK) return rc;
  if (status_out == nullptr) return SPECVERIFY_ERR_INVALID_ARG;
  DeviceGuard guard(h->cfg.device);
  int32_t st = 0;
  if (h->last_run_empty) {
    *status_out = 0;
    return SPECVERIFY_OK;
  }
  if (cudaStreamSynchronize(h->last_stream) != cudaSuccess ||
      cudaMemcpy(&st, h->cfg.sc.ctr + sv::kCntStatus, sizeof st, cudaMemcpyDeviceToHost) !=
          cudaSuccess) {
    cudaGetLastError();
    return SPECVERIFY_ERR_CUDA;
  }
  *status_out = st;
  return SPECVERIFY_OK;
}

int specverify_set_timing_events(specverify_t h, int n, void* const* start_events,
                                 void* const* stop_events) {
  int rc = check_handle(h);
  if (rc != SPECVERIFY_OK) return rc;
  if (n < 0 || n > 64) return SPECVERIFY_ERR_INVALID_ARG;
  if (n > 0 && (!start_events || !stop_events)) return SPECVERIFY_ERR_INVALID_ARG;
  for (int i = 0; i < n; ++i) {
    if (!start_events[i] || !stop_events[i]) return SPECVERIFY_ERR_INVALID_ARG;
    h->ev_start[i] = reinterpret_cast<cudaEvent_t>(start_events[i]);
    h->ev_stop[i] = reinterpret_cast<cudaEvent_t>(stop_events[i]);
  }
  h->n_events = n;
  h->run_counter = 0;
  return SPECVERIFY_OK;
}

int specverify_set_depth(specverify_t h, int depth) {
  int rc = check_handle(h);
  if (rc != SPECVERIFY_OK) return rc;
  if (depth < 0 || depth > h->cfg.max_k + 1) return SPECVERIFY_ERR_INVALID_ARG;
  h->cfg.depth_setting = depth;
  return SPECVERIFY_OK;
}

int specverify_set_host_reads(specverify_t h, int mode) {
  int rc = check_handle(h);
  if (rc != SPECVERIFY_OK) return rc;
  if (mode != SPECVERIFY_HOST_READS_AUTO && mode != SPECVERIFY_HOST_READS_STAGE)
    return SPECVERIFY_ERR_INVALID_ARG;
  h->host_reads = mode;
  return SPECVERIFY_OK;
}

int specverify_wave_depth(specverify_t h, int batch, int* depth_out) {
  int rc = check_handle(h);
  if (rc != SPECVERIFY_OK) return rc;
  if (depth_out == nullptr || batch < 0 || batch > h->cfg.max_batch)
    return SPECVERIFY_ERR_INVALID_ARG;
  *depth_out = run_depth(h->cfg, batch);
  return SPECVERIFY_OK;
}

int specverify_last_host_reads(specverify_t h, int* in_place_out) {
  int rc = check_handle(h);
  if (rc != SPECVERIFY_OK) return rc;
  if (in_place_out == nullptr) return SPECVERIFY_ERR_INVALID_ARG;
  *in_place_out = h->last_host_place;
  return SPECVERIFY_OK;
}

int specverify_set_schedule(specverify_t h, int schedule) {
  int rc = check_handle(h);
  if (rc != SPECVERIFY_OK) return rc;
  if (schedule != SPECVERIFY_SCHEDULE_AUTO && schedule != SPECVERIFY_SCHEDULE_WAVES)
    return SPECVERIFY_ERR_INVALID_ARG;
  return SPECVERIFY_OK;
}

int specverify_launches_per_run(specverify_t h, int batch, int* launches_out) {
  int rc = check_handle(h);
  if (rc != SPECVERIFY_OK) return rc;
  if (launches_out == nullptr || batch < 0 || batch > h->cfg.max_batch)
    return SPECVERIFY_ERR_INVALID_ARG;
  *launches_out = batch == 0 ? 0 : 1 + sv::wave_count(h->cfg.max_k, run_depth(h->cfg, batch));
  return SPECVERIFY_OK;
}

int specverify_destroy(specverify_t h) {
  int rc = check_handle(h);
  if (rc != SPECVERIFY_OK) return rc;
  DeviceGuard guard(h->cfg.device);
  // the small host record is kept (marked dead) so later calls report
  // SPECVERIFY_ERR_DESTROYED instead of touching freed memory
  h->magic = kDeadMagic;
  bool ok = cudaDeviceSynchronize() == cudaSuccess;
  if (h->scratch) ok = (cudaFree(h->scratch) == cudaSuccess) && ok;
  if (h->stage) ok = (cudaFree(h->stage) == cudaSuccess) && ok;
  h->scratch = nullptr;
  h->stage = nullptr;
  if (!ok) {
    cudaGetLastError();
    return SPECVERIFY_ERR_CUDA;
  }
  return SPECVERIFY_OK;
}

int specverify_metrics(const int32_t* accepted_len, const int32_t* num_draft, int batch,
                       int max_k, uint64_t* hist, uint64_t* proposed, uint64_t* accepted,
                       double* summary, void* stream) {
  if (batch < 0 || max_k < 0 || max_k > sv::kMetricsMaxK || hist == nullptr ||
      (max_k > 0 && (proposed == nullptr || accepted == nullptr)))
    return SPECVERIFY_ERR_INVALID_ARG;
  if (batch > 0 && (accepted_len == nullptr || num_draft == nullptr))
    return SPECVERIFY_ERR_INVALID_ARG;
  if (batch == 0 && summary == nullptr) return SPECVERIFY_OK;
  sv::sv_metrics<<<1, sv::kMetricsThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      accepted_len, num_draft, batch, max_k, reinterpret_cast<unsigned long long*>(hist),
      reinterpret_cast<unsigned long long*>(proposed),
      reinterpret_cast<unsigned long long*>(accepted), summary);
  if (cudaGetLastError() != cudaSuccess) return SPECVERIFY_ERR_CUDA;
  return SPECVERIFY_OK;
}

int specverify_tree_create(specverify_tree_t* out, int device, int max_batch, int max_nodes,
                           int vocab, int dtype) {
  if (out == nullptr) return SPECVERIFY_ERR_INVALID_ARG;
  *out = nullptr;
  if (dtype != SPECVERIFY_F32 && dtype != SPECVERIFY_BF16) return SPECVERIFY_ERR_DTYPE;
  if (max_batch < 1 || max_batch > sv::kMaxBatch || max_nodes < 0 ||
      max_nodes > sv::kTreeMaxNodes || vocab < 1 || vocab > (1 << 30))
    return SPECVERIFY_ERR_INVALID_ARG;
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess || device < 0 || device >= ndev) {
    cudaGetLastError();
    return SPECVERIFY_ERR_CUDA;
  }
  DeviceGuard guard(device);
  specverify_tree_ctx* h = new (std::nothrow) specverify_tree_ctx();
  if (!h) return SPECVERIFY_ERR_CUDA;
  h->device = device;
  h->max_batch = max_batch;
  h->max_nodes = max_nodes;
  h->vocab = vocab;
  h->dtype = dtype;
  h->elem_bytes = dtype == SPECVERIFY_BF16 ? 2 : 4;
  h->last_stream = nullptr;
  h->last_run_empty = true;
  if (cudaDeviceGetAttribute(&h->sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess ||
      h->sms < 1) {
    cudaGetLastError();
    delete h;
    return SPECVERIFY_ERR_CUDA;
  }
  size_t off = 0;
  const size_t o_t = off;
  off = align_up(off + sizeof(int) * ((size_t)max_batch + 1), 256);
  const size_t o_n = off;
  off = align_up(off + sizeof(int) * ((size_t)max_batch + 1), 256);
  const size_t o_c = off;
  off = align_up(off + sizeof(int) * 4, 256);
  if (cudaMalloc(&h->scratch, off) != cudaSuccess ||
      cudaMemset(h->scratch, 0, off) != cudaSuccess) {
    cudaGetLastError();
    if (h->scratch) cudaFree(h->scratch);
    delete h;
    return SPECVERIFY_ERR_CUDA;
  }
  char* b = static_cast<char*>(h->scratch);
  h->t_off = reinterpret_cast<int*>(b + o_t);
  h->n_off = reinterpret_cast<int*>(b + o_n);
  h->ctr = reinterpret_cast<int*>(b + o_c);
  h->magic = kLiveMagic;
  *out = h;
  return SPECVERIFY_OK;
}

int specverify_tree_run(specverify_tree_t h, const void* target_logits, const int32_t* num_nodes,
                        const int32_t* parent, const int32_t* node_tokens, int batch,
                        int total_nodes, int32_t* accepted_len, int32_t* path,
                        int32_t* committed, int32_t* req_status, void* stream) {
  int rc = check_tree(h);
  if (rc != SPECVERIFY_OK) return rc;
  if (batch < 0 || batch > h->max_batch || total_nodes < 0 ||
      (long long)total_nodes > (long long)batch * h->max_nodes)
    return SPECVERIFY_ERR_INVALID_ARG;
  if (batch == 0) {
    h->last_run_empty = true;
    return SPECVERIFY_OK;
  }
  if (!target_logits || !num_nodes || !accepted_len || !committed ||
      (h->max_nodes > 0 && !path) || (total_nodes > 0 && (!parent || !node_tokens)))
    return SPECVERIFY_ERR_INVALID_ARG;
  if ((uintptr_t)target_logits & (uintptr_t)(h->elem_bytes - 1)) return SPECVERIFY_ERR_INVALID_ARG;
  DeviceGuard guard(h->device);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  sv::TreeParams P;
  std::memset(&P, 0, sizeof P);
  P.target = target_logits;
  P.num_nodes = num_nodes;
  P.parent = parent;
  P.tokens = node_tokens;
  P.batch = batch;
  P.total_nodes = total_nodes;
  P.max_nodes = h->max_nodes;
  P.vocab = h->vocab;
  P.nvec = (int)((size_t)h->vocab * h->elem_bytes / 16);
  P.rows = batch + total_nodes;
  P.accepted_len = accepted_len;
  P.path = path;
  P.committed = committed;
  P.req_status = req_status;
  P.t_off = h->t_off;
  P.n_off = h->n_off;
  P.ctr = h->ctr;
  const bool aligned = ((size_t)h->vocab * h->elem_bytes) % 16 == 0 &&
                       ((uintptr_t)target_logits & 15u) == 0;
  // a cluster of cs CTAs per tree: the largest power of two up to 8 that still
  // lets every tree's cluster be resident at once (two CTAs per SM)
  const int resident = 2 * h->sms;
  int cs = 1;
  while (cs < sv::kPathMaxCluster && (long long)batch * cs * 2 <= resident) cs *= 2;
  const int clusters = std::max(1, std::min(batch, resident / cs));
  sv::sv_tree_plan<<<1, sv::kPlanThreads, 0, s>>>(P);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(clusters * cs));
  cfg.blockDim = dim3(sv::kPathThreads);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e;
  if (h->dtype == SPECVERIFY_BF16)
    e = aligned ? cudaLaunchKernelEx(&cfg, sv::sv_tree_path<sv::BF16, true>, P)
                : cudaLaunchKernelEx(&cfg, sv::sv_tree_path<sv::BF16, false>, P);
  else
    e = aligned ? cudaLaunchKernelEx(&cfg, sv::sv_tree_path<sv::F32, true>, P)
                : cudaLaunchKernelEx(&cfg, sv::sv_tree_path<sv::F32, false>, P);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return SPECVERIFY_ERR_CUDA;
  }
  h->last_stream = s;
  h->last_run_empty = false;
  return cudaGetLastError() == cudaSuccess ? SPECVERIFY_OK : SPECVERIFY_ERR_CUDA;
}

int specverify_tree_status(specverify_tree_t h, int32_t* status_out) {
  int rc = check_tree(h);
  if (rc != SPECVERIFY_OK) return rc;
  if (status_out == nullptr) return SPECVERIFY_ERR_INVALID_ARG;
  if (h->last_run_empty) {
    *status_out = 0;
    return SPECVERIFY_OK;
  }
  DeviceGuard guard(h->device);
  int32_t st = 0;
  if (cudaStreamSynchronize(h->last_stream) != cudaSuccess ||
      cudaMemcpy(&st, h->ctr, sizeof st, cudaMemcpyDeviceToHost) != cudaSuccess) {
    cudaGetLastError();
    return SPECVERIFY_ERR_CUDA;
  }
  *status_out = st;
  return SPECVERIFY_OK;
}

int specverify_tree_destroy(specverify_tree_t h) {
  int rc = check_tree(h);
  if (rc != SPECVERIFY_OK) return rc;
  DeviceGuard guard(h->device);
  h->magic = kDeadMagic;
  bool ok = cudaDeviceSynchronize() == cudaSuccess;
  if (h->scratch) ok = (cudaFree(h->scratch) == cudaSuccess) && ok;
  h->scratch = nullptr;
  if (!ok) {
    cudaGetLastError();
    return SPECVERIFY_ERR_CUDA;
  }
  return SPECVERIFY_OK;
}

int specverify_truncate(int dtype, int vocab, const void* target_in, const void* draft_in,
                        const int32_t* num_draft, const float* temperature, const int32_t* top_k,
                        const float* top_p, int batch, int total_draft, void* target_out,
                        void* draft_out, int32_t* status, void* stream) {
  if (dtype != SPECVERIFY_F32 && dtype != SPECVERIFY_BF16) return SPECVERIFY_ERR_DTYPE;
  if (vocab < 1 || vocab > (1 << 30) || batch < 0 || total_draft < 0)
    return SPECVERIFY_ERR_INVALID_ARG;
  if (batch == 0) return SPECVERIFY_OK;
  if (!target_in || !target_out || !num_draft || !temperature || !top_k || !top_p ||
      (draft_in != nullptr) != (draft_out != nullptr))
    return SPECVERIFY_ERR_INVALID_ARG;
  const int es = dtype == SPECVERIFY_BF16 ? 2 : 4;
  const uintptr_t mask = 15u;
  const bool aligned = ((size_t)vocab * es) % 16 == 0 && ((uintptr_t)target_in & mask) == 0 &&
                       ((uintptr_t)target_out & mask) == 0 &&
                       ((uintptr_t)draft_in & mask) == 0 && ((uintptr_t)draft_out & mask) == 0;
  if (((uintptr_t)target_in | (uintptr_t)target_out | (uintptr_t)draft_in |
       (uintptr_t)draft_out) & (uintptr_t)(es - 1))
    return SPECVERIFY_ERR_INVALID_ARG;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return SPECVERIFY_ERR_CUDA;
  }
  sv::TruncParams P{};  // every field set, the threshold outputs NULL (copy mode)
  P.target_in = target_in;
  P.draft_in = total_draft > 0 ? draft_in : nullptr;
  P.target_out = target_out;
  P.draft_out = total_draft > 0 ? draft_out : nullptr;
  P.num_draft = num_draft;
  P.temperature = temperature;
  P.top_k = top_k;
  P.top_p = top_p;
  P.batch = batch;
  P.total_draft = total_draft;
  P.vocab = vocab;
  P.status = status;
  P.thr_target = nullptr;
  P.thr_draft = nullptr;
  // two CTAs per SM, a row each at a time: the rows in flight stay in L2 across
  // the passes, and one CTA's scans overlap the other's loads
  const long long rows = (long long)batch + 2ll * total_draft;
  const int grid = (int)std::min<long long>(rows, 2ll * sms);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (dtype == SPECVERIFY_BF16) {
    if (aligned)
      sv::sv_truncate<sv::BF16, true><<<grid, sv::kTruncThreads, 0, s>>>(P);
    else
      sv::sv_truncate<sv::BF16, false><<<grid, sv::kTruncThreads, 0, s>>>(P);
  } else {
    if (aligned)
      sv::sv_truncate<sv::F32, true><<<grid, sv::kTruncThreads, 0, s>>>(P);
    else
      sv::sv_truncate<sv::F32, false><<<grid, sv::kTruncThreads, 0, s>>>(P);
  }
  return cudaGetLastError() == cudaSuccess ? SPECVERIFY_OK : SPECVERIFY_ERR_CUDA;
}

const char* specverify_error_string(int code) {
  switch (code) {
    case SPECVERIFY_OK: return "ok";
    case SPECVERIFY_ERR_INVALID_ARG: return "invalid argument";
    case SPECVERIFY_ERR_DTYPE: return "unknown dtype";
    case SPECVERIFY_ERR_CUDA: return "CUDA runtime error";
    case SPECVERIFY_ERR_DESTROYED: return "handle already destroyed";
    case SPECVERIFY_ERR_NO_STAGING: return "handle has no host staging buffers";
    case SPECVERIFY_ERR_TOO_LARGE:
      return "batch or max_k above the static scratch limits (SPECVERIFY_STATIC_MAX_BATCH, "
             "SPECVERIFY_STATIC_MAX_K)";
    default: return "unknown error code";
  }
}

}  // extern "C"
