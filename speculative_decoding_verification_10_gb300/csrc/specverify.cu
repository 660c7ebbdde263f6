// specverify.cu -- host side of the C ABI declared in include/specverify.h.
//
// Argument checking, scratch ownership and the launches of a verify round
// (a plan launch and one wave launch per draft position).  All device work
// lives in sv_kernels.cuh.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <new>

#include "specverify.h"
#include "sv_kernels.cuh"

namespace {

constexpr uint32_t kLiveMagic = 0x53564c56u;  // "SVLV"
constexpr uint32_t kDeadMagic = 0x53564444u;  // "SVDD"

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

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

}  // namespace

struct specverify_ctx {
  uint32_t magic;
  int device, max_batch, max_k, vocab, dtype, elem_bytes;
  int num_sms, grid_aligned, grid_scalar;
  int depth_setting;  // 0: chosen per run from the batch size
  void* scratch;
  size_t scratch_bytes;
  sv::Entry* lists;
  int* list_cnt;
  sv::ResEntry* res;
  int* res_cnt;
  unsigned long long* pos_cnt;
  unsigned long long* rcnt;
  sv::Partial* part;
  sv::Partial* rpart;
  int* ctr;
  uint32_t epoch;
  // staging for specverify_run_host
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

static int check_handle(specverify_t h) {
  if (h == nullptr) return SPECVERIFY_ERR_INVALID_ARG;
  if (h->magic == kDeadMagic) return SPECVERIFY_ERR_DESTROYED;
  if (h->magic != kLiveMagic) return SPECVERIFY_ERR_INVALID_ARG;
  return SPECVERIFY_OK;
}

static size_t ring_bytes() {
  return sizeof(uint4) * sv::kStages * sv::kStageVecs * sv::kThreads;
}

// The kernels of one dtype: the wave kernel for 16-byte aligned rows and the
// scalar one for any other row layout.
template <typename E>
struct Kernels {
  static void* wave(bool aligned) {
    return aligned ? reinterpret_cast<void*>(sv::sv_wave<E, true>)
                   : reinterpret_cast<void*>(sv::sv_wave<E, false>);
  }
};

// Batches whose whole verify window (every row of every position) is at most
// this many bytes are verified in one wave of all positions: reading rows past
// a rejection costs less than a launch per position there.
constexpr double kShallowBytes = 192.0 * (1 << 20);

// Positions per wave for a run of `batch` requests.
static int run_depth(const specverify_ctx* h, int batch) {
  if (h->depth_setting > 0) return h->depth_setting;
  const double window = (double)batch * (2.0 * h->max_k + 1.0) * h->vocab * h->elem_bytes;
  return window <= kShallowBytes ? h->max_k + 1 : 1;
}

// A wave launch that may begin while the previous launch of the stream is
// finishing (programmatic dependent launch; the kernel waits for it first).
template <typename K>
static cudaError_t launch_wave(K kernel, int grid, size_t smem, cudaStream_t s,
                               const sv::Params& P) {
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
// returns at once).
template <typename E>
static int launch_round(specverify_ctx* h, sv::Params P, bool aligned, cudaStream_t s) {
  const int slot = h->n_events > 0 ? (int)(h->run_counter % (unsigned long long)h->n_events) : -1;
  h->run_counter++;
  if (slot >= 0 && cudaEventRecord(h->ev_start[slot], s) != cudaSuccess) return SPECVERIFY_ERR_CUDA;
  sv::sv_plan<<<1, sv::kPlanThreads, 0, s>>>(P);
  const size_t smem = aligned ? ring_bytes() : 0;
  const int grid = aligned ? h->grid_aligned : h->grid_scalar;
  for (int w = 0; w < P.n_waves; ++w) {
    P.wave = w;
    P.pos0 = std::min(w * P.depth, h->max_k + 1);
    P.pos1 = std::min((w + 1) * P.depth, h->max_k + 1);
    const cudaError_t e = aligned ? launch_wave(sv::sv_wave<E, true>, grid, smem, s, P)
                                  : launch_wave(sv::sv_wave<E, false>, grid, smem, s, P);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return SPECVERIFY_ERR_CUDA;
    }
  }
  if (slot >= 0 && cudaEventRecord(h->ev_stop[slot], s) != cudaSuccess) return SPECVERIFY_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? SPECVERIFY_OK : SPECVERIFY_ERR_CUDA;
}

static int run_impl(specverify_t h, const void* target_logits, const void* draft_logits,
                    const int32_t* draft_tokens, const int32_t* num_draft,
                    const float* temperature, uint64_t seed, int batch, int total_draft,
                    int32_t* accepted_len, int32_t* committed_tokens, uint8_t* accept_flags,
                    const int64_t* request_ids, float* p_y, float* q_y, float* u,
                    int32_t* req_status, void* stream) {
  int rc = check_handle(h);
  if (rc != SPECVERIFY_OK) return rc;
  if (batch < 0 || batch > h->max_batch) return SPECVERIFY_ERR_INVALID_ARG;
  if (total_draft < 0 || (long long)total_draft > (long long)batch * h->max_k)
    return SPECVERIFY_ERR_INVALID_ARG;
  if (batch == 0) {
    h->last_run_empty = true;
    return SPECVERIFY_OK;
  }
  if (!target_logits || !num_draft || !temperature || !accepted_len || !committed_tokens)
    return SPECVERIFY_ERR_INVALID_ARG;
  if (total_draft > 0 && (!draft_tokens || !accept_flags)) return SPECVERIFY_ERR_INVALID_ARG;
  const uintptr_t ea = (uintptr_t)(h->elem_bytes - 1);
  if (((uintptr_t)target_logits & ea) || ((uintptr_t)draft_logits & ea))
    return SPECVERIFY_ERR_INVALID_ARG;

  sv::Params P;
  std::memset(&P, 0, sizeof P);
  P.target = target_logits;
  P.draft = total_draft > 0 ? draft_logits : nullptr;
  P.tokens = draft_tokens;
  P.num_draft = num_draft;
  P.temperature = temperature;
  P.request_ids = request_ids;
  P.key = sv::PhiloxKey{(uint32_t)(seed & 0xffffffffu), (uint32_t)(seed >> 32)};
  P.batch = batch;
  P.total_draft = total_draft;
  P.max_k = h->max_k;
  P.vocab = h->vocab;
  P.epoch = ++h->epoch;  // never 0: 0 is the initial value of every tag
  P.depth = run_depth(h, batch);
  P.n_waves = sv::wave_count(h->max_k, P.depth);
  P.list_cap = 2 * P.depth * h->max_batch;
  P.nb = (h->vocab + sv::kRaceBlock - 1) / sv::kRaceBlock;
  P.nvec = (int)((size_t)h->vocab * h->elem_bytes / 16);
  const int block_bytes = sv::kRaceBlock * h->elem_bytes;
  P.min_span = std::max(1, sv::kMinSpanBytes / block_bytes);
  P.min_span_res = std::max(1, sv::kMinSpanBytes / (2 * block_bytes));
  P.stride = h->max_batch;
  P.accepted_len = accepted_len;
  P.committed = committed_tokens;
  P.flags = accept_flags;
  P.p_y = p_y;
  P.q_y = q_y;
  P.u_dbg = u;
  P.req_status = req_status;
  P.lists = h->lists;
  P.list_cnt = h->list_cnt;
  P.res = h->res;
  P.res_cnt = h->res_cnt;
  P.pos_cnt = h->pos_cnt;
  P.rcnt = h->rcnt;
  P.part = h->part;
  P.rpart = h->rpart;
  P.ctr = h->ctr;
  // the vector path needs every row on a 16-byte boundary
  const bool aligned = ((size_t)h->vocab * h->elem_bytes) % 16 == 0 &&
                       ((uintptr_t)target_logits & 15u) == 0 &&
                       ((uintptr_t)P.draft & 15u) == 0;

  DeviceGuard guard(h->device);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  rc = h->dtype == SPECVERIFY_BF16 ? launch_round<sv::BF16>(h, P, aligned, s)
                                   : launch_round<sv::F32>(h, P, aligned, s);
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
  if (max_batch < 1 || max_batch > sv::kMaxBatch || max_k < 0 || max_k > 31 || vocab < 1 ||
      vocab > (1 << 30))
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
  h->device = device;
  h->max_batch = max_batch;
  h->max_k = max_k;
  h->vocab = vocab;
  h->dtype = dtype;
  h->elem_bytes = dtype == SPECVERIFY_BF16 ? 2 : 4;
  h->last_stream = nullptr;
  h->n_events = 0;
  h->run_counter = 0;

  h->last_run_empty = true;
  h->depth_setting = 0;
  bool ok = cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, device) ==
            cudaSuccess;
  int occ_a = 0, occ_s = 0;
  const size_t smem = ring_bytes();
  for (int a = 0; a < 2 && ok; ++a) {
    const void* fn = dtype == SPECVERIFY_BF16 ? Kernels<sv::BF16>::wave(a == 1)
                                              : Kernels<sv::F32>::wave(a == 1);
    const size_t sm = a == 1 ? smem : 0;
    ok = cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout,
                              cudaSharedmemCarveoutMaxShared) == cudaSuccess;
    ok = ok && cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm) ==
                   cudaSuccess;
    ok = ok && cudaOccupancyMaxActiveBlocksPerMultiprocessor(a == 1 ? &occ_a : &occ_s, fn,
                                                             sv::kBlock, sm) == cudaSuccess;
  }
  if (!ok || occ_a < 1 || occ_s < 1) {
    cudaGetLastError();
    delete h;
    return SPECVERIFY_ERR_CUDA;
  }
  // one wave of CTAs, all resident at once
  h->grid_aligned = occ_a * h->num_sms;
  h->grid_scalar = occ_s * h->num_sms;
  const int grid = std::max(h->grid_aligned, h->grid_scalar);
  const size_t row_bytes = (size_t)vocab * h->elem_bytes;

  // one scratch allocation, carved into aligned pieces
  size_t off = 0;
  auto carve = [&](size_t bytes) {
    const size_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  };
  // sized for every wave depth D = 1 .. max_k + 1
  const size_t mb = (size_t)max_batch;
  size_t list_entries = 0, max_waves = 0, max_cap = 0;
  for (int d = 1; d <= max_k + 1; ++d) {
    const size_t w = (size_t)sv::wave_count(max_k, d), cap = 2 * (size_t)d * mb;
    list_entries = std::max(list_entries, w * cap);
    max_waves = std::max(max_waves, w);
    max_cap = std::max(max_cap, cap);
  }
  const size_t o_lists = carve(sizeof(sv::Entry) * list_entries);
  const size_t o_lcnt = carve(sizeof(int) * max_waves);
  const size_t o_res = carve(sizeof(sv::ResEntry) * max_waves * mb);
  const size_t o_rcnt = carve(sizeof(int) * max_waves);
  const size_t o_poscnt = carve(sizeof(unsigned long long) * ((size_t)max_k + 1) * mb);
  const size_t o_rescnt = carve(sizeof(unsigned long long) * mb);
  const size_t o_part = carve(sizeof(sv::Partial) * ((size_t)grid + max_cap));
  const size_t o_rpart = carve(sizeof(sv::Partial) * ((size_t)grid + mb));
  const size_t o_ctr = carve(sizeof(int) * sv::kCntCount);
  h->scratch_bytes = off;
  if (cudaMalloc(&h->scratch, h->scratch_bytes) != cudaSuccess) {
    cudaGetLastError();
    delete h;
    return SPECVERIFY_ERR_CUDA;
  }
  if (cudaMemset(h->scratch, 0, h->scratch_bytes) != cudaSuccess) {
    cudaGetLastError();
    cudaFree(h->scratch);
    delete h;
    return SPECVERIFY_ERR_CUDA;
  }
  char* b = static_cast<char*>(h->scratch);
  h->lists = reinterpret_cast<sv::Entry*>(b + o_lists);
  h->list_cnt = reinterpret_cast<int*>(b + o_lcnt);
  h->res = reinterpret_cast<sv::ResEntry*>(b + o_res);
  h->res_cnt = reinterpret_cast<int*>(b + o_rcnt);
  h->pos_cnt = reinterpret_cast<unsigned long long*>(b + o_poscnt);
  h->rcnt = reinterpret_cast<unsigned long long*>(b + o_rescnt);
  h->part = reinterpret_cast<sv::Partial*>(b + o_part);
  h->rpart = reinterpret_cast<sv::Partial*>(b + o_rpart);
  h->ctr = reinterpret_cast<int*>(b + o_ctr);
  h->epoch = 0u;

  h->stage = nullptr;
  if (flags & SPECVERIFY_CREATE_HOST_STAGING) {
    size_t so = 0;
    auto scarve = [&](size_t bytes) {
      const size_t o = so;
      so = align_up(so + bytes, 256);
      return o;
    };
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
  return run_impl(h, target_logits, draft_logits, draft_tokens, num_draft, temperature, seed,
                  batch, total_draft, accepted_len, committed_tokens, accept_flags, nullptr,
                  nullptr, nullptr, nullptr, nullptr, stream);
}

int specverify_run_ex(specverify_t h, const void* target_logits, const void* draft_logits,
                      const int32_t* draft_tokens, const int32_t* num_draft,
                      const float* temperature, uint64_t seed, int batch, int total_draft,
                      int32_t* accepted_len, int32_t* committed_tokens, uint8_t* accept_flags,
                      const int64_t* request_ids, float* p_y, float* q_y, float* u,
                      int32_t* req_status, void* stream) {
  return run_impl(h, target_logits, draft_logits, draft_tokens, num_draft, temperature, seed,
                  batch, total_draft, accepted_len, committed_tokens, accept_flags, request_ids,
                  p_y, q_y, u, req_status, stream);
}

int specverify_run_host(specverify_t h, const void* target_logits, const void* draft_logits,
                        const int32_t* draft_tokens, const int32_t* num_draft,
                        const float* temperature, uint64_t seed, int batch, int total_draft,
                        int32_t* accepted_len, int32_t* committed_tokens,
                        uint8_t* accept_flags, void* stream) {
  int rc = check_handle(h);
  if (rc != SPECVERIFY_OK) return rc;
  if (h->stage == nullptr) return SPECVERIFY_ERR_NO_STAGING;
  if (batch < 0 || batch > h->max_batch) return SPECVERIFY_ERR_INVALID_ARG;
  if (total_draft < 0 || (long long)total_draft > (long long)batch * h->max_k)
    return SPECVERIFY_ERR_INVALID_ARG;
  if (batch == 0) return SPECVERIFY_OK;
  if (!target_logits || !num_draft || !temperature || !accepted_len || !committed_tokens)
    return SPECVERIFY_ERR_INVALID_ARG;
  if (total_draft > 0 && (!draft_tokens || !accept_flags)) return SPECVERIFY_ERR_INVALID_ARG;

  DeviceGuard guard(h->device);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const size_t row_bytes = (size_t)h->vocab * h->elem_bytes;
  bool ok = true;
  auto h2d = [&](void* dst, const void* src, size_t n) {
    if (n && ok) ok = cudaMemcpyAsync(dst, src, n, cudaMemcpyHostToDevice, s) == cudaSuccess;
  };
  auto d2h = [&](void* dst, const void* src, size_t n) {
    if (n && ok) ok = cudaMemcpyAsync(dst, src, n, cudaMemcpyDeviceToHost, s) == cudaSuccess;
  };
  h2d(h->st_target, target_logits, (size_t)(batch + total_draft) * row_bytes);
  const bool has_draft = draft_logits != nullptr && total_draft > 0;
  if (has_draft) h2d(h->st_draft, draft_logits, (size_t)total_draft * row_bytes);
  h2d(h->st_tokens, draft_tokens, sizeof(int32_t) * (size_t)total_draft);
  h2d(h->st_num_draft, num_draft, sizeof(int32_t) * (size_t)batch);
  h2d(h->st_temperature, temperature, sizeof(float) * (size_t)batch);
  if (!ok) {
    cudaGetLastError();
    return SPECVERIFY_ERR_CUDA;
  }
  rc = run_impl(h, h->st_target, has_draft ? h->st_draft : nullptr, h->st_tokens,
                h->st_num_draft, h->st_temperature, seed, batch, total_draft, h->st_accepted,
                h->st_committed, h->st_flags, nullptr, nullptr, nullptr, nullptr, nullptr,
                stream);
  if (rc != SPECVERIFY_OK) return rc;
  d2h(accepted_len, h->st_accepted, sizeof(int32_t) * (size_t)batch);
  d2h(committed_tokens, h->st_committed, sizeof(int32_t) * (size_t)batch * (h->max_k + 1));
  d2h(accept_flags, h->st_flags, (size_t)total_draft);
  if (ok) ok = cudaStreamSynchronize(s) == cudaSuccess;
  if (!ok) {
    cudaGetLastError();
    return SPECVERIFY_ERR_CUDA;
  }
  return SPECVERIFY_OK;
}

int specverify_status(specverify_t h, int32_t* status_out) {
  int rc = check_handle(h);
  if (rc != SPECVERIFY_OK) return rc;
  if (status_out == nullptr) return SPECVERIFY_ERR_INVALID_ARG;
  DeviceGuard guard(h->device);
  int32_t st = 0;
  if (h->last_run_empty) {
    *status_out = 0;
    return SPECVERIFY_OK;
  }
  if (cudaStreamSynchronize(h->last_stream) != cudaSuccess ||
      cudaMemcpy(&st, h->ctr + sv::kCntStatus, sizeof st, cudaMemcpyDeviceToHost) !=
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
  if (depth < 0 || depth > h->max_k + 1) return SPECVERIFY_ERR_INVALID_ARG;
  h->depth_setting = depth;
  return SPECVERIFY_OK;
}

int specverify_launches_per_run(specverify_t h, int batch, int* launches_out) {
  int rc = check_handle(h);
  if (rc != SPECVERIFY_OK) return rc;
  if (launches_out == nullptr || batch < 0 || batch > h->max_batch)
    return SPECVERIFY_ERR_INVALID_ARG;
  *launches_out = batch == 0 ? 0 : 1 + sv::wave_count(h->max_k, run_depth(h, batch));
  return SPECVERIFY_OK;
}

int specverify_destroy(specverify_t h) {
  int rc = check_handle(h);
  if (rc != SPECVERIFY_OK) return rc;
  DeviceGuard guard(h->device);
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

const char* specverify_error_string(int code) {
  switch (code) {
    case SPECVERIFY_OK: return "ok";
    case SPECVERIFY_ERR_INVALID_ARG: return "invalid argument";
    case SPECVERIFY_ERR_DTYPE: return "unknown dtype";
    case SPECVERIFY_ERR_CUDA: return "CUDA runtime error";
    case SPECVERIFY_ERR_DESTROYED: return "handle already destroyed";
    case SPECVERIFY_ERR_NO_STAGING: return "handle has no host staging buffers";
    default: return "unknown error code";
  }
}

}  // extern "C"
