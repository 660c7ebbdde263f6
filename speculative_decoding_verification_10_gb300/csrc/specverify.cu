// specverify.cu -- host side of the C ABI declared in include/specverify.h.
//
// Argument checking, scratch ownership and the single launch of a verify
// round.  All device work lives in sv_kernels.cuh.
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
constexpr int kMaxNper = 256;                  // 16-byte vectors per thread per chunk (896 KB of logits)
constexpr size_t kJobChunkBytes = 128 * 1024;  // bytes of each row in one residual job chunk
constexpr size_t kPartialBudget = size_t(256) << 20;
constexpr int kSpinLimit = 1 << 16;

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
  int num_sms, grid, max_nch;
  size_t max_rows, smem_bytes_max;
  void* scratch;
  size_t scratch_bytes;
  sv::Partial* part;
  sv::Partial* rowres;
  unsigned long long* row_cnt;
  unsigned long long* pos_cnt;
  uint32_t* done;
  uint32_t epoch;
  unsigned long long* res_slots;
  sv::Partial* part2;
  int* res_cnt;
  int* ctr;
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
  // optional timing events around the verify kernel
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

// Balanced chunking of a row into n chunks: vectors per thread per chunk.
static int chunk_nper(long long nvec, long long n) {
  const long long step = (long long)sv::kStageVecs * sv::kThreads;  // vectors per stage
  const long long chv = ((nvec + n - 1) / n + step - 1) / step * step;
  return (int)(chv / sv::kThreads);
}
static int chunks_of(long long nvec, int nper) {
  const long long chv = (long long)nper * sv::kThreads;
  return (int)((nvec + chv - 1) / chv);
}

// Items: the fewest chunks per row (whole rows when possible) such that the
// first wave -- a target and a draft row per request -- still gives every CTA
// two items.  Residual jobs: chunks of about kJobChunkBytes of each row, and
// at least as many as the items have.
static void choose_chunks(const specverify_ctx* h, int batch, int* nper, int* nch, int* jnper,
                          int* jnch) {
  const long long nvec = std::max<long long>(1, (long long)h->vocab * h->elem_bytes / 16);
  const long long step = (long long)sv::kStageVecs * sv::kThreads;
  const long long n_max = std::max<long long>(1, std::min<long long>(h->max_nch, (nvec + step - 1) / step));
  const long long rows0 = 2LL * batch;
  long long n = (nvec + (long long)kMaxNper * sv::kThreads - 1) / ((long long)kMaxNper * sv::kThreads);
  while (n < n_max && rows0 * n < 2LL * h->grid) ++n;
  n = std::min(n, n_max);
  *nper = chunk_nper(nvec, n);
  *nch = chunks_of(nvec, *nper);
  long long jn = std::max<long long>(1, ((long long)h->vocab * h->elem_bytes + kJobChunkBytes / 2) / kJobChunkBytes);
  jn = std::min(std::max<long long>(jn, *nch), n_max);
  *jnper = chunk_nper(nvec, jn);
  *jnch = chunks_of(nvec, *jnper);
}

template <typename E>
static int launch_round(specverify_ctx* h, const sv::Params& P, cudaStream_t s) {
  const size_t smem = ring_bytes() + sizeof(int) * ((size_t)P.batch + 1);
  const long long items = (long long)(h->max_k + 1) * 2 * P.batch * P.nch;
  const int grid = (int)std::max<long long>(1, std::min<long long>(h->grid, items));
  const int slot = h->n_events > 0 ? (int)(h->run_counter % (unsigned long long)h->n_events) : -1;
  h->run_counter++;
  if (slot >= 0 && cudaEventRecord(h->ev_start[slot], s) != cudaSuccess) return SPECVERIFY_ERR_CUDA;
  sv::sv_verify<E><<<grid, sv::kBlock, smem, s>>>(P);
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
  choose_chunks(h, batch, &P.nper, &P.nch, &P.jnper, &P.jnch);
  {
    const int spi = P.nper / sv::kStageVecs;
    P.fill = std::min(sv::kQueue - 2, (sv::kStages - 1 + spi - 1) / spi + 1);
  }
  P.spin_limit = kSpinLimit;
  P.accepted_len = accepted_len;
  P.committed = committed_tokens;
  P.flags = accept_flags;
  P.p_y = p_y;
  P.q_y = q_y;
  P.u_dbg = u;
  P.req_status = req_status;
  P.part = h->part;
  P.rowres = h->rowres;
  P.row_cnt = h->row_cnt;
  P.pos_cnt = h->pos_cnt;
  P.done = h->done;
  P.epoch = ++h->epoch;  // never 0: 0 is the initial value of every tag
  P.res_slots = h->res_slots;
  P.part2 = h->part2;
  P.res_cnt = h->res_cnt;
  P.ctr = h->ctr;

  DeviceGuard guard(h->device);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  rc = h->dtype == SPECVERIFY_BF16 ? launch_round<sv::BF16>(h, P, s)
                                   : launch_round<sv::F32>(h, P, s);
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
  h->smem_bytes_max = ring_bytes() + sizeof(int) * ((size_t)max_batch + 1);
  int occ = 0;
  bool ok = cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, device) ==
            cudaSuccess;
  if (dtype == SPECVERIFY_BF16) {
    ok = ok && cudaFuncSetAttribute(sv::sv_verify<sv::BF16>,
                                    cudaFuncAttributePreferredSharedMemoryCarveout,
                                    cudaSharedmemCarveoutMaxShared) == cudaSuccess;
    ok = ok && cudaFuncSetAttribute(sv::sv_verify<sv::BF16>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)h->smem_bytes_max) == cudaSuccess;
    ok = ok && cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, sv::sv_verify<sv::BF16>,
                                                             sv::kBlock, h->smem_bytes_max) ==
                   cudaSuccess;
  } else {
    ok = ok && cudaFuncSetAttribute(sv::sv_verify<sv::F32>,
                                    cudaFuncAttributePreferredSharedMemoryCarveout,
                                    cudaSharedmemCarveoutMaxShared) == cudaSuccess;
    ok = ok && cudaFuncSetAttribute(sv::sv_verify<sv::F32>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)h->smem_bytes_max) == cudaSuccess;
    ok = ok && cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, sv::sv_verify<sv::F32>,
                                                             sv::kBlock, h->smem_bytes_max) ==
                   cudaSuccess;
  }
  if (!ok || occ < 1) {
    cudaGetLastError();
    delete h;
    return SPECVERIFY_ERR_CUDA;
  }
  // persistent grid: every CTA resident at once
  h->grid = occ * h->num_sms;

  // row slots: waves 0..max_k, a target and a draft slot per request each
  h->max_rows = (size_t)max_batch * 2 * ((size_t)max_k + 1);
  const size_t row_bytes = (size_t)vocab * h->elem_bytes;
  const size_t nvec = std::max<size_t>(1, row_bytes / 16);
  const size_t min_chv = (size_t)sv::kStageVecs * sv::kThreads;
  size_t max_nch = (nvec + min_chv - 1) / min_chv;
  max_nch = std::min<size_t>(max_nch, std::max<size_t>(
                                          (nvec + (size_t)kMaxNper * sv::kThreads - 1) /
                                              ((size_t)kMaxNper * sv::kThreads),
                                          kPartialBudget / sizeof(sv::Partial) / h->max_rows));
  h->max_nch = (int)std::max<size_t>(1, max_nch);

  // one scratch allocation, carved into aligned pieces
  size_t off = 0;
  auto carve = [&](size_t bytes) {
    const size_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  };
  const size_t o_part = carve(sizeof(sv::Partial) * h->max_rows * h->max_nch);
  const size_t o_rowres = carve(sizeof(sv::Partial) * h->max_rows);
  const size_t o_rowcnt = carve(sizeof(unsigned long long) * h->max_rows);
  const size_t o_poscnt = carve(sizeof(unsigned long long) * (size_t)max_batch * (max_k + 1));
  const size_t o_done = carve(sizeof(uint32_t) * max_batch);
  // job slots: at most one residual job per request
  const size_t o_slots = carve(sizeof(unsigned long long) * (size_t)max_batch);
  const size_t o_part2 = carve(sizeof(sv::Partial) * (size_t)max_batch * h->max_nch);
  const size_t o_rescnt = carve(sizeof(int) * (size_t)max_batch);
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
  h->part = reinterpret_cast<sv::Partial*>(b + o_part);
  h->rowres = reinterpret_cast<sv::Partial*>(b + o_rowres);
  h->row_cnt = reinterpret_cast<unsigned long long*>(b + o_rowcnt);
  h->pos_cnt = reinterpret_cast<unsigned long long*>(b + o_poscnt);
  h->done = reinterpret_cast<uint32_t*>(b + o_done);
  h->epoch = 0u;
  h->res_slots = reinterpret_cast<unsigned long long*>(b + o_slots);
  h->part2 = reinterpret_cast<sv::Partial*>(b + o_part2);
  h->res_cnt = reinterpret_cast<int*>(b + o_rescnt);
  h->ctr = reinterpret_cast<int*>(b + o_ctr);

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
      cudaMemcpy(&st, h->ctr + sv::kCntLastStatus, sizeof st, cudaMemcpyDeviceToHost) !=
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

int specverify_launches_per_run(void) { return 1; }

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
