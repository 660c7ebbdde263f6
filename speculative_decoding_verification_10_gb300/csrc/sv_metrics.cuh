// sv_metrics.cuh -- acceptance statistics of verify rounds, on the device.
//
// "Speculative Decoding on AMD GPUs" (vLLM blog), "Monitor acceptance
// behavior" and the appendix tables: the signals to watch are the mean
// accepted length (MAL), the overall acceptance rate and the per-position
// acceptance rates; the printed rows satisfy MAL = 1 + the sum of the
// per-position rates, i.e. MAL counts the target's own token of the round.
// One launch adds a batch of round outputs (accepted_len, num_draft) to
// running counts and, optionally, writes the summary of the counts so far:
//   hist[a]        rounds that accepted a draft tokens (a = 0..max_k),
//   hist[max_k+1]  requests that were skipped (accepted_len = -1),
//   proposed[j]    rounds with a draft at position j   (num_draft > j),
//   accepted[j]    rounds that accepted position j     (accepted_len > j),
//   summary        MAL, acceptance rate, per-position rates, rounds, skipped.
// A num_draft above max_k counts only up to max_k; an accepted_len above
// max_k lands in hist[max_k].
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace sv {

constexpr int kMetricsThreads = 1024;
constexpr int kMetricsMaxK = 31;

// One CTA: warp-aggregated counts in shared memory, then added to the running
// counts, then (thread 0) the summary from the updated counts.
__global__ void __launch_bounds__(kMetricsThreads)
    sv_metrics(const int32_t* accepted_len, const int32_t* num_draft, int batch, int max_k,
               unsigned long long* hist, unsigned long long* proposed,
               unsigned long long* accepted, double* summary) {
  __shared__ unsigned int s_hist[kMetricsMaxK + 2];
  __shared__ unsigned int s_prop[kMetricsMaxK];
  __shared__ unsigned int s_acc[kMetricsMaxK];
  const int tid = threadIdx.x, lane = tid & 31;
  if (tid < kMetricsMaxK + 2) s_hist[tid] = 0u;
  if (tid < kMetricsMaxK) {
    s_prop[tid] = 0u;
    s_acc[tid] = 0u;
  }
  __syncthreads();
  for (int base = tid - lane; base < batch; base += kMetricsThreads) {
    const int r = base + lane;
    const bool in = r < batch;
    const int a = in ? accepted_len[r] : -2;
    const int k = in ? num_draft[r] : 0;
    const bool ok = in && a >= 0;
    // the bucket of this request: 0..max_k, max_k + 1 when skipped
    const int bucket = !in ? -1 : (ok ? min(a, max_k) : max_k + 1);
    for (int h = 0; h <= max_k + 1; ++h) {
      const unsigned n = __popc(__ballot_sync(0xffffffffu, bucket == h));
      if (lane == 0 && n) atomicAdd(&s_hist[h], n);
    }
    const int kk = ok ? min(k, max_k) : 0;
    for (int j = 0; j < max_k; ++j) {
      const unsigned np = __popc(__ballot_sync(0xffffffffu, kk > j));
      const unsigned na = __popc(__ballot_sync(0xffffffffu, kk > j && a > j));
      if (lane == 0 && np) atomicAdd(&s_prop[j], np);
      if (lane == 0 && na) atomicAdd(&s_acc[j], na);
    }
  }
  __syncthreads();
  if (tid <= max_k + 1 && s_hist[tid]) atomicAdd(&hist[tid], (unsigned long long)s_hist[tid]);
  if (tid < max_k) {
    if (s_prop[tid]) atomicAdd(&proposed[tid], (unsigned long long)s_prop[tid]);
    if (s_acc[tid]) atomicAdd(&accepted[tid], (unsigned long long)s_acc[tid]);
  }
  if (summary == nullptr) return;
  __threadfence();
  __syncthreads();
  if (tid != 0) return;
  const double nan = __longlong_as_double(0x7ff8000000000000ll);
  double rounds = 0.0, tokens = 0.0;
  for (int h = 0; h <= max_k; ++h) {
    const double c = (double)__ldcg(&hist[h]);
    rounds += c;
    tokens += (double)h * c;
  }
  double prop = 0.0, acc = 0.0;
  for (int j = 0; j < max_k; ++j) {
    const double p = (double)__ldcg(&proposed[j]), q = (double)__ldcg(&accepted[j]);
    prop += p;
    acc += q;
    summary[2 + j] = p > 0.0 ? q / p : nan;
  }
  summary[0] = rounds > 0.0 ? 1.0 + tokens / rounds : nan;
  summary[1] = prop > 0.0 ? acc / prop : nan;
  summary[2 + max_k] = rounds;
  summary[3 + max_k] = (double)__ldcg(&hist[max_k + 1]);
}

}  // namespace sv
