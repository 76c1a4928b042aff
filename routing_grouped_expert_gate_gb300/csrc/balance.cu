// Load-balance bookkeeping on the device: int64 token counts per expert, the
// aux-loss-free expert-bias update and MaxVio.
//
// The Ultimate MoE Training Handbook §3.3 "Load balancing", part "Loss-free
// bias": the router keeps an int64 token count per expert, adds every
// micro-batch's counts to it, and after the step moves each expert's bias by
// a fixed rate towards balance, bias += sign(total - count[e] * E) * rate,
// comparing the integers (count * E against the total) rather than a
// floating-point mean. §3.2 "Routing strategy", part "Who selects": MaxVio =
// (busiest expert's load - mean load) / mean load.
//
// E <= 256: one CTA does each job; every sum runs in a fixed order.
#include "common.cuh"
#include "internal.h"

namespace moe {

__global__ void tokens_accumulate(const int32_t* __restrict__ counts, int64_t* __restrict__ acc,
                                  int E) {
  for (int e = threadIdx.x; e < E; e += blockDim.x) acc[e] += (int64_t)counts[e];
}

__device__ __forceinline__ int64_t ordered_total(const int64_t* __restrict__ tpe, int E,
                                                 int64_t* shared_total) {
  if (threadIdx.x == 0) {
    int64_t t = 0;
    for (int e = 0; e < E; ++e) t += tpe[e];
    *shared_total = t;
  }
  __syncthreads();
  return *shared_total;
}

__global__ void expert_bias_update_kernel(const int64_t* __restrict__ tpe,
                                          float* __restrict__ bias, int E, float rate) {
  __shared__ int64_t total_s;
  const int64_t total = ordered_total(tpe, E, &total_s);
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const int64_t ce = tpe[e] * (int64_t)E;
    const int dir = (total > ce) - (total < ce);
    bias[e] = __fadd_rn(bias[e], (float)dir * rate);
  }
}

__global__ void max_vio_kernel(const int64_t* __restrict__ tpe, int E, float* __restrict__ out) {
  if (threadIdx.x != 0 || blockIdx.x != 0) return;
  int64_t total = 0, mx = 0;
  for (int e = 0; e < E; ++e) {
    total += tpe[e];
    if (e == 0 || tpe[e] > mx) mx = tpe[e];
  }
  // (max - total / E) / (total / E) = (max E - total) / total, in fp64
  *out = total > 0 ? (float)((double)(mx * (int64_t)E - total) / (double)total) : 0.f;
}

cudaError_t launch_tokens_accumulate(const Ctx& c, const moe_cfg& cfg, const int32_t* counts,
                                     int64_t* tokens_per_expert) {
  tokens_accumulate<<<1, 256, 0, c.stream>>>(counts, tokens_per_expert, cfg.E);
  note_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_expert_bias_update(const Ctx& c, const moe_cfg& cfg,
                                      const int64_t* tokens_per_expert, float* expert_bias,
                                      float rate) {
  expert_bias_update_kernel<<<1, 256, 0, c.stream>>>(tokens_per_expert, expert_bias, cfg.E, rate);
  note_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_max_vio(const Ctx& c, const moe_cfg& cfg, const int64_t* tokens_per_expert,
                           float* out) {
  max_vio_kernel<<<1, 32, 0, c.stream>>>(tokens_per_expert, cfg.E, out);
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace moe
