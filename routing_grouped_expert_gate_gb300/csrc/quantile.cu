// Quantile balancing: the per-expert bias solved from the micro-batch.
//
// The Ultimate MoE Training Handbook §3.3 "Load balancing", part "Quantile":
// the router ranks k + 1 experts per token on score - beta (the top-k kernel
// with a quantile bias, router.cu), keeps the first k and the (k+1)-th key as
// the token's threshold alpha; then, for each expert, it ranks the micro-
// batch's tokens by score - alpha and reads off the (col_target + 1)-th
// largest, col_target = T k / E: the value only the expert's target share of
// tokens beats. The solutions of the micro-batches are averaged, mixed into
// the running beta by an EMA and centred to zero mean.
//
// Per expert the quantile is found by an exact radix select on the fp32 bit
// patterns (four 8-bit digits, most significant first), one CTA per expert;
// the histograms use integer atomics, so the result does not depend on
// thread order.
#include "common.cuh"
#include "internal.h"

namespace moe {

// fp32 -> uint32 with the same order (larger float <-> larger key)
__device__ __forceinline__ uint32_t order_key(float v) {
  const uint32_t u = __float_as_uint(v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t k) {
  const uint32_t u = (k & 0x80000000u) ? (k & 0x7fffffffu) : ~k;
  return __uint_as_float(u);
}

// the selection score of one logit: the logit itself (softmax) or the
// sigmoid-like score, by the same function the top-k kernel uses, so that
// score - alpha is computed from the very values alpha was ranked on
__device__ __forceinline__ float select_score(const float* __restrict__ row, int e,
                                              int score_fn) {
  const float l = row[e];
  return score_fn == MOE_SCORE_SOFTMAX ? l : bias_score(l, score_fn);
}

__global__ void __launch_bounds__(256)
quantile_solve_kernel(const float* __restrict__ logits, const float* __restrict__ alpha,
                      int64_t T, int E, int score_fn, int64_t r, float* __restrict__ beta_local) {
  __shared__ uint32_t hist[256];
  __shared__ uint32_t s_prefix, s_mask;
  __shared__ int64_t s_rem;
  const int e = blockIdx.x;
  if (threadIdx.x == 0) {
    s_prefix = 0u;
    s_mask = 0u;
    s_rem = r;
  }
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = threadIdx.x; i < 256; i += blockDim.x) hist[i] = 0u;
    __syncthreads();
    const uint32_t prefix = s_prefix, mask = s_mask;
    for (int64_t t = threadIdx.x; t < T; t += blockDim.x) {
      const float v = __fsub_rn(select_score(logits + t * E, e, score_fn), alpha[t]);
      const uint32_t key = order_key(v);
      if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      int64_t rem = s_rem;
      int digit = 0;
      for (int b = 255; b >= 0; --b) {
        if (rem <= (int64_t)hist[b]) {
          digit = b;
          break;
        }
        rem -= hist[b];
      }
      s_rem = rem;
      s_prefix = prefix | ((uint32_t)digit << shift);
      s_mask = mask | (255u << shift);
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) beta_local[e] = key_value(s_prefix);
}

__global__ void quantile_accumulate_kernel(const float* __restrict__ beta_local,
                                           float* __restrict__ accum, int32_t* __restrict__ count,
                                           int E) {
  for (int e = threadIdx.x; e < E; e += blockDim.x) accum[e] += beta_local[e];
  if (threadIdx.x == 0) *count += 1;
}

__global__ void quantile_update_kernel(float* __restrict__ beta, float* __restrict__ accum,
                                       int32_t* __restrict__ count, int E, float ema) {
  __shared__ float nb[kMaxE];
  __shared__ float mean_s;
  const int n = *count > 1 ? *count : 1;
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    nb[e] = ema * beta[e] + (1.f - ema) * (accum[e] / (float)n);
  __syncthreads();
  if (threadIdx.x == 0) {
    double s = 0.0;
    for (int e = 0; e < E; ++e) s += (double)nb[e];
    mean_s = (float)(s / (double)E);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    beta[e] = nb[e] - mean_s;
    accum[e] = 0.f;
  }
  __syncthreads();
  if (threadIdx.x == 0) *count = 0;
}

cudaError_t launch_quantile_solve(const Ctx& c, const moe_cfg& cfg, const float* logits,
                                  const float* alpha, float* beta_local) {
  const int64_t r = cfg.T * (int64_t)cfg.k / cfg.E + 1;  // the (col_target + 1)-th largest
  quantile_solve_kernel<<<cfg.E, 256, 0, c.stream>>>(logits, alpha, cfg.T, cfg.E, cfg.score_fn,
                                                      r, beta_local);
  note_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_quantile_accumulate(const Ctx& c, const moe_cfg& cfg, const float* beta_local,
                                       float* accum, int32_t* count) {
  quantile_accumulate_kernel<<<1, 256, 0, c.stream>>>(beta_local, accum, count, cfg.E);
  note_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_quantile_beta_update(const Ctx& c, const moe_cfg& cfg, float* beta,
                                        float* accum, int32_t* count, float ema) {
  quantile_update_kernel<<<1, 256, 0, c.stream>>>(beta, accum, count, cfg.E, ema);
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace moe
