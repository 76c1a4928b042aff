// The shared expert's sigmoid gate (Megatron's --moe-shared-expert-gate).
//
// The Ultimate MoE Training Handbook §3.4 "Shared experts": with the gate the
// shared expert's output is multiplied per token by sigmoid(x · w_gate), a [d]
// gate weight (a [1, d] linear layer); without it the output is added at
// weight 1.
//   forward   gate[t] = sigmoid(<x[t], w_gate>)           (fp32 dot, one warp per token)
//   backward  d_gate_logit[t] = <dy[t], y_s[t]> gate (1 - gate);  dy_s[t] = gate dy[t]
// The gate weight's gradient sum_t d_gate_logit[t] x[t] and the input's
// d_gate_logit[t] w_gate are taken elsewhere (the router's dW kernel for one
// expert; the permute backward).
#include "common.cuh"
#include "internal.h"

namespace moe {

static unsigned gate_grid(const Ctx& c, int64_t T) {
  const int64_t blocks = (T + 7) / 8;
  const int64_t cap = (int64_t)c.sm_count * 8;
  return (unsigned)(blocks < cap ? (blocks > 0 ? blocks : 1) : cap);
}

template <typename T>
__global__ void __launch_bounds__(256)
shared_gate_fwd(const T* __restrict__ x, const float* __restrict__ w_gate,
                float* __restrict__ gate, int64_t Tn, int d) {
  pdl_wait();  // a dependent launch: inputs come from the kernels before
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int ng = d >> 3;
  for (int64_t t = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < Tn; t += nwarps) {
    float acc = 0.f;
    for (int g = lane; g < ng; g += 32) {
      float xv[8], wv[8];
      load8(x + t * d + 8 * g, xv);
      load8(w_gate + 8 * g, wv);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc = fmaf(xv[i], wv[i], acc);
    }
    acc = warp_sum(acc);
    if (lane == 0) gate[t] = sigmoidf_acc(acc);
  }
}

template <typename T>
__global__ void __launch_bounds__(256)
shared_gate_bwd_tok(const T* __restrict__ dy, const T* __restrict__ y_s,
                    const float* __restrict__ gate, T* __restrict__ dy_s,
                    float* __restrict__ d_gate_logit, int64_t Tn, int d) {
  pdl_wait();  // a dependent launch: inputs come from the kernels before
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int ng = d >> 3;
  for (int64_t t = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < Tn; t += nwarps) {
    const float gt = gate[t];
    float dot = 0.f;
    for (int g = lane; g < ng; g += 32) {
      float dv[8], sv[8], o[8];
      load8(dy + t * d + 8 * g, dv);
      load8(y_s + t * d + 8 * g, sv);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        dot = fmaf(dv[i], sv[i], dot);
        o[i] = gt * dv[i];
      }
      store8(dy_s + t * d + 8 * g, o);
    }
    dot = warp_sum(dot);
    if (lane == 0) d_gate_logit[t] = dot * gt * (1.f - gt);
  }
}

cudaError_t launch_shared_gate(const Ctx& c, const moe_cfg& cfg, const void* x,
                               const float* w_gate, float* gate) {
  if (cfg.T == 0) return cudaSuccess;
  if (cfg.act_dtype == MOE_BF16)
    launch_dependent(shared_gate_fwd<bf16>, dim3(gate_grid(c, cfg.T)), dim3(256), 0, c.stream,
        static_cast<const bf16*>(x), w_gate, gate, cfg.T, cfg.d);
  else
    launch_dependent(shared_gate_fwd<float>, dim3(gate_grid(c, cfg.T)), dim3(256), 0, c.stream,
        static_cast<const float*>(x), w_gate, gate, cfg.T, cfg.d);
  note_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_shared_gate_bwd_tokens(const Ctx& c, const moe_cfg& cfg, const void* dy,
                                          const void* shared_out, const float* gate,
                                          void* dy_shared, float* d_gate_logit) {
  if (cfg.T == 0) return cudaSuccess;
  if (cfg.act_dtype == MOE_BF16)
    launch_dependent(shared_gate_bwd_tok<bf16>, dim3(gate_grid(c, cfg.T)), dim3(256), 0, c.stream,
        static_cast<const bf16*>(dy), static_cast<const bf16*>(shared_out), gate,
        static_cast<bf16*>(dy_shared), d_gate_logit, cfg.T, cfg.d);
  else
    launch_dependent(shared_gate_bwd_tok<float>, dim3(gate_grid(c, cfg.T)), dim3(256), 0, c.stream,
        static_cast<const float*>(dy), static_cast<const float*>(shared_out), gate,
        static_cast<float*>(dy_shared), d_gate_logit, cfg.T, cfg.d);
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace moe
