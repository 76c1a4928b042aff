// Shared device helpers for the MoE layer kernels (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "moe.h"

namespace moe {

typedef __nv_bfloat16 bf16;

constexpr int kMaxE = 256;
constexpr int kMaxK = 8;

// ---------------------------------------------------------------- status word
// status[0]: first error code recorded (0 = none); status[1]: its detail.
__device__ __forceinline__ void record_error(int* status, int code, int detail) {
  if (status != nullptr && atomicCAS(status, 0, code) == 0) {
    atomicExch(status + 1, detail);
  }
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------- conversions
template <typename T> __device__ __forceinline__ float to_f32(T v);
template <> __device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ float to_f32<bf16>(bf16 v) { return __bfloat162float(v); }

template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ bf16 from_f32<bf16>(float v) { return __float2bfloat16_rn(v); }

// Eight consecutive elements <-> eight floats. Pointers are 16-byte aligned
// for bf16 (one 16-byte access) and 32-byte aligned for fp32 (two accesses).
__device__ __forceinline__ void load8(const bf16* p, float (&v)[8]) {
  uint4 r = *reinterpret_cast<const uint4*>(p);
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&r);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 f = __bfloat1622float2(h[i]);
    v[2 * i] = f.x;
    v[2 * i + 1] = f.y;
  }
}
__device__ __forceinline__ void load8(const float* p, float (&v)[8]) {
  float4 a = *reinterpret_cast<const float4*>(p);
  float4 b = *reinterpret_cast<const float4*>(p + 4);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
__device__ __forceinline__ void store8(bf16* p, const float (&v)[8]) {
  uint4 r;
  __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&r);
#pragma unroll
  for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
  *reinterpret_cast<uint4*>(p) = r;
}
__device__ __forceinline__ void store8(float* p, const float (&v)[8]) {
  *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
  *reinterpret_cast<float4*>(p + 4) = make_float4(v[4], v[5], v[6], v[7]);
}

// Eight consecutive elements held raw (as loaded), converted to float later, so
// that several rows' loads can be in flight before any of them is used.
template <typename T> struct Raw8;
template <> struct Raw8<bf16> {
  uint4 a;
  __device__ __forceinline__ void load(const bf16* p) { a = __ldg(reinterpret_cast<const uint4*>(p)); }
  __device__ __forceinline__ void zero() { a = make_uint4(0, 0, 0, 0); }
  __device__ __forceinline__ void to_float(float (&v)[8]) const {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&a);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float2 f = __bfloat1622float2(h[i]);
      v[2 * i] = f.x;
      v[2 * i + 1] = f.y;
    }
  }
};
template <> struct Raw8<float> {
  float4 a, b;
  __device__ __forceinline__ void load(const float* p) {
    a = __ldg(reinterpret_cast<const float4*>(p));
    b = __ldg(reinterpret_cast<const float4*>(p + 4));
  }
  __device__ __forceinline__ void zero() { a = b = make_float4(0.f, 0.f, 0.f, 0.f); }
  __device__ __forceinline__ void to_float(float (&v)[8]) const {
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  }
};

// Raw 16-byte row-chunk copy type: a row of n elements is n*sizeof(T)/16 chunks.
template <typename T> struct Vec16 { static constexpr int kElems = 16 / sizeof(T); };

// ---------------------------------------------------------------- error-free sums
// Knuth's TwoSum: s + e == a + b exactly (round-to-nearest, no overflow).
// The _rn intrinsics keep the compiler from contracting or reassociating.
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = __fadd_rn(a, b);
  float bb = __fsub_rn(s, a);
  e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

// (hi, lo) += c, keeping hi + lo as an unevaluated sum with fp32 error terms.
__device__ __forceinline__ void comp_add(float& hi, float& lo, float c) {
  float s, e;
  two_sum(hi, c, s, e);
  hi = s;
  lo = __fadd_rn(lo, e);
}

// ---------------------------------------------------------------- warp helpers
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float sigmoidf_acc(float z) { return 1.0f / (1.0f + expf(-z)); }

// sqrt(softplus(z)) = sqrt(log(1 + exp(z))); softplus(z) = z + log1p(exp(-z))
// for z > 0 (no overflow), log1p(exp(z)) otherwise.
__device__ __forceinline__ float sqrt_softplusf(float z) {
  const float sp = z > 0.f ? z + log1pf(expf(-z)) : log1pf(expf(z));
  return sqrtf(sp);
}

// Score of one logit for the sigmoid-like score functions (sigmoid and
// sqrt(softplus)); d score / d logit through `deriv`.
__device__ __forceinline__ float bias_score(float z, int score_fn) {
  return score_fn == MOE_SCORE_SQRT_SOFTPLUS ? sqrt_softplusf(z) : sigmoidf_acc(z);
}
__device__ __forceinline__ float bias_score_deriv(float z, float s, int score_fn) {
  // sigmoid: s (1 - s); sqrt(softplus): sigmoid(z) / (2 s)
  return score_fn == MOE_SCORE_SQRT_SOFTPLUS ? sigmoidf_acc(z) / (2.f * s) : s * (1.f - s);
}

// ---------------------------------------------------------------- W_r staging
// W [E][d] fp32 (global) -> sW [E][2][d/8] float4 (shared): the two halves of
// each 8-element group in separate planes, so that lanes taking consecutive
// groups read consecutive 16-byte words. Each thread keeps eight loads in
// flight before storing them (one load at a time would leave the copy bound by
// memory latency). Ends with __syncthreads().
__device__ __forceinline__ void stage_w_planes(float4* sW, const float* __restrict__ W, int E,
                                               int d) {
  const float4* W4 = reinterpret_cast<const float4*>(W);
  const int q = d >> 2, ng = d >> 3;
  const int n4 = E * q;
  for (int i0 = threadIdx.x; i0 < n4; i0 += 8 * blockDim.x) {
    float4 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = i0 + u * blockDim.x;
      if (i < n4) v[u] = __ldg(W4 + i);
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = i0 + u * blockDim.x;
      if (i < n4) {
        const int e = i / q, r = i - e * q;
        sW[(e * 2 + (r & 1)) * ng + (r >> 1)] = v[u];
      }
    }
  }
  __syncthreads();
}

// ---------------------------------------------------------------- dependent launches
// A kernel launched with launch_dependent may start while the previous kernel
// on the stream is still running; before it reads anything that kernel (or an
// earlier one) wrote, it must pass pdl_wait(), which returns once the previous
// grid has finished and its writes are visible. pdl_launch_dependents() lets
// the next dependent grid be scheduled early. Both are no-ops in a kernel
// launched the ordinary way.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
static inline cudaError_t launch_dependent(void (*kern)(KArgs...), dim3 grid, dim3 block,
                                           size_t smem, cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

}  // namespace moe
