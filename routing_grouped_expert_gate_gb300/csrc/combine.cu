// Weighted unpermute-combine (S6) and its backward (B6).
//
// MoE training cluster: routing, load balancing (LeCompute), "An expert
// transforms numbers inside the model": the block returns each chosen expert's
// output times its weight, summed coordinate by coordinate. The Ultimate MoE
// Training Handbook, §3.4 "Shared experts": the shared expert's output is added
// at weight 1, or times sigmoid(x · w_gate) with the shared-expert gate.
//
// Both kernels run one warp per token with 16-byte accesses (8 bf16 or 4+4
// fp32 per lane per step): the gather, the scaling and the accumulation happen
// in one pass, so each expert output row is read once and y is written once.
#include "common.cuh"
#include "internal.h"

namespace moe {

static unsigned token_grid(const Ctx& c, int64_t T) {
  const int64_t blocks = (T + 7) / 8;
  const int64_t cap = (int64_t)c.sm_count * 8;
  return (unsigned)(blocks < cap ? (blocks > 0 ? blocks : 1) : cap);
}

// Rows of one token: the k row indices (validated) and their weights.
template <int KK>
__device__ __forceinline__ void token_rows(const int32_t* __restrict__ row_of,
                                           const float* __restrict__ w, int64_t t, int k,
                                           int64_t A, int lane, int* status, int64_t (&rows)[KK],
                                           float (&wj)[KK]) {
#pragma unroll
  for (int j = 0; j < KK; ++j) {
    int r = -1;
    wj[j] = 0.f;
    if (j < k) {
      r = row_of[t * k + j];
      wj[j] = w[t * k + j];
      if (r < 0 || r >= A) {
        if (lane == 0) record_error(status, MOE_ERR_DEVICE_INDEX, (int)t);
        r = -1;
      }
    }
    rows[j] = r;
  }
}

// KK: compile-time bound on k. Each lane handles U = 8 / KK (at least 1)
// 8-element groups per step, so about nine or more 16-byte loads are in
// flight per lane whatever k is; all of them are issued before any is used.
template <typename T, int KK>
__global__ void __launch_bounds__(256)
combine_kernel(const T* __restrict__ out_perm, const int32_t* __restrict__ row_of,
               const float* __restrict__ w, const T* __restrict__ shared_out,
               const float* __restrict__ shared_gate, T* __restrict__ y, int64_t Tn, int k,
               int d, int64_t A, int* status) {
  pdl_wait();  // a dependent launch: inputs come from the kernels before
  constexpr int U = KK >= 8 ? 1 : 8 / KK;
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int ng = d >> 3;
  for (int64_t t = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < Tn; t += nwarps) {
    int64_t rows[KK];
    float wj[KK];
    token_rows<KK>(row_of, w, t, k, A, lane, status, rows, wj);
    const float gs = shared_gate != nullptr ? shared_gate[t] : 1.f;
    for (int g0 = 0; g0 < ng; g0 += 32 * U) {
      Raw8<T> raw[U][KK], sraw[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int g = g0 + 32 * u + lane;
#pragma unroll
        for (int j = 0; j < KK; ++j) {
          if (g < ng && j < k && rows[j] >= 0) raw[u][j].load(out_perm + rows[j] * d + 8 * g);
          else raw[u][j].zero();
        }
        if (g < ng && shared_out != nullptr) sraw[u].load(shared_out + t * d + 8 * g);
        else sraw[u].zero();
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int g = g0 + 32 * u + lane;
        if (g >= ng) continue;
        float acc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = 0.f;
#pragma unroll
        for (int j = 0; j < KK; ++j) {
          if (j < k) {
            float v[8];
            raw[u][j].to_float(v);
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] = fmaf(wj[j], v[i], acc[i]);
          }
        }
        float sv[8];
        sraw[u].to_float(sv);
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = fmaf(gs, sv[i], acc[i]);
        store8(y + t * d + 8 * g, acc);
      }
    }
  }
}

// d_out_perm[row] = w * dy[t] (rounded to the act dtype); dw[t, j] = <dy[t], out_perm[row]>
// with per-lane partial sums in a fixed order and a butterfly at the end.
template <typename T, int KK>
__global__ void __launch_bounds__(256)
combine_bwd_kernel(const T* __restrict__ dy, const T* __restrict__ out_perm,
                   const int32_t* __restrict__ row_of, const float* __restrict__ w,
                   T* __restrict__ d_out_perm, float* __restrict__ dw, int64_t Tn, int k,
                   int d, int64_t A, int* status) {
  pdl_wait();  // a dependent launch: inputs come from the kernels before
  constexpr int U = KK >= 8 ? 1 : 8 / KK;
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int ng = d >> 3;
  for (int64_t t = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < Tn; t += nwarps) {
    int64_t rows[KK];
    float wj[KK], dot[KK];
    token_rows<KK>(row_of, w, t, k, A, lane, status, rows, wj);
#pragma unroll
    for (int j = 0; j < KK; ++j) dot[j] = 0.f;
    for (int g0 = 0; g0 < ng; g0 += 32 * U) {
      Raw8<T> graw[U], raw[U][KK];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int g = g0 + 32 * u + lane;
        if (g < ng) graw[u].load(dy + t * d + 8 * g);
        else graw[u].zero();
#pragma unroll
        for (int j = 0; j < KK; ++j) {
          if (g < ng && j < k && rows[j] >= 0) raw[u][j].load(out_perm + rows[j] * d + 8 * g);
          else raw[u][j].zero();
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int g = g0 + 32 * u + lane;
        if (g >= ng) continue;
        float g8[8];
        graw[u].to_float(g8);
#pragma unroll
        for (int j = 0; j < KK; ++j) {
          if (j < k && rows[j] >= 0) {
            float v[8], o[8];
            raw[u][j].to_float(v);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              dot[j] = fmaf(g8[i], v[i], dot[j]);
              o[i] = wj[j] * g8[i];
            }
            store8(d_out_perm + rows[j] * d + 8 * g, o);
          }
        }
      }
    }
#pragma unroll
    for (int j = 0; j < KK; ++j) {
      if (j < k) {
        const float sum = warp_sum(dot[j]);
        if (lane == j) dw[t * k + j] = sum;
      }
    }
  }
}

#define MOE_BY_K(k, MACRO) \
  do {                     \
    if ((k) <= 1) {        \
      MACRO(1);            \
    } else if ((k) <= 2) { \
      MACRO(2);            \
    } else if ((k) <= 4) { \
      MACRO(4);            \
    } else {               \
      MACRO(8);            \
    }                      \
  } while (0)

cudaError_t launch_combine(const Ctx& c, const moe_cfg& cfg, const void* out_perm,
                           const int32_t* row_of, const float* w, const void* shared_out,
                           const float* shared_gate, void* y) {
  if (cfg.T == 0) return cudaSuccess;
  const int64_t A = cfg.T * cfg.k;
  const unsigned grid = token_grid(c, cfg.T);
#define MOE_COMBINE(KK)                                                                       \
  if (cfg.act_dtype == MOE_BF16)                                                             \
    launch_dependent(combine_kernel<bf16, KK>, dim3(grid), dim3(256), 0, c.stream,          \
        static_cast<const bf16*>(out_perm), row_of, w, static_cast<const bf16*>(shared_out), \
        shared_gate, static_cast<bf16*>(y), cfg.T, cfg.k, cfg.d, A, c.status);               \
  else                                                                                       \
    launch_dependent(combine_kernel<float, KK>, dim3(grid), dim3(256), 0, c.stream,         \
        static_cast<const float*>(out_perm), row_of, w,                                      \
        static_cast<const float*>(shared_out), shared_gate, static_cast<float*>(y), cfg.T,   \
        cfg.k, cfg.d, A, c.status)
  MOE_BY_K(cfg.k, MOE_COMBINE);
#undef MOE_COMBINE
  note_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_combine_bwd(const Ctx& c, const moe_cfg& cfg, const void* dy,
                               const void* out_perm, const int32_t* row_of, const float* w,
                               void* d_out_perm, float* dw) {
  if (cfg.T == 0) return cudaSuccess;
  const int64_t A = cfg.T * cfg.k;
  const unsigned grid = token_grid(c, cfg.T);
#define MOE_COMBINE_BWD(KK)                                                                 \
  if (cfg.act_dtype == MOE_BF16)                                                           \
    launch_dependent(combine_bwd_kernel<bf16, KK>, dim3(grid), dim3(256), 0, c.stream,    \
        static_cast<const bf16*>(dy), static_cast<const bf16*>(out_perm), row_of, w,       \
        static_cast<bf16*>(d_out_perm), dw, cfg.T, cfg.k, cfg.d, A, c.status);             \
  else                                                                                     \
    launch_dependent(combine_bwd_kernel<float, KK>, dim3(grid), dim3(256), 0, c.stream,   \
        static_cast<const float*>(dy), static_cast<const float*>(out_perm), row_of, w,     \
        static_cast<float*>(d_out_perm), dw, cfg.T, cfg.k, cfg.d, A, c.status)
  MOE_BY_K(cfg.k, MOE_COMBINE_BWD);
#undef MOE_COMBINE_BWD
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace moe
