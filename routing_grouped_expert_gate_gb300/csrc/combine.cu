// Weighted unpermute-combine (S6) and its backward (B6).
//
// MoE training cluster: routing, load balancing (LeCompute), "An expert
// transforms numbers inside the model": the block returns each chosen expert's
// output times its weight, summed coordinate by coordinate. The Ultimate MoE
// Training Handbook, §3.4 "Shared experts": the shared expert's output is added
// at weight 1.
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

template <typename T>
__global__ void __launch_bounds__(256)
combine_kernel(const T* __restrict__ out_perm, const int32_t* __restrict__ row_of,
               const float* __restrict__ w, const T* __restrict__ shared_out,
               T* __restrict__ y, int64_t Tn, int k, int d, int64_t A, int* status) {
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int ng = d >> 3;
  for (int64_t t = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < Tn; t += nwarps) {
    int64_t rows[kMaxK];
    float wj[kMaxK];
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) {
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
    // one 8-element group per lane per step; the k rows (and the shared row)
    // are all loaded before any is used
    for (int g = lane; g < ng; g += 32) {
      Raw8<T> raw[kMaxK];
      Raw8<T> sraw;
#pragma unroll
      for (int j = 0; j < kMaxK; ++j) {
        if (j < k && rows[j] >= 0) raw[j].load(out_perm + rows[j] * d + 8 * g);
        else raw[j].zero();
      }
      if (shared_out != nullptr) sraw.load(shared_out + t * d + 8 * g);
      else sraw.zero();
      float acc[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = 0.f;
#pragma unroll
      for (int j = 0; j < kMaxK; ++j) {
        if (j < k) {
          float v[8];
          raw[j].to_float(v);
#pragma unroll
          for (int i = 0; i < 8; ++i) acc[i] = fmaf(wj[j], v[i], acc[i]);
        }
      }
      float sv[8];
      sraw.to_float(sv);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] += sv[i];
      store8(y + t * d + 8 * g, acc);
    }
  }
}

// d_out_perm[row] = w * dy[t] (rounded to the act dtype); dw[t, j] = <dy[t], out_perm[row]>
// with per-lane partial sums in a fixed order and a butterfly at the end.
template <typename T>
__global__ void __launch_bounds__(256)
combine_bwd_kernel(const T* __restrict__ dy, const T* __restrict__ out_perm,
                   const int32_t* __restrict__ row_of, const float* __restrict__ w,
                   T* __restrict__ d_out_perm, float* __restrict__ dw, int64_t Tn, int k,
                   int d, int64_t A, int* status) {
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int ng = d >> 3;
  for (int64_t t = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < Tn; t += nwarps) {
    int64_t rows[kMaxK];
    float wj[kMaxK], dot[kMaxK];
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) {
      int r = -1;
      wj[j] = 0.f;
      dot[j] = 0.f;
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
    for (int g = lane; g < ng; g += 32) {
      Raw8<T> graw, raw[kMaxK];
      graw.load(dy + t * d + 8 * g);
#pragma unroll
      for (int j = 0; j < kMaxK; ++j) {
        if (j < k && rows[j] >= 0) raw[j].load(out_perm + rows[j] * d + 8 * g);
        else raw[j].zero();
      }
      float g8[8];
      graw.to_float(g8);
#pragma unroll
      for (int j = 0; j < kMaxK; ++j) {
        if (j < k && rows[j] >= 0) {
          float v[8], o[8];
          raw[j].to_float(v);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            dot[j] = fmaf(g8[i], v[i], dot[j]);
            o[i] = wj[j] * g8[i];
          }
          store8(d_out_perm + rows[j] * d + 8 * g, o);
        }
      }
    }
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) {
      if (j < k) {
        const float s = warp_sum(dot[j]);
        if (lane == j) dw[t * k + j] = s;
      }
    }
  }
}

cudaError_t launch_combine(const Ctx& c, const moe_cfg& cfg, const void* out_perm,
                           const int32_t* row_of, const float* w, const void* shared_out,
                           void* y) {
  if (cfg.T == 0) return cudaSuccess;
  const int64_t A = cfg.T * cfg.k;
  if (cfg.act_dtype == MOE_BF16)
    combine_kernel<bf16><<<token_grid(c, cfg.T), 256, 0, c.stream>>>(
        static_cast<const bf16*>(out_perm), row_of, w, static_cast<const bf16*>(shared_out),
        static_cast<bf16*>(y), cfg.T, cfg.k, cfg.d, A, c.status);
  else
    combine_kernel<float><<<token_grid(c, cfg.T), 256, 0, c.stream>>>(
        static_cast<const float*>(out_perm), row_of, w, static_cast<const float*>(shared_out),
        static_cast<float*>(y), cfg.T, cfg.k, cfg.d, A, c.status);
  note_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_combine_bwd(const Ctx& c, const moe_cfg& cfg, const void* dy,
                               const void* out_perm, const int32_t* row_of, const float* w,
                               void* d_out_perm, float* dw) {
  if (cfg.T == 0) return cudaSuccess;
  const int64_t A = cfg.T * cfg.k;
  if (cfg.act_dtype == MOE_BF16)
    combine_bwd_kernel<bf16><<<token_grid(c, cfg.T), 256, 0, c.stream>>>(
        static_cast<const bf16*>(dy), static_cast<const bf16*>(out_perm), row_of, w,
        static_cast<bf16*>(d_out_perm), dw, cfg.T, cfg.k, cfg.d, A, c.status);
  else
    combine_bwd_kernel<float><<<token_grid(c, cfg.T), 256, 0, c.stream>>>(
        static_cast<const float*>(dy), static_cast<const float*>(out_perm), row_of, w,
        static_cast<float*>(d_out_perm), dw, cfg.T, cfg.k, cfg.d, A, c.status);
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace moe
