// Register-tiled SIMT GEMM with fp32 accumulation, plus the SwiGLU elementwise
// steps used around it.
//
// Serves the parts of the layer that are not bf16 tensor-core contractions:
//   * the fp32 expert path (grouped over expert segments along M for fc1/fc2
//     and their dgrad, along K for the weight gradients), and
//   * the router backward: dx_router = d_logits · W_r (K = E) and
//     dW_r = d_logitsᵀ · x (K = T, split over K with partials reduced in a fixed
//     order so the result is deterministic).
//
// A CTA computes a 128 x 64 tile of C with 256 threads (4 x 8 per thread: rows
// 4ty..4ty+3, columns {4tx..4tx+3} and {32+4tx..32+4tx+3}, so the eight threads
// of one shared-memory phase read 128 consecutive bytes); K advances 32 at a
// time through shared memory. Operands are addressed through
// element strides, so the same kernel reads K-contiguous or M/N-contiguous
// matrices; consecutive threads always touch consecutive addresses.
#include "common.cuh"
#include "internal.h"
#include "glu_act.cuh"

namespace moe {

constexpr int SG_BM = 128, SG_BN = 64, SG_KC = 32;

template <typename T>
__device__ __forceinline__ float ldf(const void* p, int64_t i) {
  return to_f32<T>(static_cast<const T*>(p)[i]);
}

template <typename TA, typename TB, typename TC>
__global__ void __launch_bounds__(256, 2) simt_gemm_kernel(SimtGemm g, int mode, int* status) {
  __shared__ __align__(16) float As[SG_KC][SG_BM + 4];
  __shared__ __align__(16) float Bs[SG_KC][SG_BN + 4];
  __shared__ int s_info[4];

  const int tid = threadIdx.x;
  const int ty = tid >> 3, tx = tid & 7;

  int64_t m0 = 0, m_lim = g.M, k_beg = 0, k_end = g.K;
  const void* Ap = g.A;
  const void* Bp = g.B;
  void* Cp = g.C;
  const int n0 = blockIdx.y * SG_BN;

  if (mode == kGroupM) {
    // map this CTA's virtual tile to (group, first row) by walking the segments
    if (tid == 0) {
      int found = -1, row0 = 0, rowlim = 0;
      int64_t acc = 0;
      const int vt = blockIdx.x;
      for (int i = 0; i < g.n_groups; ++i) {
        const int a = g.offsets ? g.offsets[i] : 0;
        const int b = g.offsets ? g.offsets[i + 1] : g.M;
        if (b < a || a < 0 || b > g.M) {
          record_error(status, MOE_ERR_DEVICE_INDEX, i);
          continue;
        }
        const int64_t tiles = (b - a + SG_BM - 1) / SG_BM;
        if (vt < acc + tiles) {
          found = i;
          row0 = a + (int)(vt - acc) * SG_BM;
          rowlim = b;
          break;
        }
        acc += tiles;
      }
      s_info[0] = found;
      s_info[1] = row0;
      s_info[2] = rowlim;
    }
    __syncthreads();
    const int grp = s_info[0];
    if (grp < 0) return;
    m0 = s_info[1];
    m_lim = s_info[2];
    Bp = static_cast<const char*>(g.B) + (int64_t)grp * g.b_sg * (int64_t)sizeof(TB);
  } else if (mode == kGroupK) {
    const int grp = blockIdx.z;
    m0 = (int64_t)blockIdx.x * SG_BM;
    const int a = g.offsets ? g.offsets[grp] : 0;
    const int b = g.offsets ? g.offsets[grp + 1] : g.K;
    if (b < a || a < 0 || b > g.K) {
      if (tid == 0) record_error(status, MOE_ERR_DEVICE_INDEX, grp);
      return;
    }
    k_beg = a;
    k_end = b;
    Cp = static_cast<char*>(g.C) + (int64_t)grp * g.c_sg * (int64_t)sizeof(TC);
  } else {
    m0 = (int64_t)blockIdx.x * SG_BM;
    if (g.split_k > 1) {
      const int64_t chunk = ((g.K + g.split_k - 1) / g.split_k + SG_KC - 1) / SG_KC * SG_KC;
      k_beg = (int64_t)blockIdx.z * chunk;
      k_end = k_beg + chunk < g.K ? k_beg + chunk : g.K;
      Cp = static_cast<char*>(g.C) + (int64_t)blockIdx.z * g.c_sg * (int64_t)sizeof(TC);
    }
  }
  if (m0 >= m_lim) return;

  const bool a_kc = (g.a_sk == 1);
  const bool b_kc = (g.b_sk == 1);
  float acc[4][8];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;

  for (int64_t k0 = k_beg; k0 < k_end; k0 += SG_KC) {
    // A: 128 x 32 elements, 16 per thread; B: 64 x 32, 8 per thread. Consecutive
    // threads read consecutive addresses whichever way the operand is laid out.
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      const int lin = tid + 256 * r;
      int mm, kk;
      if (a_kc) { mm = lin >> 5; kk = lin & 31; } else { kk = lin >> 7; mm = lin & 127; }
      const int64_t gm = m0 + mm, gk = k0 + kk;
      As[kk][mm] = (gm < m_lim && gk < k_end) ? ldf<TA>(Ap, gm * g.a_sm + gk * g.a_sk) : 0.f;
    }
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const int lin = tid + 256 * r;
      int nn, kk;
      if (b_kc) { nn = lin >> 5; kk = lin & 31; } else { kk = lin >> 6; nn = lin & 63; }
      const int64_t gn = n0 + nn, gk = k0 + kk;
      Bs[kk][nn] = (gn < g.N && gk < k_end) ? ldf<TB>(Bp, gn * g.b_sn + gk * g.b_sk) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < SG_KC; ++kk) {
      const float4 a = *reinterpret_cast<const float4*>(&As[kk][4 * ty]);
      const float4 b0 = *reinterpret_cast<const float4*>(&Bs[kk][4 * tx]);
      const float4 b1 = *reinterpret_cast<const float4*>(&Bs[kk][32 + 4 * tx]);
      const float av[4] = {a.x, a.y, a.z, a.w};
      const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    __syncthreads();
  }

  TC* C = static_cast<TC*>(Cp);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t gm = m0 + 4 * ty + i;
    if (gm >= m_lim) continue;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int64_t gn = n0 + (j < 4 ? 4 * tx + j : 32 + 4 * tx + (j - 4));
      if (gn >= g.N) continue;
      float v = g.alpha * acc[i][j];
      TC* dst = C + gm * g.c_sm + gn * (g.c_sn ? g.c_sn : 1);
      if (g.accumulate) v += to_f32<TC>(*dst);
      *dst = from_f32<TC>(v);
    }
  }
}

cudaError_t launch_simt_gemm(const Ctx& c, const SimtGemm& g) {
  if (g.M <= 0 || g.N <= 0) return cudaSuccess;
  const int mode = g.mode;
  dim3 grid;
  const unsigned gn = (unsigned)((g.N + SG_BN - 1) / SG_BN);
  if (mode == kGroupK) {
    // one z-slice per group; an empty group still runs and writes zeros
    grid = dim3((unsigned)((g.M + SG_BM - 1) / SG_BM), gn, (unsigned)g.n_groups);
  } else if (mode == kGroupM) {
    // sum_g ceil(n_g / 64) <= M / 64 + n_groups virtual tiles; the surplus exits
    const int64_t vt = (g.M + SG_BM - 1) / SG_BM + g.n_groups;
    grid = dim3((unsigned)vt, gn, 1);
  } else {
    grid = dim3((unsigned)((g.M + SG_BM - 1) / SG_BM), gn,
                (unsigned)(g.split_k > 1 ? g.split_k : 1));
  }
#define MOE_SG(TA, TB, TC) simt_gemm_kernel<TA, TB, TC><<<grid, 256, 0, c.stream>>>(g, mode, c.status)
  if (g.dtA == kF32 && g.dtB == kF32 && g.dtC == kF32) MOE_SG(float, float, float);
  else if (g.dtA == kBF16 && g.dtB == kBF16 && g.dtC == kBF16) MOE_SG(bf16, bf16, bf16);
  else if (g.dtA == kBF16 && g.dtB == kBF16 && g.dtC == kF32) MOE_SG(bf16, bf16, float);
  else if (g.dtA == kF32 && g.dtB == kBF16 && g.dtC == kF32) MOE_SG(float, bf16, float);
  else if (g.dtA == kF32 && g.dtB == kF32 && g.dtC == kBF16) MOE_SG(float, float, bf16);
  else if (g.dtA == kBF16 && g.dtB == kF32 && g.dtC == kF32) MOE_SG(bf16, float, float);
  else return cudaErrorInvalidValue;
#undef MOE_SG
  note_launches(1);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ reduce
template <typename TO>
__global__ void __launch_bounds__(256)
reduce_partials_kernel(const float* __restrict__ part, int64_t stride, int nz, int64_t n,
                       TO* __restrict__ out, int accumulate) {
  pdl_wait();  // a dependent launch: inputs come from the kernels before
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    // the partials added in slice order, sixteen loads in flight at a time
    float v = 0.f;
    for (int z0 = 0; z0 < nz; z0 += 16) {
      float p[16];
#pragma unroll
      for (int u = 0; u < 16; ++u) p[u] = z0 + u < nz ? part[(int64_t)(z0 + u) * stride + i] : 0.f;
#pragma unroll
      for (int u = 0; u < 16; ++u)
        if (z0 + u < nz) v += p[u];
    }
    if (accumulate) v += to_f32<TO>(out[i]);
    out[i] = from_f32<TO>(v);
  }
}

cudaError_t launch_reduce_partials(const Ctx& c, const float* part, int64_t stride, int nz,
                                   int64_t n, void* out, int dt_out, int accumulate) {
  if (n <= 0) return cudaSuccess;
  const int64_t blocks = (n + 255) / 256;
  const unsigned grid = (unsigned)(blocks < (int64_t)c.sm_count * 8 ? blocks : c.sm_count * 8);
  if (dt_out == kF32)
    launch_dependent(reduce_partials_kernel<float>, dim3(grid), dim3(256), 0, c.stream, part,
                     stride, nz, n, static_cast<float*>(out), accumulate);
  else
    launch_dependent(reduce_partials_kernel<bf16>, dim3(grid), dim3(256), 0, c.stream, part,
                     stride, nz, n, static_cast<bf16*>(out), accumulate);
  note_launches(1);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ SwiGLU elementwise
// Handbook §3.4 "Activation": the first half of fc1's output is the gate,
// h = act(gate, up): SwiGLU or one of its variants (glu_fwd).
template <typename T>
__global__ void __launch_bounds__(256)
swiglu_fwd_elem(const T* __restrict__ pre, T* __restrict__ h, int64_t rows, int F, GluAct act) {
  const int64_t n = rows * F;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / F;
    const int f = (int)(i - r * F);
    const float gt = to_f32<T>(pre[r * 2 * F + f]);
    const float up = to_f32<T>(pre[r * 2 * F + F + f]);
    h[i] = from_f32<T>(glu_fwd(gt, up, act));
  }
}

// d_pre = [dh * d h / d g | dh * d h / d u] of the activation (glu_bwd)
template <typename T>
__global__ void __launch_bounds__(256)
swiglu_bwd_elem(const float* __restrict__ dh, const T* __restrict__ pre, T* __restrict__ d_pre,
                int64_t rows, int F, GluAct act) {
  const int64_t n = rows * F;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / F;
    const int f = (int)(i - r * F);
    const float gt = to_f32<T>(pre[r * 2 * F + f]);
    const float up = to_f32<T>(pre[r * 2 * F + F + f]);
    float dg, du;
    glu_bwd(gt, up, dh[i], act, dg, du);
    d_pre[r * 2 * F + f] = from_f32<T>(dg);
    d_pre[r * 2 * F + F + f] = from_f32<T>(du);
  }
}

static unsigned elem_grid(const Ctx& c, int64_t n) {
  const int64_t blocks = (n + 255) / 256;
  const int64_t cap = (int64_t)c.sm_count * 16;
  return (unsigned)(blocks < cap ? (blocks > 0 ? blocks : 1) : cap);
}

cudaError_t launch_swiglu_fwd_elem(const Ctx& c, int dt, const void* pre_gu, void* h,
                                   int64_t rows, int F) {
  if (rows * F == 0) return cudaSuccess;
  if (dt == kBF16)
    swiglu_fwd_elem<bf16><<<elem_grid(c, rows * F), 256, 0, c.stream>>>(
        static_cast<const bf16*>(pre_gu), static_cast<bf16*>(h), rows, F, c.act);
  else
    swiglu_fwd_elem<float><<<elem_grid(c, rows * F), 256, 0, c.stream>>>(
        static_cast<const float*>(pre_gu), static_cast<float*>(h), rows, F, c.act);
  note_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_swiglu_bwd_elem(const Ctx& c, int dt, const float* dh, const void* pre_gu,
                                   void* d_pre, int64_t rows, int F) {
  if (rows * F == 0) return cudaSuccess;
  if (dt == kBF16)
    swiglu_bwd_elem<bf16><<<elem_grid(c, rows * F), 256, 0, c.stream>>>(
        dh, static_cast<const bf16*>(pre_gu), static_cast<bf16*>(d_pre), rows, F, c.act);
  else
    swiglu_bwd_elem<float><<<elem_grid(c, rows * F), 256, 0, c.stream>>>(
        dh, static_cast<const float*>(pre_gu), static_cast<float*>(d_pre), rows, F, c.act);
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace moe
