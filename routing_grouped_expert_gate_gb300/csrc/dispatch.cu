// Dispatch (S3) and its backward (B1).
//
// MoE training cluster: routing, load balancing (LeCompute): "Four GPUs, with
// one holding up the group" counts the T*k token-expert assignments of each
// expert; "Read the timeline before blaming the network" groups the token rows
// by expert before the expert GEMMs and restores the order afterwards.
//
// Four launches, all on the caller's stream, no host sync:
//   count : per block of 128 tokens, a bitmask per expert of which tokens in the
//           block chose it (shared memory), popcounts -> per-block counts
//   scan  : one CTA; per expert, exclusive scan over blocks; exclusive scan over
//           experts -> counts, offsets, absolute base row of each (block, expert)
//   rank  : rebuilds the block's bitmasks; the rank of token t among the tokens
//           of its block that chose e is a popcount of the bits below t, so
//           row(t, e) = base(block, e) + rank: expert-contiguous, stable
//   copy  : one warp per token reads its row once and writes it to its k rows
//           with 16-byte accesses (the HBM-bound part)
#include "common.cuh"
#include "internal.h"

namespace moe {

constexpr int PB_TOK = 128;           // tokens per count/rank block
constexpr int PB_WORDS = PB_TOK / 32;  // bitmask words per expert

static int64_t permute_blocks(int64_t T) { return (T + PB_TOK - 1) / PB_TOK; }

size_t permute_ws_bytes(const moe_cfg& cfg) {
  const size_t n = (size_t)permute_blocks(cfg.T) * (size_t)cfg.E * sizeof(int32_t);
  return (n + 255) & ~(size_t)255;
}

__device__ __forceinline__ void build_masks(uint32_t (*masks)[PB_WORDS], const int32_t* idx,
                                            int64_t T, int k, int E, int* status,
                                            bool record) {
  for (int i = threadIdx.x; i < E * PB_WORDS; i += blockDim.x) masks[i / PB_WORDS][i % PB_WORDS] = 0u;
  __syncthreads();
  const int64_t t_base = (int64_t)blockIdx.x * PB_TOK;
  for (int i = threadIdx.x; i < PB_TOK * k; i += blockDim.x) {
    const int tl = i / k;
    const int64_t t = t_base + tl;
    if (t >= T) continue;
    const int e = idx[t * k + (i - tl * k)];
    if (e < 0 || e >= E) {
      if (record) record_error(status, MOE_ERR_DEVICE_INDEX, (int)t);
      continue;
    }
    const uint32_t bit = 1u << (tl & 31);
    const uint32_t old = atomicOr(&masks[e][tl >> 5], bit);
    if ((old & bit) && record) record_error(status, MOE_ERR_DEVICE_INDEX, (int)t);  // repeated expert
  }
  __syncthreads();
}

__global__ void __launch_bounds__(256)
permute_count(const int32_t* __restrict__ idx, int64_t T, int k, int E,
              int32_t* __restrict__ block_counts, int* status) {
  __shared__ uint32_t masks[kMaxE][PB_WORDS];
  build_masks(masks, idx, T, k, E, status, true);
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int c = 0;
#pragma unroll
    for (int w = 0; w < PB_WORDS; ++w) c += __popc(masks[e][w]);
    block_counts[(int64_t)blockIdx.x * E + e] = c;
  }
}

__global__ void __launch_bounds__(256)
permute_scan(int32_t* __restrict__ block_counts, int64_t nblk, int E,
             int32_t* __restrict__ counts, int32_t* __restrict__ offsets) {
  __shared__ int32_t tot[kMaxE];
  __shared__ int32_t base[kMaxE];
  const int e = threadIdx.x;
  int run = 0;
  if (e < E) {
    // eight independent loads in flight, then the running sum over them
    for (int64_t b0 = 0; b0 < nblk; b0 += 8) {
      int v[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = (b0 + i < nblk) ? block_counts[(b0 + i) * E + e] : 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        if (b0 + i < nblk) {
          block_counts[(b0 + i) * E + e] = run;
          run += v[i];
        }
      }
    }
    counts[e] = run;
    tot[e] = run;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int acc = 0;
    for (int i = 0; i < E; ++i) {
      base[i] = acc;
      offsets[i] = acc;
      acc += tot[i];
    }
    offsets[E] = acc;
  }
  __syncthreads();
  if (e < E) {
    const int base_e = base[e];
    for (int64_t b0 = 0; b0 < nblk; b0 += 8) {
      int v[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = (b0 + i < nblk) ? block_counts[(b0 + i) * E + e] : 0;
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (b0 + i < nblk) block_counts[(b0 + i) * E + e] = v[i] + base_e;
    }
  }
}

__global__ void __launch_bounds__(256)
permute_rank(const int32_t* __restrict__ idx, int64_t T, int k, int E,
             const int32_t* __restrict__ block_base, int32_t* __restrict__ row_of,
             int32_t* __restrict__ src_tok, int* status) {
  __shared__ uint32_t masks[kMaxE][PB_WORDS];
  build_masks(masks, idx, T, k, E, status, false);
  const int64_t t_base = (int64_t)blockIdx.x * PB_TOK;
  for (int i = threadIdx.x; i < PB_TOK * k; i += blockDim.x) {
    const int tl = i / k;
    const int64_t t = t_base + tl;
    if (t >= T) continue;
    const int j = i - tl * k;
    const int e = idx[t * k + j];
    if (e < 0 || e >= E) {
      row_of[t * k + j] = -1;
      continue;
    }
    int rank = __popc(masks[e][tl >> 5] & ((1u << (tl & 31)) - 1u));
    for (int w = 0; w < (tl >> 5); ++w) rank += __popc(masks[e][w]);
    const int row = block_base[(int64_t)blockIdx.x * E + e] + rank;
    row_of[t * k + j] = row;
    src_tok[row] = (int32_t)t;
  }
}

// One warp per token; 4 x 16 B loads in flight per lane before the k stores.
template <typename T>
__global__ void __launch_bounds__(256)
permute_copy(const T* __restrict__ x, const int32_t* __restrict__ row_of, T* __restrict__ x_perm,
             int64_t Tn, int k, int d, int64_t A) {
  const int lane = threadIdx.x & 31;
  const int nvec = d * (int)sizeof(T) / 16;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t t = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < Tn; t += nwarps) {
    int64_t rows[kMaxK];
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) {
      int r = (j < k) ? row_of[t * k + j] : -1;
      rows[j] = (r >= 0 && r < A) ? r : -1;
    }
    const uint4* src = reinterpret_cast<const uint4*>(x + t * d);
    for (int v0 = 0; v0 < nvec; v0 += 128) {
      uint4 buf[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int v = v0 + u * 32 + lane;
        if (v < nvec) buf[u] = __ldg(src + v);
      }
#pragma unroll
      for (int j = 0; j < kMaxK; ++j) {
        if (j < k && rows[j] >= 0) {
          uint4* dst = reinterpret_cast<uint4*>(x_perm + rows[j] * d);
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int v = v0 + u * 32 + lane;
            if (v < nvec) dst[v] = buf[u];
          }
        }
      }
    }
  }
}

static unsigned copy_grid(const Ctx& c, int64_t warps) {
  const int64_t blocks = (warps + 7) / 8;
  const int64_t cap = (int64_t)c.sm_count * 8;
  return (unsigned)(blocks < cap ? (blocks > 0 ? blocks : 1) : cap);
}

cudaError_t launch_permute(const Ctx& c, const moe_cfg& cfg, const void* x, const int32_t* idx,
                           int32_t* counts, int32_t* offsets, int32_t* row_of,
                           int32_t* src_tok, void* x_perm, void* ws) {
  const int64_t nblk = permute_blocks(cfg.T);
  int32_t* block_counts = static_cast<int32_t*>(ws);
  if (nblk > 0) {
    permute_count<<<(unsigned)nblk, 256, 0, c.stream>>>(idx, cfg.T, cfg.k, cfg.E, block_counts,
                                                         c.status);
  }
  permute_scan<<<1, 256, 0, c.stream>>>(block_counts, nblk, cfg.E, counts, offsets);
  if (nblk > 0) {
    permute_rank<<<(unsigned)nblk, 256, 0, c.stream>>>(idx, cfg.T, cfg.k, cfg.E, block_counts,
                                                        row_of, src_tok, c.status);
    const int64_t A = cfg.T * cfg.k;
    if (cfg.act_dtype == MOE_BF16)
      permute_copy<bf16><<<copy_grid(c, cfg.T), 256, 0, c.stream>>>(
          static_cast<const bf16*>(x), row_of, static_cast<bf16*>(x_perm), cfg.T, cfg.k, cfg.d, A);
    else
      permute_copy<float><<<copy_grid(c, cfg.T), 256, 0, c.stream>>>(
          static_cast<const float*>(x), row_of, static_cast<float*>(x_perm), cfg.T, cfg.k, cfg.d,
          A);
  }
  note_launches(nblk > 0 ? 4 : 1);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ B1
// dx[t] = dx_router[t] + sum_j dx_perm[row_of[t, j]] + dx_shared[t], in fp32 in
// that order, rounded once. One warp per token, 8 elements per lane per step.
template <typename T, int KK>
__global__ void __launch_bounds__(256)
permute_bwd_kernel(const T* __restrict__ dx_perm, const int32_t* __restrict__ row_of,
                   const float* __restrict__ dx_router, const T* __restrict__ dx_shared,
                   const float* __restrict__ d_gate_logit, const float* __restrict__ w_gate,
                   T* __restrict__ dx, int64_t Tn, int k, int d, int64_t A, int* status) {
  constexpr int U = KK >= 8 ? 1 : 8 / KK;  // 8-element groups per lane per step
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int ng = d >> 3;
  for (int64_t t = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < Tn; t += nwarps) {
    int64_t rows[KK];
#pragma unroll
    for (int j = 0; j < KK; ++j) {
      int r = (j < k) ? row_of[t * k + j] : -1;
      if (j < k && (r < 0 || r >= A)) {
        if (lane == 0) record_error(status, MOE_ERR_DEVICE_INDEX, (int)t);
        r = -1;
      }
      rows[j] = r;
    }
    const float dgl = d_gate_logit != nullptr ? d_gate_logit[t] : 0.f;
    for (int g0 = 0; g0 < ng; g0 += 32 * U) {
      Raw8<T> raw[U][KK], sraw[U];
      Raw8<float> rraw[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int g = g0 + 32 * u + lane;
        if (g < ng && dx_router != nullptr) rraw[u].load(dx_router + t * d + 8 * g);
        else rraw[u].zero();
#pragma unroll
        for (int j = 0; j < KK; ++j) {
          if (g < ng && j < k && rows[j] >= 0) raw[u][j].load(dx_perm + rows[j] * d + 8 * g);
          else raw[u][j].zero();
        }
        if (g < ng && dx_shared != nullptr) sraw[u].load(dx_shared + t * d + 8 * g);
        else sraw[u].zero();
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int g = g0 + 32 * u + lane;
        if (g >= ng) continue;
        float acc[8];
        rraw[u].to_float(acc);
#pragma unroll
        for (int j = 0; j < KK; ++j) {
          if (j < k) {
            float v[8];
            raw[u][j].to_float(v);
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] += v[i];
          }
        }
        float sv[8];
        sraw[u].to_float(sv);
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] += sv[i];
        if (d_gate_logit != nullptr) {
          // the shared-expert gate's path: d(logit) * w_gate
          float wg[8];
          load8(w_gate + 8 * g, wg);
#pragma unroll
          for (int i = 0; i < 8; ++i) acc[i] = fmaf(dgl, wg[i], acc[i]);
        }
        store8(dx + t * d + 8 * g, acc);
      }
    }
  }
}

cudaError_t launch_permute_bwd(const Ctx& c, const moe_cfg& cfg, const void* dx_perm,
                               const int32_t* row_of, const float* dx_router,
                               const void* dx_shared, const float* d_gate_logit,
                               const float* w_gate, void* dx) {
  if (cfg.T == 0) return cudaSuccess;
  const int64_t A = cfg.T * cfg.k;
  const unsigned grid = copy_grid(c, cfg.T);
#define MOE_PBWD(KK)                                                                          \
  if (cfg.act_dtype == MOE_BF16)                                                             \
    permute_bwd_kernel<bf16, KK><<<grid, 256, 0, c.stream>>>(                                 \
        static_cast<const bf16*>(dx_perm), row_of, dx_router,                                \
        static_cast<const bf16*>(dx_shared), d_gate_logit, w_gate, static_cast<bf16*>(dx),   \
        cfg.T, cfg.k, cfg.d, A, c.status);                                                   \
  else                                                                                       \
    permute_bwd_kernel<float, KK><<<grid, 256, 0, c.stream>>>(                                \
        static_cast<const float*>(dx_perm), row_of, dx_router,                               \
        static_cast<const float*>(dx_shared), d_gate_logit, w_gate, static_cast<float*>(dx), \
        cfg.T, cfg.k, cfg.d, A, c.status)
  if (cfg.k <= 1) {
    MOE_PBWD(1);
  } else if (cfg.k <= 2) {
    MOE_PBWD(2);
  } else if (cfg.k <= 4) {
    MOE_PBWD(4);
  } else {
    MOE_PBWD(8);
  }
#undef MOE_PBWD
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace moe
