// Dispatch (S3) and its backward (B1).
//
// MoE training cluster: routing, load balancing (LeCompute): "Four GPUs, with
// one holding up the group" counts the T*k token-expert assignments of each
// expert; "Read the timeline before blaming the network" groups the token rows
// by expert before the expert GEMMs and restores the order afterwards.
//
// Two launches on the caller's stream, no host sync, the second a programmatic
// dependent launch of the first (scheduled while it runs, waiting on
// griddepcontrol.wait for its results, which hides the launch gap):
//   count     : per block of 128 tokens, a bitmask per expert of which tokens in
//               the block chose it (shared memory), popcounts -> per-block counts
//   rank+copy : several CTAs per 128-token block. Each sums the count matrix
//               (expert totals, and per expert the blocks before its own), scans
//               the totals over experts -> the base row of each expert in its
//               block (CTA 0 writes counts and offsets); rebuilds the block's
//               bitmasks: the rank of token t among the block's tokens that
//               chose e is a popcount of the bits below t, so row(t, e) =
//               base(block, e) + rank: expert-contiguous and stable. Each CTA
//               then copies its share of the block's tokens, one warp per token
//               reading the row once and writing its k copies with 16-byte
//               accesses (the HBM-bound part).
// Beyond 16384 (block, expert) cells the per-CTA sums would grow too large and
// the older four-launch form runs: count, a one-thread-per-expert scan, rank,
// copy.
#include <type_traits>

#include "common.cuh"
#include "internal.h"
#include "tc_ptx.cuh"

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
  pdl_wait();  // idx comes from the kernel before (when launched as a dependent)
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

// CTA (block b, part p) of `parts`, from the per-(block, expert) counts of
// permute_count: the base rows it needs, then the bitmasks of block b, then for
// the tokens of part p the rows row(t, j) = base(b, e) + rank (written to
// row_of and src_tok) and the copy x_perm[row(t, j)] = x[t], one warp per token.
// base(b, e) = offsets[e] + sum_{b' < b} cnt[b'][e], offsets the exclusive scan
// of the expert totals: every CTA sums the count matrix itself (threads split
// it by expert and by chunks of blocks), which takes the place of a separate
// scan launch; CTA 0 also writes counts and offsets.
template <typename T>
__global__ void __launch_bounds__(256)
permute_rank_copy(const T* __restrict__ x, const int32_t* __restrict__ idx, int64_t Tn, int k,
                  int E, int d, int parts, int nblk, const int32_t* __restrict__ block_counts,
                  int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                  int32_t* __restrict__ row_of, int32_t* __restrict__ src_tok,
                  T* __restrict__ x_perm) {
  __shared__ uint32_t masks[kMaxE][PB_WORDS];
  __shared__ int32_t s_rows[PB_TOK][kMaxK];
  __shared__ int32_t s_tot[256], s_pre[256];  // [chunk][expert] partial sums
  __shared__ int32_t s_base[kMaxE];
  pdl_wait();
  const int blk = blockIdx.x / parts;
  const int part = blockIdx.x - blk * parts;
  // ---- the count matrix: expert totals and this block's prefix, per chunk
  {
    int C = (int)blockDim.x / E;
    if (C > nblk) C = nblk;
    const int e = threadIdx.x % E, c = threadIdx.x / E;
    if (c < C) {
      const int b0 = (int)((int64_t)nblk * c / C), b1 = (int)((int64_t)nblk * (c + 1) / C);
      int tot = 0, pre = 0;
      for (int i0 = b0; i0 < b1; i0 += 16) {
        int v[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          v[i] = (i0 + i < b1) ? block_counts[(int64_t)(i0 + i) * E + e] : 0;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          tot += v[i];
          pre += (i0 + i < blk) ? v[i] : 0;
        }
      }
      s_tot[c * E + e] = tot;
      s_pre[c * E + e] = pre;
    }
    for (int i = threadIdx.x; i < E * PB_WORDS; i += blockDim.x) masks[i / PB_WORDS][i % PB_WORDS] = 0u;
    __syncthreads();
    if (threadIdx.x < E) {
      int tot = 0, pre = 0;
      for (int cc = 0; cc < C; ++cc) {
        tot += s_tot[cc * E + threadIdx.x];
        pre += s_pre[cc * E + threadIdx.x];
      }
      s_base[threadIdx.x] = tot;  // the total, scanned below
      s_pre[threadIdx.x] = pre;   // (row 0 of s_pre: this thread's own cell)
    }
    __syncthreads();
    if (threadIdx.x < 32) {  // exclusive scan of the totals over experts, one warp
      const int per = (E + 31) / 32;
      const int lo = threadIdx.x * per;
      int loc = 0;
      for (int i = lo; i < lo + per && i < E; ++i) loc += s_base[i];
      int incl = loc;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int w = __shfl_up_sync(0xffffffffu, incl, off);
        if ((int)threadIdx.x >= off) incl += w;
      }
      int run = incl - loc;
      for (int i = lo; i < lo + per && i < E; ++i) {
        const int w = s_base[i];
        if (blockIdx.x == 0) {
          counts[i] = w;
          offsets[i] = run;
        }
        s_base[i] = run + s_pre[i];  // base row of (this block, expert i)
        run += w;
      }
      if (blockIdx.x == 0 && threadIdx.x == 31) offsets[E] = incl;
    }
  }
  // ---- bitmasks of the block (the block's indices kept for the ranks)
  const int64_t t_base = (int64_t)blk * PB_TOK;
  for (int i = threadIdx.x; i < PB_TOK * k; i += blockDim.x) {
    const int tl = i / k;
    const int64_t t = t_base + tl;
    if (t >= Tn) continue;
    const int e = idx[t * k + (i - tl * k)];
    if (e >= 0 && e < E) atomicOr(&masks[e][tl >> 5], 1u << (tl & 31));
  }
  __syncthreads();
  const int per = PB_TOK / parts;
  const int tl0 = part * per;
  for (int i = threadIdx.x; i < per * k; i += blockDim.x) {
    const int tl = tl0 + i / k;
    const int j = i % k;
    const int64_t t = t_base + tl;
    if (t >= Tn) continue;
    const int e = idx[t * k + j];
    int row = -1;
    if (e >= 0 && e < E) {
      int rank = __popc(masks[e][tl >> 5] & ((1u << (tl & 31)) - 1u));
      for (int w = 0; w < (tl >> 5); ++w) rank += __popc(masks[e][w]);
      row = s_base[e] + rank;
      src_tok[row] = (int32_t)t;
    }
    row_of[t * k + j] = row;
    s_rows[tl][j] = row;
  }
  if (x_perm == nullptr) return;  // the index outputs only
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nvec = d * (int)sizeof(T) / 16;
  for (int tl = tl0 + warp; tl < tl0 + per; tl += (int)(blockDim.x >> 5)) {
    const int64_t t = t_base + tl;
    if (t >= Tn) break;
    int64_t rows[kMaxK];
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) rows[j] = (j < k) ? s_rows[tl][j] : -1;
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
  const int64_t A = cfg.T * cfg.k;
  if (nblk > 0 && nblk * cfg.E <= 16384) {
    // count (one CTA per 128-token block), then rank + copy, which also turns
    // the counts into base rows: a dependent launch of the count
    cudaError_t e = launch_dependent(permute_count, dim3((unsigned)nblk), dim3(256), 0, c.stream,
                                     idx, cfg.T, cfg.k, cfg.E, block_counts, c.status);
    if (e != cudaSuccess) return e;
    // CTAs per 128-token block: about four waves of the SMs in all
    int64_t parts = ((int64_t)4 * c.sm_count + nblk - 1) / nblk;
    parts = parts < 1 ? 1 : (parts > 16 ? 16 : parts);
    while (PB_TOK % parts) --parts;
    const unsigned grid = (unsigned)(nblk * parts);
    if (cfg.act_dtype == MOE_BF16)
      e = launch_dependent(permute_rank_copy<bf16>, dim3(grid), dim3(256), 0, c.stream,
                           static_cast<const bf16*>(x), idx, cfg.T, cfg.k, cfg.E, cfg.d,
                           (int)parts, (int)nblk, static_cast<const int32_t*>(block_counts),
                           counts, offsets, row_of, src_tok, static_cast<bf16*>(x_perm));
    else
      e = launch_dependent(permute_rank_copy<float>, dim3(grid), dim3(256), 0, c.stream,
                           static_cast<const float*>(x), idx, cfg.T, cfg.k, cfg.E, cfg.d,
                           (int)parts, (int)nblk, static_cast<const int32_t*>(block_counts),
                           counts, offsets, row_of, src_tok, static_cast<float*>(x_perm));
    note_launches(2);
    return e;
  }
  if (nblk > 0) {
    permute_count<<<(unsigned)nblk, 256, 0, c.stream>>>(idx, cfg.T, cfg.k, cfg.E, block_counts,
                                                         c.status);
  }
  permute_scan<<<1, 256, 0, c.stream>>>(block_counts, nblk, cfg.E, counts, offsets);
  if (nblk > 0) {
    permute_rank<<<(unsigned)nblk, 256, 0, c.stream>>>(idx, cfg.T, cfg.k, cfg.E, block_counts,
                                                        row_of, src_tok, c.status);
    if (x_perm == nullptr) {
      note_launches(3);
      return cudaGetLastError();
    }
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
  pdl_wait();  // a dependent launch: inputs come from the kernels before
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

// B1 with the router's share formed here (few experts): dx[t] = r[t] +
// sum_j dx_perm[row_of[t, j]] + dx_shared[t] (+ d_gate_logit[t] w_gate),
// where r[t] = d_logits[t] · W_r is computed per element with fp32 FMAs over
// the experts in order from 0 (the value the router backward would have
// written as dx_router), and the rest is added in the same order as in
// permute_bwd_kernel, so dx is the same bit for bit while the fp32 [T, d]
// round trip through HBM is gone. W_r sits in shared memory ([E][2][d/8]
// float4 planes, lanes reading consecutive words) when w_smem is set, else it
// is read from global memory. A warp takes TB tokens at a time so that each W
// value read from shared memory serves TB tokens, and U groups of 8 elements
// per lane per step so that enough row loads are in flight.
template <typename T, int KK, int EMAX, int TB>
__global__ void __launch_bounds__(256, 1)
permute_bwd_router(const T* __restrict__ dx_perm, const int32_t* __restrict__ row_of,
                   const T* __restrict__ dx_shared, const float* __restrict__ d_gate_logit,
                   const float* __restrict__ w_gate, const float* __restrict__ d_logits,
                   const float* __restrict__ w_router, T* __restrict__ dx, int64_t Tn, int k,
                   int d, int64_t A, int E, int w_smem, int* status) {
  constexpr int U = sizeof(T) == 2 ? 2 : 1;
  extern __shared__ float4 sW[];
  pdl_wait();  // a dependent launch: inputs come from the kernels before
  if (w_smem) stage_w_planes(sW, w_router, E, d);
  const int lane = threadIdx.x & 31;
  const int ng = d >> 3;
  const int64_t n_tg = (Tn + TB - 1) / TB;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t tg = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); tg < n_tg;
       tg += warps) {
    const int64_t t0 = tg * TB;
    int64_t rows[TB][KK];
    float dl[TB][EMAX], dgl[TB];
#pragma unroll
    for (int a = 0; a < TB; ++a) {
      const int64_t t = t0 + a;
      const bool tv = t < Tn;
#pragma unroll
      for (int j = 0; j < KK; ++j) {
        int r = (tv && j < k) ? row_of[t * k + j] : -1;
        if (tv && j < k && (r < 0 || r >= A)) {
          if (lane == 0) record_error(status, MOE_ERR_DEVICE_INDEX, (int)t);
          r = -1;
        }
        rows[a][j] = r;
      }
#pragma unroll
      for (int e = 0; e < EMAX; ++e) dl[a][e] = (tv && e < E) ? __ldg(d_logits + t * E + e) : 0.f;
      dgl[a] = (tv && d_gate_logit != nullptr) ? d_gate_logit[t] : 0.f;
    }
    for (int g0 = 0; g0 < ng; g0 += 32 * U) {
      Raw8<T> raw[U][TB][KK];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int g = g0 + 32 * u + lane;
#pragma unroll
        for (int a = 0; a < TB; ++a)
#pragma unroll
          for (int j = 0; j < KK; ++j) {
            if (g < ng && j < k && rows[a][j] >= 0)
              raw[u][a][j].load(dx_perm + rows[a][j] * d + 8 * g);
            else
              raw[u][a][j].zero();
          }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int g = g0 + 32 * u + lane;
        if (g >= ng) continue;
        float acc[TB][8];
#pragma unroll
        for (int a = 0; a < TB; ++a)
#pragma unroll
          for (int i = 0; i < 8; ++i) acc[a][i] = 0.f;
#pragma unroll
        for (int e = 0; e < EMAX; ++e) {
          if (e < E) {
            float4 w0, w1;
            if (w_smem) {
              w0 = sW[(e * 2) * ng + g];
              w1 = sW[(e * 2 + 1) * ng + g];
            } else {
              w0 = __ldg(reinterpret_cast<const float4*>(w_router + (int64_t)e * d + 8 * g));
              w1 = __ldg(reinterpret_cast<const float4*>(w_router + (int64_t)e * d + 8 * g + 4));
            }
            const float wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
            for (int a = 0; a < TB; ++a)
#pragma unroll
              for (int i = 0; i < 8; ++i) acc[a][i] = fmaf(dl[a][e], wv[i], acc[a][i]);
          }
        }
        float wg[8];
        if (d_gate_logit != nullptr) load8(w_gate + 8 * g, wg);
#pragma unroll
        for (int a = 0; a < TB; ++a) {
          if (t0 + a >= Tn) continue;
#pragma unroll
          for (int j = 0; j < KK; ++j) {
            if (j < k) {
              float v[8];
              raw[u][a][j].to_float(v);
#pragma unroll
              for (int i = 0; i < 8; ++i) acc[a][i] += v[i];
            }
          }
          Raw8<T> sraw;
          if (dx_shared != nullptr) sraw.load(dx_shared + (t0 + a) * d + 8 * g);
          else sraw.zero();
          float sv[8];
          sraw.to_float(sv);
#pragma unroll
          for (int i = 0; i < 8; ++i) acc[a][i] += sv[i];
          if (d_gate_logit != nullptr) {
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[a][i] = fmaf(dgl[a], wg[i], acc[a][i]);
          }
          store8(dx + (t0 + a) * d + 8 * g, acc[a]);
        }
      }
    }
  }
}

// N = 4 or 8 consecutive bf16 in shared memory <-> N floats (one 8- or
// 16-byte access); stores round to nearest like store8.
template <int N>
__device__ __forceinline__ void load_smem_bf16(const uint8_t* p, float (&v)[N]) {
  static_assert(N == 4 || N == 8, "4 or 8 elements");
  if constexpr (N == 8) {
    load8(reinterpret_cast<const bf16*>(p), v);
  } else {
    const uint2 r = *reinterpret_cast<const uint2*>(p);
    const float2 f0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&r.x));
    const float2 f1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&r.y));
    v[0] = f0.x; v[1] = f0.y; v[2] = f1.x; v[3] = f1.y;
  }
}
template <int N>
__device__ __forceinline__ void store_bf16_n(bf16* p, const float (&v)[N]) {
  static_assert(N == 4 || N == 8, "4 or 8 elements");
  if constexpr (N == 8) {
    store8(p, v);
  } else {
    uint2 r;
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&r);
    h[0] = __floats2bfloat162_rn(v[0], v[1]);
    h[1] = __floats2bfloat162_rn(v[2], v[3]);
    *reinterpret_cast<uint2*>(p) = r;
  }
}

// The same sums for bf16 rows streamed through shared memory. A CTA takes a
// 1024-column slice of d and a slice of the tokens. The slice's rows, d_logits
// and gate logits are staged in shared memory once at the start; then a
// producer warp copies, per ring slot of TS tokens, each token's k row slices
// of dx_perm (and the one of dx_shared) with one bulk copy each, without
// waiting on any load, while sixteen consumer warps keep their lanes' columns
// of W_r (EMAX x CPL values) and of w_gate in registers for the whole kernel
// (so W_r is read once per CTA) and add the slot's rows. The work is bound by
// instruction issue (EMAX FMAs per element): sixteen warps of 4 columns per
// lane measured 25.7 us at T = 4096, d = 4096, E = 8, k = 2 against 31.1 us
// for eight warps of 8 columns. Per element the
// arithmetic is that of permute_bwd_router, in the same order: dx is the same
// bit for bit. Every mbarrier wait is bounded (MOE_ERR_TIMEOUT + abort flag).
constexpr int kPbCols = 1024;       // columns per CTA
constexpr int kPbRowsPerSlot = 16;  // row slices per slot (TS tokens x (k + shared))
constexpr int kPbMaxSlots = 6;
constexpr int kPbConsumers = 16;    // consumer warps
constexpr int kPbThreads = 32 * (kPbConsumers + 1);  // + 1 producer warp
constexpr size_t kPbRingSmem = 192 * 1024;
constexpr size_t kPbTableSmem = 32 * 1024;

struct PbParams {
  int64_t T, A;
  int d, k, E, ns, tok_per_cta;
  int* status;
  uint64_t timeout_ns;
};

template <int KK, int EMAX, bool SH>
struct PbTile {
  static constexpr int CPL = 4;                       // columns per lane
  static constexpr int WCOLS = 32 * CPL;              // columns per warp
  static constexpr int QUARTERS = kPbCols / WCOLS;    // warps across the slice: 8
  static constexpr int TGROUPS = kPbConsumers / QUARTERS;  // token classes: 2
  static constexpr int RPT = KK + (SH ? 1 : 0);       // row slices per token (+ shared)
  static constexpr int TS = kPbRowsPerSlot / RPT > 0 ? kPbRowsPerSlot / RPT : 1;  // tokens per slot
  static constexpr int kSlot = TS * RPT * kPbCols * 2;  // bytes
};

template <int KK, int EMAX, bool SH>
__global__ void __launch_bounds__(kPbThreads, 1)
permute_bwd_router_stream(const bf16* __restrict__ dx_perm, const int32_t* __restrict__ row_of,
                          const bf16* __restrict__ dx_shared, const float* __restrict__ d_gate_logit,
                          const float* __restrict__ w_gate, const float* __restrict__ d_logits,
                          const float* __restrict__ w_router, bf16* __restrict__ dx,
                          const PbParams P) {
  using PT = PbTile<KK, EMAX, SH>;
  constexpr int TS = PT::TS, RPT = PT::RPT, CPL = PT::CPL;
  static_assert(TS * RPT <= 32, "one row slice per producer lane");
  extern __shared__ __align__(128) uint8_t sm_raw[];
  __shared__ __align__(8) uint64_t full[kPbMaxSlots], empty[kPbMaxSlots];
  __shared__ int abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int d = P.d, k = P.k, E = P.E, ns = P.ns;
  const int c0 = blockIdx.x * kPbCols;
  const int cols = d - c0 < kPbCols ? d - c0 : kPbCols;
  const int64_t t_beg = (int64_t)blockIdx.y * P.tok_per_cta;
  const int64_t t_end = t_beg + P.tok_per_cta < P.T ? t_beg + P.tok_per_cta : P.T;
  const int ntok = (int)(t_end - t_beg);
  const int nslots = (ntok + TS - 1) / TS;
  // the CTA's tokens' rows, d_logits and gate logits, after the ring
  int* s_rows = reinterpret_cast<int*>(sm_raw + (size_t)ns * PT::kSlot);  // [tok][KK]
  float* s_dl = reinterpret_cast<float*>(s_rows + (size_t)P.tok_per_cta * KK);  // [tok][EMAX]
  float* s_dgl = s_dl + (size_t)P.tok_per_cta * EMAX;                            // [tok]

  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int s = 0; s < ns; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], kPbConsumers);  // one arrival per consumer warp
    }
    tc::fence_barrier_init();
  }
  pdl_wait();  // a dependent launch: inputs come from the kernels before
  for (int i = threadIdx.x; i < ntok * KK; i += blockDim.x) {
    const int a = i / KK, j = i - a * KK;
    const int64_t t = t_beg + a;
    int r = j < k ? row_of[t * k + j] : -1;
    if (j < k && (r < 0 || r >= P.A)) {
      record_error(P.status, MOE_ERR_DEVICE_INDEX, (int)t);
      r = -1;
    }
    s_rows[i] = r;
  }
  for (int i = threadIdx.x; i < ntok * EMAX; i += blockDim.x) {
    const int a = i / EMAX, e = i - a * EMAX;
    s_dl[i] = e < E ? d_logits[(t_beg + a) * E + e] : 0.f;
  }
  for (int i = threadIdx.x; i < ntok; i += blockDim.x)
    s_dgl[i] = d_gate_logit != nullptr ? d_gate_logit[t_beg + i] : 0.f;
  __syncthreads();

  if (warp == kPbConsumers) {
    // ---------------- producer: one bulk copy per row slice, lane = (token, row)
    int slot = 0;
    uint32_t ph = 0;
    bool ok = true;
    const int a = lane / RPT, j = lane - (lane / RPT) * RPT;
    for (int i = 0; i < nslots; ++i) {
      int w_ok = 1;
      if (lane == 0) w_ok = tc::mbar_wait(&empty[slot], ph ^ 1, abort_flag, P, 51) ? 1 : 0;
      if (!__shfl_sync(0xffffffffu, w_ok, 0)) { ok = false; break; }
      const int ta = i * TS + a;  // the lane's token within the CTA
      int64_t src = -1;           // element offset of the slice's source row
      if (a < TS && ta < ntok) {
        if (j < KK) {
          const int r = j < k ? s_rows[ta * KK + j] : -1;
          if (r >= 0) src = (int64_t)r * d + c0;
        } else if (SH) {
          src = (t_beg + ta) * d + c0;
        }
      }
      const uint32_t bytes = (uint32_t)cols * 2;
      const unsigned issue = __ballot_sync(0xffffffffu, src >= 0);
      if (lane == 0) tc::mbar_expect_tx(&full[slot], bytes * (uint32_t)__popc(issue));
      __syncwarp();
      if (src >= 0) {
        const bf16* g = (j < KK) ? dx_perm + src : dx_shared + src;
        tc::bulk_load_1d(sm_raw + (size_t)slot * PT::kSlot + (size_t)(a * RPT + j) * (kPbCols * 2),
                         g, bytes, &full[slot]);
      }
      if (++slot == ns) { slot = 0; ph ^= 1; }
    }
    if (!ok && lane == 0) {
      // let the copies already in flight land before the CTA exits
      const uint64_t t_start = global_timer_ns();
      while (global_timer_ns() - t_start < 2000000ull) { }
    }
  } else {
    // ---------------- consumers
    const int q = warp % PT::QUARTERS, tg = warp / PT::QUARTERS;
    const int cl = q * PT::WCOLS + lane * CPL;  // column within the slice
    const int col = c0 + cl;
    const bool active = cl < cols;
    float w[EMAX][CPL], wg[CPL];
#pragma unroll
    for (int e = 0; e < EMAX; ++e)
#pragma unroll
      for (int i = 0; i < CPL; ++i)
        w[e][i] = (active && e < E) ? __ldg(w_router + (int64_t)e * d + col + i) : 0.f;
#pragma unroll
    for (int i = 0; i < CPL; ++i)
      wg[i] = (active && d_gate_logit != nullptr) ? __ldg(w_gate + col + i) : 0.f;
    int slot = 0;
    uint32_t ph = 0;
    for (int i = 0; i < nslots; ++i) {
      if (!tc::mbar_wait(&full[slot], ph, abort_flag, P, 52)) break;
      const uint8_t* base = sm_raw + (size_t)slot * PT::kSlot + (size_t)cl * 2;
      for (int a = tg; a < TS; a += PT::TGROUPS) {
        const int ta = i * TS + a;
        if (ta >= ntok || !active) continue;
        float acc[CPL];
#pragma unroll
        for (int ii = 0; ii < CPL; ++ii) acc[ii] = 0.f;
#pragma unroll
        for (int e = 0; e < EMAX; ++e) {
          if (e < E) {
            const float dl = s_dl[ta * EMAX + e];
#pragma unroll
            for (int ii = 0; ii < CPL; ++ii) acc[ii] = fmaf(dl, w[e][ii], acc[ii]);
          }
        }
#pragma unroll
        for (int j = 0; j < KK; ++j) {
          if (j < k && s_rows[ta * KK + j] >= 0) {
            float v[CPL];
            load_smem_bf16<CPL>(base + (size_t)(a * RPT + j) * (kPbCols * 2), v);
#pragma unroll
            for (int ii = 0; ii < CPL; ++ii) acc[ii] += v[ii];
          } else if (j < k) {
#pragma unroll
            for (int ii = 0; ii < CPL; ++ii) acc[ii] += 0.f;
          }
        }
        float sv[CPL];
        if (SH) {
          load_smem_bf16<CPL>(base + (size_t)(a * RPT + (SH ? KK : 0)) * (kPbCols * 2), sv);
        } else {
#pragma unroll
          for (int ii = 0; ii < CPL; ++ii) sv[ii] = 0.f;
        }
#pragma unroll
        for (int ii = 0; ii < CPL; ++ii) acc[ii] += sv[ii];
        if (d_gate_logit != nullptr) {
          const float dgl = s_dgl[ta];
#pragma unroll
          for (int ii = 0; ii < CPL; ++ii) acc[ii] = fmaf(dgl, wg[ii], acc[ii]);
        }
        store_bf16_n<CPL>(dx + (t_beg + ta) * d + col, acc);
      }
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&empty[slot]);
      if (++slot == ns) { slot = 0; ph ^= 1; }
    }
  }
}

template <int KK, int EMAX, bool SH>
static cudaError_t launch_permute_bwd_stream(const Ctx& c, const moe_cfg& cfg, const bf16* dx_perm,
                                             const int32_t* row_of, const bf16* dx_shared,
                                             const float* d_gate_logit, const float* w_gate,
                                             const float* d_logits, const float* w_router,
                                             bf16* dx) {
  using PT = PbTile<KK, EMAX, SH>;
  auto kern = permute_bwd_router_stream<KK, EMAX, SH>;
  static bool attr_done[64];
  int dev = 0;
  cudaGetDevice(&dev);
  if (!attr_done[dev & 63]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)(kPbRingSmem + kPbTableSmem));
    if (e != cudaSuccess) return e;
    attr_done[dev & 63] = true;
  }
  size_t ns = kPbRingSmem / PT::kSlot;
  if (ns > (size_t)kPbMaxSlots) ns = kPbMaxSlots;
  // about one CTA per SM: 1024-column slices x token slices of a multiple of
  // TS, with the slice's per-token tables (rows, d_logits, gate logit) within
  // kPbTableSmem
  const size_t per_tok = (size_t)KK * 4 + (size_t)EMAX * 4 + 4;
  const int64_t cap = (int64_t)(kPbTableSmem / per_tok) / PT::TS * PT::TS;
  const int64_t n_cs = (cfg.d + kPbCols - 1) / kPbCols;
  const int64_t want = c.sm_count / n_cs > 1 ? c.sm_count / n_cs : 1;
  int64_t tpc = ((cfg.T + want - 1) / want + PT::TS - 1) / PT::TS * PT::TS;
  if (tpc > cap) tpc = cap;
  if (tpc < PT::TS) tpc = PT::TS;
  const int64_t n_ts = (cfg.T + tpc - 1) / tpc;
  const size_t smem = ns * PT::kSlot + (size_t)tpc * per_tok;
  PbParams P{};
  P.T = cfg.T;
  P.A = cfg.T * cfg.k;
  P.d = cfg.d;
  P.k = cfg.k;
  P.E = cfg.E;
  P.ns = (int)ns;
  P.tok_per_cta = (int)tpc;
  P.status = c.status;
  P.timeout_ns = c.timeout_ns;
  return launch_dependent(kern, dim3((unsigned)n_cs, (unsigned)n_ts), dim3(kPbThreads), smem,
                          c.stream, dx_perm, row_of, dx_shared, d_gate_logit, w_gate, d_logits,
                          w_router, dx, P);
}

// Shared memory the router-fused form may take for W_r.
constexpr size_t kPermBwdWSmem = 160 * 1024;

template <typename T, int KK, int EMAX>
static cudaError_t launch_permute_bwd_router(const Ctx& c, const moe_cfg& cfg, const T* dx_perm,
                                             const int32_t* row_of, const T* dx_shared,
                                             const float* d_gate_logit, const float* w_gate,
                                             const float* d_logits, const float* w_router,
                                             T* dx) {
  // tokens per warp: each W value read serves TB tokens; fewer with many rows
  constexpr int TB0 = KK >= 8 ? 1 : (KK >= 4 ? 2 : 4);
  constexpr int TB = EMAX > 8 && TB0 > 2 ? 2 : TB0;
  auto kern = permute_bwd_router<T, KK, EMAX, TB>;
  static bool attr_done[64];
  int dev = 0;
  cudaGetDevice(&dev);
  if (!attr_done[dev & 63]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kPermBwdWSmem);
    if (e != cudaSuccess) return e;
    attr_done[dev & 63] = true;
  }
  if constexpr (std::is_same<T, bf16>::value) {
    // bf16 rows, 16-byte aligned, d a multiple of 8: the streamed form
    const auto al = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
    if (cfg.d % 8 == 0 && cfg.T <= (int64_t)INT32_MAX && al(dx_perm) && al(dx) &&
        (dx_shared == nullptr || al(dx_shared))) {
      return dx_shared != nullptr
                 ? launch_permute_bwd_stream<KK, EMAX, true>(c, cfg, dx_perm, row_of, dx_shared,
                                                             d_gate_logit, w_gate, d_logits,
                                                             w_router, dx)
                 : launch_permute_bwd_stream<KK, EMAX, false>(c, cfg, dx_perm, row_of, dx_shared,
                                                              d_gate_logit, w_gate, d_logits,
                                                              w_router, dx);
    }
  }
  const size_t wbytes = (size_t)cfg.E * cfg.d * sizeof(float);
  const bool in_smem = wbytes <= kPermBwdWSmem;
  // W_r staged once per CTA: one CTA per SM, its eight warps walking the tokens
  const int64_t need = ((cfg.T + TB - 1) / TB + 7) / 8;
  const int64_t cap = in_smem ? (int64_t)c.sm_count : (int64_t)c.sm_count * 4;
  const unsigned grid = (unsigned)(need < cap ? (need > 0 ? need : 1) : cap);
  return launch_dependent(kern, dim3(grid), dim3(256), in_smem ? wbytes : 0, c.stream, dx_perm,
                          row_of, dx_shared, d_gate_logit, w_gate, d_logits, w_router, dx, cfg.T,
                          cfg.k, cfg.d, cfg.T * cfg.k, cfg.E, in_smem ? 1 : 0, c.status);
}

bool permute_bwd_forms_router_dx(const moe_cfg& cfg) { return cfg.E <= 16; }

cudaError_t launch_permute_bwd(const Ctx& c, const moe_cfg& cfg, const void* dx_perm,
                               const int32_t* row_of, const float* dx_router,
                               const void* dx_shared, const float* d_gate_logit,
                               const float* w_gate, const float* d_logits,
                               const float* w_router, void* dx) {
  if (cfg.T == 0) return cudaSuccess;
  const int64_t A = cfg.T * cfg.k;
  if (d_logits != nullptr) {
    if (cfg.E > 16) return cudaErrorInvalidValue;  // refused by the entry point first
    cudaError_t e;
#define MOE_PBWDR(TT, KK)                                                                     \
  e = cfg.E <= 8 ? launch_permute_bwd_router<TT, KK, 8>(                                      \
      c, cfg, static_cast<const TT*>(dx_perm), row_of, static_cast<const TT*>(dx_shared),     \
      d_gate_logit, w_gate, d_logits, w_router, static_cast<TT*>(dx))                        \
                 : launch_permute_bwd_router<TT, KK, 16>(                                     \
      c, cfg, static_cast<const TT*>(dx_perm), row_of, static_cast<const TT*>(dx_shared),     \
      d_gate_logit, w_gate, d_logits, w_router, static_cast<TT*>(dx))
#define MOE_PBWDR_K(TT)                                              \
  if (cfg.k <= 1) { MOE_PBWDR(TT, 1); }                              \
  else if (cfg.k <= 2) { MOE_PBWDR(TT, 2); }                         \
  else if (cfg.k <= 4) { MOE_PBWDR(TT, 4); }                         \
  else { MOE_PBWDR(TT, 8); }
    if (cfg.act_dtype == MOE_BF16) {
      MOE_PBWDR_K(bf16)
    } else {
      MOE_PBWDR_K(float)
    }
#undef MOE_PBWDR_K
#undef MOE_PBWDR
    note_launches(1);
    return e;
  }
  const unsigned grid = copy_grid(c, cfg.T);
#define MOE_PBWD(KK)                                                                          \
  if (cfg.act_dtype == MOE_BF16)                                                             \
    launch_dependent(permute_bwd_kernel<bf16, KK>, dim3(grid), dim3(256), 0, c.stream,       \
                     static_cast<const bf16*>(dx_perm), row_of, dx_router,                   \
                     static_cast<const bf16*>(dx_shared), d_gate_logit, w_gate,              \
                     static_cast<bf16*>(dx), cfg.T, cfg.k, cfg.d, A, c.status);              \
  else                                                                                       \
    launch_dependent(permute_bwd_kernel<float, KK>, dim3(grid), dim3(256), 0, c.stream,      \
                     static_cast<const float*>(dx_perm), row_of, dx_router,                  \
                     static_cast<const float*>(dx_shared), d_gate_logit, w_gate,             \
                     static_cast<float*>(dx), cfg.T, cfg.k, cfg.d, A, c.status)
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
